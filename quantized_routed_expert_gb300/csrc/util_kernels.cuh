#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

cudaError_t launch_dequant(const void* blocks, int64_t n_blocks, int mode, void* out,
                           int num_sms, cudaStream_t stream);
cudaError_t launch_sanitize(const int32_t* ids, const float* w, int64_t n, int E,
                            int32_t* ids_out, float* w_out, uint32_t* status, int num_sms,
                            cudaStream_t stream);

}  // namespace moe
