// Router launch interface.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

struct RouteParams {
  int H, E, k, T;
  const uint16_t* Wr;
  const float* bias;
  const uint16_t* x;
  int32_t* ids;
  float* w;
};

cudaError_t launch_route(const RouteParams& p, bool pdl, cudaStream_t stream);
// Chunks of at least 256 tokens with at most 256 experts: scores on tensor
// cores (prefill.cu).
bool route_mma_supported(const RouteParams& p);
cudaError_t launch_route_mma(const RouteParams& p, bool pdl, cudaStream_t stream);

}  // namespace moe
