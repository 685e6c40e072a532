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

}  // namespace moe
