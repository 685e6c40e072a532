// Prefill path of libmoe: workspace layout and launch interface.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

constexpr int kPrefillMaxTokens = 16384;

struct PrefillLayout {
  int64_t counts, offsets, perm, comb, x16, h16, o, sched, total;  // byte offsets
};

PrefillLayout prefill_layout(const moe_shape& s, int64_t T);
int prefill_launches(const moe_shape& s, int T);
bool prefill_supported(const moe_shape& s);

cudaError_t launch_prefill(const moe_shape& s, const moe_expert_weights& w, const uint16_t* x,
                           int T, const int32_t* ids, const float* weights, float* y,
                           uint8_t* ws, const PrefillLayout& L, uint32_t* status, int num_sms,
                           bool pdl, cudaStream_t stream);

}  // namespace moe
