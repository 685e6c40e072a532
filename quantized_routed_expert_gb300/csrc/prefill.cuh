// Prefill path of libmoe: workspace layout and launch interface.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

constexpr int kPrefillMaxTokens = 16384;

struct PrefillLayout {
  int64_t counts, offsets, perm, comb, x16, h16, o, sched, total;  // byte offsets
  // E4M3 operands only (fp8 layout): codes of x and h, h as fp32, exponents
  int64_t x8, h8, h32, bexp, hexp;
};

// fp8: the layout of the E4M3-operand prefill (adds the regions above).
PrefillLayout prefill_layout(const moe_shape& s, int64_t T, bool fp8 = false);
bool prefill_fp8_supported(const moe_shape& s);
// Per-row exponents of every weight matrix (the E4M3 prefill's weight scales):
// int8 per row, gate [E][F], up [E][F], down [E][H], then the shared expert's
// gate [Fs], up [Fs], down [H].
int64_t fp8_row_exponent_count(const moe_shape& s);
cudaError_t launch_fp8_row_exponents(const moe_shape& s, const moe_expert_weights& w,
                                     int8_t* out, cudaStream_t stream);
// The E4M3 weight decoder on its own: row exponents of rows x K weights, then
// every weight's code (the functions the fp8 prefill producers call).
cudaError_t launch_dequant_e4m3(const void* mat, int64_t rows, int K, int8_t* row_exp,
                                uint8_t* out, int num_sms, cudaStream_t stream);
cudaError_t launch_prefill_fp8(const moe_shape& s, const moe_expert_weights& w,
                               const int8_t* row_exp, const uint16_t* x, int T,
                               const int32_t* ids, const float* weights, float* y, uint8_t* ws,
                               const PrefillLayout& L, uint32_t* status, int num_sms, bool pdl,
                               cudaStream_t stream);
int prefill_launches(const moe_shape& s, int T);
bool prefill_supported(const moe_shape& s);

cudaError_t launch_prefill(const moe_shape& s, const moe_expert_weights& w, const uint16_t* x,
                           int T, const int32_t* ids, const float* weights, float* y,
                           uint8_t* ws, const PrefillLayout& L, uint32_t* status, int num_sms,
                           bool pdl, cudaStream_t stream);

}  // namespace moe
