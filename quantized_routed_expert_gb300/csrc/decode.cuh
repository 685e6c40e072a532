// Decode path of libmoe: parameters, workspace layout and launch helpers.
#pragma once

#include <cstddef>
#include <cstdint>

#include "moe.h"

namespace moe {

constexpr int kMaxPairs = MOE_MAX_DECODE_TOKENS * MOE_MAX_TOP_K;  // T*k

inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Bytes of one IQ4_NL row with K inputs.
inline int64_t row_bytes(int64_t K) { return K / 32 * 18; }
// Rows per alignment granule: the smallest g with g*row_bytes(K) % 16 == 0.
inline int row_granule(int64_t K) {
  const int64_t rb = row_bytes(K);
  int g = 1;
  while ((g * rb) % 16) g *= 2;
  return g;
}
// Lanes per row in the down kernels (and the quantised vector layout): a power
// of two, at most 8 and at most the number of block pairs of the row.
inline int lanes_per_row(int64_t K) {
  int l = 8;
  while (l > K / 64) l >>= 1;
  return l;
}
// Words of one quantised vector record (int16 pairs + fp32 scales), 16-byte padded.
inline int64_t qvec_words(int64_t K) {
  const int64_t lpr = lanes_per_row(K);
  const int64_t groups = (K / 64 + lpr - 1) / lpr;
  return groups * lpr * 32 + align_up(K / 32, 4);
}

struct DecodeLayout {
  int64_t h_r, h_s, rec_r, rec_s, sync, scores, xrec, part, tscores, xc, total;  // byte offsets
};

inline DecodeLayout decode_layout(const moe_shape& s, int64_t T) {
  DecodeLayout L{};
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const int64_t Fs = s.n_shared ? s.ffn_shared : 0;
  L.h_r = take(T * s.top_k * s.ffn * 4);
  L.h_s = take(T * Fs * 4);
  L.rec_r = take(T * s.top_k * qvec_words(s.ffn) * 4);
  L.rec_s = take(Fs ? T * qvec_words(Fs) * 4 : 0);
  L.sync = take(64);                       // grid-barrier counters of the fused kernel
  L.scores = take(T * s.n_experts * 4);    // router scores of the routed fused kernel
  L.xrec = take(T * qvec_words(s.hidden) * 4);   // quantised x, when it does not fit on chip
  L.part = take((T * s.top_k + (Fs ? T : 0)) * s.hidden * 4);   // down partials per pair
  L.tscores = take(2 * T * s.n_experts * 8);   // tagged router scores (multi-layer kernel)
  L.xc = take(T * s.hidden * 2);               // chained bf16 input (multi-layer, launch per layer)
  L.total = off;
  return L;
}

struct DecodeParams {
  int H, F, Fs, E, k, n_shared, T;
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const uint8_t* sh_gate;
  const uint8_t* sh_up;
  const uint8_t* sh_down;
  const uint16_t* x;
  const int32_t* ids;
  const float* weights;
  float* y;
  float* h_r;        // [T*k][F]
  float* h_s;        // [T][Fs]
  uint32_t* rec_r;   // [T*k][qvec_words(F)]
  uint32_t* rec_s;   // [T][qvec_words(Fs)]
  uint32_t* sync;    // [0..3]: h arrivals, departures, score arrivals (fused kernel);
                     // [4..7]: h arrivals, y arrivals, departures, epoch (multi-layer kernel)
  uint32_t* status;
  uint32_t* xrec;    // [T][qvec_words(H)]: quantised x (gate/up kernel without room for it)
  float* part;       // [T*k (+T)][H]: down partials per pair (two-kernel path)
  // routing inside the fused kernel (route != 0)
  int route;
  const uint16_t* Wr;    // bf16 [E][H]
  const float* bias;     // [E] or NULL
  int32_t* ids_out;      // [T][k]
  float* w_out;          // [T][k]
  float* scores;         // workspace [T][E]
  // launch-derived
  int gu_nblk;       // gate/up kernel: 32-row blocks a CTA may get
  int dn_rows_max;   // max output rows per down CTA
  int fz_rg;         // fused kernel: output rows per down unit
  uint64_t wait_ns;  // limit of a CTA's waits on other CTAs (grid barriers)
  // several layers in one call (moe_iq4nl_decode_layers)
  int L;             // layers
  int chained;       // 1: layer l + 1's input is bf16(y_l)
  uint64_t* tscores; // workspace [2][T][E]: score | tag << 32
  uint16_t* xc;      // workspace [T][H]: chained input, launch-per-layer path
};

// Per-layer pointers of a multi-layer call (kernel parameter space).
struct LayerPtrs {
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const uint8_t* sh_gate;
  const uint8_t* sh_up;
  const uint8_t* sh_down;
  const uint16_t* Wr;
  const float* bias;
};
struct LayerTable {
  LayerPtrs layer[MOE_MAX_LAYERS];
};

cudaError_t launch_decode(const DecodeParams& p, int num_sms, bool pdl, cudaStream_t stream);
// Kernel launches of one launch_decode call (route = 0) for these sizes.
int decode_launches(const DecodeParams& p, int num_sms);
bool fused_decode_supported(const DecodeParams& p, int num_sms, size_t* smem, int* rg,
                            int* rows_max);
bool fused_resident(const DecodeParams& p, size_t smem);
cudaError_t launch_decode_routed(const DecodeParams& p, int num_sms, bool pdl,
                                 cudaStream_t stream);
cudaError_t launch_decode_fused(const DecodeParams& p, int num_sms, size_t smem, bool pdl,
                                cudaStream_t stream);
bool layers_supported(const DecodeParams& p, int num_sms, size_t* smem, int* rg, int* rows_max);
int layers_launches(const DecodeParams& p, int num_sms);
cudaError_t launch_decode_layers(const DecodeParams& p, const LayerTable& lt, int num_sms,
                                 bool pdl, cudaStream_t stream);

}  // namespace moe
