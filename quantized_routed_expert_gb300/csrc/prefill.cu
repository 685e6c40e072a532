// Prefill path of libmoe (sm_103a): bucket a token chunk by expert, run each
// expert's tokens as a grouped tensor-core contraction (tcgen05, fp16 operands,
// fp32 accumulation in TMEM) on IQ4_NL weights dequantised on the fly, then a
// gather-combine in the fixed per-token order.
//
// Prior art: the Xolotl blog ("Prompts: fast, and exact") streams each layer's
// experts once per chunk into one batched multiply on tensor cores; Red Lite
// ("What we learned", section 3) uses batched matrix kernels for experts over
// 2048-token chunks. Here the chunk is bucketed with a stable counting sort
// (no atomics decide any position), and the weights are dequantised by
// producer warps straight into the 128-byte-swizzled shared-memory layout that
// the MMA reads, while token rows arrive by TMA.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "prefill.cuh"
#include "tc.cuh"

namespace moe {

namespace {
int64_t up256(int64_t v) { return (v + 255) / 256 * 256; }
}  // namespace

// Per-tile stamps of the GEMM kernels (builds with MOE_PROFILE only), read back
// with moe_profile_prefill: [gate/up, down][CTA < 256][tile < 15, 15 = kernel]
// [8]: 0 MMA tile start, 1 MMA last commit, 2 dequant start, 3 dequant done,
// 4 accumulator seen by the epilogue, 5 epilogue done, 6 tokens, 7 bucket.
#ifdef MOE_PROFILE
__device__ uint64_t g_pfprof[2 * 256 * 16 * 8];
#define PF_STAMP(tile, k, v)                                                            \
  do {                                                                                  \
    if (blockIdx.x < 256 && (tile) < 15)                                                \
      g_pfprof[(((size_t)(GATEUP ? 0 : 1) * 256 + blockIdx.x) * 16 + (tile)) * 8 + (k)] = \
          (v);                                                                          \
  } while (0)
#define PF_STAMP_K(k, v)                                                                \
  do {                                                                                  \
    if (blockIdx.x < 256)                                                               \
      g_pfprof[(((size_t)(GATEUP ? 0 : 1) * 256 + blockIdx.x) * 16 + 15) * 8 + (k)] = (v); \
  } while (0)
#else
#define PF_STAMP(tile, k, v) \
  do {                       \
  } while (0)
#define PF_STAMP_K(k, v) \
  do {                   \
  } while (0)
#endif

PrefillLayout prefill_layout(const moe_shape& s, int64_t T, bool fp8) {
  PrefillLayout L{};
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off = up256(off + bytes);
    return o;
  };
  const int64_t E = s.n_experts, k = s.top_k, H = s.hidden, F = s.ffn;
  const int64_t Fs = s.n_shared ? s.ffn_shared : 0;
  const int64_t rows = T * k + (s.n_shared ? T : 0);
  const int64_t fmax = F > Fs ? F : Fs;
  L.counts = take((E + 2) * 4);                 // bucket row offsets [E+2]
  L.offsets = take(T * k * 4);                  // row of each (token, slot) pair, -1 invalid
  L.perm = take(rows * 4);                      // token of each bucketed row
  L.comb = take(T * (k + 1) * 8);               // per token: rows and weights, combine order
  L.x16 = take(rows * H * 2);                   // activations in bucket order, fp16
  L.h16 = take(rows * fmax * 2);                // h in bucket order, fp16
  L.o = take(rows * H * 4);                     // expert outputs in bucket order, fp32
  L.sched = 0;
  if (fp8) {
    L.x8 = take(rows * H);                      // E4M3 codes of x 2^-X, bucket order
    L.h8 = take(rows * fmax);                   // E4M3 codes of h 2^-X
    L.h32 = take(rows * fmax * 4);              // h, fp32, bucket order
    L.bexp = take(rows * 4);                    // each bucket row's x exponent
    L.hexp = take(rows * 4);                    // each bucket row's h exponent (it enters the
                                                // combine weights; kept for inspection)
  }
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------
// 1. Bucketing: a stable counting sort of the valid (token, slot) pairs by
// expert (ties by pair index). Routed buckets 0..E-1 occupy rows
// [0, n_valid); the shared expert's bucket (every token, in order) follows.
struct BucketParams {
  const int32_t* ids;
  int T, k, E, n_shared;
  int32_t* bucket_off;   // [E+2]
  int32_t* row_of;       // [T*k]
  int32_t* row_tok;      // [rows]
  uint32_t* status;
};

constexpr int kBucketThreads = 1024;
constexpr int kBucketWarps = kBucketThreads / 32;

// Counting sort of the (token, expert) pairs by expert, stable in the pair
// index, in one CTA with three passes: every warp counts its contiguous share
// of the pairs per expert (match_any groups one round of 32 pairs; no atomics
// decide any order); the per-expert totals are scanned into bucket starts and
// the per-warp counts into each warp's offsets within every bucket; every warp
// then walks its share again and places each pair at its bucket start + its
// warp's offset + the pairs of that expert before it in the warp. Dynamic
// shared memory: kBucketWarps x E counters.
__global__ void __launch_bounds__(kBucketThreads) pf_bucket_kernel(BucketParams p) {
  extern __shared__ int wc[];                   // [kBucketWarps][E]
  __shared__ int start[MOE_MAX_EXPERTS + 2];
  __shared__ int wsum[32];
  __shared__ int invalid;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = p.T * p.k, E = p.E;
#pragma unroll 1
  for (int i = tid; i < kBucketWarps * E; i += kBucketThreads) wc[i] = 0;
  if (tid == 0) invalid = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int per = (P + kBucketWarps - 1) / kBucketWarps;
  const int p0 = warp * per, p1 = p0 + per < P ? p0 + per : P;
  int* mine = wc + warp * E;
  // the ids of 8 rounds of 32 pairs, all loads in flight at once
  constexpr int kR = 8;
  auto load_ids = [&](int r0, int (&e)[kR]) {
#pragma unroll
    for (int u = 0; u < kR; ++u) {
      const int pi = r0 + 32 * u + lane;
      const int id = pi < p1 ? p.ids[pi] : -1;
      e[u] = pi < p1 && id >= 0 && id < E ? id : (pi < p1 ? -2 : -1);   // -2: invalid pair
    }
  };
  // pass 1: per-warp counts
  int bad = 0;
#pragma unroll 1
  for (int r0 = p0; r0 < p1; r0 += 32 * kR) {
    int e[kR];
    load_ids(r0, e);
#pragma unroll
    for (int u = 0; u < kR; ++u) {
      bad += e[u] == -2;
      const uint32_t m = __match_any_sync(0xFFFFFFFFu, e[u]);
      if (e[u] >= 0 && (m & ((1u << lane) - 1u)) == 0) mine[e[u]] += __popc(m);
      __syncwarp();
    }
  }
  bad = __reduce_add_sync(0xFFFFFFFFu, (unsigned)bad);
  if (lane == 0 && bad) atomicAdd(&invalid, bad);
  __syncthreads();
  // pass 2: per-expert totals -> bucket starts; per-warp offsets within them
  {
    int c = 0;
    if (tid < E) {
      int run = 0;
#pragma unroll 1
      for (int w = 0; w < kBucketWarps; ++w) {
        const int v = wc[w * E + tid];
        wc[w * E + tid] = run;
        run += v;
      }
      c = run;
    }
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = wsum[lane];
      int s2 = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, s2, o);
        if (lane >= o) s2 += u;
      }
      wsum[lane] = s2 - v;
    }
    __syncthreads();
    if (tid < E) start[tid] = incl - c + wsum[warp];
  }
  const int n_valid = P - invalid;
  if (tid == 0) {
    start[E] = n_valid;
    start[E + 1] = n_valid + (p.n_shared ? p.T : 0);
  }
  __syncthreads();
  for (int i = tid; i < E + 2; i += kBucketThreads) p.bucket_off[i] = start[i];
  // pass 3: places
#pragma unroll 1
  for (int r0 = p0; r0 < p1; r0 += 32 * kR) {
    int e[kR];
    load_ids(r0, e);
#pragma unroll
    for (int u = 0; u < kR; ++u) {
      const int pi = r0 + 32 * u + lane;
      const uint32_t m = __match_any_sync(0xFFFFFFFFu, e[u]);
      const int before = __popc(m & ((1u << lane) - 1u));
      if (e[u] >= 0) {
        const int row = start[e[u]] + mine[e[u]] + before;
        p.row_of[pi] = row;
        p.row_tok[row] = pi / p.k;
      } else if (e[u] == -2) {
        p.row_of[pi] = -1;
      }
      __syncwarp();
      if (e[u] >= 0 && before == 0) mine[e[u]] += __popc(m);
      __syncwarp();
    }
  }
  if (p.n_shared)
    for (int t = tid; t < p.T; t += kBucketThreads) p.row_tok[n_valid + t] = t;
  if (tid == 0 && p.status && invalid)
    atomicAdd(p.status, (uint32_t)(invalid < 0xFFFF ? invalid : 0xFFFF));
}

// ---------------------------------------------------------------------------
// 2. Activations in bucket order, fp16 (round to nearest even from bf16), and
// each token's combine list: its rows in the fixed order of the sum (shared
// expert first, then experts ascending: rows are grouped by expert, so
// ascending rows) with their weights.
struct CombineListParams {
  const int32_t* row_of;   // [T*k], -1 for an invalid pair
  const float* w;          // [T*k]
  int T, k, n_shared;
  int32_t* comb_row;       // [T][k+1]
  float* comb_w;           // [T][k+1]
};
// F8: the bucket rows are E4M3 codes of x 2^-X_t, X_t = floor(log2 max|x_t|)
// - 6 (0 for a zero row), in the E4M3 block order of K (e4m3_block_pos_value),
// and each row's X_t goes to bexp. The token's warp finds the maximum in a
// first pass over x_t (|bf16| bits widened to fp32 order like the values); the
// second pass converts (its loads hit L1) and writes every row of the token.
struct Gather8 {
  int32_t* bexp;             // [rows]
  uint8_t* x8;               // [rows][H]
};
template <bool F8>
__global__ void pf_gather_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ bucket_off,
                                 int E, int H, __half* xs,
                                 const CombineListParams cl, const Gather8 g8) {
  pdl_wait();
  pdl_trigger();
  {
    const int n_valid = bucket_off[E];
    const int kk = cl.k + 1;
    const int first = cl.n_shared ? 1 : 0;
#pragma unroll 1
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < cl.T; t += gridDim.x * blockDim.x) {
      int32_t* cr = cl.comb_row + (size_t)t * kk;
      float* cw = cl.comb_w + (size_t)t * kk;
      if (cl.n_shared) {
        cr[0] = n_valid + t;
        cw[0] = 1.0f;
      }
      int rows[MOE_MAX_TOP_K];
#pragma unroll
      for (int j = 0; j < MOE_MAX_TOP_K; ++j) rows[j] = j < cl.k ? cl.row_of[t * cl.k + j] : -1;
      int nv = 0;
#pragma unroll
      for (int j = 0; j < MOE_MAX_TOP_K; ++j) {
        if (rows[j] < 0) continue;
        int rank = 0;
#pragma unroll
        for (int i = 0; i < MOE_MAX_TOP_K; ++i) rank += rows[i] >= 0 && rows[i] < rows[j];
        cr[first + rank] = rows[j];
        cw[first + rank] = cl.w[t * cl.k + j];
        ++nv;
      }
      for (int j = first + nv; j < kk; ++j) {
        cr[j] = -1;
        cw[j] = 0.0f;
      }
    }
  }
  // one warp per token: its x row is read once and written to each of its
  // bucket rows (lane j < k: the row of slot j, -1 for an invalid pair; lane k:
  // the shared expert's row)
  const int n_valid = bucket_off[E];
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int h8 = H / 8;
  for (int t = gw; t < cl.T; t += nw) {
    int myrow = -1;
    if (lane < cl.k) myrow = cl.row_of[(size_t)t * cl.k + lane];
    else if (lane == cl.k && cl.n_shared) myrow = n_valid + t;
    const uint32_t have = __ballot_sync(0xFFFFFFFFu, myrow >= 0);
    if constexpr (F8) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
      uint32_t m = 0;
      for (int c = lane; c < h8; c += 32) {
        const uint4 v = src[c];
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          m = max(m, max((in[i] << 16) & 0x7FFFFFFFu, in[i] & 0x7FFF0000u));
      }
      const int X = vec_exponent_bits(__reduce_max_sync(0xFFFFFFFFu, m));
      const float sx = pow2_of(-X);
      if (myrow >= 0) g8.bexp[myrow] = X;
      // positions 8c .. 8c + 7 of the E4M3 block order: values 4j .. 4j + 3
      // and 4j + 16 .. 4j + 19 of block c / 4 (j = c % 4), interleaved
      const uint2* src2 = reinterpret_cast<const uint2*>(x + (size_t)t * H);
      for (int c = lane; c < h8; c += 32) {
        const int v0 = (c >> 2) * 32 + (c & 3) * 4;
        const uint2 a = src2[v0 / 4], b = src2[(v0 + 16) / 4];
        const uint32_t lo[4] = {a.x << 16, a.x & 0xFFFF0000u, a.y << 16, a.y & 0xFFFF0000u};
        const uint32_t hi[4] = {b.x << 16, b.x & 0xFFFF0000u, b.y << 16, b.y & 0xFFFF0000u};
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)      // values 4j + i (low byte) and 4j + 16 + i
          pk[i] = cvt_e4m3x2(pow2_scale(__uint_as_float(hi[i]), -X, sx),
                             pow2_scale(__uint_as_float(lo[i]), -X, sx));
        const uint2 v = make_uint2(pk[0] | (pk[1] << 16), pk[2] | (pk[3] << 16));
        for (uint32_t rem = have; rem; rem &= rem - 1) {
          const int r = __shfl_sync(0xFFFFFFFFu, myrow, __ffs(rem) - 1);
          reinterpret_cast<uint2*>(g8.x8 + (size_t)r * H)[c] = v;
        }
      }
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
      for (int c = lane; c < h8; c += 32) {
        const uint4 v = src[c];
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half lo = __float2half_rn(__uint_as_float(in[i] << 16));
          const __half hi = __float2half_rn(__uint_as_float(in[i] & 0xFFFF0000u));
          out[i] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
        }
        const uint4 o = make_uint4(out[0], out[1], out[2], out[3]);
        for (uint32_t rem = have; rem; rem &= rem - 1) {
          const int r = __shfl_sync(0xFFFFFFFFu, myrow, __ffs(rem) - 1);
          reinterpret_cast<uint4*>(xs + (size_t)r * H)[c] = o;
        }
      }
    }
  }
}

// E4M3 operands: h (fp32, written by the gate/up GEMM) to E4M3 codes of
// h 2^-X_p in the E4M3 block order of K, X_p from the row's largest |h|, one
// warp per bucket row. The down outputs then lack the factor 2^X_p: the row's
// combine weight w (its token's slot in the combine list) becomes w 2^X_p, the
// same product as scaling the outputs whenever w 2^X_p is a normal fp32 (each
// fp32 rounding commutes with a power of two). A first
// pass over the row finds the largest |h| (as fp32 bits, which order like the
// values), the second converts (its loads hit L1).
__global__ void pf8_hconv_kernel(const float* __restrict__ h32,
                                 const int32_t* __restrict__ bucket_off, int E, int ld, int F,
                                 int Fs, uint8_t* __restrict__ h8, int32_t* __restrict__ hexp,
                                 const int32_t* __restrict__ row_tok,
                                 const int32_t* __restrict__ comb_row, float* __restrict__ comb_w,
                                 int kk) {
  pdl_wait();
  pdl_trigger();
  const int rows = bucket_off[E + 1], n_valid = bucket_off[E];
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int r = gw; r < rows; r += nw) {
    const int K = r < n_valid ? F : Fs;
    const float4* src = reinterpret_cast<const float4*>(h32 + (size_t)r * ld);
    uint32_t m = 0;
    for (int c = lane; c < K / 4; c += 32) {
      const float4 a = src[c];
      m = max(m, max(max(__float_as_uint(fabsf(a.x)), __float_as_uint(fabsf(a.y))),
                     max(__float_as_uint(fabsf(a.z)), __float_as_uint(fabsf(a.w)))));
    }
    const int X = vec_exponent_bits(__reduce_max_sync(0xFFFFFFFFu, m));
    const float sx = pow2_of(-X);
    if (lane == 0) hexp[r] = X;
    if (lane < kk) {                           // this row's slot in its token's list
      const size_t slot = (size_t)row_tok[r] * kk + lane;
      if (comb_row[slot] == r) {
        const float w = comb_w[slot];
        comb_w[slot] = X >= -126 ? w * exp2i(X) : ldexpf(w, X);
      }
    }
    uint2* dst = reinterpret_cast<uint2*>(h8 + (size_t)r * ld);
    for (int c = lane; c < K / 8; c += 32) {
      // the E4M3 block order: values 4j + i and 4j + 16 + i of block c / 4
      const int v0 = (c >> 2) * 32 + (c & 3) * 4;
      const float4 a = src[v0 / 4], b = src[(v0 + 16) / 4];
      const uint32_t p0 = cvt_e4m3x2(pow2_scale(b.x, -X, sx), pow2_scale(a.x, -X, sx));
      const uint32_t p1 = cvt_e4m3x2(pow2_scale(b.y, -X, sx), pow2_scale(a.y, -X, sx));
      const uint32_t p2 = cvt_e4m3x2(pow2_scale(b.z, -X, sx), pow2_scale(a.z, -X, sx));
      const uint32_t p3 = cvt_e4m3x2(pow2_scale(b.w, -X, sx), pow2_scale(a.w, -X, sx));
      dst[c] = make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
    }
  }
}

// ---------------------------------------------------------------------------
// 3. Grouped GEMM on tcgen05. Tiles: (bucket, 128 weight rows, 256 tokens).
//   D[m][n] = sum_k A[m][k] B[n][k]: A = dequantised weights (fp16, rows of the
//   expert matrix), B = token rows (fp16, bucket order), fp32 in TMEM.
//   gate/up: two accumulators (columns 0..255 gate, 256..511 up), epilogue
//   h = silu(g) u -> fp16. down: one accumulator, epilogue -> fp32 o.
// Warps: 0 loads token tiles (TMA), 1 owns TMEM and issues the MMAs, 2..9
// dequantise weight tiles and run the epilogue.
constexpr int kTM = 128;
constexpr int kTN = 256;
constexpr int kTK = 64;

struct GemmParams {
  int E, n_shared;
  int M, Ms;             // weight rows: routed, shared
  int K, Ks;             // reduction length: routed, shared
  const uint8_t* a0;     // routed gate (or down)   [E][M][K/32]
  const uint8_t* a1;     // routed up               (gate/up only)
  const uint8_t* s0;     // shared gate (or down)   [Ms][Ks/32]
  const uint8_t* s1;     // shared up
  const int32_t* bucket_off;
  __half* h;             // gate/up out: [rows][ldh]
  int ldh;
  float* o;              // down out: [rows][ldo]
  int ldo;
  uint32_t* status;
  // E4M3 operands only: each weight row's exponent (routed [E][M], shared
  // [Ms]) for a0, a1, s0, s1; gate/up: x's exponent per bucket row (its
  // token's), and h written as fp32 [rows][ldh]
  const int8_t *e0, *e1, *se0, *se1;
  const int32_t* bexp;
  float* h32;
};

// Shared memory and warp roles of the GEMM kernels. RAW: the IQ4_NL rows of the
// weight tile arrive by 2D bulk copies, four K-steps (144 bytes) per row per
// copy, into a ring the dequantising warps read (the reduction length is a
// multiple of 256 so the row pitch is a multiple of 16 bytes); otherwise each
// dequantising thread loads its own row from global memory.
template <bool GATEUP, bool RAW>
struct GemmCfg {
  static constexpr int kCtl = RAW ? 3 : 2;                        // control warps
  static constexpr int kDq = (RAW && GATEUP) ? 16 : 8;            // dequantising warps
  // Down: four epilogue warps of their own and two accumulators (N <= 256
  // columns each), so that a tile's epilogue overlaps the next tile's MMAs.
  // Gate/up needs all 512 TMEM columns for one tile: its dequantising warps
  // run the epilogue.
  static constexpr int kEpi = GATEUP ? 0 : 4;
  static constexpr int kAcc = GATEUP ? 1 : 2;
  static constexpr int kThreads = (kCtl + kDq + kEpi) * 32;
  static constexpr int kA = kTM * kTK * 2;                        // 16 KB
  static constexpr int kB = kTN * kTK * 2;                        // 32 KB
  static constexpr int kStage = (GATEUP ? 2 : 1) * kA + kB;
  static constexpr int kStages = RAW ? (GATEUP ? 2 : 3) : (GATEUP ? 3 : 4);
  static constexpr int kRawGroup = 4;                             // K-steps per raw copy
  static constexpr int kRawMat = kTM * kRawGroup * kPairB;        // 18 KB per matrix
  static constexpr int kRawStage = (GATEUP ? 2 : 1) * kRawMat;
  static constexpr int kRawRing = 2;                              // raw ring depth
  static constexpr int kRawStages = RAW ? kRawRing : 0;           // raw stages allocated
  static constexpr int kBars = 3 * kStages + 2 * kAcc + 2 * kRawStages;
  static constexpr size_t kTotal =
      1024 /*align slack*/ + (size_t)kStages * kStage + (size_t)kRawStages * kRawStage + 4096;
};

__device__ __forceinline__ void sw128_store_chunk(uint8_t* tile, int r, int c, uint4 v) {
  *reinterpret_cast<uint4*>(tile + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4)) = v;
}

// Dequantise one 32-weight block (4 index words, fp16 scale bits) into four
// 16-byte chunks (8 fp16 each, K order) of row r, chunks c0..c0+3.
__device__ __forceinline__ void dequant_block_to_tile(const uint32_t (&q)[4], uint16_t dbits,
                                                      uint8_t* tile, int r, int c0) {
  uint32_t w[16];
  dequant_block_half(q, dbits, w);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    sw128_store_chunk(tile, r, c0 + c, make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]));
}

struct TileInfo {
  int bucket, m0, n0, nvalid, row0;
};

// silu(g) u in the GEMM epilogues, on the hardware exp2 and reciprocal (a few
// fp32 ulps): h is rounded to fp16 or E4M3 right after, far coarser. For g
// below about -87, 1 + e^-g exceeds 2^126 and the quotient is a signed zero,
// where the exact value is below 1e-36 in magnitude.
__device__ __forceinline__ float silu_mul_fast(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Token tiles are loaded with the smallest of four box heights that covers
// the tile's tokens, and the MMA runs with N = tokens rounded up to 16: with
// skewed routing most buckets hold far fewer than 256 tokens.
constexpr int kNumBoxes = 4;                 // 32, 64, 128, 256 rows
struct TmapSet {
  CUtensorMap m[kNumBoxes];   // token rows, by box height
  CUtensorMap raw[4];         // IQ4_NL rows (bytes): routed gate|down, routed up, shared gate|down, shared up
};
__device__ __forceinline__ int box_index(int n) {
  return n <= 32 ? 0 : (n <= 64 ? 1 : (n <= 128 ? 2 : 3));
}

// F8: E4M3 operands (kind::f8f6f4). A K-step is then 128 values, the same 128
// bytes of every row as a 64-value fp16 step, so the stages, rings and
// barriers are the same; a raw copy (four pairs of blocks) feeds two steps.
// Each weight row is scaled by 2^-E_row before rounding and each B row by
// 2^-bexp; the epilogue multiplies the accumulator back by 2^(E_row + bexp).
template <bool GATEUP, bool RAW, bool F8>
__global__ void __launch_bounds__(GemmCfg<GATEUP, RAW>::kThreads, 1)
pf_gemm_kernel(const __grid_constant__ TmapSet tmaps, const GemmParams p) {
  using S = GemmCfg<GATEUP, RAW>;
  static_assert(!F8 || RAW, "E4M3 operands need the raw-row ring");
  constexpr int kTKe = F8 ? 128 : kTK;                     // K values per stage
  constexpr int kStepsPerRaw = F8 ? 2 : S::kRawGroup;      // stages per raw copy
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* raw = smem + (size_t)S::kStages * S::kStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + (size_t)S::kRawStages * S::kRawStage);
  uint64_t* full_a = bars;
  uint64_t* full_b = bars + S::kStages;
  uint64_t* empty = bars + 2 * S::kStages;
  uint64_t* acc_full = bars + 3 * S::kStages;       // [kAcc]
  uint64_t* acc_empty = acc_full + S::kAcc;         // [kAcc]
  uint64_t* full_raw = acc_empty + S::kAcc;
  uint64_t* empty_raw = full_raw + S::kRawStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + S::kBars);
  int* boff = reinterpret_cast<int*>(tmem_slot + 4);           // [E+2] bucket offsets
  int* tpre = boff + (p.E + 2);                                 // [E+2] tile prefix

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(&full_a[s], S::kDq);
      mbar_init(&full_b[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < S::kAcc; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], S::kEpi ? S::kEpi : S::kDq);
    }
    for (int s = 0; s < S::kRawStages; ++s) {
      mbar_init(&full_raw[s], 1);
      mbar_init(&empty_raw[s], S::kDq);
    }
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) PF_STAMP_K(0, global_timer_ns());
  // bucket offsets and the tile prefix (tiles of a bucket: weight tiles x token tiles)
  const int nb = p.E + p.n_shared;
  for (int i = threadIdx.x; i < p.E + 2; i += S::kThreads) boff[i] = p.bucket_off[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < nb; ++b) {
      tpre[b] = acc;
      const int n = boff[b + 1] - boff[b];
      const int mt = (b < p.E ? p.M : p.Ms) / kTM;
      acc += mt * ((n + kTN - 1) / kTN);
    }
    tpre[nb] = acc;
  }
  __syncthreads();
  const int ntiles = tpre[nb];
  const uint32_t tmem = *tmem_slot;

  auto tile_info = [&](int t) {
    int lo = 0, hi = nb - 1;                     // last bucket with tpre[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tpre[mid] <= t) lo = mid; else hi = mid - 1;
    }
    TileInfo ti;
    ti.bucket = lo;
    const int n = boff[lo + 1] - boff[lo];
    const int nt = (n + kTN - 1) / kTN;
    const int local = t - tpre[lo];
    const int mi = local / nt, ni = local - mi * nt;
    ti.m0 = mi * kTM;
    ti.n0 = ni * kTN;
    ti.nvalid = n - ti.n0 < kTN ? n - ti.n0 : kTN;
    ti.row0 = boff[lo];
    return ti;
  };

  if (warp == 0) {
    // ---- token tiles by TMA
    if (lane == 0) {
      int it = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const TileInfo ti = tile_info(t);
        const int K = ti.bucket < p.E ? p.K : p.Ks;
        for (int ks = 0; ks < K / kTKe; ++ks, ++it) {
          const int s = it % S::kStages;
          if (!mbar_wait(&empty[s], ((it / S::kStages) & 1) ^ 1, p.status)) {
            t = ntiles;                          // give up; fall through to the exit barrier
            break;
          }
          uint8_t* b = stages + (size_t)s * S::kStage + (GATEUP ? 2 : 1) * S::kA;
          const int bx = box_index(ti.nvalid);
          mbar_arrive_expect_tx(&full_b[s], (uint32_t)((32 << bx) * 128));   // 128 B a row
          tma_load_2d(b, &tmaps.m[bx], ks * kTKe, ti.row0 + ti.n0, &full_b[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issue (one thread)
    if (lane == 0) {
      int it = 0, tc = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tc) {
        const TileInfo ti = tile_info(t);
        const int K = ti.bucket < p.E ? p.K : p.Ks;
        const uint32_t idesc = idesc_f16_f32(kTM, (ti.nvalid + 15) & ~15);
        const int ab = tc % S::kAcc;
        const uint32_t acc = tmem + (uint32_t)(ab * kTN);
        if (!mbar_wait(&acc_empty[ab], ((tc / S::kAcc) & 1) ^ 1, p.status)) break;
        tc_fence_after();
        PF_STAMP(tc, 0, global_timer_ns());
        PF_STAMP(tc, 6, (uint64_t)ti.nvalid);
        PF_STAMP(tc, 7, (uint64_t)ti.bucket);
        for (int ks = 0; ks < K / kTKe; ++ks, ++it) {
          const int s = it % S::kStages;
          const uint32_t par = (it / S::kStages) & 1;
          if (!mbar_wait(&full_a[s], par, p.status) || !mbar_wait(&full_b[s], par, p.status)) {
            tc = -1;
            break;
          }
          tc_fence_after();
          uint8_t* st = stages + (size_t)s * S::kStage;
          const uint64_t ad0 = sw128_kmajor_desc(smem_u32(st));
          const uint64_t ad1 = sw128_kmajor_desc(smem_u32(st + S::kA));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(st + (GATEUP ? 2 : 1) * S::kA));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {          // 32 bytes of K per MMA
            const uint32_t accum = (ks > 0 || kk > 0) ? 1u : 0u;
            if constexpr (F8) {
              tc_mma_f8(acc, ad0 + 2 * kk, bd + 2 * kk, idesc, accum);
              if (GATEUP) tc_mma_f8(acc + kTN, ad1 + 2 * kk, bd + 2 * kk, idesc, accum);
            } else {
              tc_mma_f16(acc, ad0 + 2 * kk, bd + 2 * kk, idesc, accum);
              if (GATEUP) tc_mma_f16(acc + kTN, ad1 + 2 * kk, bd + 2 * kk, idesc, accum);
            }
          }
          tc_commit(&empty[s]);
        }
        if (tc < 0) break;
        PF_STAMP(tc, 1, global_timer_ns());
        tc_commit(&acc_full[ab]);
      }
    }
  } else if (RAW && warp == 2) {
    // ---- IQ4_NL rows of the weight tiles by TMA, four K-steps per copy
    if (lane == 0) {
      int it = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const TileInfo ti = tile_info(t);
        const bool sh = ti.bucket >= p.E;
        const int K = sh ? p.Ks : p.K;
        const int row = (sh ? 0 : ti.bucket * p.M) + ti.m0;
        bool ok = true;
        for (int g = 0; g < K / (kTK * S::kRawGroup); ++g, ++it) {
          const int s = it % S::kRawRing;
          if (!mbar_wait(&empty_raw[s], ((it / S::kRawRing) & 1) ^ 1, p.status)) {
            ok = false;
            break;
          }
          uint8_t* dst = raw + (size_t)s * S::kRawStage;
          mbar_arrive_expect_tx(&full_raw[s], (uint32_t)S::kRawStage);
          tma_load_2d(dst, &tmaps.raw[sh ? 2 : 0], g * S::kRawGroup * kPairB, row, &full_raw[s]);
          if (GATEUP)
            tma_load_2d(dst + S::kRawMat, &tmaps.raw[sh ? 3 : 1], g * S::kRawGroup * kPairB, row,
                        &full_raw[s]);
        }
        if (!ok) break;
      }
    }
  } else if (warp < S::kCtl + S::kDq) {
    // ---- dequantise weight tiles (and, for gate/up, the epilogue of each tile)
    const int d = threadIdx.x - S::kCtl * 32;
    const int dw = warp - S::kCtl;
    const int r = d & (kTM - 1);
    // RAW gate/up: (row, matrix, block of the pair) per thread; otherwise
    // gate/up: (row, matrix), a whole pair per K-step; down: (row, block).
    const int part = (RAW && GATEUP) ? ((d >> 7) & 1) : (d >> 7);
    const int blkh = (RAW && GATEUP) ? (d >> 8) : part;
    int it = 0, itr = 0, tc = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x, ++tc) {
      const TileInfo ti = tile_info(t);
      const bool sh = ti.bucket >= p.E;
      const int K = sh ? p.Ks : p.K;
      const int nks = K / kTKe;
      // E4M3: the exponent of this thread's weight row
      int erow = 0;
      if constexpr (F8) {
        const int8_t* et = sh ? ((GATEUP && part) ? p.se1 : p.se0)
                              : ((GATEUP && part) ? p.e1 : p.e0);
        erow = et[(sh ? 0 : (size_t)ti.bucket * p.M) + ti.m0 + r];
      }
      if (warp == S::kCtl && lane == 0) PF_STAMP(tc, 2, global_timer_ns());
      // publish one dequantised K-step of this thread
      auto publish = [&](int s) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_a[s]);
        ++it;
      };
      if constexpr (RAW) {
        for (int g = 0; ok && g < nks / kStepsPerRaw; ++g, ++itr) {
          const int sr = itr % S::kRawRing;
          if (!mbar_wait(&full_raw[sr], (itr / S::kRawRing) & 1, p.status)) { ok = false; break; }
          const uint8_t* rrow = raw + (size_t)sr * S::kRawStage + (GATEUP ? part * S::kRawMat : 0) +
                                (size_t)r * S::kRawGroup * kPairB;
#pragma unroll
          for (int j = 0; j < kStepsPerRaw; ++j) {
            const int s = it % S::kStages;
            if (!mbar_wait(&empty[s], ((it / S::kStages) & 1) ^ 1, p.status)) { ok = false; break; }
            uint8_t* tile = stages + (size_t)s * S::kStage + (GATEUP ? part * S::kA : 0);
            if constexpr (F8) {
              // the step's four blocks are pairs 2j and 2j + 1 of the copy; this
              // thread takes pair 2j + blkh: 64 codes, chunks 4 blkh .. 4 blkh + 3
              const uint32_t* pw = reinterpret_cast<const uint32_t*>(rrow + (2 * j + blkh) * kPairB);
              uint32_t w9[9];
#pragma unroll
              for (int i = 0; i < 9; ++i) w9[i] = pw[i];
              uint32_t q0[4], q1[4], o0[8], o1[8];
#pragma unroll
              for (int i = 0; i < 4; ++i) q0[i] = prmt(w9[i], w9[i + 1], 0x5432u);
#pragma unroll
              for (int i = 0; i < 4; ++i) q1[i] = w9[5 + i];
              dequant_block_e4m3(q0, (uint16_t)(w9[0] & 0xFFFFu), erow, o0);
              dequant_block_e4m3(q1, (uint16_t)(w9[4] >> 16), erow, o1);
              const int c0 = 4 * blkh;
              sw128_store_chunk(tile, r, c0, make_uint4(o0[0], o0[1], o0[2], o0[3]));
              sw128_store_chunk(tile, r, c0 + 1, make_uint4(o0[4], o0[5], o0[6], o0[7]));
              sw128_store_chunk(tile, r, c0 + 2, make_uint4(o1[0], o1[1], o1[2], o1[3]));
              sw128_store_chunk(tile, r, c0 + 3, make_uint4(o1[4], o1[5], o1[6], o1[7]));
              publish(s);
              continue;
            }
            const uint32_t* w = reinterpret_cast<const uint32_t*>(rrow + j * kPairB + (blkh ? 16 : 0));
            uint32_t q[4];
            uint16_t dbits;
            if (blkh == 0) {
              const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
              dbits = (uint16_t)(w0 & 0xFFFFu);
              q[0] = prmt(w0, w1, 0x5432u);
              q[1] = prmt(w1, w2, 0x5432u);
              q[2] = prmt(w2, w3, 0x5432u);
              q[3] = prmt(w3, w4, 0x5432u);
            } else {
              dbits = (uint16_t)(w[0] >> 16);
              q[0] = w[1]; q[1] = w[2]; q[2] = w[3]; q[3] = w[4];
            }
            dequant_block_to_tile(q, dbits, tile, r, 4 * blkh);
            publish(s);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_raw[sr]);
        }
      } else {
        const size_t rb = (size_t)(K / 32) * kBlockB;
        const int M = sh ? p.Ms : p.M;
        const uint8_t* mat;
        if (GATEUP) mat = sh ? (part ? p.s1 : p.s0) : (part ? p.a1 : p.a0);
        else mat = sh ? p.s0 : p.a0;
        const uint8_t* row = mat + ((sh ? 0 : (size_t)ti.bucket * M) + ti.m0 + r) * rb;
        // One K-step: wait for the stage, dequantise this thread's weights
        // (one block pair, nine words w) into the swizzled A tile, publish.
        auto step = [&](const uint32_t (&w)[9]) -> bool {
          const int s = it % S::kStages;
          if (!mbar_wait(&empty[s], ((it / S::kStages) & 1) ^ 1, p.status)) return false;
          uint8_t* st = stages + (size_t)s * S::kStage;
          uint32_t q0[4], q1[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) q0[i] = prmt(w[i], w[i + 1], 0x5432u);
#pragma unroll
          for (int i = 0; i < 4; ++i) q1[i] = w[5 + i];
          const uint16_t d0 = (uint16_t)(w[0] & 0xFFFFu), d1 = (uint16_t)(w[4] >> 16);
          if (GATEUP) {
            uint8_t* tile = st + part * S::kA;
            dequant_block_to_tile(q0, d0, tile, r, 0);
            dequant_block_to_tile(q1, d1, tile, r, 4);
          } else {
            if (part == 0) dequant_block_to_tile(q0, d0, st, r, 0);
            else dequant_block_to_tile(q1, d1, st, r, 4);
          }
          publish(s);
          return true;
        };
        if ((nks & 3) == 0) {
          // raw bytes four K-steps (144 bytes) at a time, double-buffered in
          // registers; the four steps of a group are unrolled so that every
          // word comes from a fixed register
          uint4 cur[9], nxt[9];
          auto load_group = [&](int g, uint4 (&dst)[9]) {
            const uint4* src = reinterpret_cast<const uint4*>(row + (size_t)g * 4 * kPairB);
#pragma unroll
            for (int i = 0; i < 9; ++i) dst[i] = __ldg(src + i);
          };
          load_group(0, nxt);
#pragma unroll 1
          for (int g = 0; ok && g < nks / 4; ++g) {
#pragma unroll
            for (int i = 0; i < 9; ++i) cur[i] = nxt[i];
            if (g + 1 < nks / 4) load_group(g + 1, nxt);
            const uint32_t* cw = reinterpret_cast<const uint32_t*>(cur);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t w[9];
#pragma unroll
              for (int i = 0; i < 9; ++i) w[i] = cw[9 * j + i];
              if (!step(w)) { ok = false; break; }
            }
          }
        } else {
#pragma unroll 1
          for (int ks = 0; ok && ks < nks; ++ks) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(row + (size_t)ks * kPairB);
            uint32_t w[9];
#pragma unroll
            for (int i = 0; i < 9; ++i) w[i] = __ldg(src + i);
            if (!step(w)) ok = false;
          }
        }
      }
      if (!ok) break;
      if (warp == S::kCtl && lane == 0) PF_STAMP(tc, 3, global_timer_ns());
      if constexpr (S::kEpi == 0) {
      // epilogue: TMEM lanes of this warp's quarter; the tile's token columns
      // in units of 8, dealt round-robin to the warps of the quarter, so that
      // a tile of few tokens still spreads over all the dequantising warps
      constexpr int kShares = S::kDq / 4;       // warps per TMEM lane quarter
      const int q = warp & 3;
      const int ch = dw >> 2;                   // this warp's units: ch, ch + kShares, ...
      const int mrow = ti.m0 + q * 32 + lane;   // weight row of this thread
      const int nunits = (ti.nvalid + 7) >> 3;
      const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
      // E4M3: 2^(gate, up row exponents); the exponents of this warp's
      // columns, lane l holding column l % 8 of unit ch + 4 (l / 8) (bxa) and
      // of unit ch + 16 + 4 (l / 8) (bxb), loaded before the accumulator wait
      float sg = 1.f, su = 1.f;
      int bxa = 0, bxb = 0;
      if constexpr (F8) {
        static_assert(kShares == 4, "the exponent prefetch below deals units over four warps");
        const size_t er = (sh ? 0 : (size_t)ti.bucket * p.M) + mrow;
        sg = exp2i((sh ? p.se0 : p.e0)[er]);
        su = exp2i((sh ? p.se1 : p.e1)[er]);
        const int ca = (ch + 4 * (lane >> 3)) * 8 + (lane & 7);
        if (ca < ti.nvalid) bxa = p.bexp[ti.row0 + ti.n0 + ca];
        if (ca + 128 < ti.nvalid) bxb = p.bexp[ti.row0 + ti.n0 + ca + 128];
      }
      if (!mbar_wait(acc_full, tc & 1, p.status)) { ok = false; break; }
      tc_fence_after();
      if (warp == S::kCtl && lane == 0) PF_STAMP(tc, 4, global_timer_ns());
#pragma unroll 1
      for (int i = 0; i < (kTN / 8) / kShares; ++i) {
        const int unit = ch + kShares * i;
        if (unit >= nunits) break;              // warp-uniform
        const int col = unit * 8;
        uint32_t g[8], u[8];
        tmem_ld8(tq + col, g);
        tmem_ld8(tq + kTN + col, u);
        tmem_ld_wait();
        const size_t row0 = (size_t)(ti.row0 + ti.n0 + col);
        if constexpr (F8) {
          // h = silu(g) u with g, u scaled back by 2^(row + column exponents);
          // lanes 0..7 (and their copies) get the unit's eight exponents
          const int bx8 = __shfl_sync(0xFFFFFFFFu, i < 4 ? bxa : bxb, ((i & 3) << 3) + (lane & 7));
          const float st8 = pow2_of(bx8);
          if (__all_sync(0xFFFFFFFFu, bx8 >= -126 && bx8 <= 127)) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (col + j < ti.nvalid) {
                const float st = __shfl_sync(0xFFFFFFFFu, st8, j);
                p.h32[(row0 + j) * p.ldh + mrow] = silu_mul_fast(__uint_as_float(g[j]) * sg * st,
                                                                 __uint_as_float(u[j]) * su * st);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (col + j < ti.nvalid) {
                const int bx = __shfl_sync(0xFFFFFFFFu, bx8, j);
                const float st = pow2_of(bx);
                p.h32[(row0 + j) * p.ldh + mrow] =
                    silu_mul_fast(scale_acc(__uint_as_float(g[j]), sg, bx, st),
                                  scale_acc(__uint_as_float(u[j]), su, bx, st));
              }
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (col + j < ti.nvalid) {
              const float hv = silu_mul_fast(__uint_as_float(g[j]), __uint_as_float(u[j]));
              p.h[(row0 + j) * p.ldh + mrow] = __float2half_rn(hv);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (warp == S::kCtl && lane == 0) PF_STAMP(tc, 5, global_timer_ns());
      if (lane == 0) mbar_arrive(acc_empty);
      }
    }
  }
  if constexpr (S::kEpi > 0) {
    if (warp >= S::kCtl + S::kDq) {
      // ---- epilogue warps: each takes its TMEM lane quarter (32 weight rows)
      // and every token column of the tile, from the tile's accumulator
      const int q = warp & 3;
      int tc = 0;
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tc) {
        const TileInfo ti = tile_info(t);
        const int ab = tc % S::kAcc;
        const int mrow = ti.m0 + q * 32 + lane;
        // E4M3: 2^(the down row's exponent), loaded before the accumulator
        // wait; the columns' (h rows') exponents scale the combine weights
        float sd = 1.f;
        if constexpr (F8) {
          const bool sh = ti.bucket >= p.E;
          sd = exp2i((sh ? p.se0 : p.e0)[(sh ? 0 : (size_t)ti.bucket * p.M) + mrow]);
        }
        if (!mbar_wait(&acc_full[ab], (tc / S::kAcc) & 1, p.status)) break;
        tc_fence_after();
        if (warp == S::kCtl + S::kDq && lane == 0) PF_STAMP(tc, 4, global_timer_ns());
        const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * kTN);
        for (int col = 0; col < kTN; col += 32) {
          if (col >= ti.nvalid) break;            // warp-uniform
          uint32_t g[32];
          tmem_ld32(base + col, g);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col + j < ti.nvalid) {
              const size_t row = (size_t)(ti.row0 + ti.n0 + col + j);
              p.o[row * p.ldo + mrow] = F8 ? __uint_as_float(g[j]) * sd : __uint_as_float(g[j]);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (warp == S::kCtl + S::kDq && lane == 0) PF_STAMP(tc, 5, global_timer_ns());
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) PF_STAMP_K(1, global_timer_ns());
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// 4. Combine: y[t] = o[shared row] + sum over routed rows (experts ascending) w o.
__global__ void pf_combine_kernel(const float* __restrict__ o, const int32_t* __restrict__ comb_row,
                                  const float* __restrict__ comb_w, int T, int kk, int H,
                                  float* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int h4 = H / 4;
  const int64_t total = (int64_t)T * h4;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / h4), c = (int)(i - (int64_t)t * h4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int32_t* cr = comb_row + (size_t)t * kk;
    const float* cw = comb_w + (size_t)t * kk;
    // rows in groups of four: the group's loads are all in flight before the
    // first of its terms is added (terms in the fixed order)
    for (int j0 = 0; j0 < kk; j0 += 4) {
      int r[4];
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) r[u] = j0 + u < kk ? cr[j0 + u] : -1;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[u] = r[u] >= 0 ? reinterpret_cast<const float4*>(o + (size_t)r[u] * H)[c]
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (r[u] < 0) break;
        const float wv = cw[j0 + u];
        acc.x = fmaf(wv, v[u].x, acc.x);
        acc.y = fmaf(wv, v[u].y, acc.y);
        acc.z = fmaf(wv, v[u].z, acc.z);
        acc.w = fmaf(wv, v[u].w, acc.w);
      }
      if (r[3] < 0) break;
    }
    reinterpret_cast<float4*>(y + (size_t)t * H)[c] = acc;
  }
}

// ---------------------------------------------------------------------------
// E4M3 weight scales: each row's exponent, the largest floor(log2 d) of its
// blocks' fp16 scales (-14 for a subnormal or zero d), one warp per row.
struct RowExpJob {
  const uint8_t* mat;
  int64_t rows;
  int K;
  int8_t* out;
};
struct RowExpJobs {
  RowExpJob j[6];
  int n;
};
__global__ void pf8_row_exp_kernel(const __grid_constant__ RowExpJobs jobs) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int q = 0; q < jobs.n; ++q) {
    const RowExpJob& J = jobs.j[q];
    const int nb = J.K / 32;
    for (int64_t r = gw; r < J.rows; r += nw) {
      const uint8_t* row = J.mat + r * nb * kBlockB;
      int e = -1000;
      for (int b = lane; b < nb; b += 32) {
        const uint16_t d = (uint16_t)(row[(size_t)b * kBlockB] | (row[(size_t)b * kBlockB + 1] << 8));
        const int f = (d >> 10) & 0x1F;
        const int eb = f == 0 ? -14 : f - 15;
        e = eb > e ? eb : e;
      }
      e = __reduce_max_sync(0xFFFFFFFFu, (unsigned)(e + 1024)) - 1024;
      if (lane == 0) J.out[r] = (int8_t)e;
    }
  }
}

// Each thread: one block of a row, through dequant_block_e4m3 with the row's
// exponent (written by pf8_row_exp_kernel first); its codes are written back in
// K order.
__global__ void pf8_dequant_kernel(const uint8_t* __restrict__ mat, int64_t rows, int K,
                                   const int8_t* __restrict__ row_exp, uint8_t* __restrict__ out) {
  const int nb = K / 32;
  const int64_t n = rows * nb;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nb;
    const uint8_t* b = mat + i * kBlockB;
    const uint16_t d = (uint16_t)(b[0] | (b[1] << 8));
    uint32_t q[4];
#pragma unroll
    for (int w = 0; w < 4; ++w)
      q[w] = (uint32_t)b[2 + 4 * w] | ((uint32_t)b[3 + 4 * w] << 8) |
             ((uint32_t)b[4 + 4 * w] << 16) | ((uint32_t)b[5 + 4 * w] << 24);
    uint32_t c[8];
    dequant_block_e4m3(q, d, row_exp[r], c);
    uint8_t* o = out + i * 32;                 // 32 codes, back in K order
#pragma unroll
    for (int p = 0; p < 32; ++p) o[e4m3_block_pos_value(p)] = (uint8_t)(c[p >> 2] >> (8 * (p & 3)));
  }
}

// ---------------------------------------------------------------------------
// Host side.
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// fp16 [rows][cols] row-major, box 64 columns x 256 rows, 128-byte swizzle.
bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// E4M3 codes [rows][cols] row-major (cols bytes a row), box 128 columns x
// box_rows rows, 128-byte swizzle.
bool make_tmap_u8(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// IQ4_NL rows (bytes) of a stacked weight matrix: rows x (K/32 * 18) bytes;
// boxes of 144 bytes (four block pairs) x 128 rows. Needs the row pitch to be
// a multiple of 16 bytes (K a multiple of 256).
bool make_raw_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t K) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int64_t rb = K / 32 * kBlockB;
  cuuint64_t dims[2] = {(cuuint64_t)rb, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)rb};
  cuuint32_t box[2] = {(cuuint32_t)(4 * kPairB), (cuuint32_t)kTM};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern kernel, dim3 grid, dim3 block, size_t smem, bool pdl,
                      cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <bool GATEUP, bool RAW, bool F8 = false>
cudaError_t launch_gemm(int num_sms, int E, bool pdl, cudaStream_t stream, const TmapSet& tm,
                        const GemmParams& g) {
  using S = GemmCfg<GATEUP, RAW>;
  const size_t sm = S::kTotal + (size_t)(E + 2) * 8;
  const cudaError_t e =
      ensure_smem_attr(reinterpret_cast<const void*>(pf_gemm_kernel<GATEUP, RAW, F8>), sm);
  if (e != cudaSuccess) return e;
  return launch_ex(pf_gemm_kernel<GATEUP, RAW, F8>, dim3(num_sms), dim3(S::kThreads), sm, pdl,
                   stream, tm, g);
}

}  // namespace

bool prefill_supported(const moe_shape& s) {
  return s.hidden % kTM == 0 && s.ffn % kTM == 0 && (!s.n_shared || s.ffn_shared % kTM == 0);
}

int prefill_launches(const moe_shape& s, int T) {
  if (T <= 0) return 0;
  return prefill_supported(s) ? 5 : 0;
}

cudaError_t launch_prefill(const moe_shape& s, const moe_expert_weights& w, const uint16_t* x,
                           int T, const int32_t* ids, const float* weights, float* y,
                           uint8_t* ws, const PrefillLayout& L, uint32_t* status, int num_sms,
                           bool pdl, cudaStream_t stream) {
  if (!prefill_supported(s)) return cudaErrorNotSupported;
  const int E = s.n_experts, k = s.top_k, H = s.hidden, F = s.ffn;
  const int Fs = s.n_shared ? s.ffn_shared : 0;
  const int fmax = F > Fs ? F : Fs;
  const int64_t rows = (int64_t)T * k + (s.n_shared ? T : 0);
  int32_t* boff = reinterpret_cast<int32_t*>(ws + L.counts);
  int32_t* row_of = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* row_tok = reinterpret_cast<int32_t*>(ws + L.perm);
  int32_t* comb_row = reinterpret_cast<int32_t*>(ws + L.comb);
  float* comb_w = reinterpret_cast<float*>(ws + L.comb + (int64_t)T * (k + 1) * 4);
  __half* x16 = reinterpret_cast<__half*>(ws + L.x16);
  __half* h16 = reinterpret_cast<__half*>(ws + L.h16);
  float* o = reinterpret_cast<float*>(ws + L.o);

  BucketParams bp{ids, T, k, E, s.n_shared, boff, row_of, row_tok, status};
  const size_t bsm = (size_t)kBucketWarps * E * 4;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(pf_bucket_kernel), bsm);
  if (e != cudaSuccess) return e;
  e = launch_ex(pf_bucket_kernel, dim3(1), dim3(kBucketThreads), bsm, pdl, stream, bp);
  if (e != cudaSuccess) return e;
  const CombineListParams cl{(const int32_t*)row_of, weights, T, k, s.n_shared, comb_row, comb_w};
  e = launch_ex(pf_gather_kernel<false>, dim3(num_sms * 4), dim3(256), 0, pdl, stream, x,
                (const int32_t*)boff, E, H, x16, cl, Gather8{});
  if (e != cudaSuccess) return e;

  TmapSet tm_x, tm_h;
  for (int b = 0; b < kNumBoxes; ++b)
    if (!make_tmap(&tm_x.m[b], x16, rows, H, 32 << b) ||
        !make_tmap(&tm_h.m[b], h16, rows, fmax, 32 << b))
      return cudaErrorInvalidValue;
  GemmParams g1{};
  g1.E = E;
  g1.n_shared = s.n_shared;
  g1.M = F;
  g1.Ms = Fs;
  g1.K = H;
  g1.Ks = H;
  g1.a0 = reinterpret_cast<const uint8_t*>(w.gate);
  g1.a1 = reinterpret_cast<const uint8_t*>(w.up);
  g1.s0 = reinterpret_cast<const uint8_t*>(w.sh_gate);
  g1.s1 = reinterpret_cast<const uint8_t*>(w.sh_up);
  g1.bucket_off = boff;
  g1.h = h16;
  g1.ldh = fmax;
  g1.status = status;
  // raw-weight copies when the reduction lengths keep row pitches 16-byte aligned
  const bool raw1 = H % 256 == 0;
  const bool raw2 = F % 256 == 0 && (!s.n_shared || Fs % 256 == 0);
  if (raw1 && (!make_raw_tmap(&tm_x.raw[0], w.gate, (int64_t)E * F, H) ||
               !make_raw_tmap(&tm_x.raw[1], w.up, (int64_t)E * F, H) ||
               (s.n_shared && (!make_raw_tmap(&tm_x.raw[2], w.sh_gate, Fs, H) ||
                               !make_raw_tmap(&tm_x.raw[3], w.sh_up, Fs, H)))))
    return cudaErrorInvalidValue;
  if (raw2 && (!make_raw_tmap(&tm_h.raw[0], w.down, (int64_t)E * H, F) ||
               (s.n_shared && !make_raw_tmap(&tm_h.raw[2], w.sh_down, H, Fs))))
    return cudaErrorInvalidValue;
  e = raw1 ? launch_gemm<true, true>(num_sms, E, pdl, stream, tm_x, g1)
           : launch_gemm<true, false>(num_sms, E, pdl, stream, tm_x, g1);
  if (e != cudaSuccess) return e;

  GemmParams g2 = g1;
  g2.M = H;
  g2.Ms = H;
  g2.K = F;
  g2.Ks = Fs;
  g2.a0 = reinterpret_cast<const uint8_t*>(w.down);
  g2.a1 = nullptr;
  g2.s0 = reinterpret_cast<const uint8_t*>(w.sh_down);
  g2.s1 = nullptr;
  g2.h = nullptr;
  g2.o = o;
  g2.ldo = H;
  e = raw2 ? launch_gemm<false, true>(num_sms, E, pdl, stream, tm_h, g2)
           : launch_gemm<false, false>(num_sms, E, pdl, stream, tm_h, g2);
  if (e != cudaSuccess) return e;

  const int64_t total = (int64_t)T * (H / 4);
  int64_t grid = (total + 255) / 256;
  if (grid > (int64_t)num_sms * 8) grid = (int64_t)num_sms * 8;
  return launch_ex(pf_combine_kernel, dim3((unsigned)grid), dim3(256), 0, pdl, stream,
                   (const float*)o, (const int32_t*)comb_row, (const float*)comb_w, T, k + 1, H,
                   y);
}

// ---------------------------------------------------------------------------
// The prefill with E4M3 operands: the same bucketing, tiles and combine; the
// weights' row scales come from a table made once for the weights
// (launch_fp8_row_exponents).
bool prefill_fp8_supported(const moe_shape& s) {
  // the raw-row ring (reduction lengths multiples of 256) feeds the E4M3 producers
  return prefill_supported(s) && s.hidden % 256 == 0 && s.ffn % 256 == 0 &&
         (!s.n_shared || s.ffn_shared % 256 == 0);
}

int64_t fp8_row_exponent_count(const moe_shape& s) {
  const int64_t E = s.n_experts, H = s.hidden, F = s.ffn;
  const int64_t Fs = s.n_shared ? s.ffn_shared : 0;
  return E * F * 2 + E * H + (s.n_shared ? 2 * Fs + H : 0);
}

cudaError_t launch_fp8_row_exponents(const moe_shape& s, const moe_expert_weights& w,
                                     int8_t* out, cudaStream_t stream) {
  const int64_t E = s.n_experts, H = s.hidden, F = s.ffn;
  const int64_t Fs = s.n_shared ? s.ffn_shared : 0;
  RowExpJobs jobs{};
  int64_t off = 0;
  auto add = [&](const void* m, int64_t rows, int K) {
    jobs.j[jobs.n++] = RowExpJob{reinterpret_cast<const uint8_t*>(m), rows, K, out + off};
    off += rows;
  };
  add(w.gate, E * F, (int)H);
  add(w.up, E * F, (int)H);
  add(w.down, E * H, (int)F);
  if (s.n_shared) {
    add(w.sh_gate, Fs, (int)H);
    add(w.sh_up, Fs, (int)H);
    add(w.sh_down, H, (int)Fs);
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  pf8_row_exp_kernel<<<sms * 8, 256, 0, stream>>>(jobs);
  return cudaGetLastError();
}

cudaError_t launch_dequant_e4m3(const void* mat, int64_t rows, int K, int8_t* row_exp,
                                uint8_t* out, int num_sms, cudaStream_t stream) {
  RowExpJobs jobs{};
  jobs.j[0] = RowExpJob{reinterpret_cast<const uint8_t*>(mat), rows, K, row_exp};
  jobs.n = 1;
  pf8_row_exp_kernel<<<num_sms * 8, 256, 0, stream>>>(jobs);
  int64_t grid = (rows * (K / 32) + 255) / 256;
  if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
  pf8_dequant_kernel<<<(unsigned)grid, 256, 0, stream>>>(reinterpret_cast<const uint8_t*>(mat),
                                                        rows, K, row_exp, out);
  return cudaGetLastError();
}

cudaError_t launch_prefill_fp8(const moe_shape& s, const moe_expert_weights& w,
                               const int8_t* row_exp, const uint16_t* x, int T,
                               const int32_t* ids, const float* weights, float* y, uint8_t* ws,
                               const PrefillLayout& L, uint32_t* status, int num_sms, bool pdl,
                               cudaStream_t stream) {
  if (!prefill_fp8_supported(s)) return cudaErrorNotSupported;
  const int E = s.n_experts, k = s.top_k, H = s.hidden, F = s.ffn;
  const int Fs = s.n_shared ? s.ffn_shared : 0;
  const int fmax = F > Fs ? F : Fs;
  const int64_t rows = (int64_t)T * k + (s.n_shared ? T : 0);
  int32_t* boff = reinterpret_cast<int32_t*>(ws + L.counts);
  int32_t* row_of = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* row_tok = reinterpret_cast<int32_t*>(ws + L.perm);
  int32_t* comb_row = reinterpret_cast<int32_t*>(ws + L.comb);
  float* comb_w = reinterpret_cast<float*>(ws + L.comb + (int64_t)T * (k + 1) * 4);
  float* o = reinterpret_cast<float*>(ws + L.o);
  uint8_t* x8 = ws + L.x8;
  uint8_t* h8 = ws + L.h8;
  float* h32 = reinterpret_cast<float*>(ws + L.h32);
  int32_t* bexp = reinterpret_cast<int32_t*>(ws + L.bexp);
  int32_t* hexp = reinterpret_cast<int32_t*>(ws + L.hexp);
  const int64_t EF = (int64_t)E * F, EH = (int64_t)E * H;
  const int8_t* ex_gate = row_exp;
  const int8_t* ex_up = row_exp + EF;
  const int8_t* ex_down = row_exp + 2 * EF;
  const int8_t* ex_sg = row_exp + 2 * EF + EH;
  const int8_t* ex_su = ex_sg + Fs;
  const int8_t* ex_sd = ex_su + Fs;

  BucketParams bp{ids, T, k, E, s.n_shared, boff, row_of, row_tok, status};
  const size_t bsm = (size_t)kBucketWarps * E * 4;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(pf_bucket_kernel), bsm);
  if (e != cudaSuccess) return e;
  e = launch_ex(pf_bucket_kernel, dim3(1), dim3(kBucketThreads), bsm, pdl, stream, bp);
  if (e != cudaSuccess) return e;
  const CombineListParams cl{(const int32_t*)row_of, weights, T, k, s.n_shared, comb_row, comb_w};
  const Gather8 g8{bexp, x8};
  e = launch_ex(pf_gather_kernel<true>, dim3(num_sms * 4), dim3(256), 0, pdl, stream, x,
                (const int32_t*)boff, E, H, (__half*)nullptr, cl, g8);
  if (e != cudaSuccess) return e;

  TmapSet tm_x, tm_h;
  for (int b = 0; b < kNumBoxes; ++b)
    if (!make_tmap_u8(&tm_x.m[b], x8, rows, H, 32 << b) ||
        !make_tmap_u8(&tm_h.m[b], h8, rows, fmax, 32 << b))
      return cudaErrorInvalidValue;
  if (!make_raw_tmap(&tm_x.raw[0], w.gate, (int64_t)E * F, H) ||
      !make_raw_tmap(&tm_x.raw[1], w.up, (int64_t)E * F, H) ||
      (s.n_shared && (!make_raw_tmap(&tm_x.raw[2], w.sh_gate, Fs, H) ||
                      !make_raw_tmap(&tm_x.raw[3], w.sh_up, Fs, H))) ||
      !make_raw_tmap(&tm_h.raw[0], w.down, (int64_t)E * H, F) ||
      (s.n_shared && !make_raw_tmap(&tm_h.raw[2], w.sh_down, H, Fs)))
    return cudaErrorInvalidValue;
  GemmParams g1{};
  g1.E = E;
  g1.n_shared = s.n_shared;
  g1.M = F;
  g1.Ms = Fs;
  g1.K = H;
  g1.Ks = H;
  g1.a0 = reinterpret_cast<const uint8_t*>(w.gate);
  g1.a1 = reinterpret_cast<const uint8_t*>(w.up);
  g1.s0 = reinterpret_cast<const uint8_t*>(w.sh_gate);
  g1.s1 = reinterpret_cast<const uint8_t*>(w.sh_up);
  g1.bucket_off = boff;
  g1.ldh = fmax;
  g1.status = status;
  g1.e0 = ex_gate;
  g1.e1 = ex_up;
  g1.se0 = ex_sg;
  g1.se1 = ex_su;
  g1.bexp = bexp;
  g1.h32 = h32;
  e = launch_gemm<true, true, true>(num_sms, E, pdl, stream, tm_x, g1);
  if (e != cudaSuccess) return e;
  e = launch_ex(pf8_hconv_kernel, dim3(num_sms * 4), dim3(256), 0, pdl, stream,
                (const float*)h32, (const int32_t*)boff, E, fmax, F, Fs,
                h8, hexp, (const int32_t*)row_tok, (const int32_t*)comb_row, comb_w, k + 1);
  if (e != cudaSuccess) return e;

  GemmParams g2 = g1;
  g2.M = H;
  g2.Ms = H;
  g2.K = F;
  g2.Ks = Fs;
  g2.a0 = reinterpret_cast<const uint8_t*>(w.down);
  g2.a1 = nullptr;
  g2.s0 = reinterpret_cast<const uint8_t*>(w.sh_down);
  g2.s1 = nullptr;
  g2.e0 = ex_down;
  g2.e1 = nullptr;
  g2.se0 = ex_sd;
  g2.se1 = nullptr;
  g2.bexp = nullptr;                 // the h rows' exponents enter in the combine
  g2.h32 = nullptr;
  g2.o = o;
  g2.ldo = H;
  e = launch_gemm<false, true, true>(num_sms, E, pdl, stream, tm_h, g2);
  if (e != cudaSuccess) return e;

  const int64_t total = (int64_t)T * (H / 4);
  int64_t grid = (total + 255) / 256;
  if (grid > (int64_t)num_sms * 8) grid = (int64_t)num_sms * 8;
  return launch_ex(pf_combine_kernel, dim3((unsigned)grid), dim3(256), 0, pdl, stream,
                   (const float*)o, (const int32_t*)comb_row, (const float*)comb_w, T, k + 1, H,
                   y);
}

}  // namespace moe

#ifdef MOE_PROFILE
// Copies the GEMM tile stamps (uint64 [2][256][16][8], ns of %globaltimer).
// Profiling builds only.
extern "C" int moe_profile_prefill(void* host, size_t bytes) {
  const size_t n = sizeof(moe::g_pfprof) < bytes ? sizeof(moe::g_pfprof) : bytes;
  return cudaMemcpyFromSymbol(host, moe::g_pfprof, n) == cudaSuccess ? 0 : -1;
}
#endif
