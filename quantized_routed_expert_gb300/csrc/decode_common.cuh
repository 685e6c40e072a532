// Device helpers shared by the decode kernels: the route table built from
// ids, the 16-bit block-quantised vector layout, row splitting and the
// deferred F-block arrivals that quantise h.
#pragma once

#include "common.cuh"
#include "decode.cuh"

namespace moe {

// A named barrier over NT threads (id 0 with all threads of the CTA is
// __syncthreads).
template <int BAR, int NT>
__device__ __forceinline__ void bar_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT) : "memory");
}

// ---------------------------------------------------------------------------
// Route table built in shared memory from ids (route sanitising: an id outside
// [0, E) is dropped, i.e. routed to expert 0 with weight 0).
struct RouteTable {
  int n_slots;                 // distinct routed experts, ascending
  int n_valid;
  int invalid;
  uint32_t bitmap[MOE_MAX_EXPERTS / 32];
  int word_off[MOE_MAX_EXPERTS / 32];
  int sid[kMaxPairs];          // sanitised expert id per pair, -1 if invalid
  float wt[kMaxPairs];         // weight per pair
  int slot_expert[kMaxPairs];
  int slot_off[kMaxPairs + 1]; // CSR offsets into list
  int list[kMaxPairs];         // pair indices grouped by slot, ascending within a slot
};

__device__ __forceinline__ int slot_of_expert(const RouteTable& rt, int e) {
  const uint32_t w = rt.bitmap[e >> 5];
  return rt.word_off[e >> 5] + __popc(w & ((1u << (e & 31)) - 1u));
}

// Called by NT threads (named barrier BAR). P = T*k <= 256.
template <int NT, int BAR>
__device__ void build_route_table(RouteTable& rt, const int32_t* __restrict__ ids,
                                  const float* __restrict__ wts, int P, int E) {
  const int tid = threadIdx.x;
  if (tid < MOE_MAX_EXPERTS / 32) rt.bitmap[tid] = 0u;
  if (tid == 0) rt.invalid = 0;
  bar_sync<BAR, NT>();
  for (int i = tid; i < P; i += NT) {
    const int id = ids[i];
    const bool ok = id >= 0 && id < E;
    rt.sid[i] = ok ? id : -1;
    rt.wt[i] = ok ? wts[i] : 0.0f;
    if (ok) atomicOr(&rt.bitmap[id >> 5], 1u << (id & 31));
    else atomicAdd(&rt.invalid, 1);
  }
  bar_sync<BAR, NT>();
  if (tid < 32) {
    const int nw = (E + 31) >> 5;
    const int c = tid < nw ? __popc(rt.bitmap[tid]) : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (tid >= o) incl += v;
    }
    const int excl = incl - c;
    if (tid < nw) {
      rt.word_off[tid] = excl;
      uint32_t bits = rt.bitmap[tid];
      int pos = excl;
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1u;
        rt.slot_expert[pos++] = tid * 32 + b;
      }
    }
    if (tid == 31) rt.n_slots = incl;
  }
  bar_sync<BAR, NT>();
  // stable counting sort of the valid pairs by expert: rank = #smaller experts
  // + #earlier pairs of the same expert
  for (int p = tid; p < P; p += NT) {
    const int e = rt.sid[p];
    if (e < 0) continue;
    int rank = 0;
    bool first = true;
    for (int q = 0; q < P; ++q) {
      const int eq = rt.sid[q];
      if (eq < 0) continue;
      rank += (eq < e) || (eq == e && q < p);
      first = first && !(eq == e && q < p);
    }
    rt.list[rank] = p;
    if (first) rt.slot_off[slot_of_expert(rt, e)] = rank;
  }
  if (tid == 0) {
    rt.n_valid = P - rt.invalid;
    rt.slot_off[rt.n_slots] = rt.n_valid;
  }
  bar_sync<BAR, NT>();
}

__host__ __device__ __forceinline__ size_t align_up_dev(size_t v, size_t a) {
  return (v + a - 1) / a * a;
}
__host__ __device__ __forceinline__ int row_granule_dev(int K) {
  const int rb = K / 32 * kBlockB;
  int g = 1;
  while ((g * rb) % 16) g *= 2;
  return g;
}

// ---------------------------------------------------------------------------
// Quantised vector layout: the int16 pair words of block pair q, 16-byte chunk
// c (0..7), live at uint4 index ((q / lpr) * 8 + c) * lpr + q % lpr, so that
// lanes reading consecutive pairs read consecutive 16-byte chunks. Scales
// (one fp32 per 32 values) follow the pair words.
// lpr is a power of two: ((q / lpr) * 8 + c) * lpr + q % lpr without division.
__device__ __forceinline__ int qv_base(int q, int lpr) {
  return ((q & ~(lpr - 1)) << 3) + (q & (lpr - 1));
}
__device__ __forceinline__ int qv_u4(int q, int c, int lpr) { return qv_base(q, lpr) + c * lpr; }
// Lanes that share one row in the down kernels, and the interleave width of
// the quantised vector layout: a power of two (the reduction is an xor
// butterfly), at most 8 (a lane then walks several block pairs of its row) and
// at most the number of block pairs in the row.
__host__ __device__ __forceinline__ int dlanes_per_row(int K) {
  int l = 8;
  while (l > K / 64) l >>= 1;
  return l;
}
__host__ __device__ __forceinline__ int dqvec_pair_words(int K) {
  const int lpr = dlanes_per_row(K);
  return (K / 64 + lpr - 1) / lpr * lpr * 32;
}
__host__ __device__ __forceinline__ int dqvec_words(int K) {
  return dqvec_pair_words(K) + ((K / 32 + 3) & ~3);
}

// Quantise 32 consecutive values (one per lane) of block b of a K-vector into
// the record `rec` (shared or global). All 32 lanes participate.
__device__ __forceinline__ void quant_block_store(float v, int b, int K, uint32_t* rec) {
  const int lane = threadIdx.x & 31;
  const uint32_t e = (__float_as_uint(v) >> 23) & 0xFFu;
  const uint32_t emax = __reduce_max_sync(0xFFFFFFFFu, e);
  const int m = quant_one(v, emax);
  const int hi = __shfl_down_sync(0xFFFFFFFFu, m, 16);
  const int lpr = dlanes_per_row(K);
  if (lane < 16) {
    const int q = b >> 1;
    const int w = 16 * (b & 1) + lane;          // word within the pair
    const uint32_t word = (uint32_t)(m & 0xFFFF) | ((uint32_t)hi << 16);
    rec[qv_u4(q, w >> 2, lpr) * 4 + (w & 3)] = word;
  }
  if (lane == 0) reinterpret_cast<float*>(rec + dqvec_pair_words(K))[b] = quant_scale(emax);
}


// Quantise T bf16 rows of K values into records in shared memory. Each lane
// loads 8 consecutive values (16 bytes); four lanes form one 32-value block, so
// a warp covers 8 blocks per load; four such groups are loaded before any is
// used, to keep loads in flight.
__device__ __forceinline__ void quant_group(const uint4 raw, bool ok, int b, int K,
                                            uint32_t* rec) {
  const int lane = threadIdx.x & 31;
  const int s = lane & 3;
  const uint32_t r[4] = {raw.x, raw.y, raw.z, raw.w};
  float v[8];
  uint32_t e = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(r[i] << 16);
    v[2 * i + 1] = __uint_as_float(r[i] & 0xFFFF0000u);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t ei = (__float_as_uint(v[i]) >> 23) & 0xFFu;
    e = ei > e ? ei : e;
  }
  uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, e, 1);
  e = o > e ? o : e;
  o = __shfl_xor_sync(0xFFFFFFFFu, e, 2);
  e = o > e ? o : e;
  int m[8], m2[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = quant_one(v[i], e);
#pragma unroll
  for (int i = 0; i < 8; ++i) m2[i] = __shfl_down_sync(0xFFFFFFFFu, m[i], 2);
  const int lpr = dlanes_per_row(K);
  if (ok && s < 2) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (uint32_t)(m[i] & 0xFFFF) | ((uint32_t)m2[i] << 16);
    const int q = b >> 1;
    const int c0 = 4 * (b & 1) + 2 * s;
    uint4* r4 = reinterpret_cast<uint4*>(rec);
    r4[qv_u4(q, c0, lpr)] = make_uint4(w[0], w[1], w[2], w[3]);
    r4[qv_u4(q, c0 + 1, lpr)] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  if (ok && s == 0) reinterpret_cast<float*>(rec + dqvec_pair_words(K))[b] = quant_scale(e);
}

__device__ __forceinline__ void quant_x_to_smem(const uint16_t* __restrict__ x, int T, int K,
                                                uint32_t* xq, int xq_words, int warp,
                                                int nwarps) {
  const int lane = threadIdx.x & 31;
  const int nb = K / 32;
  const int gpr = (nb + 7) / 8;                 // 8-block groups per row
  const int total = T * gpr;
  for (int g0 = warp; g0 < total; g0 += 4 * nwarps) {
    uint4 raw[4];
    bool ok[4];
    int bb[4], tt[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * nwarps;
      tt[u] = g / gpr;
      bb[u] = (g - tt[u] * gpr) * 8 + (lane >> 2);
      ok[u] = g < total && bb[u] < nb;
      raw[u] = ok[u] ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)tt[u] * K + bb[u] * 32 +
                                                            (lane & 3) * 8))
                     : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (g0 + u * nwarps < total)       // warp-uniform
        quant_group(raw[u], ok[u], bb[u], K, xq + (size_t)(tt[u] < T ? tt[u] : 0) * xq_words);
    }
  }
}

// ---------------------------------------------------------------------------
// Gate/up work: shared-expert rows are split evenly over the CTAs (known before
// the routes are), routed rows (slots x F, slot-major) likewise after.
struct Chunk {
  int slot;   // -1 = shared expert, else routed slot index
  int f0;
  int rows;
};

struct RowRange {
  int a, b;   // [a, b) in flattened rows
};

__device__ __forceinline__ RowRange split_rows(int total, int g, int cta, int ncta) {
  const int units = total / g;
  const long long ua = (long long)units * cta / ncta;
  const long long ub = (long long)units * (cta + 1) / ncta;
  return RowRange{(int)ua * g, (int)ub * g};
}

// The next chunk of [row, end) of a slot-major space with rows_per_slot rows.
__device__ __forceinline__ Chunk next_chunk(int row, int end, int rows_per_slot, bool shared) {
  Chunk c;
  const int s = row / rows_per_slot;
  c.slot = shared ? -1 : s;
  c.f0 = row - s * rows_per_slot;
  int n = rows_per_slot - c.f0;
  if (end - row < n) n = end - row;
  c.rows = n < kChunkRows ? n : kChunkRows;
  return c;
}

// Arrivals on F-blocks, deferred: a warp records the rows it finished and
// publishes them in batches behind one fence. The 32nd arrival on a block
// quantises the block for every token of the slot and resets its counter.
constexpr int kPendMax = 8;
struct Pending {
  int n;
  int slot[kPendMax];
  int f[kPendMax];
};

inline __device__ void flush_arrivals(const DecodeParams& p, const RouteTable& rt,
                                            Pending& pd) {
  const int lane = threadIdx.x & 31;
  __threadfence();                       // this warp's h stores, before its arrivals
  __syncwarp();
  const int fmax = p.F > p.Fs ? p.F : p.Fs;
  // lane i arrives for entry i (all arrivals in flight at once)
  uint32_t old = 0;
  if (lane < pd.n) {
    const int slot = pd.slot[lane];
    const int cid = slot < 0 ? p.E : rt.slot_expert[slot];
    old = atomicAdd(p.cnt + (size_t)cid * (fmax / 32) + pd.f[lane] / 32, 1u);
  }
  const uint32_t last = __ballot_sync(0xFFFFFFFFu, lane < pd.n && old == 31u);
  if (last) __threadfence();
  // (entry, token) blocks to quantise, gathered in batches so that their loads
  // are all in flight before the first block is reduced
  constexpr int kBatch = 8;
  int ent[kBatch], tokj[kBatch];
  int nb = 0;
  auto drain = [&]() {
    const float* src[kBatch];
    uint32_t* dst[kBatch];
    int Fb[kBatch], blk[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = ent[u < nb ? u : 0], j = tokj[u < nb ? u : 0];
      const int slot = pd.slot[i];
      const bool shared = slot < 0;
      const int F = shared ? p.Fs : p.F;
      const int words = dqvec_words(F);
      const int pr = shared ? j : rt.list[rt.slot_off[slot] + j];
      src[u] = shared ? p.h_s + (size_t)j * p.Fs : p.h_r + (size_t)pr * p.F;
      dst[u] = shared ? p.rec_s + (size_t)j * words : p.rec_r + (size_t)pr * words;
      Fb[u] = F;
      blk[u] = pd.f[i] / 32;
    }
    float v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) v[u] = u < nb ? __ldcg(src[u] + blk[u] * 32 + lane) : 0.f;
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (u < nb) quant_block_store(v[u], blk[u], Fb[u], dst[u]);
    nb = 0;
  };
  for (int i = 0; i < pd.n; ++i) {
    if (!((last >> i) & 1u)) continue;
    const int slot = pd.slot[i];
    const int ntok = slot < 0 ? p.T : rt.slot_off[slot + 1] - rt.slot_off[slot];
    for (int j = 0; j < ntok; ++j) {
      ent[nb] = i;
      tokj[nb] = j;
      if (++nb == kBatch) drain();
    }
  }
  if (nb) drain();
  // reset the counters of the blocks this warp completed
  if (lane < pd.n && old == 31u) {
    const int slot = pd.slot[lane];
    const int cid = slot < 0 ? p.E : rt.slot_expert[slot];
    p.cnt[(size_t)cid * (fmax / 32) + pd.f[lane] / 32] = 0u;
  }
  __syncwarp();
  pd.n = 0;
}


}  // namespace moe
