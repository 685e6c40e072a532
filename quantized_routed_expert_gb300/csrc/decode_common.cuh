// Device helpers shared by the decode kernels: the route table built from
// ids, the 16-bit block-quantised vector layout, x quantisation, row
// splitting and the gate/up unit.
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

// A named barrier over n threads (n a multiple of 32), id and n at run time.
__device__ __forceinline__ void bar_sync_n(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
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

// Called by the nt threads 0..nt-1 (named barrier BAR; nt a multiple of 32).
// P = T*k <= 256.
template <int BAR>
__device__ void build_route_table(RouteTable& rt, const int32_t* __restrict__ ids,
                                  const float* __restrict__ wts, int P, int E, int nt) {
  const int tid = threadIdx.x;
  if (tid < MOE_MAX_EXPERTS / 32) rt.bitmap[tid] = 0u;
  if (tid == 0) rt.invalid = 0;
  bar_sync_n(BAR, nt);
  for (int i = tid; i < P; i += nt) {
    const int id = ids[i];
    const bool ok = id >= 0 && id < E;
    rt.sid[i] = ok ? id : -1;
    rt.wt[i] = ok ? wts[i] : 0.0f;
    if (ok) atomicOr(&rt.bitmap[id >> 5], 1u << (id & 31));
    else atomicAdd(&rt.invalid, 1);
  }
  bar_sync_n(BAR, nt);
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
  bar_sync_n(BAR, nt);
  // stable counting sort of the valid pairs by expert: rank = #smaller experts
  // + #earlier pairs of the same expert
  for (int p = tid; p < P; p += nt) {
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
  bar_sync_n(BAR, nt);
}

// The same table built by one warp, for P <= 64 pairs (T <= 4 tokens): two
// pairs per lane, ranks by shuffles, slot boundaries by ballots. No CTA
// barrier; the caller synchronises before other warps read the table.
// (bitmap and word_off are not filled.)
__device__ __forceinline__ void build_route_table_warp(RouteTable& rt,
                                                       const int32_t* __restrict__ ids,
                                                       const float* __restrict__ wts, int P,
                                                       int E) {
  const int lane = threadIdx.x & 31;
  const int p1 = lane + 32;
  int e0 = -1, e1 = -1;
  if (lane < P) {
    const int id = ids[lane];
    e0 = id >= 0 && id < E ? id : -1;
    rt.sid[lane] = e0;
    rt.wt[lane] = e0 >= 0 ? wts[lane] : 0.0f;
  }
  if (p1 < P) {
    const int id = ids[p1];
    e1 = id >= 0 && id < E ? id : -1;
    rt.sid[p1] = e1;
    rt.wt[p1] = e1 >= 0 ? wts[p1] : 0.0f;
  }
  const int inv = __popc(__ballot_sync(0xFFFFFFFFu, lane < P && e0 < 0)) +
                  __popc(__ballot_sync(0xFFFFFFFFu, p1 < P && e1 < 0));
  // stable rank by (expert, pair index) among the valid pairs
  int r0 = 0, r1 = 0;
#pragma unroll 1
  for (int q = 0; q < P; ++q) {
    const int eq = __shfl_sync(0xFFFFFFFFu, q < 32 ? e0 : e1, q & 31);
    if (eq >= 0) {
      r0 += (eq < e0) || (eq == e0 && q < lane);
      r1 += (eq < e1) || (eq == e1 && q < p1);
    }
  }
  if (lane < P && e0 >= 0) rt.list[r0] = lane;
  if (p1 < P && e1 >= 0) rt.list[r1] = p1;
  __syncwarp();
  const int nv = P - inv;
  int es0 = -1, es1 = -1;
  bool f0 = false, f1 = false;
  if (lane < nv) {
    es0 = rt.sid[rt.list[lane]];
    f0 = lane == 0 || rt.sid[rt.list[lane - 1]] != es0;
  }
  if (p1 < nv) {
    es1 = rt.sid[rt.list[p1]];
    f1 = rt.sid[rt.list[p1 - 1]] != es1;
  }
  const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, f0);
  const uint32_t b1 = __ballot_sync(0xFFFFFFFFu, f1);
  const uint32_t below = (1u << lane) - 1u;
  if (f0) {
    const int sl = __popc(b0 & below);
    rt.slot_expert[sl] = es0;
    rt.slot_off[sl] = lane;
  }
  if (f1) {
    const int sl = __popc(b0) + __popc(b1 & below);
    rt.slot_expert[sl] = es1;
    rt.slot_off[sl] = p1;
  }
  if (lane == 0) {
    const int ns = __popc(b0) + __popc(b1);
    rt.n_slots = ns;
    rt.slot_off[ns] = nv;
    rt.n_valid = nv;
    rt.invalid = inv;
  }
  __syncwarp();
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
#ifdef __CUDA_ARCH__
  const int m = (K >> 6) < 8 ? (K >> 6) : 8;      // K is a multiple of 64
  return 1 << (31 - __clz(m));
#else
  int l = 8;
  while (l > K / 64) l >>= 1;
  return l;
#endif
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


// Four lanes per 32-value block: lane s = lane & 3 holds values 8s..8s+7 of
// block b. The largest exponent is combined over the four lanes by two
// shuffles; lanes 0 and 1 of the group write the pair words (value j with
// value j + 16, taken from lane s + 2), lane 0 the scale. All 32 lanes of the
// warp call it (ok = false: a lane without a block).
__device__ __forceinline__ void quant_group8(const float (&v)[8], bool ok, int b, int K,
                                             uint32_t* rec) {
  const int s = threadIdx.x & 3;
  uint32_t e = 0;
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
  if (ok && s < 2) {
    const int lpr = dlanes_per_row(K);
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

// Quantise T bf16 rows of K values (16-byte aligned) into records (shared or
// global memory), four lanes per 32-value block (16 bytes each); all threads
// tid, tid + nt, ... (nt a multiple of 32). Each thread has kXLoads loads in
// flight before it quantises any of them.
template <int kXLoads>
__device__ __forceinline__ void quant_x_lanes(const uint16_t* __restrict__ x, int T, int K,
                                              uint32_t* xq, int xq_words, int tid, int nt) {
  const int nb = K / 32;
  const int n = T * nb * 4;
#pragma unroll 1
  for (int i0 = tid & ~31; i0 < n; i0 += kXLoads * nt) {
    uint4 raw[kXLoads];
#pragma unroll
    for (int u = 0; u < kXLoads; ++u) {
      const int i = i0 + u * nt + (tid & 31);
      raw[u] = make_uint4(0, 0, 0, 0);
      if (i < n) {
        const int blk = i >> 2, t = blk / nb, b = blk - t * nb;
        raw[u] = __ldcg(reinterpret_cast<const uint4*>(x + (size_t)t * K + b * 32) + (i & 3));
      }
    }
#pragma unroll
    for (int u = 0; u < kXLoads; ++u) {
      if (i0 + u * nt < n) {                 // warp-uniform: i0 + u * nt is a multiple of 32
        const int i = i0 + u * nt + (tid & 31);
        const bool ok = i < n;
        const int blk = ok ? i >> 2 : 0;
        const int t = blk / nb, b = blk - t * nb;
        const uint32_t r[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
        float v[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[2 * j] = __uint_as_float(r[j] << 16);
          v[2 * j + 1] = __uint_as_float(r[j] & 0xFFFF0000u);
        }
        quant_group8(v, ok, b, K, xq + (size_t)t * xq_words);
      }
    }
  }
}

// The down rows of one expert, [0, nrows) of `wrows` (K inputs each), for its
// ntok tokens: rec_of(j) is token j's quantised h record, store(j, row, v) takes
// the row's dot product. Lanes split a row lpr ways (pairs q = q0, q0 + lpr,
// ..., accumulated in that order, then an xor butterfly); NPS tokens share each
// decoded block; LPR = lpr when known at compile time, else 0.
template <int NPS, int LPR, typename RecOf, typename Store>
__device__ __forceinline__ void down_rows(const uint8_t* wrows, int K, int nrows, int ntok,
                                          RecOf rec_of, Store store) {
  const int lane = threadIdx.x & 31;
  const int rbK = (K >> 5) * kBlockB;
  const int lpr = LPR ? LPR : dlanes_per_row(K);
  const int rpw = 32 / lpr;
  const int npq = K >> 6;
  const int pw = dqvec_pair_words(K);
  const int q0 = lane & (lpr - 1);
#pragma unroll 1
  for (int g0 = 0; g0 < ntok; g0 += NPS) {
    const int np = ntok - g0 < NPS ? ntok - g0 : NPS;
    const uint32_t* rp[NPS];
#pragma unroll
    for (int j = 0; j < NPS; ++j) rp[j] = rec_of(g0 + (j < np ? j : 0));
#pragma unroll 1
    for (int rb = 0; rb < nrows; rb += rpw) {
      const int rl = rb + lane / lpr;
      const bool active = rl < nrows;
      float acc[NPS];
#pragma unroll
      for (int j = 0; j < NPS; ++j) acc[j] = 0.0f;
      if (active) {
        const uint8_t* row = wrows + (size_t)rl * rbK;
        if (NPS == 1 || np == 1) {
          // one token: the split-table dot products (same integers as below)
          for (int q = q0; q < npq; q += lpr) {
            const int qbase = qv_base(q, lpr);
            uint32_t w[9];
            load_pair_smem(row + q * kPairB, w);
            float d0, d1;
            pair_scales(w, d0, d1);
            const uint4* r4 = reinterpret_cast<const uint4*>(rp[0]) + qbase;
            uint32_t v[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 t4 = r4[c * lpr];
              v[4 * c] = t4.x; v[4 * c + 1] = t4.y; v[4 * c + 2] = t4.z; v[4 * c + 3] = t4.w;
            }
            const float2 sc = reinterpret_cast<const float2*>(rp[0] + pw)[q];
            int i0, i1;
            iq4_pair_dot1(w, v, i0, i1);
            acc[0] = fmaf((float)i0, d0 * sc.x, acc[0]);
            acc[0] = fmaf((float)i1, d1 * sc.y, acc[0]);
          }
        } else {
        for (int q = q0; q < npq; q += lpr) {
          const int qbase = qv_base(q, lpr);
          uint32_t w[9];
          float d0, d1;
          uint32_t a0[4], a1[4];
          uint32_t t0[8], t1[8];
          load_pair_smem(row + q * kPairB, w);
          split_pair(w, d0, d1, a0, a1);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            iq4_lookup8(a0[i], t0[2 * i], t0[2 * i + 1]);
            iq4_lookup8(a1[i], t1[2 * i], t1[2 * i + 1]);
          }
#pragma unroll
          for (int j = 0; j < NPS; ++j) {
            if (j < np) {
              const uint4* r4 = reinterpret_cast<const uint4*>(rp[j]) + qbase;
              uint32_t v[32];
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const uint4 t4 = r4[c * lpr];
                v[4 * c] = t4.x; v[4 * c + 1] = t4.y; v[4 * c + 2] = t4.z; v[4 * c + 3] = t4.w;
              }
              const float2 sc = reinterpret_cast<const float2*>(rp[j] + pw)[q];
              const int i0 = iq4_dot_block(t0, v);
              const int i1 = iq4_dot_block(t1, v + 16);
              acc[j] = fmaf((float)i0, d0 * sc.x, acc[j]);
              acc[j] = fmaf((float)i1, d1 * sc.y, acc[j]);
            }
          }
        }
        }
      }
#pragma unroll
      for (int j = 0; j < NPS; ++j)
        if (j < np) {
#pragma unroll
          for (int o = (LPR ? LPR : 8) >> 1; o > 0; o >>= 1)
            if (LPR || o < lpr) acc[j] += __shfl_xor_sync(0xFFFFFFFFu, acc[j], o);
        }
      if (active && q0 == 0) {
#pragma unroll
        for (int j = 0; j < NPS; ++j)
          if (j < np) store(g0 + j, rl, acc[j]);
      }
    }
  }
}


// ---------------------------------------------------------------------------
// Gate/up work: shared-expert rows are split evenly over the CTAs (known before
// the routes are), routed rows (slots x F, slot-major) likewise after.
struct RowRange {
  int a, b;   // [a, b) in flattened rows
};

__device__ __forceinline__ RowRange split_rows(int total, int g, int cta, int ncta) {
  const int units = total / g;
  const long long ua = (long long)units * cta / ncta;
  const long long ub = (long long)units * (cta + 1) / ncta;
  return RowRange{(int)ua * g, (int)ub * g};
}

// One gate/up unit: the warp's f-row (gate row at `g`, up row at `u`) for every
// token of the slot; writes h (fp32) for each (token, slot) pair. LPR is the
// interleave width of the quantised x records (dlanes_per_row(H)); 0 = known
// only at run time.
template <int MAXT, int LPR>
__device__ __forceinline__ void gateup_unit_t(const DecodeParams& p, const RouteTable& rt,
                                           const uint8_t* g, const uint8_t* u, int slot, int f,
                                           const uint32_t* xq, int xq_words) {
  const int lane = threadIdx.x & 31;
  const int H = p.H;
  const int npairs = H >> 6;
  const int lpr = LPR ? LPR : dlanes_per_row(H);
  const bool shared = slot < 0;
  const int ntok = shared ? p.T : rt.slot_off[slot + 1] - rt.slot_off[slot];
  const int lbase = shared ? 0 : rt.slot_off[slot];
  const int xs_off = dqvec_pair_words(H);
#pragma unroll 1
  for (int g0 = 0; g0 < ntok; g0 += MAXT) {
    const int ng = ntok - g0 < MAXT ? ntok - g0 : MAXT;
    const uint32_t* rec[MAXT];
#pragma unroll
    for (int j = 0; j < MAXT; ++j) {
      const int jj = g0 + (j < ng ? j : 0);
      const int tok = shared ? jj : rt.list[lbase + jj] / p.k;
      rec[j] = xq + (size_t)tok * xq_words;
    }
    float ag[MAXT], au[MAXT];
#pragma unroll
    for (int j = 0; j < MAXT; ++j) ag[j] = au[j] = 0.0f;
    if (MAXT == 1 || ng == 1) {
      // one token: the split-table dot products (fewer ALU-pipe operations;
      // the same integers, so the same h as the general loop below)
      for (int q = lane; q < npairs; q += 32) {
        const int qbase = qv_base(q, lpr);
        uint32_t wg[9], wu[9];
        load_pair_smem(g + q * kPairB, wg);
        load_pair_smem(u + q * kPairB, wu);
        float dg0, dg1, du0, du1;
        pair_scales(wg, dg0, dg1);
        pair_scales(wu, du0, du1);
        const uint4* r4 = reinterpret_cast<const uint4*>(rec[0]) + qbase;
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 t4 = r4[c * lpr];
          v[4 * c] = t4.x; v[4 * c + 1] = t4.y; v[4 * c + 2] = t4.z; v[4 * c + 3] = t4.w;
        }
        const float2 sc = reinterpret_cast<const float2*>(rec[0] + xs_off)[q];
        int ig0, ig1, iu0, iu1;
        iq4_pair_dot1(wg, v, ig0, ig1);
        iq4_pair_dot1(wu, v, iu0, iu1);
        ag[0] = fmaf((float)ig0, dg0 * sc.x, ag[0]);
        ag[0] = fmaf((float)ig1, dg1 * sc.y, ag[0]);
        au[0] = fmaf((float)iu0, du0 * sc.x, au[0]);
        au[0] = fmaf((float)iu1, du1 * sc.y, au[0]);
      }
    } else {
    for (int q = lane; q < npairs; q += 32) {
      const int qbase = qv_base(q, lpr);
      uint32_t w[9];
      float dg0, dg1, du0, du1;
      uint32_t a0[4], a1[4];
      uint32_t tg0[8], tg1[8], tu0[8], tu1[8];
      load_pair_smem(g + q * kPairB, w);
      split_pair(w, dg0, dg1, a0, a1);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        iq4_lookup8(a0[i], tg0[2 * i], tg0[2 * i + 1]);
        iq4_lookup8(a1[i], tg1[2 * i], tg1[2 * i + 1]);
      }
      load_pair_smem(u + q * kPairB, w);
      split_pair(w, du0, du1, a0, a1);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        iq4_lookup8(a0[i], tu0[2 * i], tu0[2 * i + 1]);
        iq4_lookup8(a1[i], tu1[2 * i], tu1[2 * i + 1]);
      }
#pragma unroll
      for (int j = 0; j < MAXT; ++j) {
        if (j < ng) {
          const uint4* r4 = reinterpret_cast<const uint4*>(rec[j]) + qbase;
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 t4 = r4[c * lpr];
            v[4 * c] = t4.x; v[4 * c + 1] = t4.y; v[4 * c + 2] = t4.z; v[4 * c + 3] = t4.w;
          }
          const float2 sc = reinterpret_cast<const float2*>(rec[j] + xs_off)[q];
          const int ig0 = iq4_dot_block(tg0, v);
          const int ig1 = iq4_dot_block(tg1, v + 16);
          const int iu0 = iq4_dot_block(tu0, v);
          const int iu1 = iq4_dot_block(tu1, v + 16);
          ag[j] = fmaf((float)ig0, dg0 * sc.x, ag[j]);
          ag[j] = fmaf((float)ig1, dg1 * sc.y, ag[j]);
          au[j] = fmaf((float)iu0, du0 * sc.x, au[j]);
          au[j] = fmaf((float)iu1, du1 * sc.y, au[j]);
        }
      }
    }
    }
#pragma unroll
    for (int j = 0; j < MAXT; ++j) {
      if (j < ng) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ag[j] += __shfl_xor_sync(0xFFFFFFFFu, ag[j], o);
          au[j] += __shfl_xor_sync(0xFFFFFFFFu, au[j], o);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < MAXT; ++j) {
      if (j < ng && lane == j) {
        const float hv = silu_mul(ag[j], au[j]);
        if (shared) p.h_s[(size_t)(g0 + j) * p.Fs + f] = hv;
        else p.h_r[(size_t)rt.list[lbase + g0 + j] * p.F + f] = hv;
      }
    }
  }
}


// h rows of this call into records in shared memory, in the layout the down
// units read: the routed pairs' records (indexed by pair), then the shared
// expert's (by token). Four lanes per 32-value block. STAGED: the rows sit in
// shared memory in list order (the valid routed pairs as rt.list orders them,
// F values each, then the shared expert's rows, Fs values each); otherwise
// they are read from global memory through L2 (written by other CTAs).
// Two lanes per 32-value block: lane s = lane & 1 quantises values 8s..8s+7
// and 16+8s..16+8s+7, i.e. exactly the pair words 8s..8s+7 (value j with
// value j + 16); the block's largest exponent is combined by one shuffle.
__device__ __forceinline__ void quant_half_block(const float4 (&f)[4], bool ok, int b, int K,
                                                 uint32_t* rec) {
  const int s = threadIdx.x & 1;
  const float v[16] = {f[0].x, f[0].y, f[0].z, f[0].w, f[1].x, f[1].y, f[1].z, f[1].w,
                       f[2].x, f[2].y, f[2].z, f[2].w, f[3].x, f[3].y, f[3].z, f[3].w};
  uint32_t e = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t ei = (__float_as_uint(v[i]) >> 23) & 0xFFu;
    e = ei > e ? ei : e;
  }
  const uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, e, 1);
  e = o > e ? o : e;
  if (ok) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = (uint32_t)(quant_one(v[i], e) & 0xFFFF) | ((uint32_t)quant_one(v[8 + i], e) << 16);
    const int lpr = dlanes_per_row(K);
    const int q = b >> 1;
    const int c0 = 4 * (b & 1) + 2 * s;
    uint4* r4 = reinterpret_cast<uint4*>(rec);
    r4[qv_u4(q, c0, lpr)] = make_uint4(w[0], w[1], w[2], w[3]);
    r4[qv_u4(q, c0 + 1, lpr)] = make_uint4(w[4], w[5], w[6], w[7]);
    if (s == 0) reinterpret_cast<float*>(rec + dqvec_pair_words(K))[b] = quant_scale(e);
  }
}

// floor(n / d) for 0 <= n < 2^16 and 1 <= d < 2^16 with inv = ceil(2^32 / d).
__device__ __forceinline__ int div_by_inv(int n, uint32_t inv) {
  return (int)__umulhi((uint32_t)n, inv);
}

template <bool STAGED>
__device__ __forceinline__ void quant_h(const DecodeParams& p, const RouteTable& rt,
                                        const float* stage, uint32_t* recs, int tid, int nt) {
  const int nbF = p.F / 32;
  const int nbS = p.n_shared ? p.Fs / 32 : 1;
  const uint32_t invF = 0xFFFFFFFFu / (uint32_t)nbF + 1u;
  const uint32_t invS = 0xFFFFFFFFu / (uint32_t)nbS + 1u;
  const int wF = dqvec_words(p.F);
  const int wS = p.n_shared ? dqvec_words(p.Fs) : 0;
  uint32_t* rec_sh = recs + (size_t)p.T * p.k * wF;
  const int nr = rt.n_valid * nbF;
  const int total = nr + (p.n_shared ? p.T * nbS : 0);
#pragma unroll 1
  for (int i0 = tid & ~31; i0 < total * 2; i0 += nt) {
    const int i = i0 + (tid & 31);
    const bool ok = i < total * 2;
    const int blk = ok ? i >> 1 : 0;
    const int s = i & 1;
    uint32_t* dst;
    const float* row;
    int b, K;
    if (blk < nr) {
      const int e = div_by_inv(blk, invF);
      b = blk - e * nbF;
      K = p.F;
      dst = recs + (size_t)rt.list[e] * wF;
      row = p.h_r + (size_t)rt.list[e] * p.F;
    } else {
      const int j = div_by_inv(blk - nr, invS);
      b = (blk - nr) - j * nbS;
      K = p.Fs;
      dst = rec_sh + (size_t)j * wS;
      row = p.h_s + (size_t)j * p.Fs;
    }
    float4 f[4];
    const float* src = STAGED ? stage + (size_t)blk * 32 : row + b * 32;
    const float4* s4 = reinterpret_cast<const float4*>(src + 8 * s);
    if (STAGED) {
      f[0] = s4[0]; f[1] = s4[1]; f[2] = s4[4]; f[3] = s4[5];
    } else if (ok) {
      f[0] = __ldcg(s4); f[1] = __ldcg(s4 + 1); f[2] = __ldcg(s4 + 4); f[3] = __ldcg(s4 + 5);
    } else {
      f[0] = f[1] = f[2] = f[3] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    quant_half_block(f, ok, b, K, dst);
  }
}

// ---------------------------------------------------------------------------
// Pieces shared by the single-launch decode kernels.

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One down unit: rows [r0, r0 + nrows) (CTA-local indices) of the slot's W_d at
// `wrows`; for every pair of the slot, the row dot products into `part`.
// NPS pairs share each decoded block; LPR as for gate/up (0 = run time).
template <int NPS, int LPR>
__device__ __forceinline__ void down_unit_t(const DecodeParams& p, const RouteTable& rt,
                                         const uint8_t* wrows, int slot, int r0, int nrows,
                                         const uint32_t* recs, float* part, int rows_max) {
  const bool shared = slot < 0;
  const int K = shared ? p.Fs : p.F;
  const int words = dqvec_words(K);
  const int P = p.T * p.k;
  const int ntok = shared ? p.T : rt.slot_off[slot + 1] - rt.slot_off[slot];
  const int lbase = shared ? 0 : rt.slot_off[slot];
  const uint32_t* rec_sh = recs + (size_t)P * dqvec_words(p.F);
  auto pidx = [&](int jj) { return shared ? P + jj : rt.list[lbase + jj]; };
  down_rows<NPS, LPR>(
      wrows, K, nrows, ntok,
      [&](int jj) { return shared ? rec_sh + (size_t)jj * words : recs + (size_t)pidx(jj) * words; },
      [&](int jj, int rl, float v) { part[(size_t)pidx(jj) * rows_max + r0 + rl] = v; });
}

}  // namespace moe
