// Decode kernels of libmoe (sm_103a): gate/up + SwiGLU, then down + combine.
//
// Each distinct expert's IQ4_NL rows are streamed from HBM once per call by
// 1D bulk copies (TMA) into a shared-memory ring; each block is decoded once
// (a byte_perm table lookup to int8) and its exact integer dot product with
// every token routed to that expert is taken with dp2a against 16-bit block-
// quantised activations. This is the paired-token decode of the Red Lite page
// ("What we learned", section 4: decode each weight block once for both
// tokens, and merge the tokens' experts into one dispatch), for 1..16 tokens.
#include <cstdio>

#include "common.cuh"
#include "decode.cuh"
#include "decode_common.cuh"
#include "route.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Gate/up + SwiGLU for the shapes and token counts the fused kernel does not
// take. Every warp streams its own units as the fused kernel does (g
// consecutive f-rows of one expert per unit, g the rows that make a copy a
// multiple of 16 bytes; two bulk-copy slots per warp) and computes each row
// with the same per-row code, so every h value is bitwise the fused kernel's.
//
// Work goes to CTAs in whole 32-row blocks (the quantisation blocks of h), so
// each block of h is completed inside one CTA: a shared-memory counter per
// block collects the rows, and the warp that adds the last row quantises the
// block for every token of its expert into the records the down kernel reads.
// The shared expert's blocks go one each to the last CTAs (evenly, if there
// are more blocks than CTAs); the routed blocks (slot-major) are then split so
// that every CTA gets about the same compute, by the measured cost of a row
// for n tokens (gu_cost, in tenths of a one-token row).
constexpr int kGuSlots = 2;
constexpr int kGuMaxT = 4;        // tokens per pass over a row (more: several passes)

// Cost of a row with n tokens: one token 10 (its own code path); otherwise
// passes of up to 4 tokens, a full pass 24 and a last pass of 1, 2 or 3
// tokens 12, 18, 21 (rates of the unit code on the GPU).
__host__ __device__ inline int gu_cost(int n) {
  if (n <= 1) return 10;
  const int r = n & 3;
  return (n >> 2) * 24 + (r == 0 ? 0 : r == 1 ? 12 : r == 2 ? 18 : 21);
}

__host__ __device__ inline int gu_shared_cum(int S, int c, int G) {
  return S <= G ? (c > G - S ? c - (G - S) : 0) : S * c / G;
}
// Routed blocks of CTAs 0..c-1 (non-decreasing in c; all routed blocks at
// c = G). bps: blocks per slot. All 32 lanes of a warp call it and get the
// same value. 32-bit arithmetic suffices: the total cost is below 2^22 (at
// most 256 slots x 256 blocks x cost 12 per token) and G below 2^9.
__device__ __forceinline__ int gu_routed_cum(const RouteTable& rt, int bps, int S, int T, int c,
                                             int G) {
  const int lane = threadIdx.x & 31;
  const int ns = rt.n_slots;
  // slot costs: lane l sums slots 8l .. 8l+7; exclusive scan over lanes
  int mine = 0;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int sl = lane * 8 + m;
    if (sl < ns) mine += bps * gu_cost(rt.slot_off[sl + 1] - rt.slot_off[sl]);
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  const int rcost = __shfl_sync(0xFFFFFFFFu, incl, 31);
  const int ws = gu_cost(T);
  const int tot = S * ws + rcost;
  // the routed cost that CTAs 0..c-1 take, made non-decreasing
  int best = 0;
#pragma unroll 1
  for (int i = 1 + lane; i <= c; i += 32) {
    int v = tot * i / G - ws * gu_shared_cum(S, i, G);
    v = v > rcost ? rcost : v;
    best = v > best ? v : best;
  }
  const int X = (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)best);
  if (X >= rcost) return ns * bps;
  // the slot holding cost X, and the whole blocks of it below X
  int res = 0;
  const int start = incl - mine;
  const bool here = start <= X && X < incl;
  if (here) {
    int pc = start;
#pragma unroll 1
    for (int m = 0; m < 8; ++m) {
      const int sl = lane * 8 + m;
      const int cs = gu_cost(rt.slot_off[sl + 1] - rt.slot_off[sl]);
      if (X < pc + bps * cs) {
        res = sl * bps + (X - pc) / cs;
        break;
      }
      pc += bps * cs;
    }
  }
  const unsigned who = __ballot_sync(0xFFFFFFFFu, here);
  return __shfl_sync(0xFFFFFFFFu, res, __ffs(who) - 1);
}
// Most 32-row blocks any CTA can get (slots_max routed experts, P pairs): a
// CTA takes about tot / G of the cost, a routed block costs at least 10 and
// all of them at most 12 per pair, and the floors and the block granularity
// add a few.
inline int gu_blocks_max(int S, int bps, int slots_max, int P, int T, int G) {
  const int rmax = bps * (10 * slots_max > 12 * P ? 10 * slots_max : 12 * P);
  const int tot = S * gu_cost(T) + rmax;
  const int sh = S <= G ? (S > 0 ? 1 : 0) : (S + G - 1) / G;
  return tot / (10 * G) + 4 + gu_cost(T) / 10 + sh;
}

struct GuSmem {
  size_t xq, slots, bars, cnt, total, slot_bytes;
};
// xs: the quantised x records sit in shared memory; otherwise the kernel reads
// them from the workspace, where quant_x_kernel wrote them. nblk: the block
// counters a CTA needs.
__host__ __device__ inline GuSmem gu_smem(int H, int T, int nw, bool xs, int g, int nblk) {
  GuSmem m;
  m.slot_bytes = align_up_dev((size_t)2 * g * (H / 32) * kBlockB, 128);
  m.xq = align_up_dev(sizeof(RouteTable), 128);
  m.slots = align_up_dev(m.xq + (xs ? (size_t)T * dqvec_words(H) * 4 : 0), 128);
  m.bars = m.slots + (size_t)nw * kGuSlots * m.slot_bytes;
  m.cnt = m.bars + (size_t)nw * kGuSlots * 8;
  m.total = m.cnt + (size_t)nblk * 4;
  return m;
}

// x -> quantised records in the workspace.
__global__ void __launch_bounds__(256) quant_x_kernel(const __grid_constant__ DecodeParams p) {
  pdl_wait();
  pdl_trigger();
  quant_x_lanes(p.x, p.T, p.H, p.xrec, dqvec_words(p.H), blockIdx.x * blockDim.x + threadIdx.x,
                gridDim.x * blockDim.x);
}

// Block fb (32 h values) of a slot -> its records, for every token of the slot
// (one warp; the values were written by warps of this CTA).
__device__ __noinline__ void quant_h_block(const DecodeParams& p, const RouteTable& rt, int slot,
                                           int fb) {
  const int lane = threadIdx.x & 31;
  const bool shared = slot < 0;
  const int F = shared ? p.Fs : p.F;
  const int words = dqvec_words(F);
  const int ntok = shared ? p.T : rt.slot_off[slot + 1] - rt.slot_off[slot];
  const int lbase = shared ? 0 : rt.slot_off[slot];
  constexpr int kBatch = 8;      // loads in flight before the first reduction
#pragma unroll 1
  for (int j0 = 0; j0 < ntok; j0 += kBatch) {
    float v[kBatch];
    uint32_t* dst[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = j0 + u < ntok ? j0 + u : j0;
      const int pr = shared ? j : rt.list[lbase + j];
      const float* src = shared ? p.h_s + (size_t)j * p.Fs : p.h_r + (size_t)pr * p.F;
      dst[u] = shared ? p.rec_s + (size_t)j * words : p.rec_r + (size_t)pr * words;
      v[u] = src[fb * 32 + lane];
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (j0 + u < ntok) quant_block_store(v[u], fb, F, dst[u]);
  }
}

template <int LPR, bool XS>
__global__ void __launch_bounds__(512, 1) gu_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = p.H;
  const int nw = blockDim.x >> 5;
  const int g = row_granule_dev(H);
  const GuSmem L = gu_smem(H, p.T, nw, XS, g, p.gu_nblk);
  RouteTable& rt = *reinterpret_cast<RouteTable*>(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int xq_words = dqvec_words(H);
  const size_t rbH = (size_t)(H / 32) * kBlockB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint32_t* bcnt = reinterpret_cast<uint32_t*>(smem + L.cnt);
  uint8_t* myslots = smem + L.slots + (size_t)warp * kGuSlots * L.slot_bytes;
  uint64_t* mybar = bars + warp * kGuSlots;

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int i = 0; i < nw * kGuSlots; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
  }
#pragma unroll 1
  for (int i = threadIdx.x; i < p.gu_nblk; i += blockDim.x) bcnt[i] = 0u;
  __syncthreads();

  // this CTA's blocks: shared [sb0, sb1) of the shared expert, then routed
  // [rb0, rb1) of the slot-major routed rows; its units (g rows each) are
  // numbered in that order and dealt round-robin to the warps
  const int G = gridDim.x, c = blockIdx.x;
  const int S = p.n_shared ? p.Fs / 32 : 0;
  const int sb0 = gu_shared_cum(S, c, G), sb1 = gu_shared_cum(S, c + 1, G);
  const int upb = 32 / g;                      // units per block
  const int n_sh_u = (sb1 - sb0) * upb;
  int rb0 = 0, n_u = n_sh_u;
  auto count = [&](int nu) { return warp < nu ? (nu - warp + nw - 1) / nw : 0; };
  const int n_sh = count(n_sh_u);
  int n_tot = n_sh;
  int issued = 0, consumed = 0;
  bool ok = true;
  const uint64_t pol = l2_evict_first_policy();   // weights: read once per call
  // a warp's units, in order: u = warp, warp + nw, ... of the CTA's units;
  // slot (-1 shared) and first f-row, kept up to date without divisions
  const int lg_upb = 5 - (31 - __clz(g));        // log2 of the units per block
  struct Cursor {
    int u, sl, f;
  };
  auto cur_get = [&](Cursor& k, int& sl, int& f) {
    if (k.u < n_sh_u) {
      sl = -1;
      f = sb0 * 32 + k.u * g;
      return;
    }
    if (k.sl < 0) {
      const int r = rb0 * 32 + (k.u - n_sh_u) * g;
      k.sl = r / p.F;
      k.f = r - k.sl * p.F;
    }
    sl = k.sl;
    f = k.f;
  };
  auto cur_next = [&](Cursor& k) {
    if (k.sl >= 0) {
      k.f += nw * g;
      while (k.f >= p.F) {
        k.f -= p.F;
        ++k.sl;
      }
    }
    k.u += nw;
  };
  Cursor ci{warp, -1, 0}, cc{warp, -1, 0};        // next unit to issue, to compute
  const uint32_t ubytes = (uint32_t)(g * rbH);     // a multiple of 16
  auto issue_upto = [&](int limit) {
    while (issued < limit && issued - consumed < kGuSlots) {
      int sl, f;
      cur_get(ci, sl, f);
      if (lane == 0) {
        const size_t row = sl < 0 ? (size_t)f : (size_t)rt.slot_expert[sl] * p.F + f;
        const int s = issued % kGuSlots;
        uint8_t* dst = myslots + (size_t)s * L.slot_bytes;
        mbar_arrive_expect_tx(&mybar[s], 2 * ubytes);
        bulk_g2s_hint(dst, (sl < 0 ? p.sh_gate : p.gate) + row * rbH, ubytes, &mybar[s], pol);
        bulk_g2s_hint(dst + ubytes, (sl < 0 ? p.sh_up : p.up) + row * rbH, ubytes, &mybar[s],
                      pol);
      }
      cur_next(ci);
      ++issued;
    }
  };

  issue_upto(n_sh);
  pdl_wait();
  pdl_trigger();
  uint32_t* xq = XS ? reinterpret_cast<uint32_t*>(smem + L.xq) : p.xrec;
  if (XS) quant_x_lanes(p.x, p.T, H, xq, xq_words, threadIdx.x, blockDim.x);
  if (p.T * p.k <= 64) {
    if (warp == 0) build_route_table_warp(rt, p.ids, p.weights, p.T * p.k, p.E);
    __syncthreads();
  } else {
    build_route_table<0>(rt, p.ids, p.weights, p.T * p.k, p.E, blockDim.x);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.status && rt.invalid)
    atomicAdd(p.status, (uint32_t)(rt.invalid < 0xFFFF ? rt.invalid : 0xFFFF));
  int rb1 = 0;
  {
    rb0 = gu_routed_cum(rt, p.F / 32, S, p.T, c, G);
    rb1 = gu_routed_cum(rt, p.F / 32, S, p.T, c + 1, G);
    // never more blocks than the counters the launch provided (only a route
    // table the host bound did not foresee could ask for more)
    if (rb1 - rb0 + (sb1 - sb0) > p.gu_nblk) {
      rb1 = rb0 + (p.gu_nblk - (sb1 - sb0));
      if (blockIdx.x == 0 && threadIdx.x == 0 && p.status) atomicOr(p.status, MOE_STATUS_TIMEOUT);
    }
    n_u = n_sh_u + (rb1 - rb0) * upb;
  }
  n_tot = count(n_u);
  issue_upto(n_tot);

#pragma unroll 1
  for (int j = 0; ok && j < n_tot; ++j) {
    ok = mbar_wait(&mybar[j % kGuSlots], (uint32_t)((j / kGuSlots) & 1), p.status);
    if (!ok) break;
    const uint8_t* d = myslots + (size_t)(j % kGuSlots) * L.slot_bytes;
    int sl, f;
    cur_get(cc, sl, f);
    const int blk = cc.u >> lg_upb;
    cur_next(cc);
    // one-token experts (most of them) take the code built for one token
    const int ntok = sl < 0 ? p.T : rt.slot_off[sl + 1] - rt.slot_off[sl];
#pragma unroll 1
    for (int i = 0; i < g; ++i) {
      if (ntok == 1)
        gateup_unit_t<1, LPR>(p, rt, d + i * rbH, d + (g + i) * rbH, sl, f + i, xq, xq_words);
      else
        gateup_unit_t<kGuMaxT, LPR>(p, rt, d + i * rbH, d + (g + i) * rbH, sl, f + i, xq,
                                    xq_words);
    }
    __syncwarp();
    ++consumed;
    issue_upto(n_tot);
    // this warp's h stores, then its rows' arrival on the block
    __threadfence_block();
    __syncwarp();
    if (lane == 0) atomicAdd(&bcnt[blk], (uint32_t)g);
  }
  // after a timeout: no bulk copy of this warp stays in flight
  while (consumed < issued) {
    mbar_wait(&mybar[consumed % kGuSlots], (uint32_t)((consumed / kGuSlots) & 1), p.status);
    ++consumed;
  }
  // Quantise the CTA's blocks of h, block b by warp b % nw once all 32 of its
  // rows have arrived (spread evenly: the warp that happens to add the last
  // row would otherwise collect most of them and fall behind).
  const int nsb = sb1 - sb0, nb = nsb + (rb1 - rb0);
  const int bps = p.F / 32;
#pragma unroll 1
  for (int b = warp; ok && b < nb; b += nw) {
    ok = wait_count_cta(&bcnt[b], 32u, p.status);
    if (!ok) break;
    if (b < nsb) {
      quant_h_block(p, rt, -1, sb0 + b);
    } else {
      const int rb = rb0 + b - nsb;
      const int sl = rb / bps;
      quant_h_block(p, rt, sl, rb - sl * bps);
    }
  }
}

struct DnSmem {
  size_t yacc, bar, ring, stage, total;
};
__host__ __device__ inline DnSmem dn_smem(int F, int Fs, int n_shared, int T, int rows_max,
                                          int nst) {
  DnSmem m;
  m.yacc = align_up_dev(sizeof(RouteTable), 16);
  m.bar = align_up_dev(m.yacc + (size_t)rows_max * T * 4, 16);
  m.ring = align_up_dev(m.bar + (size_t)16 * nst, 128);
  size_t rb = (size_t)(F / 32) * kBlockB;
  size_t rec = (size_t)dqvec_words(F) * 4;
  if (n_shared) {
    const size_t rbs = (size_t)(Fs / 32) * kBlockB;
    const size_t recs = (size_t)dqvec_words(Fs) * 4;
    rb = rb > rbs ? rb : rbs;
    rec = rec > recs ? rec : recs;
  }
  m.stage = align_up_dev(align_up_dev((size_t)rows_max * rb, 16) + kPairsPerStage * rec, 128);
  m.total = m.ring + (size_t)nst * m.stage;
  return m;
}

// ---------------------------------------------------------------------------
// Down + combine. Each CTA owns output rows [n0, n1) and walks the stages:
// the shared expert (if any) first, then the routed experts in ascending id;
// each stage holds those rows of one expert's W_d and the quantised h of up
// to kPairsPerStage of its (token, slot) pairs.
struct StageIt {
  int slot;  // -1 = shared expert
  int g0;
};

__device__ __forceinline__ int stage_ntok(const DecodeParams& p, const RouteTable& rt, int slot) {
  return slot < 0 ? p.T : rt.slot_off[slot + 1] - rt.slot_off[slot];
}
__device__ __forceinline__ StageIt stage_first(const DecodeParams& p, const RouteTable& rt) {
  if (p.n_shared && p.T > 0) return StageIt{-1, 0};
  return StageIt{0, 0};
}
__device__ __forceinline__ bool stage_done(const RouteTable& rt, const StageIt& s) {
  return s.slot >= rt.n_slots;
}
__device__ __forceinline__ void stage_next(const DecodeParams& p, const RouteTable& rt,
                                           StageIt& s) {
  s.g0 += kPairsPerStage;
  if (s.g0 >= stage_ntok(p, rt, s.slot)) {
    s.slot += 1;
    s.g0 = 0;
  }
}

template <int NPS>
__global__ void __launch_bounds__(kThreads, 2) down_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = p.H;
  const int NST = p.dn_stages;
  const DnSmem L = dn_smem(p.F, p.Fs, p.n_shared, p.T, p.dn_rows_max, NST);
  RouteTable& rt = *reinterpret_cast<RouteTable*>(smem);
  float* yacc = reinterpret_cast<float*>(smem + L.yacc);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* empty = full + NST;
  uint8_t* ring = smem + L.ring;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int gd = row_granule_dev(p.F);
  if (p.n_shared && row_granule_dev(p.Fs) > gd) gd = row_granule_dev(p.Fs);
  const RowRange rows = split_rows(H, gd, blockIdx.x, gridDim.x);
  const int n0 = rows.a;
  const int nrows = rows.b - rows.a;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    all_sync_named();  // route table ready (ids come from the router, already complete)
    if (lane == 0) {
      auto desc = [&](const StageIt& si, const uint8_t*& wsrc, uint32_t& wbytes, int& np,
                      uint32_t& rbytes) {
        const bool sh = si.slot < 0;
        const int K = sh ? p.Fs : p.F;
        const int rbK = K / 32 * kBlockB;
        const int64_t erow = sh ? 0 : (int64_t)rt.slot_expert[si.slot] * H;
        wsrc = (sh ? p.sh_down : p.down) + (erow + n0) * rbK;
        wbytes = (uint32_t)(nrows * rbK);
        const int nt = stage_ntok(p, rt, si.slot) - si.g0;
        np = nt < NPS ? nt : NPS;
        rbytes = (uint32_t)dqvec_words(K) * 4;
      };
      auto issue_recs = [&](const StageIt& si, int s) {
        const uint8_t* wsrc;
        uint32_t wbytes, rbytes;
        int np;
        desc(si, wsrc, wbytes, np, rbytes);
        uint8_t* dst = ring + (size_t)s * L.stage + wbytes;
        for (int j = 0; j < np; ++j) {
          const uint32_t* src;
          if (si.slot < 0) src = p.rec_s + (size_t)(si.g0 + j) * (rbytes / 4);
          else src = p.rec_r + (size_t)rt.list[rt.slot_off[si.slot] + si.g0 + j] * (rbytes / 4);
          bulk_g2s(dst + (size_t)j * rbytes, src, rbytes, &full[s]);
        }
      };
      const uint64_t pol = l2_evict_first_policy();   // weights: read once per call
      int it = 0;
      bool waited = false;
      StageIt si = stage_first(p, rt);
      while (!stage_done(rt, si)) {
        const int s = it % NST;
        const uint32_t par = ((it / NST) & 1) ^ 1;
        if (!mbar_wait(&empty[s], par, p.status)) break;
        const uint8_t* wsrc;
        uint32_t wbytes, rbytes;
        int np;
        desc(si, wsrc, wbytes, np, rbytes);
        mbar_arrive_expect_tx(&full[s], wbytes + np * rbytes);
        if (wbytes) bulk_g2s_hint(ring + (size_t)s * L.stage, wsrc, wbytes, &full[s], pol);
        if (waited) issue_recs(si, s);
        ++it;
        stage_next(p, rt, si);
        if (!waited && (it == NST || stage_done(rt, si))) {
          // the quantised h comes from the gate/up kernel: wait for it
          pdl_wait();
          waited = true;
          StageIt sj = stage_first(p, rt);
          for (int j = 0; j < it; ++j) {
            issue_recs(sj, j);
            stage_next(p, rt, sj);
          }
        }
      }
    }
    __syncwarp();
    pdl_wait();
    pdl_trigger();
    return;
  }

  // Consumers.
  build_route_table<1>(rt, p.ids, p.weights, p.T * p.k, p.E, kConsumers);
  for (int i = threadIdx.x; i < nrows * p.T; i += kConsumers) yacc[i] = 0.0f;
  consumers_sync();
  all_sync_named();
  pdl_wait();
  pdl_trigger();

  int it = 0;
  for (StageIt si = stage_first(p, rt); !stage_done(rt, si); stage_next(p, rt, si), ++it) {
    const int s = it % NST;
    if (!mbar_wait(&full[s], (it / NST) & 1, p.status)) break;
    const bool sh = si.slot < 0;
    const int K = sh ? p.Fs : p.F;
    const int rbK = K / 32 * kBlockB;
    const int lpr = dlanes_per_row(K);
    const int rpw = 32 / lpr;
    const int npq = K / 64;
    const int words = dqvec_words(K);
    const int pw = dqvec_pair_words(K);
    const int nt = stage_ntok(p, rt, si.slot) - si.g0;
    const int np = nt < NPS ? nt : NPS;
    const uint8_t* wst = ring + (size_t)s * L.stage;
    const uint32_t* recs = reinterpret_cast<const uint32_t*>(wst + (size_t)nrows * rbK);
    int tok[NPS];
    float wgt[NPS];
#pragma unroll
    for (int j = 0; j < NPS; ++j) {
      const int jj = si.g0 + (j < np ? j : 0);
      if (sh) {
        tok[j] = jj;
        wgt[j] = 1.0f;
      } else {
        const int pr = rt.list[rt.slot_off[si.slot] + jj];
        tok[j] = pr / p.k;
        wgt[j] = rt.wt[pr];
      }
    }
    const int q0 = lane % lpr;
    for (int rbase = warp * rpw; rbase < nrows; rbase += (kConsumers / 32) * rpw) {
      const int r = rbase + lane / lpr;
      const bool active = r < nrows;
      float acc[NPS];
#pragma unroll
      for (int j = 0; j < NPS; ++j) acc[j] = 0.0f;
      if (active && np == 1) {
        // one token: the split-table dot products (same integers as below)
        const uint8_t* row = wst + (size_t)r * rbK;
        const float* sc = reinterpret_cast<const float*>(recs + pw);
#pragma unroll 1
        for (int q = q0; q < npq; q += lpr) {
          const int qbase = qv_base(q, lpr);
          uint32_t w[9];
          load_pair_smem(row + q * kPairB, w);
          float d0, d1;
          pair_scales(w, d0, d1);
          const uint4* r4 = reinterpret_cast<const uint4*>(recs) + qbase;
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 u = r4[c * lpr];
            v[4 * c] = u.x; v[4 * c + 1] = u.y; v[4 * c + 2] = u.z; v[4 * c + 3] = u.w;
          }
          int i0, i1;
          iq4_pair_dot1(w, v, i0, i1);
          acc[0] = fmaf((float)i0, d0 * sc[2 * q], acc[0]);
          acc[0] = fmaf((float)i1, d1 * sc[2 * q + 1], acc[0]);
        }
      } else if (active) {
        const uint8_t* row = wst + (size_t)r * rbK;
#pragma unroll 1
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
              const uint32_t* rec = recs + (size_t)j * words;
              const uint4* r4 = reinterpret_cast<const uint4*>(rec) + qbase;
              uint32_t v[32];
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const uint4 u = r4[c * lpr];
                v[4 * c] = u.x; v[4 * c + 1] = u.y; v[4 * c + 2] = u.z; v[4 * c + 3] = u.w;
              }
              const float* sc = reinterpret_cast<const float*>(rec + pw);
              const int i0 = iq4_dot_block(t0, v);
              const int i1 = iq4_dot_block(t1, v + 16);
              acc[j] = fmaf((float)i0, d0 * sc[2 * q], acc[j]);
              acc[j] = fmaf((float)i1, d1 * sc[2 * q + 1], acc[j]);
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NPS; ++j)
        if (j < np)
          for (int o = lpr >> 1; o > 0; o >>= 1) acc[j] += __shfl_xor_sync(0xFFFFFFFFu, acc[j], o);
      if (active && q0 == 0) {
#pragma unroll
        for (int j = 0; j < NPS; ++j)
          if (j < np) yacc[r * p.T + tok[j]] += wgt[j] * acc[j];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  consumers_sync();
  for (int i = threadIdx.x; i < nrows * p.T; i += kConsumers) {
    const int t = i / nrows, r = i - t * nrows;
    p.y[(size_t)t * H + n0 + r] = yacc[r * p.T + t];
  }
}

// ---------------------------------------------------------------------------
// Host side.
namespace {
constexpr size_t kSmemMax = 227 * 1024;

template <typename K>
cudaError_t launch(K kernel, int grid, int threads, size_t smem, bool pdl, cudaStream_t stream,
                   const DecodeParams& p) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Warps per CTA and where x lives for the gate/up kernel: 16 warps, with x in
// shared memory if it fits beside their slots, else in the workspace; 8 or 4
// warps when even that does not fit.
bool gu_config(const DecodeParams& p, int num_sms, int* nw, bool* xs, size_t* smem,
               int* nblk) {
  const int g = row_granule_dev(p.H);
  const int slots_max = p.T * p.k < p.E ? p.T * p.k : p.E;
  *nblk = gu_blocks_max(p.n_shared ? p.Fs / 32 : 0, p.F / 32, slots_max, p.T * p.k, p.T, num_sms);
  const int ws[3] = {16, 8, 4};
  for (int i = 0; i < 3; ++i) {
    for (int pass = 0; pass < 2; ++pass) {
      const bool x_on_chip = pass == 0;
      const size_t t = gu_smem(p.H, p.T, ws[i], x_on_chip, g, *nblk).total;
      if (t <= kSmemMax) {
        *nw = ws[i];
        *xs = x_on_chip;
        *smem = t;
        return true;
      }
    }
  }
  return false;
}

int down_stages(const DnSmem& one, int lo, int hi) {
  int n = hi;
  while (n > lo && one.ring + (size_t)n * one.stage > kSmemMax) --n;
  return n;
}
}  // namespace

int decode_launches(const DecodeParams& p, int num_sms) {
  size_t fsm = 0;
  int rg = 0, rmax = 0;
  if (fused_decode_supported(p, num_sms, &fsm, &rg, &rmax)) return 1;
  int nw = 0, nblk = 0;
  bool xs = true;
  size_t sm = 0;
  if (!gu_config(p, num_sms, &nw, &xs, &sm, &nblk)) return 2;
  return xs ? 2 : 3;
}

cudaError_t launch_decode(const DecodeParams& p0, int num_sms, bool pdl, cudaStream_t stream) {
  DecodeParams p = p0;
  p.route = 0;
  {
    size_t fsm = 0;
    int rg = 0, rmax = 0;
    if (fused_decode_supported(p, num_sms, &fsm, &rg, &rmax)) {
      p.fz_rg = rg;
      p.dn_rows_max = rmax;
      return launch_decode_fused(p, num_sms, fsm, pdl, stream);
    }
  }
  // gate/up
  int nw = 0;
  bool xs = true;
  size_t gsm = 0;
  if (!gu_config(p, num_sms, &nw, &xs, &gsm, &p.gu_nblk)) return cudaErrorInvalidConfiguration;
  // down
  int gd = row_granule_dev(p.F);
  if (p.n_shared && row_granule_dev(p.Fs) > gd) gd = row_granule_dev(p.Fs);
  const int units = p.H / gd;
  const int grid_dn = units < num_sms ? units : num_sms;
  p.dn_rows_max = (units + grid_dn - 1) / grid_dn * gd;
  const DnSmem d1 = dn_smem(p.F, p.Fs, p.n_shared, p.T, p.dn_rows_max, 1);
  p.dn_stages = down_stages(d1, 1, 8);
  const size_t dsm = dn_smem(p.F, p.Fs, p.n_shared, p.T, p.dn_rows_max, p.dn_stages).total;
  if (dsm > kSmemMax) return cudaErrorInvalidConfiguration;

  cudaError_t e;
  const bool w8 = dlanes_per_row(p.H) == 8;
  if (!xs) {
    const int n = p.T * (p.H / 32) * 4;             // four threads per 32-value block
    int grid = (n + 255) / 256;
    if (grid > num_sms) grid = num_sms;
    e = launch(quant_x_kernel, grid, 256, 0, pdl, stream, p);
    if (e != cudaSuccess) return e;
  }
  if (w8) e = xs ? launch(gu_kernel<8, true>, num_sms, nw * 32, gsm, pdl, stream, p)
                 : launch(gu_kernel<8, false>, num_sms, nw * 32, gsm, pdl, stream, p);
  else e = xs ? launch(gu_kernel<0, true>, num_sms, nw * 32, gsm, pdl, stream, p)
              : launch(gu_kernel<0, false>, num_sms, nw * 32, gsm, pdl, stream, p);
  if (e != cudaSuccess) return e;
  return launch(down_kernel<kPairsPerStage>, grid_dn, kThreads, dsm, pdl, stream, p);
}

// Route + layer in one call: one fused launch when the shape allows, else the
// router kernel followed by the decode kernels.
cudaError_t launch_decode_routed(const DecodeParams& p0, int num_sms, bool pdl,
                                 cudaStream_t stream) {
  DecodeParams p = p0;
  p.route = 1;
  size_t fsm = 0;
  int rg = 0, rmax = 0;
  if (fused_decode_supported(p, num_sms, &fsm, &rg, &rmax)) {
    p.fz_rg = rg;
    p.dn_rows_max = rmax;
    return launch_decode_fused(p, num_sms, fsm, pdl, stream);
  }
  RouteParams rp{p.H, p.E, p.k, p.T, p.Wr, p.bias, p.x, p.ids_out, p.w_out};
  cudaError_t e = launch_route(rp, pdl, stream);
  if (e != cudaSuccess) return e;
  p.route = 0;
  p.ids = p.ids_out;
  p.weights = p.w_out;
  return launch_decode(p, num_sms, pdl, stream);
}

}  // namespace moe
