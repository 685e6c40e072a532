// Decode kernels of libmoe (sm_103a) for the batches and shapes the fused
// kernel does not take: gate/up + SwiGLU, then down, then the combine.
//
// Each distinct expert's IQ4_NL rows are streamed from HBM once per call by
// 1D bulk copies (TMA) into per-warp shared-memory slots; each block is
// decoded once (prmt table lookups to int8) and its exact integer dot product
// with every token routed to that expert is taken with dp2a against 16-bit
// block-quantised activations. This is the paired-token decode of the Red
// Lite page ("What we learned", section 4: decode each weight block once for
// both tokens, and merge the tokens' experts into one dispatch), for 1..16
// tokens.
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

// The gate/up and down kernels run nw warps per CTA: nw - 1 compute, and the
// last one issues every weight copy. A bulk copy is taken in by the copy
// engine no faster than memory delivers, so the issuing thread stalls
// meanwhile; with each computing warp issuing its own rows, that took about as
// many cycles as its dot products. Lane w of the copy warp keeps computing
// warp w's slots filled in the warp's unit order, each slot once the warp has
// released its previous unit (an mbarrier arrival).
struct CopyWarpSmem {
  size_t ebars, stop, iss;      // slot-free barriers, stop flag, units issued per warp
};
__host__ __device__ inline size_t copy_warp_smem(size_t at, int nc, CopyWarpSmem& c) {
  c.ebars = align_up_dev(at, 8);
  c.stop = c.ebars + (size_t)nc * kGuSlots * 8;
  c.iss = c.stop + 4;
  return align_up_dev(c.iss + (size_t)nc * 4, 16);
}

struct GuSmem {
  size_t xq, slots, bars, cnt, total, slot_bytes;
  CopyWarpSmem cw;
};
// xs: the quantised x records sit in shared memory; otherwise the kernel reads
// them from the workspace, where quant_x_kernel wrote them. nblk: the block
// counters a CTA needs.
__host__ __device__ inline GuSmem gu_smem(int H, int T, int nw, bool xs, int g, int nblk) {
  GuSmem m;
  const int nc = nw - 1;
  m.slot_bytes = align_up_dev((size_t)2 * g * (H / 32) * kBlockB, 128);
  m.xq = align_up_dev(sizeof(RouteTable), 128);
  m.slots = align_up_dev(m.xq + (xs ? (size_t)T * dqvec_words(H) * 4 : 0), 128);
  m.bars = m.slots + (size_t)nc * kGuSlots * m.slot_bytes;
  m.cnt = copy_warp_smem(m.bars + (size_t)nc * kGuSlots * 8, nc, m.cw);
  m.total = m.cnt + (size_t)nblk * 4;
  return m;
}

// x -> quantised records in the workspace.
__global__ void __launch_bounds__(256) quant_x_kernel(const __grid_constant__ DecodeParams p) {
  pdl_wait();
  pdl_trigger();
  quant_x_lanes<4>(p.x, p.T, p.H, p.xrec, dqvec_words(p.H), blockIdx.x * blockDim.x + threadIdx.x,
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
  const int nw = (blockDim.x >> 5) - 1;          // computing warps; warp nw issues the copies
  const int g = row_granule_dev(H);
  const GuSmem L = gu_smem(H, p.T, nw + 1, XS, g, p.gu_nblk);
  RouteTable& rt = *reinterpret_cast<RouteTable*>(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool copier = warp == nw;
  const int xq_words = dqvec_words(H);
  const size_t rbH = (size_t)(H / 32) * kBlockB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* ebars = reinterpret_cast<uint64_t*>(smem + L.cw.ebars);
  volatile uint32_t* stop = reinterpret_cast<uint32_t*>(smem + L.cw.stop);
  volatile uint32_t* final_iss = reinterpret_cast<uint32_t*>(smem + L.cw.iss);
  uint32_t* bcnt = reinterpret_cast<uint32_t*>(smem + L.cnt);
  // the warp whose slots this thread fills (copy warp lane w) or computes
  const int ww = copier ? (lane < nw ? lane : 0) : warp;
  uint8_t* myslots = smem + L.slots + (size_t)ww * kGuSlots * L.slot_bytes;
  uint64_t* mybar = bars + ww * kGuSlots;

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int i = 0; i < nw * kGuSlots; ++i) {
      mbar_init(&bars[i], 1);
      mbar_init(&ebars[i], 1);
    }
    mbar_fence_init();
    *stop = 0u;
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
  auto count = [&](int nu) { return ww < nu ? (nu - ww + nw - 1) / nw : 0; };
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
  Cursor ci{ww, -1, 0}, cc{ww, -1, 0};            // next unit to issue, to compute
  const uint32_t ubytes = (uint32_t)(g * rbH);     // a multiple of 16
  // the copy warp: lane w < nw issues warp w's next units, up to `limit`, each
  // once its slot is free; true if it issued any
  auto issue_upto = [&](int limit) {
    bool any = false;
#pragma unroll 1
    for (;;) {
      bool can = lane < nw && issued < limit;
      if (can && issued >= kGuSlots)
        can = mbar_test(&ebars[ww * kGuSlots + issued % kGuSlots],
                        (uint32_t)(((issued / kGuSlots) + 1) & 1));
      if (!__any_sync(0xFFFFFFFFu, can)) break;
      if (can) {
        int sl, f;
        cur_get(ci, sl, f);
        const size_t row = sl < 0 ? (size_t)f : (size_t)rt.slot_expert[sl] * p.F + f;
        const int s = issued % kGuSlots;
        uint8_t* dst = myslots + (size_t)s * L.slot_bytes;
        mbar_arrive_expect_tx(&mybar[s], 2 * ubytes);
        bulk_g2s_hint(dst, (sl < 0 ? p.sh_gate : p.gate) + row * rbH, ubytes, &mybar[s], pol);
        bulk_g2s_hint(dst + ubytes, (sl < 0 ? p.sh_up : p.up) + row * rbH, ubytes, &mybar[s],
                      pol);
        cur_next(ci);
        ++issued;
      }
      any = true;
    }
    return any;
  };

  if (copier) issue_upto(n_sh < kGuSlots ? n_sh : kGuSlots);
  pdl_wait();
  pdl_trigger();
  uint32_t* xq = XS ? reinterpret_cast<uint32_t*>(smem + L.xq) : p.xrec;
  if (XS) quant_x_lanes<4>(p.x, p.T, H, xq, xq_words, threadIdx.x, blockDim.x);
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
  if (copier) {
    // every unit of every computing warp, as slots free up; a stop from the
    // computing warps (a failed wait) or a long idle spell ends it early
    const bool mine = lane < nw;
    uint64_t t_act = global_timer_ns();
#pragma unroll 1
    while (!__all_sync(0xFFFFFFFFu, !mine || issued >= n_tot) && !*stop) {
      const uint64_t now = global_timer_ns();
      if (issue_upto(n_tot)) {
        t_act = now;
      } else {
        if (now - t_act > 2 * kWaitLimitNs) {
          if (lane == 0 && p.status) atomicOr(p.status, MOE_STATUS_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    if (mine) final_iss[lane] = (uint32_t)issued;
    __syncthreads();     // the computing warps' final barrier
    return;
  }

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
    if (lane == 0) mbar_arrive(&ebars[warp * kGuSlots + j % kGuSlots]);   // slot free
    ++consumed;
    // this warp's h stores, then its rows' arrival on the block
    __threadfence_block();
    __syncwarp();
    if (lane == 0) atomicAdd(&bcnt[blk], (uint32_t)g);
  }
  if (!ok && lane == 0) *stop = 1u;
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
  // after a timeout: no bulk copy of this warp stays in flight
  __syncthreads();
  while (consumed < (int)final_iss[warp]) {
    mbar_wait(&mybar[consumed % kGuSlots], (uint32_t)((consumed / kGuSlots) & 1), p.status);
    ++consumed;
  }
}

// ---------------------------------------------------------------------------
// Down projection of the two-kernel path, then the combine. Work is split as
// in the gate/up kernel: 32-row blocks of every expert's W_d (H output rows),
// the shared expert's blocks on the last CTAs and the routed blocks by cost.
// Every warp streams units of RU rows (two slots) and computes them with the
// fused kernel's per-row code, reading the quantised h records from global
// memory (a CTA's blocks belong to one or two experts, so their records stay
// in L1). Each (pair, row) dot product goes to a partial buffer, which the
// combine kernel sums per token in the fixed order: shared expert first, then
// the routed experts ascending (the fused kernel's order).

// Rows per down unit for K inputs: a power of two, at least the rows that make
// a copy a multiple of 16 bytes, at most 32, and otherwise the most rows that
// fit in 4608 bytes (a gate/up unit at H = 4096).
__host__ __device__ inline int dn_rows_per_unit(int K) {
  const int rbK = K / 32 * kBlockB;
  int ru = 32;
  while (ru > 1 && ru * rbK > 4608) ru >>= 1;
  const int gd = row_granule_dev(K);
  return ru < gd ? gd : ru;
}

struct DnSmem {
  size_t slots, bars, total, slot_bytes;
  CopyWarpSmem cw;
};
__host__ __device__ inline DnSmem dn_smem(int F, int Fs, int n_shared, int nw) {
  DnSmem m;
  const int nc = nw - 1;
  size_t ub = (size_t)dn_rows_per_unit(F) * (F / 32) * kBlockB;
  if (n_shared) {
    const size_t us = (size_t)dn_rows_per_unit(Fs) * (Fs / 32) * kBlockB;
    ub = us > ub ? us : ub;
  }
  m.slot_bytes = align_up_dev(ub, 128);
  m.slots = align_up_dev(sizeof(RouteTable), 128);
  m.bars = m.slots + (size_t)nc * kGuSlots * m.slot_bytes;
  m.total = copy_warp_smem(m.bars + (size_t)nc * kGuSlots * 8, nc, m.cw);
  return m;
}

template <int LPR>
__global__ void __launch_bounds__(512, 1) dn_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = p.H;
  const int nw = (blockDim.x >> 5) - 1;          // computing warps; warp nw issues the copies
  const DnSmem L = dn_smem(p.F, p.Fs, p.n_shared, nw + 1);
  RouteTable& rt = *reinterpret_cast<RouteTable*>(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool copier = warp == nw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* ebars = reinterpret_cast<uint64_t*>(smem + L.cw.ebars);
  volatile uint32_t* stop = reinterpret_cast<uint32_t*>(smem + L.cw.stop);
  volatile uint32_t* final_iss = reinterpret_cast<uint32_t*>(smem + L.cw.iss);
  const int ww = copier ? (lane < nw ? lane : 0) : warp;
  uint8_t* myslots = smem + L.slots + (size_t)ww * kGuSlots * L.slot_bytes;
  uint64_t* mybar = bars + ww * kGuSlots;
  const int P = p.T * p.k;
  const int ru = dn_rows_per_unit(p.F), rus = p.n_shared ? dn_rows_per_unit(p.Fs) : 32;
  const uint32_t rbK = (uint32_t)(p.F / 32 * kBlockB), rbKs = (uint32_t)(p.Fs / 32 * kBlockB);

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int i = 0; i < nw * kGuSlots; ++i) {
      mbar_init(&bars[i], 1);
      mbar_init(&ebars[i], 1);
    }
    mbar_fence_init();
    *stop = 0u;
  }
  __syncthreads();

  const int G = gridDim.x, c = blockIdx.x;
  const int S = p.n_shared ? H / 32 : 0;
  const int sb0 = gu_shared_cum(S, c, G), sb1 = gu_shared_cum(S, c + 1, G);
  const int n_sh_u = (sb1 - sb0) * (32 / rus);
  int rb0 = 0, n_u = n_sh_u;
  auto count = [&](int nu) { return ww < nu ? (nu - ww + nw - 1) / nw : 0; };
  const int n_sh = count(n_sh_u);
  int n_tot = n_sh;
  int issued = 0, consumed = 0;
  bool ok = true;
  const uint64_t pol = l2_evict_first_policy();   // weights: read once per call
  // a warp's units in order (u = warp, warp + nw, ...): slot (-1 shared) and
  // first output row, kept up to date without divisions
  struct Cursor {
    int u, sl, row;
  };
  auto cur_get = [&](Cursor& k, int& sl, int& row) {
    if (k.u < n_sh_u) {
      sl = -1;
      row = sb0 * 32 + k.u * rus;
      return;
    }
    if (k.sl < 0) {
      const int r = rb0 * 32 + (k.u - n_sh_u) * ru;
      k.sl = r / H;
      k.row = r - k.sl * H;
    }
    sl = k.sl;
    row = k.row;
  };
  auto cur_next = [&](Cursor& k) {
    if (k.sl >= 0) {
      k.row += nw * ru;
      while (k.row >= H) {
        k.row -= H;
        ++k.sl;
      }
    }
    k.u += nw;
  };
  Cursor ci{ww, -1, 0}, cc{ww, -1, 0};
  // the copy warp: lane w < nw issues warp w's next units, up to `limit`, each
  // once its slot is free; true if it issued any
  auto issue_upto = [&](int limit) {
    bool any = false;
#pragma unroll 1
    for (;;) {
      bool can = lane < nw && issued < limit;
      if (can && issued >= kGuSlots)
        can = mbar_test(&ebars[ww * kGuSlots + issued % kGuSlots],
                        (uint32_t)(((issued / kGuSlots) + 1) & 1));
      if (!__any_sync(0xFFFFFFFFu, can)) break;
      if (can) {
        int sl, row;
        cur_get(ci, sl, row);
        const int s = issued % kGuSlots;
        const uint8_t* src = sl < 0 ? p.sh_down + (size_t)row * rbKs
                                    : p.down + ((size_t)rt.slot_expert[sl] * H + row) * rbK;
        const uint32_t bytes = sl < 0 ? rus * rbKs : ru * rbK;    // multiples of 16
        mbar_arrive_expect_tx(&mybar[s], bytes);
        bulk_g2s_hint(myslots + (size_t)s * L.slot_bytes, src, bytes, &mybar[s], pol);
        cur_next(ci);
        ++issued;
      }
      any = true;
    }
    return any;
  };

  if (copier) issue_upto(n_sh < kGuSlots ? n_sh : kGuSlots);
  // ids and weights come from a kernel that finished before the gate/up kernel
  // passed its own dependency wait: they may be read before this one's
  if (P <= 64) {
    if (warp == 0) build_route_table_warp(rt, p.ids, p.weights, P, p.E);
    __syncthreads();
  } else {
    build_route_table<0>(rt, p.ids, p.weights, P, p.E, blockDim.x);
  }
  {
    const int bps = H / 32;
    rb0 = gu_routed_cum(rt, bps, S, p.T, c, G);
    const int rb1 = gu_routed_cum(rt, bps, S, p.T, c + 1, G);
    n_u = n_sh_u + (rb1 - rb0) * (32 / ru);
  }
  n_tot = count(n_u);
  if (copier) {
    // every unit of every computing warp, as slots free up; a stop from the
    // computing warps (a failed wait) or a long idle spell ends it early
    const bool mine = lane < nw;
    uint64_t t_act = global_timer_ns();
#pragma unroll 1
    while (!__all_sync(0xFFFFFFFFu, !mine || issued >= n_tot) && !*stop) {
      const uint64_t now = global_timer_ns();
      if (issue_upto(n_tot)) {
        t_act = now;
      } else {
        if (now - t_act > 2 * kWaitLimitNs) {
          if (lane == 0 && p.status) atomicOr(p.status, MOE_STATUS_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    if (mine) final_iss[lane] = (uint32_t)issued;
    __syncthreads();     // the computing warps' final barrier
    return;
  }
  pdl_wait();                  // the records come from the gate/up kernel
  pdl_trigger();

  const int words = dqvec_words(p.F), words_s = dqvec_words(p.Fs);
#pragma unroll 1
  for (int j = 0; ok && j < n_tot; ++j) {
    ok = mbar_wait(&mybar[j % kGuSlots], (uint32_t)((j / kGuSlots) & 1), p.status);
    if (!ok) break;
    const uint8_t* d = myslots + (size_t)(j % kGuSlots) * L.slot_bytes;
    int sl, row;
    cur_get(cc, sl, row);
    cur_next(cc);
    const bool shared = sl < 0;
    const int ntok = shared ? p.T : rt.slot_off[sl + 1] - rt.slot_off[sl];
    const int lbase = shared ? 0 : rt.slot_off[sl];
    auto pidx = [&](int jj) { return shared ? P + jj : rt.list[lbase + jj]; };
    auto rec_of = [&](int jj) -> const uint32_t* {
      return shared ? p.rec_s + (size_t)jj * words_s : p.rec_r + (size_t)pidx(jj) * words;
    };
    auto store = [&](int jj, int rl, float v) { p.part[(size_t)pidx(jj) * H + row + rl] = v; };
    if (ntok == 1)
      down_rows<1, LPR>(d, shared ? p.Fs : p.F, shared ? rus : ru, 1, rec_of, store);
    else
      down_rows<kGuMaxT, LPR>(d, shared ? p.Fs : p.F, shared ? rus : ru, ntok, rec_of, store);
    __syncwarp();
    if (lane == 0) mbar_arrive(&ebars[warp * kGuSlots + j % kGuSlots]);   // slot free
    ++consumed;
  }
  if (!ok && lane == 0) *stop = 1u;
  // after a timeout: no bulk copy of this warp stays in flight
  __syncthreads();
  while (consumed < (int)final_iss[warp]) {
    mbar_wait(&mybar[consumed % kGuSlots], (uint32_t)((consumed / kGuSlots) & 1), p.status);
    ++consumed;
  }
}

// y[t][n] = shared expert's partial + the routed partials of token t, in the
// route table's order (experts ascending, then pair index), each times its
// weight: the fused kernel's combine. One warp per token first sorts the
// token's valid pairs into that order (ranks by ballots), which needs only the
// ids and weights; then every thread sums its outputs.
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ int tp[MOE_MAX_DECODE_TOKENS][MOE_MAX_TOP_K];   // pair indices in order
  __shared__ float tw[MOE_MAX_DECODE_TOKENS][MOE_MAX_TOP_K];
  __shared__ int tc[MOE_MAX_DECODE_TOKENS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = p.k;
  // ids and weights come from a kernel that finished before the gate/up
  // kernel passed its own dependency wait: they may be read before this one's
#pragma unroll 1
  for (int t = warp; t < p.T; t += blockDim.x >> 5) {
    const int pr = t * k + lane;
    int e = -1;
    float w = 0.0f;
    if (lane < k) {
      const int id = p.ids[pr];
      if (id >= 0 && id < p.E) {
        e = id;
        w = p.weights[pr];
      }
    }
    int rank = 0;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
      rank += ej >= 0 && (ej < e || (ej == e && j < lane));
    }
    const unsigned valid = __ballot_sync(0xFFFFFFFFu, e >= 0);
    if (e >= 0) {
      tp[t][rank] = pr;
      tw[t][rank] = w;
    }
    if (lane == 0) tc[t] = __popc(valid);
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int H = p.H, P = p.T * k;
#pragma unroll 1
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.T * H; i += gridDim.x * blockDim.x) {
    const int t = i / H, n = i - t * H;
    const int cnt = tc[t];
    float v[MOE_MAX_TOP_K];
#pragma unroll
    for (int r = 0; r < MOE_MAX_TOP_K; ++r)
      v[r] = r < cnt ? p.part[(size_t)tp[t][r] * H + n] : 0.0f;
    float acc = 0.0f;
    if (p.n_shared) acc = p.part[(size_t)(P + t) * H + n];
#pragma unroll
    for (int r = 0; r < MOE_MAX_TOP_K; ++r)
      if (r < cnt) acc += tw[t][r] * v[r];
    p.y[i] = acc;
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

}  // namespace

int decode_launches(const DecodeParams& p, int num_sms) {
  size_t fsm = 0;
  int rg = 0, rmax = 0;
  if (fused_decode_supported(p, num_sms, &fsm, &rg, &rmax)) return 1;
  int nw = 0, nblk = 0;
  bool xs = true;
  size_t sm = 0;
  if (!gu_config(p, num_sms, &nw, &xs, &sm, &nblk)) return 3;
  return xs ? 3 : 4;
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
  int dnw = 16;
  while (dnw > 4 && dn_smem(p.F, p.Fs, p.n_shared, dnw).total > kSmemMax) dnw >>= 1;
  const size_t dsm = dn_smem(p.F, p.Fs, p.n_shared, dnw).total;
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
  const bool d8 = lanes_per_row(p.F) == 8 && (!p.n_shared || lanes_per_row(p.Fs) == 8);
  e = d8 ? launch(dn_kernel<8>, num_sms, dnw * 32, dsm, pdl, stream, p)
         : launch(dn_kernel<0>, num_sms, dnw * 32, dsm, pdl, stream, p);
  if (e != cudaSuccess) return e;
  int cgrid = (p.T * p.H + 255) / 256;
  if (cgrid > num_sms) cgrid = num_sms;
  return launch(combine_kernel, cgrid, 256, 0, pdl, stream, p);
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
