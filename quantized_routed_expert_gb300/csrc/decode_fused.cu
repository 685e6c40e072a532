// Fused decode kernel of libmoe (sm_103a): gate/up + SwiGLU, a grid barrier,
// then down + combine, in one persistent launch (one CTA per SM).
//
// Every warp streams its own work units: it issues 1D bulk copies (TMA) of
// the IQ4_NL rows of its next units into two private shared-memory slots and
// computes each unit as it lands, with no barrier between warps. Units:
//   gate/up: one f-row of one expert (its gate row and its up row);
//   down:    a group of output rows of one expert's W_d.
// Each IQ4_NL block is decoded once (byte_perm table lookup) and dotted with
// every token routed to the expert by dp2a against 16-bit block-quantised
// activations (Red Lite, "What we learned", section 4: decode each weight
// block once for both tokens of a paired pass). Down-phase weights are fetched
// before the grid barrier, so they stream while the gate/up phase finishes.
// Each output is the sum, in a fixed order, of per-(pair, row) partials: the
// shared expert first, then the routed experts in ascending id.
#include "common.cuh"
#include "decode.cuh"
#include "decode_common.cuh"

#include <mutex>

namespace moe {

constexpr int kFW = 15;            // computing warps per CTA (warp 15 issues the copies)
constexpr int kFT = kFW * 32;      // computing threads per CTA
constexpr int kFTP = kFT + 32;     // threads per CTA: the computing warps and the copy warp
constexpr int kFSlots = 2;         // bulk-copy slots per computing warp
constexpr int kFBar = 2;           // named barrier of the computing warps

struct FusedSmem {
  size_t xq, slots, bars, ebars, recs, part, total, slot_bytes;
  // router scratch (routed kernel), overlaying the records area, which is used
  // only after the h barrier
  size_t r_wr, r_x, r_part, r_keys, r_ids, r_w;
  // h staging for the local quantisation (0 bytes: h is read from L2 instead)
  size_t stage, stage_bytes;
};

// Experts whose scores CTA c computes: a balanced split of E over the grid.
__host__ __device__ inline int route_e0(int E, int c, int G) { return (int)((long long)E * c / G); }

__host__ __device__ inline FusedSmem fused_smem(int H, int F, int Fs, int ns, int T, int k,
                                                int rows_max, int rg, int route, int E, int G) {
  FusedSmem m;
  const size_t rbH = (size_t)(H / 32) * kBlockB;
  size_t rbK = (size_t)(F / 32) * kBlockB;
  if (ns) {
    const size_t rbs = (size_t)(Fs / 32) * kBlockB;
    rbK = rbK > rbs ? rbK : rbs;
  }
  const size_t gu = 2 * rbH;
  const size_t dn = (size_t)rg * rbK;
  m.slot_bytes = align_up_dev(gu > dn ? gu : dn, 128);
  m.xq = align_up_dev(sizeof(RouteTable), 128);
  m.slots = align_up_dev(m.xq + (size_t)T * dqvec_words(H) * 4, 128);
  m.bars = m.slots + (size_t)kFW * kFSlots * m.slot_bytes;
  // the slots' "free" barriers, then the copy warp's words: routes known, stop,
  // units issued per computing warp, each warp's routed and down units and the
  // first routed row
  m.ebars = align_up_dev(m.bars + (size_t)(kFW * kFSlots + 4) * 8, 16);
  m.recs = align_up_dev(m.ebars + (size_t)kFW * kFSlots * 8 + 8 + (size_t)kFW * 4 +
                            (size_t)kFW * 8 + 4, 128);
  const size_t recs = (size_t)T * k * dqvec_words(F) * 4 + (ns ? (size_t)T * dqvec_words(Fs) * 4 : 0);
  m.part = align_up_dev(m.recs + recs, 16);
  size_t end = m.part + (size_t)(T * k + (ns ? T : 0)) * rows_max * 4;
  m.r_wr = m.r_x = m.r_part = m.r_keys = m.r_ids = m.r_w = 0;
  if (route) {
    const int epc = (E + G - 1) / G + 1;             // most experts any CTA scores
    m.r_wr = m.recs;
    m.r_x = align_up_dev(m.r_wr + (size_t)epc * H * 2, 128);
    m.r_part = align_up_dev(m.r_x + (size_t)T * H * 2, 16);
    m.r_keys = align_up_dev(m.r_part + (size_t)epc * 16 * T * 4, 16);
    m.r_ids = align_up_dev(m.r_keys + (size_t)2 * T * ((E + 31) & ~31) * 4, 16);  // keys, sigmoids
    m.r_w = align_up_dev(m.r_ids + (size_t)T * k * 4, 16);
    const size_t rend = m.r_w + (size_t)T * k * 4;
    end = end > rend ? end : rend;
  }
  // stage every h row of the call in shared memory when it fits
  const size_t hb = ((size_t)T * k * F + (ns ? (size_t)T * Fs : 0)) * 4;
  const size_t st = align_up_dev(end, 128);
  if (st + hb <= (size_t)227 * 1024) {
    m.stage = st;
    m.stage_bytes = hb;
    end = st + hb;
  } else {
    m.stage = 0;
    m.stage_bytes = 0;
  }
  m.total = end;
  return m;
}

// What one warp needs to issue the bulk copies of its units: the warp's unit
// sequence is its shared-expert gate/up rows, then its routed gate/up rows,
// then its down-row groups (shared expert first, then the routed slots).
struct UnitPlan {
  uint8_t* myslots;
  size_t slot_bytes;
  uint64_t* mybar;
  uint64_t pol;
  int warp, n_sh, n_rt, sh_a, rr_a, ngroups, nrows_cta, dn_a, rg;
};

// Issue unit j of a warp's sequence into slot j % kFSlots (one lane calls).
__device__ __noinline__ void issue_unit(const DecodeParams& p, const RouteTable& rt,
                                        const UnitPlan& u, int j) {
  const int s = j % kFSlots;
  uint8_t* dst = u.myslots + (size_t)s * u.slot_bytes;
  uint64_t* bar = &u.mybar[s];
  const uint32_t rbH = (uint32_t)(p.H / 32 * kBlockB);
  if (j < u.n_sh + u.n_rt) {
    const uint8_t *g, *up;
    if (j < u.n_sh) {
      const size_t f = (size_t)(u.sh_a + u.warp + kFW * j);
      g = p.sh_gate + f * rbH;
      up = p.sh_up + f * rbH;
    } else {
      const int r = u.rr_a + u.warp + kFW * (j - u.n_sh);
      const int sl = r / p.F, f = r - sl * p.F;
      const size_t row = (size_t)rt.slot_expert[sl] * p.F + f;
      g = p.gate + row * rbH;
      up = p.up + row * rbH;
    }
    mbar_arrive_expect_tx(bar, 2 * rbH);
    bulk_g2s_hint(dst, g, rbH, bar, u.pol);
    bulk_g2s_hint(dst + rbH, up, rbH, bar, u.pol);
  } else {
    const int un = u.warp + kFW * (j - u.n_sh - u.n_rt);
    const int su = un / u.ngroups, gi = un - su * u.ngroups;
    const bool sh = p.n_shared && su == 0;
    const int sl = su - p.n_shared;
    const int K = sh ? p.Fs : p.F;
    const int rbK = K / 32 * kBlockB;
    const int r0 = gi * u.rg;
    const int nr = u.nrows_cta - r0 < u.rg ? u.nrows_cta - r0 : u.rg;
    const uint8_t* src = sh ? p.sh_down + (size_t)(u.dn_a + r0) * rbK
                            : p.down + ((size_t)rt.slot_expert[sl] * p.H + u.dn_a + r0) * rbK;
    mbar_arrive_expect_tx(bar, (uint32_t)(nr * rbK));
    bulk_g2s_hint(dst, src, (uint32_t)(nr * rbK), bar, u.pol);
  }
}

template <int MAXT, bool ROUTE, int LPR>
__global__ void __launch_bounds__(kFTP, 1) decode_fused_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = p.H;
  const int rows_max = p.dn_rows_max;
  const int RG = p.fz_rg;
  const FusedSmem L = fused_smem(H, p.F, p.Fs, p.n_shared, p.T, p.k, rows_max, RG, ROUTE ? 1 : 0,
                                 p.E, gridDim.x);
  RouteTable& rt = *reinterpret_cast<RouteTable*>(smem);
  uint32_t* xq = reinterpret_cast<uint32_t*>(smem + L.xq);
  uint8_t* slots = smem + L.slots;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* recs_bar = bars + kFW * kFSlots;
  uint64_t* rwr_bar = recs_bar + 1;            // router rows of this CTA
  uint64_t* rx_bar = recs_bar + 2;             // activations for the router
  uint32_t* recs = reinterpret_cast<uint32_t*>(smem + L.recs);
  float* part = reinterpret_cast<float*>(smem + L.part);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int xq_words = dqvec_words(H);
  const int rbH = H / 32 * kBlockB;
  uint64_t* ebars = reinterpret_cast<uint64_t*>(smem + L.ebars);     // slot freed
  volatile uint32_t* routes_known = reinterpret_cast<uint32_t*>(ebars + kFW * kFSlots);
  volatile uint32_t* stop = routes_known + 1;
  volatile uint32_t* final_iss = stop + 1;
  int* plan_s = const_cast<int*>(reinterpret_cast<volatile int*>(final_iss + kFW));  // [kFW][2], rr_a
  // the warp whose slots this thread fills (copy warp lane w) or computes
  const int ww = warp == kFW ? (lane < kFW ? lane : 0) : warp;
  uint8_t* myslots = slots + (size_t)ww * kFSlots * L.slot_bytes;
  uint64_t* mybar = bars + ww * kFSlots;

  if (threadIdx.x == 0) {
    #pragma unroll 1
    for (int i = 0; i < kFW * kFSlots + 3; ++i) mbar_init(&bars[i], 1);
    #pragma unroll 1
    for (int i = 0; i < kFW * kFSlots; ++i) mbar_init(&ebars[i], 1);
    mbar_fence_init();
    *routes_known = 0u;
    *stop = 0u;
  }
  __syncthreads();

  // ---- this CTA's work
  const RowRange shr = p.n_shared ? split_rows(p.Fs, 1, blockIdx.x, gridDim.x) : RowRange{0, 0};
  const RowRange dn = split_rows(H, 1, blockIdx.x, gridDim.x);
  const int nrows_cta = dn.b - dn.a;
  const int ngroups = (nrows_cta + RG - 1) / RG;
  auto count = [&](int a, int b) { return a + ww < b ? (b - a - ww + kFW - 1) / kFW : 0; };
  const int n_sh = count(shr.a, shr.b);
  int n_rt = 0, n_tot = n_sh;      // known once the route table exists
  RowRange rr{0, 0};
  int n_dslots = 0;

  int consumed = 0;
  bool ok = true;
  const uint64_t pol = l2_evict_first_policy();   // weights are read once per call
  UnitPlan up;
  up.myslots = myslots;
  up.slot_bytes = L.slot_bytes;
  up.mybar = mybar;
  up.warp = ww;
  up.n_sh = n_sh;
  up.n_rt = 0;
  up.sh_a = shr.a;
  up.rr_a = 0;
  up.ngroups = ngroups;
  up.nrows_cta = nrows_cta;
  up.dn_a = dn.a;
  up.rg = RG;
  up.pol = pol;
  auto wait_unit = [&](int j) {
    return mbar_wait(&mybar[j % kFSlots], (uint32_t)((j / kFSlots) & 1), p.status);
  };
  auto release_unit = [&](int j) {  // the warp is done with unit j's slot
    __syncwarp();
    if (lane == 0) mbar_arrive(&ebars[warp * kFSlots + j % kFSlots]);
  };

  if (warp == kFW) {
    // ---- the copy warp. A bulk copy is taken in by the copy engine no
    // faster than memory delivers, so the issuing thread stalls meanwhile;
    // here no computing warp ever issues a weight copy. Lane w < kFW fills
    // computing warp w's two slots in its unit order, each slot once the warp
    // released the unit two back, the routed and down units once the route
    // table is built (its plan then comes from warp 0).
    const bool mine = lane < kFW;
    int iss = 0, lim = mine ? n_sh : 0;
    bool known = false;
    const uint64_t idle_ns = 2 * kWaitLimitNs + p.wait_ns;
    uint64_t t_act = global_timer_ns();
#pragma unroll 1
    for (;;) {
      bool any = false;
#pragma unroll 1
      for (;;) {
        bool can = mine && iss < lim;
        if (can && iss >= kFSlots)
          can = mbar_test(&ebars[ww * kFSlots + iss % kFSlots],
                          (uint32_t)(((iss / kFSlots) + 1) & 1));
        if (!__any_sync(0xFFFFFFFFu, can)) break;
        if (can) {
          issue_unit(p, rt, up, iss);
          ++iss;
        }
        any = true;
      }
      if (!known) {
        if (*routes_known) {
          __threadfence_block();
          if (mine) {
            up.n_rt = plan_s[2 * ww];
            up.rr_a = plan_s[2 * kFW];
            lim = n_sh + up.n_rt + plan_s[2 * ww + 1];
          }
          known = true;
          any = true;
        }
      } else if (__all_sync(0xFFFFFFFFu, !mine || iss == lim)) {
        break;                                   // every unit of the call issued
      }
      if (*stop) break;
      const uint64_t now = global_timer_ns();
      if (any) {
        t_act = now;
      } else {
        if (now - t_act > idle_ns) {
          if (lane == 0 && p.status) atomicOr(p.status, MOE_STATUS_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    if (mine) final_iss[lane] = (uint32_t)iss;
    __syncthreads();     // the computing warps' final barrier
    return;
  }

  // Router rows of this CTA's experts (constant): fetch them while the previous
  // kernel on the stream finishes.
  const int re0 = ROUTE ? route_e0(p.E, blockIdx.x, gridDim.x) : 0;
  const int re1 = ROUTE ? route_e0(p.E, blockIdx.x + 1, gridDim.x) : 0;
  if (ROUTE && threadIdx.x == 0 && re1 > re0) {
    const uint32_t bytes = (uint32_t)((re1 - re0) * H * 2);
    mbar_arrive_expect_tx(rwr_bar, bytes);
    bulk_g2s_hint(smem + L.r_wr, p.Wr + (size_t)re0 * H, bytes, rwr_bar,
                  l2_evict_first_policy());
  }
  pdl_wait();
  pdl_trigger();
  if (ROUTE && threadIdx.x == 0 && re1 > re0) {
    const uint32_t bytes = (uint32_t)(p.T * H * 2);
    mbar_arrive_expect_tx(rx_bar, bytes);
    bulk_g2s(smem + L.r_x, p.x, bytes, rx_bar);
  }
  quant_x_lanes<1>(p.x, p.T, H, xq, xq_words, threadIdx.x, kFT);

  if (ROUTE) {
    // Scores of this CTA's experts: 16 chunks of H per expert, one warp per
    // (expert, chunk), chunk partials summed in a fixed order.
    const int ne = re1 - re0;
    float* rpart = reinterpret_cast<float*>(smem + L.r_part);
    if (ne > 0) {
      ok = mbar_wait(rwr_bar, 0, p.status) && mbar_wait(rx_bar, 0, p.status);
      const uint16_t* wr_s = reinterpret_cast<const uint16_t*>(smem + L.r_wr);
      const uint16_t* x_s = reinterpret_cast<const uint16_t*>(smem + L.r_x);
      const int hc = H / 16;                     // chunk length, a multiple of 16
      #pragma unroll 1
      for (int it = warp; it < ne * 16; it += kFW) {
        const int el = it >> 4, c = it & 15;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        #pragma unroll 1
        for (int g8 = lane; g8 < hc / 8; g8 += 32) {
          const uint4 wv = reinterpret_cast<const uint4*>(wr_s + (size_t)el * H + c * hc)[g8];
          const uint32_t wr[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (t < p.T) {
              const uint4 xv = reinterpret_cast<const uint4*>(x_s + (size_t)t * H + c * hc)[g8];
              const uint32_t xr[4] = {xv.x, xv.y, xv.z, xv.w};
              float a = acc[t];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                a = fmaf(__uint_as_float(wr[i] << 16), __uint_as_float(xr[i] << 16), a);
                a = fmaf(__uint_as_float(wr[i] & 0xFFFF0000u), __uint_as_float(xr[i] & 0xFFFF0000u), a);
              }
              acc[t] = a;
            }
          }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], o);
        if (lane == 0) {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (t < p.T) rpart[(el * 16 + c) * p.T + t] = acc[t];
        }
      }
    }
    bar_sync_n(kFBar, kFT);
    #pragma unroll 1
    for (int i = threadIdx.x; i < ne * p.T; i += kFT) {
      const int el = i / p.T, t = i - el * p.T;
      float sc = 0.f;
      for (int c = 0; c < 16; ++c) sc += rpart[(el * 16 + c) * p.T + t];
      p.scores[(size_t)t * p.E + re0 + el] = sc;
    }
    __threadfence();
    bar_sync_n(kFBar, kFT);
    if (threadIdx.x == 0) atomicAdd(&p.sync[2], 1u);
  }
  bar_sync_n(kFBar, kFT);

  // ---- routing (this CTA's experts' scores were published above)
  const int32_t* ids_src = p.ids;
  const float* w_src = p.weights;
  if (ROUTE) {
    // all scores of this call -> top-k: warp t takes token t, in every CTA
    int32_t* ids_s = reinterpret_cast<int32_t*>(smem + L.r_ids);
    float* w_s = reinterpret_cast<float*>(smem + L.r_w);
    if (threadIdx.x == 0) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire_u32(&p.sync[2]) < gridDim.x) {
        if (global_timer_ns() - t0 >= p.wait_ns) {
          if (p.status) atomicOr(p.status, MOE_STATUS_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
      __threadfence();
    }
    bar_sync_n(kFBar, kFT);
    // keys p + b and sigmoids p, rows padded to E32 with -inf (keys)
    float* keys_all = reinterpret_cast<float*>(smem + L.r_keys);
    const int E32 = (p.E + 31) & ~31;
#pragma unroll 1
    for (int i = threadIdx.x; i < p.T * E32; i += kFT) {
      const int t = i / E32, e = i - t * E32;
      float key = -INFINITY, pr = 0.0f;
      if (e < p.E) {
        pr = 1.0f / (1.0f + expf(-__ldcg(p.scores + (size_t)t * p.E + e)));
        key = pr + (p.bias ? p.bias[e] : 0.0f);
      }
      keys_all[(size_t)p.T * E32 + i] = pr;
      keys_all[i] = key;
    }
    bar_sync_n(kFBar, kFT);
    if (warp < p.T) {
      const int t = warp;
      float* keys = keys_all + (size_t)t * E32;
      float* probs = keys + (size_t)p.T * E32;
      const int id = warp_topk_ids_512(keys, p.E, p.k);
      const float wv = warp_renorm(lane < p.k ? probs[id] : 0.0f, p.k);
      if (lane < p.k) {
        ids_s[t * p.k + lane] = id;
        w_s[t * p.k + lane] = wv;
        if (blockIdx.x == 0) {
          p.ids_out[(size_t)t * p.k + lane] = id;
          p.w_out[(size_t)t * p.k + lane] = wv;
        }
      }
      if (p.T > 1) bar_sync_n(1, p.T * 32);     // the token warps only
    }
    ids_src = ids_s;
    w_src = w_s;
  }
  if (warp == 0) {
    build_route_table_warp(rt, ids_src, w_src, p.T * p.k, p.E);
    // every computing warp's routed and down units, for the copy warp (the
    // row split of split_rows in 32-bit arithmetic: n_slots * F * G < 2^32)
    if (lane < kFW) {
      const uint32_t tot = (uint32_t)(rt.n_slots * p.F);
      const int a = (int)(tot * blockIdx.x / gridDim.x), b = (int)(tot * (blockIdx.x + 1) / gridDim.x);
      plan_s[2 * lane] = a + lane < b ? (b - a - lane + kFW - 1) / kFW : 0;
      const int nu = (rt.n_slots + p.n_shared) * ngroups;
      plan_s[2 * lane + 1] = lane < nu ? (nu - lane + kFW - 1) / kFW : 0;
      if (lane == 0) plan_s[2 * kFW] = a;
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      *routes_known = 1u;
    }
  }
  bar_sync_n(kFBar, kFT);
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.status && rt.invalid)
    atomicAdd(p.status, (uint32_t)(rt.invalid < 0xFFFF ? rt.invalid : 0xFFFF));
  #pragma unroll 1
  for (int i = threadIdx.x; i < (p.T * p.k + (p.n_shared ? p.T : 0)) * rows_max; i += kFT)
    part[i] = 0.0f;
  rr = split_rows(rt.n_slots * p.F, 1, blockIdx.x, gridDim.x);
  n_rt = count(rr.a, rr.b);
  up.n_rt = n_rt;
  up.rr_a = rr.a;
  n_dslots = rt.n_slots + p.n_shared;
  const int n_dn_units = n_dslots * ngroups;
  const int n_dn = warp < n_dn_units ? (n_dn_units - warp + kFW - 1) / kFW : 0;
  n_tot = n_sh + n_rt + n_dn;

  // the routed rows' copies are in flight: compute the shared expert's rows
  // (landed long ago) while they arrive, then the routed rows
  int j = 0;
#pragma unroll 1
  for (; ok && j < n_sh + n_rt; ++j) {
    ok = wait_unit(j);
    if (!ok) break;
    const uint8_t* d = myslots + (size_t)(j % kFSlots) * L.slot_bytes;
    int sl, f;
    if (j < n_sh) {
      sl = -1;
      f = shr.a + warp + kFW * j;
    } else {
      const int r = rr.a + warp + kFW * (j - n_sh);
      sl = r / p.F;
      f = r - sl * p.F;
    }
    // one-token experts (most of them) take the code built for one token
    if (MAXT == 1 || (sl < 0 ? p.T : rt.slot_off[sl + 1] - rt.slot_off[sl]) == 1)
      gateup_unit_t<1, LPR>(p, rt, d, d + rbH, sl, f, xq, xq_words);
    else
      gateup_unit_t<MAXT, LPR>(p, rt, d, d + rbH, sl, f, xq, xq_words);
    release_unit(j);
    ++consumed;
  }

  // ---- grid barrier: every h row of this call is in global memory
  bar_sync_n(kFBar, kFT);
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&p.sync[0], 1u);
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_u32(&p.sync[0]) < gridDim.x) {
      if (global_timer_ns() - t0 >= p.wait_ns) {
        if (p.status) atomicOr(p.status, MOE_STATUS_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  bar_sync_n(kFBar, kFT);
  // every CTA quantises all of h into its own records: staged in shared
  // memory by bulk copies when there is room, else read through L2
  if (L.stage_bytes) {
    float* stage = reinterpret_cast<float*>(smem + L.stage);
    if (threadIdx.x == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      const uint32_t rbF = (uint32_t)p.F * 4, rbS = (uint32_t)p.Fs * 4;
      const uint32_t total = rt.n_valid * rbF + (p.n_shared ? p.T * rbS : 0u);
      mbar_arrive_expect_tx(recs_bar, total);
      uint8_t* dst = reinterpret_cast<uint8_t*>(stage);
      for (int e = 0; e < rt.n_valid; ++e, dst += rbF)
        bulk_g2s(dst, p.h_r + (size_t)rt.list[e] * p.F, rbF, recs_bar);
      if (p.n_shared)
        for (int j = 0; j < p.T; ++j, dst += rbS)
          bulk_g2s(dst, p.h_s + (size_t)j * p.Fs, rbS, recs_bar);
    }
    // wait even after an earlier timeout: no copy of this CTA stays in flight
    const bool landed = mbar_wait(recs_bar, 0, p.status);
    ok = ok && landed;
    if (ok) quant_h<true>(p, rt, stage, recs, threadIdx.x, kFT);
  } else {
    quant_h<false>(p, rt, nullptr, recs, threadIdx.x, kFT);
  }
  bar_sync_n(kFBar, kFT);

  #pragma unroll 1
  for (int j = n_sh + n_rt; ok && j < n_tot; ++j) {
    ok = wait_unit(j);
    if (!ok) break;
    const uint8_t* d = myslots + (size_t)(j % kFSlots) * L.slot_bytes;
    const int u = warp + kFW * (j - n_sh - n_rt);
    const int su = u / ngroups, gi = u - su * ngroups;
    const bool sh = p.n_shared && su == 0;
    const int r0 = gi * RG;
    const int nr = nrows_cta - r0 < RG ? nrows_cta - r0 : RG;
    const int dsl = sh ? -1 : su - p.n_shared;
    if (MAXT == 1 || (sh ? p.T : rt.slot_off[dsl + 1] - rt.slot_off[dsl]) == 1)
      down_unit_t<1, LPR>(p, rt, d, dsl, r0, nr, recs, part, rows_max);
    else
      down_unit_t<MAXT, LPR>(p, rt, d, dsl, r0, nr, recs, part, rows_max);
    release_unit(j);
    ++consumed;
  }
  bar_sync_n(kFBar, kFT);

  // ---- combine in the fixed order: shared expert, then routed experts ascending
  #pragma unroll 1
  for (int i = threadIdx.x; i < nrows_cta * p.T; i += kFT) {
    const int t = i / nrows_cta, r = i - t * nrows_cta;
    float acc = 0.0f;
    if (p.n_shared) acc = part[(size_t)(p.T * p.k + t) * rows_max + r];
    #pragma unroll 1
    for (int e = 0; e < rt.n_valid; ++e) {
      const int pr = rt.list[e];
      if (pr / p.k == t) acc += rt.wt[pr] * part[(size_t)pr * rows_max + r];
    }
    p.y[(size_t)t * H + dn.a + r] = acc;
  }

  // ---- the copy warp stops (it has issued everything unless a wait failed)
  // and reports how many units it issued per warp; after a timeout, drain
  // this warp's bulk copies still in flight
  if (threadIdx.x == 0) {
    __threadfence_block();
    *stop = 1u;
  }
  __syncthreads();
  while (consumed < (int)final_iss[warp]) {
    wait_unit(consumed);
    ++consumed;
  }

  // ---- leave: the last CTA out resets the barrier counters for the next call
  if (threadIdx.x == 0) {
    const uint32_t old = atomicAdd(&p.sync[1], 1u);
    if (old == gridDim.x - 1) {
      p.sync[0] = 0u;
      p.sync[1] = 0u;
      p.sync[2] = 0u;
    }
  }
}

// ---------------------------------------------------------------------------
namespace {
// The instantiation a launch with these parameters uses.
const void* fused_kernel_for(const DecodeParams& p) {
  const bool w8 = lanes_per_row(p.H) == 8 && lanes_per_row(p.F) == 8 &&
                  (!p.n_shared || lanes_per_row(p.Fs) == 8);
#define MOE_FK(T_, R_, L_) reinterpret_cast<const void*>(decode_fused_kernel<T_, R_, L_>)
  const int t = p.T == 1 ? 1 : (p.T == 2 ? 2 : 4);
  if (p.route) {
    if (w8) return t == 1 ? MOE_FK(1, true, 8) : t == 2 ? MOE_FK(2, true, 8) : MOE_FK(4, true, 8);
    return t == 1 ? MOE_FK(1, true, 0) : t == 2 ? MOE_FK(2, true, 0) : MOE_FK(4, true, 0);
  }
  if (w8) return t == 1 ? MOE_FK(1, false, 8) : t == 2 ? MOE_FK(2, false, 8) : MOE_FK(4, false, 8);
  return t == 1 ? MOE_FK(1, false, 0) : t == 2 ? MOE_FK(2, false, 0) : MOE_FK(4, false, 0);
#undef MOE_FK
}
}  // namespace

// Whether one CTA of the fused kernel with `smem` bytes of shared memory fits
// on an SM of the current device (cached per kernel, device and size). The
// grid is one CTA per SM and its barriers need every CTA resident; where the
// occupancy query says no, the two-kernel path runs instead.
bool fused_resident(const DecodeParams& p, size_t smem) {
  static std::mutex mu;
  struct Entry { const void* k; int dev; size_t smem; bool ok; };
  static Entry cache[64];
  static int n = 0;
  const void* k = fused_kernel_for(p);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return false; }
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
      if (cache[i].k == k && cache[i].dev == dev && cache[i].smem == smem) return cache[i].ok;
  }
  bool ok = false;
  if (ensure_smem_attr(k, smem) == cudaSuccess) {
    int blocks = 0;
    ok = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k, kFTP, smem) == cudaSuccess &&
         blocks >= 1;
  }
  cudaGetLastError();
  std::lock_guard<std::mutex> lock(mu);
  if (n < 64) cache[n++] = Entry{k, dev, smem, ok};
  return ok;
}

bool fused_decode_supported(const DecodeParams& p, int num_sms, size_t* smem, int* rg,
                            int* rows_max) {
  if (p.T < 1 || p.T > 4) return false;
  if (p.H % 256 || p.F % 256 || (p.n_shared && p.Fs % 256)) return false;
  if (p.route && p.E > 512) return false;         // in-kernel top-k holds 16 keys a lane
  const int grid = num_sms;
  const int rmax = (p.H + grid - 1) / grid;
  // down rows per unit: one pass of a warp (32 / lanes per row rows; finer
  // units balance the down phase over the warps), unless the CTA then has
  // more than two units per warp: those beyond a warp's two slots could not be
  // fetched before the h barrier. Then whole passes are added while a unit
  // fits in max(a gate/up unit, 4608 bytes), or all of the CTA's rows.
  int K = p.F;
  if (p.n_shared && p.Fs > K) K = p.Fs;
  const int rpw = 32 / lanes_per_row(K);
  const int64_t rbK = row_bytes(K);
  int64_t budget = 2 * row_bytes(p.H);
  if (budget < 4608) budget = 4608;
  const int slots = (p.T * p.k < p.E ? p.T * p.k : p.E) + p.n_shared;
  auto units = [&](int rows) { return slots * ((rmax + rows - 1) / rows); };
  int r = rpw < rmax ? rpw : rmax;
  if (units(r) > 2 * kFW) {
    while (r + rpw <= rmax && (r + rpw) * rbK <= budget) r += rpw;
    if (rmax * rbK <= budget) r = rmax;
  }
  const FusedSmem m = fused_smem(p.H, p.F, p.Fs, p.n_shared, p.T, p.k, rmax, r, p.route, p.E,
                                 grid);
  if (m.total > 227 * 1024) return false;
  // one CTA per SM, all resident at once (the grid barriers wait for every CTA)
  if (!fused_resident(p, m.total)) return false;
  *smem = m.total;
  *rg = r;
  *rows_max = rmax;
  return true;
}

namespace {
template <int MAXT, bool ROUTE, int LPR>
cudaError_t launch_fused_t(const DecodeParams& p, const cudaLaunchConfig_t& cfg, size_t smem) {
  const cudaError_t e = ensure_smem_attr(
      reinterpret_cast<const void*>(decode_fused_kernel<MAXT, ROUTE, LPR>), smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel<MAXT, ROUTE, LPR>, p);
}
template <bool ROUTE, int LPR>
cudaError_t launch_fused_tt(const DecodeParams& p, const cudaLaunchConfig_t& cfg, size_t smem) {
  switch (p.T) {
    case 1: return launch_fused_t<1, ROUTE, LPR>(p, cfg, smem);
    case 2: return launch_fused_t<2, ROUTE, LPR>(p, cfg, smem);
    default: return launch_fused_t<4, ROUTE, LPR>(p, cfg, smem);
  }
}
}  // namespace

cudaError_t launch_decode_fused(const DecodeParams& p, int num_sms, size_t smem, bool pdl,
                                cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kFTP);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  // the record interleave width is 8 for every width of 512 and more; the
  // kernels built for it use immediate offsets, the others compute them
  const bool w8 = lanes_per_row(p.H) == 8 && lanes_per_row(p.F) == 8 &&
                  (!p.n_shared || lanes_per_row(p.Fs) == 8);
  if (p.route)
    return w8 ? launch_fused_tt<true, 8>(p, cfg, smem) : launch_fused_tt<true, 0>(p, cfg, smem);
  return w8 ? launch_fused_tt<false, 8>(p, cfg, smem) : launch_fused_tt<false, 0>(p, cfg, smem);
}

}  // namespace moe
