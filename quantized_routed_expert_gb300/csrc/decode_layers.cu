// Several decode layers in one persistent launch (moe_iq4nl_decode_layers).
//
// The PocketLLM "Xing4.0-29B-A4B" page (Performance) finds its decode step
// bound by launches: 11,536 kernel launches a step cost 178 ms of host
// submission against 46.5 ms of device work. Here one launch runs the MoE
// layers of a whole step: one CTA per SM walks the layers in order, each
// layer being route + gate/up + down + combine as in the single-layer fused
// kernel (same units, same per-row code, same fixed summation order), with
// grid-wide exchanges between the phases instead of kernel boundaries:
//   - router scores: each CTA scores its slice of the experts and publishes
//     each score together with a tag (the call's epoch plus the layer) in one
//     64-bit word; the warp that takes a token's top-k reads the words until
//     every tag is the current one, so the exchange needs no separate counter;
//   - h: a counter per call, raised by each CTA once its h rows are written;
//   - y: a second counter, raised once a CTA's rows of y are written; layer
//     l + 1 starts after every CTA raised it for layer l. With chaining, layer
//     l + 1's input is bf16(y_l) (round to nearest even); without, it is the
//     caller's x of that layer. Both orders are the same, so the layers run
//     one after another either way.
// Weights that do not depend on the routes are fetched a layer ahead: the
// next layer's router rows of this CTA once its scores are taken, and the
// next layer's shared-expert rows as soon as a warp's slots free up in the
// down phase.
//
// Fifteen warps compute; the sixteenth only issues the weight copies. A bulk
// copy is taken in by the copy engine no faster than memory delivers, so the
// thread that issues it stalls meanwhile: with every computing warp issuing
// its own rows, the issuing took as many cycles as the dot products. The
// copy warp's lane w keeps computing warp w's two slots filled in the warp's
// unit order, each slot once the warp has released its previous unit (an
// mbarrier arrival) and its rows are known (the layer's route table built).
//
// Every wait is bounded: waits on other CTAs by the host-set barrier limit,
// waits on this CTA's own copies by the fixed 2 s limit (after a timeout each
// warp still drains its copies before the kernel ends).
#include "common.cuh"
#include "decode.cuh"
#include "decode_common.cuh"
#include "route.cuh"

#include <mutex>

namespace moe {

// Phase stamps (builds with MOE_PROFILE only): thread 0 of each CTA records
// %globaltimer at each phase boundary of the first kProfLayers layers, read
// back with moe_profile_stamps. The product build has none of this.
#ifdef MOE_PROFILE
constexpr int kProfCtas = 256, kProfLayers = 64, kProfPhases = 12;
__device__ uint64_t g_prof[kProfCtas * kProfLayers * kProfPhases];
// per warp: [0] routed gate/up first unit landed, [1] routed gate/up done,
// [2] down unit landed, [3] down done, [4] top-k and weights done (token
// warps) or the shared expert's rows done (the other warps),
// [5] every score seen, [6] selection done, [7] route table built (warp 0),
// [8..11] clock64 cycles of the routed gate/up loop: waiting, computing,
// issuing copies, the whole loop; [12] its units; [13..15] the down loop's
// waiting, computing, issuing cycles; [16] / [17] written by the copy warp's
// lane w: the layer's route table seen, its first routed unit issued;
// [18] / [19] / [20] clock64 cycles of a token warp's top-k (polling
// included), of finishing its routes, of warp 0's route table build and of
// its per-warp plans for the copy warp
constexpr int kProfW = 22;
__device__ uint64_t g_profw[kProfCtas * kProfLayers * 16 * kProfW];
#define MOE_WSTAMP(l, k)                                                                      \
  do {                                                                                        \
    if ((threadIdx.x & 31) == 0 && (l) < kProfLayers && blockIdx.x < kProfCtas)              \
      g_profw[(((size_t)blockIdx.x * kProfLayers + (l)) * 16 + (threadIdx.x >> 5)) * kProfW + \
              (k)] = global_timer_ns();                                                       \
  } while (0)
#define MOE_WPUT(l, k, v)                                                                     \
  do {                                                                                        \
    if ((threadIdx.x & 31) == 0 && (l) < kProfLayers && blockIdx.x < kProfCtas)              \
      g_profw[(((size_t)blockIdx.x * kProfLayers + (l)) * 16 + (threadIdx.x >> 5)) * kProfW + \
              (k)] = (v);                                                                     \
  } while (0)
#define MOE_PSTAMP(l, w, k)                                                                   \
  do {                                                                                        \
    if ((l) < kProfLayers && blockIdx.x < kProfCtas)                                          \
      g_profw[(((size_t)blockIdx.x * kProfLayers + (l)) * 16 + (w)) * kProfW + (k)] =         \
          global_timer_ns();                                                                  \
  } while (0)
#define MOE_STAMP(l, ph)                                                                     \
  do {                                                                                       \
    if (threadIdx.x == 0 && (l) < kProfLayers && blockIdx.x < kProfCtas)                      \
      g_prof[((size_t)blockIdx.x * kProfLayers + (l)) * kProfPhases + (ph)] = global_timer_ns(); \
  } while (0)
#else
#define MOE_STAMP(l, ph) \
  do {                   \
  } while (0)
#define MOE_WSTAMP(l, k) \
  do {                   \
  } while (0)
#define MOE_WPUT(l, k, v) \
  do {                    \
  } while (0)
#define MOE_PSTAMP(l, w, k) \
  do {                      \
  } while (0)
#endif

constexpr int kLW = 15;            // computing warps per CTA (warp 15 issues the copies)
constexpr int kLT = kLW * 32;      // computing threads per CTA
constexpr int kLTP = kLT + 32;     // threads per CTA: the computing warps and the copy warp
constexpr int kLSlots = 2;         // bulk-copy slots per computing warp
constexpr int kLBar = 2;           // named barrier of the computing warps

// Sync words of this kernel in the decode workspace (after the fused
// kernel's four): h arrivals, y arrivals, departures, epoch base.
constexpr int kSyncH = 4, kSyncY = 5, kSyncOut = 6, kSyncEpoch = 7;

struct LayersSmem {
  size_t xq, slots, bars, ebars, recs, part, rwr, rx, rpart, rprob, rids, rw, rcand, stage,
      stage_bytes, total, slot_bytes;
};

// Experts whose scores CTA c takes: a balanced split of E over the grid.
__host__ __device__ inline int lr_e0(int E, int c, int G) { return (int)((long long)E * c / G); }

__host__ __device__ inline LayersSmem layers_smem(int H, int F, int Fs, int ns, int T, int k,
                                                  int rows_max, int rg, int E, int G) {
  LayersSmem m;
  const size_t rbH = (size_t)(H / 32) * kBlockB;
  size_t rbK = (size_t)(F / 32) * kBlockB;
  if (ns) {
    const size_t rbs = (size_t)(Fs / 32) * kBlockB;
    rbK = rbK > rbs ? rbK : rbs;
  }
  const size_t gu = 2 * rbH, dn = (size_t)rg * rbK;
  m.slot_bytes = align_up_dev(gu > dn ? gu : dn, 128);
  m.xq = align_up_dev(sizeof(RouteTable), 128);
  m.slots = align_up_dev(m.xq + (size_t)T * dqvec_words(H) * 4, 128);
  m.bars = m.slots + (size_t)kLW * kLSlots * m.slot_bytes;
  // the slots' "free" barriers, then the copy warp's words: the layer whose
  // routes are known, the stop flag, the units issued per computing warp, the
  // routed and down units per computing warp and the first routed row
  m.ebars = align_up_dev(m.bars + (size_t)(kLW * kLSlots + 4) * 8, 16);
  m.recs = align_up_dev(m.ebars + (size_t)kLW * kLSlots * 8 + 8 + (size_t)kLW * 4 +
                            (size_t)kLW * 8 + 4, 128);
  const size_t recs =
      (size_t)T * k * dqvec_words(F) * 4 + (ns ? (size_t)T * dqvec_words(Fs) * 4 : 0);
  m.part = align_up_dev(m.recs + recs, 16);
  size_t end = m.part + (size_t)(T * k + (ns ? T : 0)) * rows_max * 4;
  // router scratch, overlaying the records and partials: a layer's router
  // rows land there after the previous layer's combine, and the records and
  // partials of a layer are written only after its routes are known
  const int epc = (E + G - 1) / G + 1;               // most experts any CTA scores
  const int E32 = (E + 31) & ~31;
  m.rwr = m.recs;
  m.rx = align_up_dev(m.rwr + (size_t)epc * H * 2, 128);
  m.rpart = align_up_dev(m.rx + (size_t)T * H * 2, 16);
  m.rprob = align_up_dev(m.rpart + (size_t)epc * 16 * T * 4, 16);
  m.rids = align_up_dev(m.rprob + (size_t)T * E32 * 4, 16);
  m.rw = align_up_dev(m.rids + (size_t)T * k * 4, 16);
  m.rcand = align_up_dev(m.rw + (size_t)T * k * 4, 16);
  const size_t rend = m.rcand + (size_t)kLW * k * 8;
  end = end > rend ? end : rend;
  // stage every h row of a layer in shared memory when it fits
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

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Fetch bytes (a multiple of 16, 16-byte aligned) from HBM into L2 only.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// CTA barriers of the computing warps only (the copy warp never joins them).
__device__ __forceinline__ void csync() { asm volatile("bar.sync %0, %1;" ::"n"(kLBar), "n"(kLT) : "memory"); }
__device__ __forceinline__ bool csync_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "n"(kLBar), "n"(kLT)
      : "memory");
  return r != 0;
}

// What a warp needs to issue the copies of its units. Its sequence: per layer
// its shared gate/up rows, its routed gate/up rows, its down groups; then the
// next layer's shared gate/up rows (known before that layer's routes).
struct LUnitPlan {
  uint8_t* myslots;
  size_t slot_bytes;
  uint64_t* mybar;
  uint64_t pol;
  int warp, layer, ub, n_sh, n_rt, rr_a, n_dn, sh_a, sh_w, sh_nw, ngroups, nrows_cta, dn_a, rg;
};

// Issue unit j of a warp's sequence into slot j % kLSlots (one lane calls).
__device__ __noinline__ void issue_unit_layers(const DecodeParams& p, const LayerTable& lt,
                                               const RouteTable& rt, const LUnitPlan& u, int j) {
  const int s = j % kLSlots;
  uint8_t* dst = u.myslots + (size_t)s * u.slot_bytes;
  uint64_t* bar = &u.mybar[s];
  const uint32_t rbH = (uint32_t)(p.H / 32 * kBlockB);
  int lj = j - u.ub, l = u.layer;
  const int n_tot = u.n_sh + u.n_rt + u.n_dn;
  if (lj >= n_tot) {                   // the next layer's shared rows
    lj -= n_tot;
    ++l;
  }
  const LayerPtrs& W = lt.layer[l];
  if (lj < u.n_sh + u.n_rt) {
    const uint8_t *g, *up;
    if (lj < u.n_sh) {
      const size_t f = (size_t)(u.sh_a + u.sh_w + u.sh_nw * lj);
      g = W.sh_gate + f * rbH;
      up = W.sh_up + f * rbH;
    } else {
      const int r = u.rr_a + u.warp + kLW * (lj - u.n_sh);
      const int sl = r / p.F, f = r - sl * p.F;
      const size_t row = (size_t)rt.slot_expert[sl] * p.F + f;
      g = W.gate + row * rbH;
      up = W.up + row * rbH;
    }
    mbar_arrive_expect_tx(bar, 2 * rbH);
    bulk_g2s_hint(dst, g, rbH, bar, u.pol);
    bulk_g2s_hint(dst + rbH, up, rbH, bar, u.pol);
  } else {
    const int un = u.warp + kLW * (lj - u.n_sh - u.n_rt);
    const int su = un / u.ngroups, gi = un - su * u.ngroups;
    const bool sh = p.n_shared && su == 0;
    const int sl = su - p.n_shared;
    const int K = sh ? p.Fs : p.F;
    const int rbK = K / 32 * kBlockB;
    const int r0 = gi * u.rg;
    const int nr = u.nrows_cta - r0 < u.rg ? u.nrows_cta - r0 : u.rg;
    const uint8_t* src = sh ? W.sh_down + (size_t)(u.dn_a + r0) * rbK
                            : W.down + ((size_t)rt.slot_expert[sl] * p.H + u.dn_a + r0) * rbK;
    mbar_arrive_expect_tx(bar, (uint32_t)(nr * rbK));
    bulk_g2s_hint(dst, src, (uint32_t)(nr * rbK), bar, u.pol);
  }
}

// Raise a grid counter (thread 0, after a CTA barrier that follows the CTA's
// writes): a release fence at GPU scope, then a relaxed add.
__device__ __forceinline__ void grid_arrive(uint32_t* ctr) {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
}
// Wait (thread 0) until a grid counter reaches target, for at most wait_ns;
// a timeout is recorded in *status and in the CTA's flag *gave_up.
__device__ __forceinline__ void grid_wait(const uint32_t* ctr, uint32_t target, uint64_t wait_ns,
                                          uint32_t* status, volatile uint32_t* gave_up) {
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_u32(ctr) < target) {
    if (global_timer_ns() - t0 >= wait_ns) {
      if (status) atomicOr(status, MOE_STATUS_TIMEOUT);
      *gave_up = 1u;
      break;
    }
    __nanosleep(32);
  }
}

// A token's activations (bf16 from the caller, or fp32 y of the previous
// layer rounded to bf16) into the router's bf16 copy and the quantised
// records, four lanes per 32-value block, every thread of the CTA.
template <bool FROM_Y>
__device__ __forceinline__ void load_x_layer(const uint16_t* __restrict__ xb,
                                             const float* __restrict__ yf, int T, int H,
                                             uint16_t* rx, uint32_t* xq, int xq_words) {
  const int nb = H / 32;
  const int n = T * nb * 4;
#pragma unroll 1
  for (int i0 = threadIdx.x & ~31; i0 < n; i0 += kLT) {
    const int i = i0 + (threadIdx.x & 31);
    const bool ok = i < n;
    const int blk = ok ? i >> 2 : 0;
    const int t = blk / nb, b = blk - t * nb;
    const size_t off = (size_t)t * H + b * 32 + (i & 3) * 8;
    uint32_t r[4] = {0u, 0u, 0u, 0u};
    if (ok) {
      if (FROM_Y) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(yf + off));
        const float4 c = __ldcg(reinterpret_cast<const float4*>(yf + off) + 1);
        const float f[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          r[j] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f[2 * j])) |
                 ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f[2 * j + 1])) << 16);
      } else {
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(xb + off));
        r[0] = v.x; r[1] = v.y; r[2] = v.z; r[3] = v.w;
      }
      *reinterpret_cast<uint4*>(rx + off) = make_uint4(r[0], r[1], r[2], r[3]);
    }
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(r[j] << 16);
      v[2 * j + 1] = __uint_as_float(r[j] & 0xFFFF0000u);
    }
    quant_group8(v, ok, b, H, xq + (size_t)t * xq_words);
  }
}

// A token's tagged scores of all E experts, polled by one warp until every
// tag is the current one (or the wait gives up). Each polling round issues
// every lane's loads before it checks any tag. Lane l gets experts l + 32 i.
template <int NPL>
__device__ __forceinline__ void poll_scores(const uint64_t* sc, uint32_t want, int E,
                                            uint64_t (&v)[NPL], uint64_t wait_ns,
                                            uint32_t* status, volatile uint32_t* gave_up) {
  const int lane = threadIdx.x & 31;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = ld_relaxed_u64(sc + (e < E ? e : E - 1));
    }
    bool all = true;
#pragma unroll
    for (int i = 0; i < NPL; ++i) all = all && (uint32_t)(v[i] >> 32) == want;
    if (__all_sync(0xFFFFFFFFu, all)) break;
    // the give-up decision is the warp's (lane 0's clock), so every lane leaves together
    if (__shfl_sync(0xFFFFFFFFu, global_timer_ns() - t0 >= wait_ns ? 1 : 0, 0)) {
      if (lane == 0) {
        if (status) atomicOr(status, MOE_STATUS_TIMEOUT);
        *gave_up = 1u;
      }
      break;
    }
    // every CTA polls the same few lines: back off between rounds
    __nanosleep(100);
  }
}

// One token's top-k by one warp, from the tagged scores of all E experts.
// The bias is read before the wait, so that its latency overlaps it.
template <int NPL>
__device__ __forceinline__ void layer_topk(const uint64_t* sc, uint32_t want, int E, int k,
                                           const float* bias, float* prob, int& id, float& wv,
                                           uint64_t wait_ns, uint32_t* status,
                                           volatile uint32_t* gave_up, int l) {
  const int lane = threadIdx.x & 31;
  float bv[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    bv[i] = (bias && e < E) ? __ldg(bias + e) : 0.0f;
  }
  uint64_t v[NPL];
  poll_scores<NPL>(sc, want, E, v, wait_ns, status, gave_up);
  MOE_WSTAMP(l, 5);
  float kv[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    kv[i] = -INFINITY;
    if (e < E) {
      const float pr = 1.0f / (1.0f + expf(-__uint_as_float((uint32_t)v[i])));
      prob[e] = pr;
      kv[i] = pr + bv[i];
    }
  }
  id = warp_topk_regs<NPL>(kv, k);
  MOE_WSTAMP(l, 6);
  __syncwarp();
  wv = warp_renorm(lane < k ? prob[id] : 0.0f, k);
}

// The selection spread over the warps of a CTA (more than 64 experts): each
// warp takes a range of one token's experts, turns their scores into sigmoids
// and keys, and picks its own k best in the order of the one-warp selection
// (largest key first, ties to the lower expert). Lane 0 records each pick as
// (key bits << 32) | expert; a pick made after the range ran out of keys has
// key bits 0. sc_prob holds the token's scores and gets its sigmoids.
template <int NPL>
__device__ __forceinline__ void topk_part(float* sc_prob, const float (&bsel)[8], int base, int E,
                                          int k, uint64_t* cand) {
  const int lane = threadIdx.x & 31;
  uint32_t v[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = base + lane + 32 * i;
    v[i] = 0u;
    if (e < E) {
      const float pr = 1.0f / (1.0f + expf(-sc_prob[e]));
      sc_prob[e] = pr;
      const float kv = pr + bsel[i];
      v[i] = kv > -INFINITY ? ordered_key_bits(kv) : 0u;
    }
  }
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    uint32_t m[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) m[i] = v[i];
#pragma unroll
    for (int st = 1; st < NPL; st *= 2)
#pragma unroll
      for (int i = 0; i + st < NPL; i += 2 * st) m[i] = m[i] > m[i + st] ? m[i] : m[i + st];
    const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, m[0]);
    uint32_t hit = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) hit |= (v[i] == mx ? 1u : 0u) << i;
    const uint32_t c = hit ? (uint32_t)(lane + 32 * (__ffs(hit) - 1)) : 0xFFFFFFFFu;
    const uint32_t bi = __reduce_min_sync(0xFFFFFFFFu, c);
    if (lane == 0) cand[j] = ((uint64_t)mx << 32) | (uint32_t)(base + (int)bi);
    const bool mine = (int)(bi & 31u) == lane;
    const int ri = (int)(bi >> 5);
#pragma unroll
    for (int i = 0; i < NPL; ++i) v[i] = (mine && i == ri) ? 0u : v[i];
  }
}
// The token's k experts from the n candidates of its warps (stored by
// ascending expert range, so a lower position among equal keys is a lower
// expert): lane j < k gets the j-th. A choice made once no key is left is
// expert 0, as in the one-warp selection.
__device__ __forceinline__ int topk_merge(const uint64_t* cand, int n, int k) {
  const int lane = threadIdx.x & 31;
  uint32_t v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int q = lane + 32 * i;
    v[i] = q < n ? (uint32_t)(cand[q] >> 32) : 0u;
  }
  const int pos = warp_topk_bits<8>(v, k);
  const uint64_t c = cand[lane < k ? pos : 0];
  return (uint32_t)(c >> 32) == 0u ? 0 : (int)(uint32_t)c;
}

template <int MAXT, int LPR>
__global__ void __launch_bounds__(kLTP, 1)
    decode_layers_kernel(const __grid_constant__ DecodeParams p,
                         const __grid_constant__ LayerTable lt) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = p.H, G = gridDim.x, cta = blockIdx.x;
  const int rows_max = p.dn_rows_max;
  const int RG = p.fz_rg;
  const LayersSmem S =
      layers_smem(H, p.F, p.Fs, p.n_shared, p.T, p.k, rows_max, RG, p.E, G);
  RouteTable& rt = *reinterpret_cast<RouteTable*>(smem);
  uint32_t* xq = reinterpret_cast<uint32_t*>(smem + S.xq);
  uint8_t* slots = smem + S.slots;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S.bars);
  uint64_t* recs_bar = bars + kLW * kLSlots;     // staged h of a layer
  uint64_t* rwr_bar = recs_bar + 1;               // router rows of a layer
  uint32_t* epoch_s = reinterpret_cast<uint32_t*>(rwr_bar + 1);
  volatile uint32_t* gave_up = epoch_s + 1;       // this CTA saw a wait time out
  uint64_t* ebars = reinterpret_cast<uint64_t*>(smem + S.ebars);     // slot freed
  volatile uint32_t* routes_known = reinterpret_cast<uint32_t*>(ebars + kLW * kLSlots);
  volatile uint32_t* stop = routes_known + 1;
  volatile uint32_t* final_iss = stop + 1;       // units the copy warp issued, per warp
  int* plan_s = const_cast<int*>(reinterpret_cast<volatile int*>(final_iss + kLW));  // [kLW][2], rr_a
  uint32_t* recs = reinterpret_cast<uint32_t*>(smem + S.recs);
  float* part = reinterpret_cast<float*>(smem + S.part);
  uint16_t* rx = reinterpret_cast<uint16_t*>(smem + S.rx);
  float* rpart = reinterpret_cast<float*>(smem + S.rpart);
  float* rprob = reinterpret_cast<float*>(smem + S.rprob);
  int32_t* rids = reinterpret_cast<int32_t*>(smem + S.rids);
  float* rw = reinterpret_cast<float*>(smem + S.rw);
  uint64_t* rcand = reinterpret_cast<uint64_t*>(smem + S.rcand);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int xq_words = dqvec_words(H);
  const int rbH = H / 32 * kBlockB;
  const int T = p.T, k = p.k, E = p.E, Lyr = p.L;
  const int E32 = (E + 31) & ~31;

  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int i = 0; i < kLW * kLSlots + 2; ++i) mbar_init(&bars[i], 1);
#pragma unroll 1
    for (int i = 0; i < kLW * kLSlots; ++i) mbar_init(&ebars[i], 1);
    mbar_fence_init();
    *gave_up = 0u;
    *routes_known = 0u;
    *stop = 0u;
  }
  __syncthreads();

  // ---- this CTA's static share of every layer
  const RowRange shr = p.n_shared ? split_rows(p.Fs, 1, cta, G) : RowRange{0, 0};
  const RowRange dn = split_rows(H, 1, cta, G);
  const int nrows_cta = dn.b - dn.a;
  const int ngroups = (nrows_cta + RG - 1) / RG;
  // units of computing warp w among the rows [a, b) of a layer, dealt round-robin
  auto count_w = [&](int w, int a, int b) { return a + w < b ? (b - a - w + kLW - 1) / kLW : 0; };
  auto count = [&](int a, int b) { return count_w(warp, a, b); };
  // The shared expert's rows go to the warps that do not take a token's
  // top-k (warps T..kLW-1): they compute them while the scores are exchanged.
  // Warps on a scheduler (warp index mod 4) without a token warp come first,
  // so that the top-k and route table, on the path to the routed copies, do
  // not share their scheduler with these rows.
  const int sh_nw = kLW - T;
  auto sh_rank = [&](int w) {     // w's place among the shared-row warps, -1 if none
    if (w < T) return -1;
    const bool a = (w & 3) >= T;
    int r = 0;
#pragma unroll 1
    for (int v = T; v < kLW; ++v) {
      const bool av = (v & 3) >= T;
      if (a ? (av && v < w) : (av || v < w)) ++r;
    }
    return r;
  };
  auto n_sh_of = [&](int w) {
    const int sw = sh_rank(w);
    return (sw >= 0 && shr.a + sw < shr.b) ? (shr.b - shr.a - sw + sh_nw - 1) / sh_nw : 0;
  };
  const int sh_w = sh_rank(warp);
  const int n_sh = n_sh_of(warp);
  const int re0 = lr_e0(E, cta, G), re1 = lr_e0(E, cta + 1, G);
  const int ne = re1 - re0;
  const uint64_t pol = l2_evict_first_policy();

  // The unit sequence of computing warp w (per layer: its shared gate/up
  // rows, routed gate/up rows, down groups), before the layer's routes.
  auto plan_of = [&](int w) {
    LUnitPlan u;
    u.myslots = slots + (size_t)w * kLSlots * S.slot_bytes;
    u.slot_bytes = S.slot_bytes;
    u.mybar = bars + w * kLSlots;
    u.pol = pol;
    u.warp = w;
    u.layer = 0;
    u.ub = 0;
    u.n_sh = n_sh_of(w);
    u.n_rt = u.rr_a = u.n_dn = 0;
    u.sh_a = shr.a;
    u.sh_w = sh_rank(w);
    u.sh_nw = sh_nw;
    u.ngroups = ngroups;
    u.nrows_cta = nrows_cta;
    u.dn_a = dn.a;
    u.rg = RG;
    return u;
  };
  // ... and its routed and down units once the route table is built
  auto plan_slots = [&](LUnitPlan& u, int n_slots) {
    // split_rows(n_slots * F, 1, cta, G) in 32-bit arithmetic (n_slots * F * G
    // < 2^32): this is on the path from the route table to the first copy
    const uint32_t tot = (uint32_t)(n_slots * p.F);
    const RowRange rr{(int)(tot * (uint32_t)cta / (uint32_t)G),
                      (int)(tot * (uint32_t)(cta + 1) / (uint32_t)G)};
    u.n_rt = count_w(u.warp, rr.a, rr.b);
    u.rr_a = rr.a;
    const int n_dn_units = (n_slots + p.n_shared) * ngroups;
    u.n_dn = u.warp < n_dn_units ? (n_dn_units - u.warp + kLW - 1) / kLW : 0;
  };
  auto plan_routes = [&](LUnitPlan& u) { plan_slots(u, rt.n_slots); };
  // One token: the in-kernel selection gives k distinct experts except in the
  // degenerate case of NaN or -inf keys, so lane w of warp 0 keeps warp w's
  // plan for k slots from the start.
  int k_nrt = 0, k_ndn = 0, k_rra = 0;
  if (MAXT == 1 && warp == 0 && lane < kLW) {
    LUnitPlan pl;
    pl.warp = lane;
    plan_slots(pl, k);
    k_nrt = pl.n_rt;
    k_ndn = pl.n_dn;
    k_rra = pl.rr_a;
  }

  if (warp == kLW) {
    // ---- the copy warp: lane w < kLW issues computing warp w's units in
    // order, each once its slot is free (the warp's release of the unit two
    // back) and its rows are known (shared rows always, routed and down rows
    // once the layer's route table is built). The computing warps never
    // issue a weight copy, so they never stall while the copy engine takes
    // one in.
    const int w = lane;
    const bool mine = w < kLW;
    LUnitPlan u = plan_of(mine ? w : 0);
    int iss = 0, lim = mine ? u.n_sh : 0, lp = 0;
    bool known = false;
    const uint64_t idle_ns = 2 * kWaitLimitNs + p.wait_ns;
    uint64_t t_act = global_timer_ns();
#pragma unroll 1
    while (lp < Lyr) {
      bool any = false;
#pragma unroll 1
      for (;;) {
        bool can = mine && iss < lim;
        if (can && iss >= kLSlots)
          can = mbar_test(&ebars[w * kLSlots + iss % kLSlots],
                          (uint32_t)(((iss / kLSlots) + 1) & 1));
        if (!__any_sync(0xFFFFFFFFu, can)) break;
        if (can) {
#ifdef MOE_PROFILE
          if (known && iss == u.ub + u.n_sh) MOE_PSTAMP(lp, w, 17);
#endif
          issue_unit_layers(p, lt, rt, u, iss);
          ++iss;
        }
        any = true;
      }
      if (!known) {
        if (*routes_known >= (uint32_t)(lp + 1)) {     // layer lp's route table is built
          __threadfence_block();
          if (mine) MOE_PSTAMP(lp, w, 16);
          if (mine) {
            u.n_rt = plan_s[2 * w];
            u.n_dn = plan_s[2 * w + 1];
            u.rr_a = plan_s[2 * kLW];
            lim = u.ub + u.n_sh + u.n_rt + u.n_dn + (lp + 1 < Lyr ? u.n_sh : 0);
          }
          known = true;
          any = true;
        }
      } else if (__all_sync(0xFFFFFFFFu, !mine || iss == lim)) {
        // every unit of layer lp issued (and the next layer's shared rows)
        u.ub += u.n_sh + u.n_rt + u.n_dn;
        u.layer = lp + 1;
        u.n_rt = u.rr_a = u.n_dn = 0;
        ++lp;
        known = false;
        any = true;
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
    if (mine) final_iss[w] = (uint32_t)iss;
    __syncthreads();     // the computing warps' final barrier
    return;
  }

  LUnitPlan up = plan_of(warp);
  int consumed = 0;
  bool ok = true;
  int rwr_issued = -1, rwr_landed = -1;     // layers whose router rows were fetched / waited
  uint64_t wait_ns = p.wait_ns;             // 0 once this CTA saw a timeout

  auto wait_unit = [&](int j) {     // the whole warp; the result is the warp's
    return __all_sync(0xFFFFFFFFu,
                      mbar_wait(&up.mybar[j % kLSlots], (uint32_t)((j / kLSlots) & 1), p.status));
  };
  auto release_unit = [&](int j) {  // the warp is done with unit j's slot
    __syncwarp();
    if (lane == 0) mbar_arrive(&ebars[warp * kLSlots + j % kLSlots]);
  };
  auto issue_router_rows = [&](int l) {     // thread 0
    if (ne > 0) {
      const uint32_t bytes = (uint32_t)(ne * H * 2);
      mbar_arrive_expect_tx(rwr_bar, bytes);
      bulk_g2s_hint(smem + S.rwr, lt.layer[l].Wr + (size_t)re0 * H, bytes, rwr_bar, pol);
    }
  };

  // Constant weights of the first layer stream while the previous kernel on
  // the stream finishes.
  if (threadIdx.x == 0) issue_router_rows(0);
  rwr_issued = 0;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) *epoch_s = ld_acquire_u32(&p.sync[kSyncEpoch]);
  csync();
  const uint32_t epoch = *epoch_s;

#pragma unroll 1
  for (int l = 0; l < Lyr; ++l) {
    const LayerPtrs& W = lt.layer[l];
    float* yl = p.y + (size_t)l * T * H;
    MOE_STAMP(l, 0);
    // the next layer's router rows and shared down rows of this CTA into L2,
    // while this layer waits on its exchanges
    if (threadIdx.x == 0 && l + 1 < Lyr) {
      const LayerPtrs& Wn = lt.layer[l + 1];
      if (ne > 0) prefetch_l2(Wn.Wr + (size_t)re0 * H, (uint32_t)(ne * H * 2));
      if (p.n_shared && nrows_cta > 0) {
        const size_t rbS = (size_t)(p.Fs / 32) * kBlockB;
        prefetch_l2(Wn.sh_down + (size_t)dn.a * rbS, (uint32_t)(nrows_cta * rbS));
      }
    }
    // ---- this layer's input, after every CTA finished the previous layer
    if (l > 0) {
      if (threadIdx.x == 0)
        grid_wait(&p.sync[kSyncY], (uint32_t)(G * l), wait_ns, p.status, gave_up);
      csync();
      if (*gave_up) wait_ns = 0;
    }
    MOE_STAMP(l, 1);
    if (p.chained && l > 0)
      load_x_layer<true>(nullptr, p.y + (size_t)(l - 1) * T * H, T, H, rx, xq, xq_words);
    else
      load_x_layer<false>(p.x + (p.chained ? (size_t)0 : (size_t)l * T * H), nullptr, T, H, rx,
                          xq, xq_words);
    csync();
    MOE_STAMP(l, 2);

    // ---- scores of this CTA's experts: 16 chunks of H per expert, one warp
    // per (expert, chunk), chunk partials summed in a fixed order
    uint64_t* tsc = p.tscores + (size_t)(l & 1) * T * E;
    if (ne > 0) {
      const bool landed = csync_and(mbar_wait(rwr_bar, (uint32_t)(l & 1), p.status));
      rwr_landed = l;
      MOE_STAMP(l, 10);
      ok = ok && landed;
      const uint16_t* wr_s = reinterpret_cast<const uint16_t*>(smem + S.rwr);
      const int hc = H / 16;
#pragma unroll 1
      for (int it = warp; it < ne * 16; it += kLW) {
        const int el = it >> 4, c = it & 15;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int g8 = lane; g8 < hc / 8; g8 += 32) {
          const uint4 wv = reinterpret_cast<const uint4*>(wr_s + (size_t)el * H + c * hc)[g8];
          const uint32_t wr[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (t < T) {
              const uint4 xv = reinterpret_cast<const uint4*>(rx + (size_t)t * H + c * hc)[g8];
              const uint32_t xr[4] = {xv.x, xv.y, xv.z, xv.w};
              float a = acc[t];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                a = fmaf(__uint_as_float(wr[i] << 16), __uint_as_float(xr[i] << 16), a);
                a = fmaf(__uint_as_float(wr[i] & 0xFFFF0000u),
                         __uint_as_float(xr[i] & 0xFFFF0000u), a);
              }
              acc[t] = a;
            }
          }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (t < T)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], o);
        if (lane == 0) {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (t < T) rpart[(el * 16 + c) * T + t] = acc[t];
        }
      }
      csync();
      MOE_STAMP(l, 11);
#pragma unroll 1
      for (int i = threadIdx.x; i < ne * T; i += kLT) {
        const int el = i / T, t = i - el * T;
        float sc = 0.f;
        for (int c = 0; c < 16; ++c) sc += rpart[(el * 16 + c) * T + t];
        st_relaxed_u64(tsc + (size_t)t * E + re0 + el,
                       ((uint64_t)(epoch + (uint32_t)l + 1u) << 32) | __float_as_uint(sc));
      }
    }
    csync();
    MOE_STAMP(l, 3);

    // ---- top-k: warp t takes token t, in every CTA; meanwhile the other
    // warps compute the shared expert's rows (known before the routes). With
    // more than 64 experts warp t only gathers the scores, and the selection
    // is spread over all warps: kLW / T warps per token.
    const bool split_sel = E > 64;
    const int Wt = kLW / T, tt = warp / Wt;
    // experts per lane of a selecting warp: E <= 512 <= 256 Wt (Wt >= 3)
    const int nsel = E <= Wt * 32 ? 1 : (E <= Wt * 64 ? 2 : (E <= Wt * 128 ? 4 : 8));
    const int sbase = (warp - tt * Wt) * 32 * nsel;
    float bsel[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = sbase + lane + 32 * i;
      bsel[i] = (split_sel && W.bias && tt < T && i < nsel && e < E) ? __ldg(W.bias + e) : 0.0f;
    }
    if (warp >= T) {
#pragma unroll 1
      for (int j = up.ub; ok && j < up.ub + n_sh; ++j) {
        ok = wait_unit(j);
        if (!ok) break;
        const uint8_t* d = up.myslots + (size_t)(j % kLSlots) * S.slot_bytes;
        const int f = shr.a + sh_w + sh_nw * (j - up.ub);
        gateup_unit_t<1, LPR>(p, rt, d, d + rbH, -1, f, xq, xq_words);
        release_unit(j);
        ++consumed;
      }
      MOE_WSTAMP(l, 4);
    }
    auto finish_routes = [&](int id, float wv) {     // the token warps
      if (lane < k) {
        rids[warp * k + lane] = id;
        rw[warp * k + lane] = wv;
        if (cta == 0) {
          p.ids_out[((size_t)l * T + warp) * k + lane] = id;
          p.w_out[((size_t)l * T + warp) * k + lane] = wv;
        }
      }
      if (T > 1) bar_sync_n(1, T * 32);     // the token warps only
      if (MAXT == 1 && warp == 0) {
        // One token, k distinct experts (the usual case): the slots are the
        // ids in ascending order and the plans are the ones kept above, so the
        // copy warp may start on the routed rows before the rest of the table
        // is built.
        const int e = lane < k ? id : 0x7FFFFFFF;
        int r = 0;
        bool dup = false;
#pragma unroll
        for (int q = 0; q < MOE_MAX_TOP_K; ++q) {
          const int eq = __shfl_sync(0xFFFFFFFFu, e, q);
          if (q < k) {
            r += (eq < e) ? 1 : 0;
            dup = dup || (eq == e && q != lane);
          }
        }
        if (!__any_sync(0xFFFFFFFFu, lane < k && dup)) {
          if (lane < k) rt.slot_expert[r] = e;
          if (lane < kLW) {
            plan_s[2 * lane] = k_nrt;
            plan_s[2 * lane + 1] = k_ndn;
            if (lane == 0) plan_s[2 * kLW] = k_rra;
          }
          __syncwarp();
          if (lane == 0) {
            __threadfence_block();
            *routes_known = (uint32_t)(l + 1);
          }
          build_route_table_warp(rt, rids, rw, k, E);    // the same slots, and the rest
          MOE_WSTAMP(l, 7);
          return;
        }
      }
      if (warp == 0) {
#ifdef MOE_PROFILE
        const long long c0 = clock64();
#endif
        build_route_table_warp(rt, rids, rw, T * k, E);
#ifdef MOE_PROFILE
        long long c1 = clock64();
        MOE_WPUT(l, 20, (uint64_t)(c1 - c0));

#endif
        // every computing warp's routed and down units, for the copy warp,
        // which may then issue this layer's routed rows
        if (lane < kLW) {
          LUnitPlan pl;
          pl.warp = lane;
          plan_routes(pl);
          plan_s[2 * lane] = pl.n_rt;
          plan_s[2 * lane + 1] = pl.n_dn;
          if (lane == 0) plan_s[2 * kLW] = pl.rr_a;
        }
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          *routes_known = (uint32_t)(l + 1);
        }
#ifdef MOE_PROFILE
        MOE_WPUT(l, 21, (uint64_t)(clock64() - c1));
#endif
        MOE_WSTAMP(l, 7);
      }
    };
    const uint32_t want = epoch + (uint32_t)l + 1u;
    if (!split_sel) {
      if (warp < T) {
        int id;
        float wv;
#ifdef MOE_PROFILE
        const long long q0 = clock64();
#endif
        layer_topk<2>(tsc + (size_t)warp * E, want, E, k, W.bias, rprob + (size_t)warp * E32, id,
                      wv, wait_ns, p.status, gave_up, l);
        MOE_WSTAMP(l, 4);
#ifdef MOE_PROFILE
        const long long q1 = clock64();
#endif
        finish_routes(id, wv);
#ifdef MOE_PROFILE
        MOE_WPUT(l, 18, (uint64_t)(q1 - q0));
        MOE_WPUT(l, 19, (uint64_t)(clock64() - q1));
#endif
      }
    } else {
      if (warp < T) {
        uint64_t v[16];
        poll_scores<16>(tsc + (size_t)warp * E, want, E, v, wait_ns, p.status, gave_up);
        MOE_WSTAMP(l, 5);
        float* sc_s = rprob + (size_t)warp * E32;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = lane + 32 * i;
          if (e < E) sc_s[e] = __uint_as_float((uint32_t)v[i]);
        }
      }
      csync();
      if (tt < T) {
        float* sc_s = rprob + (size_t)tt * E32;
        if (nsel == 1)
          topk_part<1>(sc_s, bsel, sbase, E, k, rcand + (size_t)warp * k);
        else if (nsel == 2)
          topk_part<2>(sc_s, bsel, sbase, E, k, rcand + (size_t)warp * k);
        else if (nsel == 4)
          topk_part<4>(sc_s, bsel, sbase, E, k, rcand + (size_t)warp * k);
        else
          topk_part<8>(sc_s, bsel, sbase, E, k, rcand + (size_t)warp * k);
      }
      csync();
      if (warp < T) {
        const int id = topk_merge(rcand + (size_t)warp * Wt * k, Wt * k, k);
        MOE_WSTAMP(l, 6);
        const float* prob = rprob + (size_t)warp * E32;
        const float wv = warp_renorm(lane < k ? prob[id] : 0.0f, k);
        MOE_WSTAMP(l, 4);
        finish_routes(id, wv);
      }
    }
    csync();
    MOE_STAMP(l, 4);
    if (*gave_up) wait_ns = 0;
#pragma unroll 1
    for (int i = threadIdx.x; i < (T * k + (p.n_shared ? T : 0)) * rows_max; i += kLT)
      part[i] = 0.0f;
    plan_routes(up);
    const int ub = up.ub, n_rt = up.n_rt, rr_a = up.rr_a;
    const int n_tot = n_sh + n_rt + up.n_dn;
#ifdef MOE_PROFILE
    long long pw = 0, pc = 0, pi = 0, pl = clock64();
#endif

    // ---- gate/up: the routed rows as they arrive (the shared expert's were
    // computed above)
#pragma unroll 1
    for (int j = ub + n_sh; ok && j < ub + n_sh + n_rt; ++j) {
#ifdef MOE_PROFILE
      long long c0 = clock64();
#endif
      ok = wait_unit(j);
      if (!ok) break;
#ifdef MOE_PROFILE
      long long c1 = clock64();
      pw += c1 - c0;
#endif
      if (j == ub + n_sh) MOE_WSTAMP(l, 0);
      const uint8_t* d = up.myslots + (size_t)(j % kLSlots) * S.slot_bytes;
      const int lj = j - ub;
      const int r = rr_a + warp + kLW * (lj - n_sh);
      const int sl = r / p.F, f = r - sl * p.F;
      if (MAXT == 1 || rt.slot_off[sl + 1] - rt.slot_off[sl] == 1)
        gateup_unit_t<1, LPR>(p, rt, d, d + rbH, sl, f, xq, xq_words);
      else
        gateup_unit_t<MAXT, LPR>(p, rt, d, d + rbH, sl, f, xq, xq_words);
      release_unit(j);
      ++consumed;
#ifdef MOE_PROFILE
      pc += clock64() - c1;
#endif
    }

    MOE_WSTAMP(l, 1);
#ifdef MOE_PROFILE
    MOE_WPUT(l, 8, (uint64_t)pw);
    MOE_WPUT(l, 9, (uint64_t)pc);
    MOE_WPUT(l, 10, (uint64_t)pi);
    MOE_WPUT(l, 11, (uint64_t)(clock64() - pl));
    MOE_WPUT(l, 12, (uint64_t)n_rt);
    pw = pc = pi = 0;
#endif
    // ---- h of this layer: every CTA's rows written
    csync();
    MOE_STAMP(l, 5);
    if (threadIdx.x == 0) {
      grid_arrive(&p.sync[kSyncH]);
      grid_wait(&p.sync[kSyncH], (uint32_t)(G * (l + 1)), wait_ns, p.status, gave_up);
    }
    csync();
    MOE_STAMP(l, 6);
    if (*gave_up) wait_ns = 0;
    if (S.stage_bytes) {
      float* stage = reinterpret_cast<float*>(smem + S.stage);
      if (threadIdx.x == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        fence_proxy_async_shared();
        const uint32_t rbF = (uint32_t)p.F * 4, rbS = (uint32_t)p.Fs * 4;
        const uint32_t total = rt.n_valid * rbF + (p.n_shared ? T * rbS : 0u);
        mbar_arrive_expect_tx(recs_bar, total);
        uint8_t* dst = reinterpret_cast<uint8_t*>(stage);
        for (int e = 0; e < rt.n_valid; ++e, dst += rbF)
          bulk_g2s(dst, p.h_r + (size_t)rt.list[e] * p.F, rbF, recs_bar);
        if (p.n_shared)
          for (int j = 0; j < T; ++j, dst += rbS)
            bulk_g2s(dst, p.h_s + (size_t)j * p.Fs, rbS, recs_bar);
      }
      // wait even after an earlier timeout: no copy of this CTA stays in flight
      const bool landed = csync_and(mbar_wait(recs_bar, (uint32_t)(l & 1), p.status));
      ok = ok && landed;
      if (ok) quant_h<true>(p, rt, stage, recs, threadIdx.x, kLT);
    } else {
      quant_h<false>(p, rt, nullptr, recs, threadIdx.x, kLT);
    }
    csync();
    MOE_STAMP(l, 7);

    // ---- down
#pragma unroll 1
    for (int j = ub + n_sh + n_rt; ok && j < ub + n_tot; ++j) {
#ifdef MOE_PROFILE
      long long c0 = clock64();
#endif
      ok = wait_unit(j);
      if (!ok) break;
#ifdef MOE_PROFILE
      long long c1 = clock64();
      pw += c1 - c0;
#endif
      if (j == ub + n_sh + n_rt) MOE_WSTAMP(l, 2);
      const uint8_t* d = up.myslots + (size_t)(j % kLSlots) * S.slot_bytes;
      const int u = warp + kLW * (j - ub - n_sh - n_rt);
      const int su = u / ngroups, gi = u - su * ngroups;
      const bool sh = p.n_shared && su == 0;
      const int r0 = gi * RG;
      const int nr = nrows_cta - r0 < RG ? nrows_cta - r0 : RG;
      const int dsl = sh ? -1 : su - p.n_shared;
      if (MAXT == 1 || (sh ? T : rt.slot_off[dsl + 1] - rt.slot_off[dsl]) == 1)
        down_unit_t<1, LPR>(p, rt, d, dsl, r0, nr, recs, part, rows_max);
      else
        down_unit_t<MAXT, LPR>(p, rt, d, dsl, r0, nr, recs, part, rows_max);
      release_unit(j);
      ++consumed;
#ifdef MOE_PROFILE
      pc += clock64() - c1;
#endif
    }
    MOE_WSTAMP(l, 3);
#ifdef MOE_PROFILE
    MOE_WPUT(l, 13, (uint64_t)pw);
    MOE_WPUT(l, 14, (uint64_t)pc);
    MOE_WPUT(l, 15, (uint64_t)pi);
#endif
    csync();
    MOE_STAMP(l, 8);

    // ---- combine in the fixed order: shared expert, then routed experts ascending
#pragma unroll 1
    for (int i = threadIdx.x; i < nrows_cta * T; i += kLT) {
      const int t = i / nrows_cta, r = i - t * nrows_cta;
      float acc = 0.0f;
      if (p.n_shared) acc = part[(size_t)(T * k + t) * rows_max + r];
#pragma unroll 1
      for (int e = 0; e < rt.n_valid; ++e) {
        const int pr = rt.list[e];
        if (pr / k == t) acc += rt.wt[pr] * part[(size_t)pr * rows_max + r];
      }
      yl[(size_t)t * H + dn.a + r] = acc;
    }
    csync();
    MOE_STAMP(l, 9);
    if (threadIdx.x == 0) grid_arrive(&p.sync[kSyncY]);
    // the records and partials are read: the next layer's router rows may
    // land over them (from L2, prefetched above)
    if (ok && l + 1 < Lyr) {
      if (threadIdx.x == 0) {
        fence_proxy_async_shared();
        issue_router_rows(l + 1);
      }
      rwr_issued = l + 1;
    }
    // A failed wait on this CTA's own copies (a 2 s limit, not reached when
    // the weights are readable) ends the layers here: the slots' copy order is
    // no longer known. The counters above were still raised for this layer.
    if (!csync_and(ok)) break;

    // ---- the next layer's units follow this layer's
    up.ub += n_tot;
    up.layer = l + 1;
    up.n_rt = up.rr_a = up.n_dn = 0;
  }

  // ---- the copy warp stops (it has issued everything unless the layers
  // ended early) and reports how many units it issued per warp
  if (threadIdx.x == 0) {
    __threadfence_block();
    *stop = 1u;
  }
  __syncthreads();
  // ---- drain this warp's bulk copies still in flight (after a timeout, or
  // rows fetched ahead for a layer that did not run), then the router rows
  // fetched ahead
  while (consumed < (int)final_iss[warp]) {
    wait_unit(consumed);
    ++consumed;
  }
  if (threadIdx.x == 0 && ne > 0 && rwr_issued > rwr_landed)
    mbar_wait(rwr_bar, (uint32_t)(rwr_issued & 1), p.status);

  // ---- leave: the last CTA out resets the counters and moves the epoch on
  csync();
  if (threadIdx.x == 0) {
    const uint32_t old = atomicAdd(&p.sync[kSyncOut], 1u);
    if (old == (uint32_t)G - 1u) {
      p.sync[kSyncH] = 0u;
      p.sync[kSyncY] = 0u;
      p.sync[kSyncOut] = 0u;
      atomicAdd(&p.sync[kSyncEpoch], (uint32_t)Lyr);
    }
  }
}

// bf16 (round to nearest even) of fp32 values: the chained input of the next
// layer on the multi-launch path.
__global__ void f32_to_bf16_kernel(const float* __restrict__ y, uint16_t* __restrict__ x,
                                   int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    x[i] = __bfloat16_as_ushort(__float2bfloat16_rn(y[i]));
}

// ---------------------------------------------------------------------------
namespace {
const void* layers_kernel_for(const DecodeParams& p) {
  const bool w8 = lanes_per_row(p.H) == 8 && lanes_per_row(p.F) == 8 &&
                  (!p.n_shared || lanes_per_row(p.Fs) == 8);
  const int t = p.T == 1 ? 1 : (p.T == 2 ? 2 : 4);
#define MOE_LK(T_, L_) reinterpret_cast<const void*>(decode_layers_kernel<T_, L_>)
  if (w8) return t == 1 ? MOE_LK(1, 8) : t == 2 ? MOE_LK(2, 8) : MOE_LK(4, 8);
  return t == 1 ? MOE_LK(1, 0) : t == 2 ? MOE_LK(2, 0) : MOE_LK(4, 0);
#undef MOE_LK
}

bool layers_resident(const void* kfn, size_t smem) {
  static std::mutex mu;
  struct Entry { const void* k; int dev; size_t smem; bool ok; };
  static Entry cache[32];
  static int n = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return false; }
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
      if (cache[i].k == kfn && cache[i].dev == dev && cache[i].smem == smem) return cache[i].ok;
  }
  bool ok = false;
  if (ensure_smem_attr(kfn, smem) == cudaSuccess) {
    int blocks = 0;
    ok = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kfn, kLTP, smem) == cudaSuccess &&
         blocks >= 1;
  }
  cudaGetLastError();
  std::lock_guard<std::mutex> lock(mu);
  if (n < 32) cache[n++] = Entry{kfn, dev, smem, ok};
  return ok;
}
}  // namespace

// Whether the single-launch multi-layer kernel takes these sizes (1..4
// tokens, up to 512 experts, widths multiples of 256, shared memory within an
// SM, one CTA per SM resident); fills the launch-derived fields.
bool layers_supported(const DecodeParams& p, int num_sms, size_t* smem, int* rg,
                      int* rows_max) {
  if (p.T < 1 || p.T > 4) return false;
  if (p.H % 256 || p.F % 256 || (p.n_shared && p.Fs % 256)) return false;
  if (p.E > 512) return false;
  const int grid = num_sms;
  const int rmax = (p.H + grid - 1) / grid;
  int K = p.F;
  if (p.n_shared && p.Fs > K) K = p.Fs;
  const int rpw = 32 / lanes_per_row(K);
  const int64_t rbK = row_bytes(K);
  int64_t budget = 2 * row_bytes(p.H);
  if (budget < 4608) budget = 4608;
  const int slots = (p.T * p.k < p.E ? p.T * p.k : p.E) + p.n_shared;
  auto units = [&](int rows) { return slots * ((rmax + rows - 1) / rows); };
  // down rows per unit: one pass of a warp, grown (in whole passes, while a
  // unit fits in max(a gate/up unit, 4608 bytes)) until each warp has at most
  // one down unit: a warp fetches its down rows while it finishes gate/up, so
  // a second unit would be fetched only after the h barrier
  int r = rpw < rmax ? rpw : rmax;
  if (units(r) > kLW) {
    while (r + rpw <= rmax && (r + rpw) * rbK <= budget && units(r) > kLW) r += rpw;
    if (units(r) > kLW && rmax * rbK <= budget) r = rmax;
  }
  const LayersSmem m = layers_smem(p.H, p.F, p.Fs, p.n_shared, p.T, p.k, rmax, r, p.E, grid);
  if (m.total > 227 * 1024) return false;
  if (!layers_resident(layers_kernel_for(p), m.total)) return false;
  *smem = m.total;
  *rg = r;
  *rows_max = rmax;
  return true;
}

int layers_launches(const DecodeParams& p0, int num_sms) {
  DecodeParams p = p0;
  size_t sm = 0;
  int rg = 0, rmax = 0;
  if (layers_supported(p, num_sms, &sm, &rg, &rmax)) return 1;
  p.route = 0;
  const int per = decode_launches(p, num_sms) + 1;     // router, then the layer
  return p.L * per + (p.chained ? p.L - 1 : 0);
}

cudaError_t launch_decode_layers(const DecodeParams& p0, const LayerTable& lt, int num_sms,
                                 bool pdl, cudaStream_t stream) {
  DecodeParams p = p0;
  size_t sm = 0;
  int rg = 0, rmax = 0;
  if (layers_supported(p, num_sms, &sm, &rg, &rmax)) {
    p.fz_rg = rg;
    p.dn_rows_max = rmax;
    const void* kfn = layers_kernel_for(p);
    cudaError_t e = ensure_smem_attr(kfn, sm);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kLTP);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void* args[2] = {const_cast<DecodeParams*>(&p), const_cast<LayerTable*>(&lt)};
    return cudaLaunchKernelExC(&cfg, kfn, args);
  }
  // Otherwise one layer after another: the router, then the layer, and for a
  // chained call the bf16 rounding of y into the next layer's input.
  const int T = p.T, H = p.H;
#pragma unroll 1
  for (int l = 0; l < p.L; ++l) {
    const LayerPtrs& W = lt.layer[l];
    const uint16_t* xl = (p.chained && l > 0) ? p.xc : p.x + (p.chained ? 0 : (size_t)l * T * H);
    int32_t* ids = p.ids_out + (size_t)l * T * p.k;
    float* w = p.w_out + (size_t)l * T * p.k;
    RouteParams rp{H, p.E, p.k, T, W.Wr, W.bias, xl, ids, w};
    cudaError_t e = launch_route(rp, pdl, stream);
    if (e != cudaSuccess) return e;
    DecodeParams q = p;
    q.gate = W.gate;
    q.up = W.up;
    q.down = W.down;
    q.sh_gate = W.sh_gate;
    q.sh_up = W.sh_up;
    q.sh_down = W.sh_down;
    q.x = xl;
    q.ids = ids;
    q.weights = w;
    q.y = p.y + (size_t)l * T * H;
    q.route = 0;
    e = launch_decode(q, num_sms, pdl, stream);
    if (e != cudaSuccess) return e;
    if (p.chained && l + 1 < p.L) {
      const int n = T * H;
      f32_to_bf16_kernel<<<(n + 255) / 256, 256, 0, stream>>>(q.y, p.xc, n);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace moe

#ifdef MOE_PROFILE
// Copies the phase stamps (uint64 [256 CTAs][64 layers][12 phases], ns of
// %globaltimer) to host memory. Profiling builds only.
extern "C" int moe_profile_stamps(void* host, size_t bytes) {
  const size_t n = sizeof(moe::g_prof) < bytes ? sizeof(moe::g_prof) : bytes;
  return cudaMemcpyFromSymbol(host, moe::g_prof, n) == cudaSuccess ? 0 : -1;
}
// Per-warp stamps (uint64 [256][64][16 warps][22]).
extern "C" int moe_profile_warp_stamps(void* host, size_t bytes) {
  const size_t n = sizeof(moe::g_profw) < bytes ? sizeof(moe::g_profw) : bytes;
  return cudaMemcpyFromSymbol(host, moe::g_profw, n) == cudaSuccess ? 0 : -1;
}
#endif
