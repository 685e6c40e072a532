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

template <int MAXT>
__device__ __forceinline__ void gateup_rows(const DecodeParams& p, const RouteTable& rt,
                                            const uint8_t* stage, const Chunk& ch,
                                            const uint32_t* xq, int xq_words) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= ch.rows) return;
  const int H = p.H;
  const int rb = H / 32 * kBlockB;
  const int npairs = H / 64;
  const int lpr = dlanes_per_row(H);
  const int f = ch.f0 + warp;
  const bool shared = ch.slot < 0;
  const int F = shared ? p.Fs : p.F;
  const uint8_t* grow = stage + (size_t)warp * rb;
  const uint8_t* urow = stage + (size_t)(ch.rows + warp) * rb;
  // tokens of this slot
  const int ntok = shared ? p.T : rt.slot_off[ch.slot + 1] - rt.slot_off[ch.slot];
  const int lbase = shared ? 0 : rt.slot_off[ch.slot];
  const int xs_off = dqvec_pair_words(H);

  for (int g0 = 0; g0 < ntok; g0 += MAXT) {
    const int ng = ntok - g0 < MAXT ? ntok - g0 : MAXT;
    int tok[MAXT];
#pragma unroll
    for (int j = 0; j < MAXT; ++j) {
      const int jj = g0 + (j < ng ? j : 0);
      tok[j] = shared ? jj : rt.list[lbase + jj] / p.k;
    }
    float ag[MAXT], au[MAXT];
#pragma unroll
    for (int j = 0; j < MAXT; ++j) ag[j] = au[j] = 0.0f;

    for (int q = lane; q < npairs; q += 32) {
      const int qbase = qv_base(q, lpr);
      uint32_t w[9];
      float dg0, dg1, du0, du1;
      uint32_t a0[4], a1[4];
      uint32_t tg0[8], tg1[8], tu0[8], tu1[8];
      load_pair_smem(grow + q * kPairB, w);
      split_pair(w, dg0, dg1, a0, a1);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        iq4_lookup8(a0[i], tg0[2 * i], tg0[2 * i + 1]);
        iq4_lookup8(a1[i], tg1[2 * i], tg1[2 * i + 1]);
      }
      load_pair_smem(urow + q * kPairB, w);
      split_pair(w, du0, du1, a0, a1);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        iq4_lookup8(a0[i], tu0[2 * i], tu0[2 * i + 1]);
        iq4_lookup8(a1[i], tu1[2 * i], tu1[2 * i + 1]);
      }
#pragma unroll
      for (int j = 0; j < MAXT; ++j) {
        if (j < ng) {
          const uint32_t* rec = xq + (size_t)tok[j] * xq_words;
          const uint4* r4 = reinterpret_cast<const uint4*>(rec) + qbase;
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 u = r4[c * lpr];
            v[4 * c] = u.x; v[4 * c + 1] = u.y; v[4 * c + 2] = u.z; v[4 * c + 3] = u.w;
          }
          const float* xs = reinterpret_cast<const float*>(rec + xs_off);
          const float s0 = xs[2 * q], s1 = xs[2 * q + 1];
          const int ig0 = iq4_dot_block(tg0, v);
          const int ig1 = iq4_dot_block(tg1, v + 16);
          const int iu0 = iq4_dot_block(tu0, v);
          const int iu1 = iq4_dot_block(tu1, v + 16);
          ag[j] = fmaf((float)ig0, dg0 * s0, ag[j]);
          ag[j] = fmaf((float)ig1, dg1 * s1, ag[j]);
          au[j] = fmaf((float)iu0, du0 * s0, au[j]);
          au[j] = fmaf((float)iu1, du1 * s1, au[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < MAXT; ++j) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        ag[j] += __shfl_xor_sync(0xFFFFFFFFu, ag[j], o);
        au[j] += __shfl_xor_sync(0xFFFFFFFFu, au[j], o);
      }
    }
#pragma unroll
    for (int j = 0; j < MAXT; ++j) {
      if (j < ng && lane == j) {
        const float hv = silu_mul(ag[j], au[j]);
        if (shared) p.h_s[(size_t)tok[j] * p.Fs + f] = hv;
        else p.h_r[(size_t)rt.list[lbase + g0 + j] * p.F + f] = hv;
      }
    }
  }

}

// ---------------------------------------------------------------------------
// Shared-memory layouts (host and device agree on them).
struct GuSmem {
  size_t xq, bar, ring, stage, total;
};
__host__ __device__ inline GuSmem gu_smem(int H, int T, int nst) {
  GuSmem m;
  m.xq = align_up_dev(sizeof(RouteTable), 128);
  m.bar = align_up_dev(m.xq + (size_t)T * dqvec_words(H) * 4, 16);
  m.ring = align_up_dev(m.bar + (size_t)16 * nst, 128);
  m.stage = align_up_dev((size_t)2 * kChunkRows * (H / 32) * kBlockB, 128);
  m.total = m.ring + (size_t)nst * m.stage;
  return m;
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

template <int MAXT>
__global__ void __launch_bounds__(kThreads, 2) gateup_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = p.H;
  const int NST = p.gu_stages;
  const GuSmem L = gu_smem(H, p.T, NST);
  RouteTable& rt = *reinterpret_cast<RouteTable*>(smem);
  uint32_t* xq = reinterpret_cast<uint32_t*>(smem + L.xq);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* empty = full + NST;
  uint8_t* ring = smem + L.ring;
  const int xq_words = dqvec_words(H);
  const int rb = H / 32 * kBlockB;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = row_granule_dev(H);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    mbar_fence_init();
  }
  __syncthreads();

  const RowRange shr = p.n_shared ? split_rows(p.Fs, g, blockIdx.x, gridDim.x) : RowRange{0, 0};

  if (warp == kProducerWarp) {
    // Producer: one lane issues the bulk copies; shared-expert rows first (they
    // do not depend on the routes), then this CTA's share of the routed rows.
    const uint64_t pol = l2_evict_first_policy();   // weights: read once per call
    int it = 0;
    bool ok = true;
    auto issue = [&](const Chunk& c, const uint8_t* gbase, const uint8_t* ubase, int64_t row0) {
      const int s = it % NST;
      const uint32_t par = ((it / NST) & 1) ^ 1;
      if (!mbar_wait(&empty[s], par, p.status)) return false;
      const uint32_t bytes = (uint32_t)(c.rows * rb);
      uint8_t* dst = ring + (size_t)s * L.stage;
      mbar_arrive_expect_tx(&full[s], 2 * bytes);
      bulk_g2s_hint(dst, gbase + (row0 + c.f0) * rb, bytes, &full[s], pol);
      bulk_g2s_hint(dst + bytes, ubase + (row0 + c.f0) * rb, bytes, &full[s], pol);
      ++it;
      return true;
    };
    if (lane == 0) {
      for (int r = shr.a; ok && r < shr.b;) {
        const Chunk c = next_chunk(r, shr.b, p.Fs, true);
        ok = issue(c, p.sh_gate, p.sh_up, 0);
        r += c.rows;
      }
    }
    __syncwarp();
    pdl_wait();
    pdl_trigger();
    all_sync_named();                      // route table ready
    if (lane == 0 && ok) {
      const RowRange rr = split_rows(rt.n_slots * p.F, g, blockIdx.x, gridDim.x);
      for (int r = rr.a; ok && r < rr.b;) {
        const Chunk c = next_chunk(r, rr.b, p.F, false);
        const int64_t row0 = (int64_t)rt.slot_expert[c.slot] * p.F;
        ok = issue(c, p.gate, p.up, row0);
        r += c.rows;
      }
    }
    return;
  }

  // Consumers. Quantise x first: the inputs of this call are complete (the
  // router that precedes this kernel read them after its own dependency wait).
  quant_x_to_smem(p.x, p.T, H, xq, xq_words, warp, kConsumers / 32);
  consumers_sync();

  int it = 0;
  bool ok = true;
  Pending pd;
  pd.n = 0;
  auto consume = [&](const Chunk& c) {
    const int s = it % NST;
    const uint32_t par = (it / NST) & 1;
    if (!mbar_wait(&full[s], par, p.status)) return false;
    gateup_rows<MAXT>(p, rt, ring + (size_t)s * L.stage, c, xq, xq_words);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    ++it;
    if (warp < c.rows) {
      pd.slot[pd.n] = c.slot;
      pd.f[pd.n] = c.f0 + warp;
      if (++pd.n == kPendMax) flush_arrivals(p, rt, pd);
    }
    return true;
  };
  for (int r = shr.a; ok && r < shr.b;) {
    const Chunk c = next_chunk(r, shr.b, p.Fs, true);
    ok = consume(c);
    r += c.rows;
  }
  pdl_wait();
  pdl_trigger();
  build_route_table<kConsumers, 1>(rt, p.ids, p.weights, p.T * p.k, p.E);
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.status && rt.invalid)
    atomicAdd(p.status, (uint32_t)(rt.invalid < 0xFFFF ? rt.invalid : 0xFFFF));
  all_sync_named();
  const RowRange rr = split_rows(rt.n_slots * p.F, g, blockIdx.x, gridDim.x);
  for (int r = rr.a; ok && r < rr.b;) {
    const Chunk c = next_chunk(r, rr.b, p.F, false);
    ok = consume(c);
    r += c.rows;
  }
  if (pd.n) flush_arrivals(p, rt, pd);
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
  build_route_table<kConsumers, 1>(rt, p.ids, p.weights, p.T * p.k, p.E);
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
      if (active) {
        const uint8_t* row = wst + (size_t)r * rbK;
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
size_t gateup_smem_bytes(const DecodeParams& p, int stages) {
  return gu_smem(p.H, p.T, stages).total;
}
size_t down_smem_bytes(const DecodeParams& p, int stages) {
  return dn_smem(p.F, p.Fs, p.n_shared, p.T, p.dn_rows_max, stages).total;
}

namespace {
constexpr size_t kSmemSoft = 112 * 1024;   // two CTAs of consecutive kernels share an SM
constexpr size_t kSmemHard = 227 * 1024;

template <typename K>
cudaError_t launch(K kernel, int grid, size_t smem, bool pdl, cudaStream_t stream,
                   const DecodeParams& p) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

int pick_stages(size_t fixed, size_t stage, int lo, int hi) {
  int n = hi;
  while (n > lo && fixed + (size_t)n * stage > kSmemSoft) --n;
  while (n > 1 && fixed + (size_t)n * stage > kSmemHard) --n;
  return n;
}
}  // namespace

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
  const GuSmem g1 = gu_smem(p.H, p.T, 1);
  p.gu_stages = pick_stages(g1.ring, g1.stage, 2, 6);
  const size_t gsm = gu_smem(p.H, p.T, p.gu_stages).total;
  if (gsm > kSmemHard) return cudaErrorInvalidConfiguration;
  // down
  int gd = row_granule_dev(p.F);
  if (p.n_shared && row_granule_dev(p.Fs) > gd) gd = row_granule_dev(p.Fs);
  const int units = p.H / gd;
  const int grid_dn = units < num_sms ? units : num_sms;
  p.dn_rows_max = (units + grid_dn - 1) / grid_dn * gd;
  const DnSmem d1 = dn_smem(p.F, p.Fs, p.n_shared, p.T, p.dn_rows_max, 1);
  p.dn_stages = pick_stages(d1.ring, d1.stage, 2, 8);
  const size_t dsm = dn_smem(p.F, p.Fs, p.n_shared, p.T, p.dn_rows_max, p.dn_stages).total;
  if (dsm > kSmemHard) return cudaErrorInvalidConfiguration;

  cudaError_t e;
  const int T = p.T;
  if (T <= 1) e = launch(gateup_kernel<1>, num_sms, gsm, pdl, stream, p);
  else if (T <= 2) e = launch(gateup_kernel<2>, num_sms, gsm, pdl, stream, p);
  else if (T <= 4) e = launch(gateup_kernel<4>, num_sms, gsm, pdl, stream, p);
  else if (T <= 8) e = launch(gateup_kernel<8>, num_sms, gsm, pdl, stream, p);
  else e = launch(gateup_kernel<16>, num_sms, gsm, pdl, stream, p);
  if (e != cudaSuccess) return e;
  return launch(down_kernel<kPairsPerStage>, grid_dn, dsm, pdl, stream, p);
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
