// Router of libmoe (sm_103a): scores, sigmoid + bias, top-k, renormalised weights.
//
// PocketLLM page "Xing4.0-29B-A4B", Overview: a sigmoid-routed MoE (64 experts
// activated top-4); the choice is made on sigmoid(score) + bias, ties to the
// lower index, and the combine weights are the chosen sigmoids renormalised.
//
// A grid of thread-block clusters: the C CTAs of a cluster split the experts
// of one token tile, each keeps its scores in shared memory, and after a
// cluster barrier one warp per token reads all E scores through distributed
// shared memory and runs k rounds of a warp arg-max.
#include <cooperative_groups.h>

#include "common.cuh"
#include "route.cuh"

#include <mutex>

namespace cg = cooperative_groups;

namespace moe {

__host__ __device__ inline size_t route_smem(int H, int E, int C, int TT) {
  (void)C;
  size_t off = (size_t)TT * H * 2;                       // x tile, bf16
  off = (off + 15) & ~size_t(15);
  off += (size_t)TT * E * 4;                             // scores of the tokens this CTA owns
  off = (off + 15) & ~size_t(15);
  off += (size_t)8 * E * 4;                              // per-warp key scratch
  return off;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

template <int TT>
__global__ void __launch_bounds__(256) route_kernel(RouteParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int H = p.H, E = p.E;
  const int epc = (E + C - 1) / C;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  size_t off = ((size_t)TT * H * 2 + 15) & ~size_t(15);
  float* sc = reinterpret_cast<float*>(smem + off);      // [TT][E], rows of owned tokens
  off = (off + (size_t)TT * E * 4 + 15) & ~size_t(15);
  float* keys = reinterpret_cast<float*>(smem + off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int tile = blockIdx.x / C;
  const int t0 = tile * TT;
  const int nt = p.T - t0 < TT ? p.T - t0 : TT;
  const int e0 = rank * epc;
  const int e1 = e0 + epc < E ? e0 + epc : E;

  // Router weights are constant: warm L2 with this CTA's rows while the
  // previous kernel on the stream finishes.
  if (threadIdx.x == 0 && e1 > e0) {
    const char* base = reinterpret_cast<const char*>(p.Wr + (size_t)e0 * H);
    const size_t bytes = (size_t)(e1 - e0) * H * 2;
    for (size_t o = 0; o < bytes; o += 65536) {
      const uint32_t n = (uint32_t)(bytes - o < 65536 ? bytes - o : 65536);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + o), "r"(n & ~15u)
                   : "memory");
    }
  }
  pdl_wait();
  pdl_trigger();

  // x tile -> shared memory
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t0 * H);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    const int n16 = nt * H / 8;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();

  // Scores: lanes over H in 8-element chunks, then each score is stored
  // straight into the shared memory of the CTA that owns its token (token i of
  // the tile belongs to rank i % C). Per (expert, token) the eight products of
  // a chunk are added in element order and the chunks in lane order, then the
  // lanes by a butterfly: the same sum however the experts are grouped.
  const int h8 = H / 8;
  if (TT <= 4) {
    // Warp w takes experts e0 + w, e0 + w + 8, ... in groups of up to eight:
    // a chunk of x is unpacked once for the whole group, and the group's
    // router rows are loaded together.
    for (int g = e0 + warp; g < e1; g += 64) {
      int ng = (e1 - g + 7) / 8;
      if (ng > 8) ng = 8;
      float acc[8][TT];
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[j][t] = 0.0f;
#pragma unroll 1
      for (int c = lane; c < h8; c += 32) {
        float xf[TT][8];
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const uint4 xv = t < nt ? reinterpret_cast<const uint4*>(xs + (size_t)t * H)[c]
                                  : make_uint4(0u, 0u, 0u, 0u);
          xf[t][0] = bf16_lo(xv.x); xf[t][1] = bf16_hi(xv.x);
          xf[t][2] = bf16_lo(xv.y); xf[t][3] = bf16_hi(xv.y);
          xf[t][4] = bf16_lo(xv.z); xf[t][5] = bf16_hi(xv.z);
          xf[t][6] = bf16_lo(xv.w); xf[t][7] = bf16_hi(xv.w);
        }
        uint4 wv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < ng) wv[j] = __ldg(reinterpret_cast<const uint4*>(p.Wr + (size_t)(g + 8 * j) * H) + c);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j < ng) {
            const float w0 = bf16_lo(wv[j].x), w1 = bf16_hi(wv[j].x);
            const float w2 = bf16_lo(wv[j].y), w3 = bf16_hi(wv[j].y);
            const float w4 = bf16_lo(wv[j].z), w5 = bf16_hi(wv[j].z);
            const float w6 = bf16_lo(wv[j].w), w7 = bf16_hi(wv[j].w);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
              float a = acc[j][t];
              a = fmaf(w0, xf[t][0], a);
              a = fmaf(w1, xf[t][1], a);
              a = fmaf(w2, xf[t][2], a);
              a = fmaf(w3, xf[t][3], a);
              a = fmaf(w4, xf[t][4], a);
              a = fmaf(w5, xf[t][5], a);
              a = fmaf(w6, xf[t][6], a);
              a = fmaf(w7, xf[t][7], a);
              acc[j][t] = a;
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < ng) {
#pragma unroll
          for (int t = 0; t < TT; ++t) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
              acc[j][t] += __shfl_xor_sync(0xFFFFFFFFu, acc[j][t], o);
            if (t < nt && lane == (t & 31)) {
              float* dst = cluster.map_shared_rank(sc, t % C);
              dst[t * E + g + 8 * j] = acc[j][t];
            }
          }
        }
      }
    }
  } else
  for (int e = e0 + warp; e < e1; e += 8) {
    const uint4* wr = reinterpret_cast<const uint4*>(p.Wr + (size_t)e * H);
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.0f;
#pragma unroll 8
    for (int c = lane; c < h8; c += 32) {
      const uint4 w = __ldg(wr + c);
      const float w0 = bf16_lo(w.x), w1 = bf16_hi(w.x), w2 = bf16_lo(w.y), w3 = bf16_hi(w.y);
      const float w4 = bf16_lo(w.z), w5 = bf16_hi(w.z), w6 = bf16_lo(w.w), w7 = bf16_hi(w.w);
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        if (t < nt) {
          const uint4 xv = reinterpret_cast<const uint4*>(xs + (size_t)t * H)[c];
          float a = acc[t];
          a = fmaf(w0, bf16_lo(xv.x), a);
          a = fmaf(w1, bf16_hi(xv.x), a);
          a = fmaf(w2, bf16_lo(xv.y), a);
          a = fmaf(w3, bf16_hi(xv.y), a);
          a = fmaf(w4, bf16_lo(xv.z), a);
          a = fmaf(w5, bf16_hi(xv.z), a);
          a = fmaf(w6, bf16_lo(xv.w), a);
          a = fmaf(w7, bf16_hi(xv.w), a);
          acc[t] = a;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], o);
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      if (t < nt && lane == (t & 31)) {
        float* dst = cluster.map_shared_rank(sc, t % C);
        dst[t * E + e] = acc[t];
      }
    }
  }
  cluster.sync();

  // top-k for the tokens this CTA owns; only local shared memory from here on
  float* mykeys = keys + (size_t)warp * E;
  for (int i = rank + C * warp; i < nt; i += C * 8) {
    const float* srow = sc + (size_t)i * E;
    for (int e = lane; e < E; e += 32) {
      const float pr = 1.0f / (1.0f + expf(-srow[e]));
      mykeys[e] = pr + (p.bias ? p.bias[e] : 0.0f);
    }
    __syncwarp();
    const int id = warp_topk_ids(mykeys, E, p.k);
    const float wv = warp_renorm(lane < p.k ? 1.0f / (1.0f + expf(-srow[id])) : 0.0f, p.k);
    if (lane < p.k) {
      const size_t t = (size_t)(t0 + i);
      p.ids[t * p.k + lane] = id;
      p.w[t * p.k + lane] = wv;
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Router for token chunks on the tensor cores: D[t][e] = sum_h x[t][h] Wr[e][h]
// by mma.sync m16n8k16 (bf16 operands, fp32 accumulation). A CTA takes 16
// tokens (the MMA's M) and every expert; warp w takes expert tile n (8
// experts, the MMA's N) and one half of K when there are at most 8 tiles.
// K runs in chunks of 64: within a chunk, lane (g, c) = (lane / 4, lane % 4)
// feeds the MMA's k = 2c, 2c+1, 2c+8, 2c+9 of step s from memory positions
// 16c + 4s + 0..3 of its rows, the same positions for x and Wr, so each lane
// reads 32 contiguous bytes of a row per chunk and every product x[t][h]
// Wr[e][h] still meets its own pair. x sits in shared memory in rows padded
// by 16 bytes (the eight rows of a fragment load fall in different banks);
// Wr is read through L1/L2. Then sigmoid, bias and the warp top-k as above.
constexpr int kRmTok = 16;
constexpr int kRmWarps = 16;

__host__ __device__ inline size_t route_mma_smem(int H, int E) {
  size_t off = (size_t)kRmTok * (H * 2 + 16);           // x tile, padded rows
  off += 2 * (size_t)kRmTok * E * 4;                    // score partials (two K halves)
  off += (size_t)kRmWarps * E * 4;                      // per-warp keys
  return off;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kRmWarps * 32, 1) route_mma_kernel(RouteParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int H = p.H, E = p.E;
  const int xrow = H * 2 + 16;
  uint8_t* xs = smem;
  float* part = reinterpret_cast<float*>(smem + (size_t)kRmTok * xrow);
  float* keys = part + 2 * kRmTok * E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int t0 = blockIdx.x * kRmTok;
  const int nt = p.T - t0 < kRmTok ? p.T - t0 : kRmTok;
  const int n8 = (E + 7) >> 3;
  const int KP = n8 <= kRmWarps / 2 ? 2 : 1;
  const int nch = H >> 6;

  // Router rows are constant: a few CTAs warm L2 with them while the previous
  // kernel on the stream finishes.
  if (threadIdx.x == 0 && blockIdx.x < 8) {
    const size_t bytes = (size_t)E * H * 2;
    const size_t o0 = bytes * blockIdx.x / 8 & ~size_t(15);
    const size_t o1 = (blockIdx.x == 7 ? bytes : bytes * (blockIdx.x + 1) / 8) & ~size_t(15);
    const char* base = reinterpret_cast<const char*>(p.Wr);
    for (size_t o = o0; o < o1; o += 65536) {
      const uint32_t n = (uint32_t)(o1 - o < 65536 ? o1 - o : 65536);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + o), "r"(n)
                   : "memory");
    }
  }
  pdl_wait();
  pdl_trigger();

  // x tile -> shared memory; rows past the chunk are zero
  const int h16 = H >> 3;
  for (int i = threadIdx.x; i < kRmTok * h16; i += blockDim.x) {
    const int r = i / h16, q = i - r * h16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < nt) v = reinterpret_cast<const uint4*>(p.x + (size_t)(t0 + r) * H)[q];
    *reinterpret_cast<uint4*>(xs + (size_t)r * xrow + (size_t)q * 16) = v;
  }
  __syncthreads();

  for (int job = warp; job < n8 * KP; job += kRmWarps) {
    const int n = job % n8, kp = job / n8;
    const int ch0 = kp * nch / KP, ch1 = (kp + 1) * nch / KP;
    const int e = n * 8 + g;
    const uint4* wrow = reinterpret_cast<const uint4*>(p.Wr + (size_t)(e < E ? e : 0) * H) + 2 * c;
    const uint8_t* xa = xs + (size_t)g * xrow + 32 * c;
    const uint8_t* xb = xa + (size_t)8 * xrow;
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
    for (int ch = ch0; ch < ch1; ++ch) {
      uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
      if (e < E) {
        w0 = __ldg(wrow + (size_t)ch * 8);
        w1 = __ldg(wrow + (size_t)ch * 8 + 1);
      }
      const uint4 a0 = *reinterpret_cast<const uint4*>(xa + (size_t)ch * 128);
      const uint4 a1 = *reinterpret_cast<const uint4*>(xa + (size_t)ch * 128 + 16);
      const uint4 b0 = *reinterpret_cast<const uint4*>(xb + (size_t)ch * 128);
      const uint4 b1 = *reinterpret_cast<const uint4*>(xb + (size_t)ch * 128 + 16);
      mma_bf16_16816(d, a0.x, b0.x, a0.y, b0.y, w0.x, w0.y);
      mma_bf16_16816(d, a0.z, b0.z, a0.w, b0.w, w0.z, w0.w);
      mma_bf16_16816(d, a1.x, b1.x, a1.y, b1.y, w1.x, w1.y);
      mma_bf16_16816(d, a1.z, b1.z, a1.w, b1.w, w1.z, w1.w);
    }
    // d[0], d[1]: token g, experts 8n + 2c, 8n + 2c + 1; d[2], d[3]: token g + 8
    float* pp = part + (size_t)kp * kRmTok * E;
    const int ea = n * 8 + 2 * c;
    if (ea < E) {
      pp[g * E + ea] = d[0];
      pp[(g + 8) * E + ea] = d[2];
    }
    if (ea + 1 < E) {
      pp[g * E + ea + 1] = d[1];
      pp[(g + 8) * E + ea + 1] = d[3];
    }
  }
  __syncthreads();

  // warp w: token w of the tile
  float* mykeys = keys + (size_t)warp * E;
  for (int i = warp; i < nt; i += kRmWarps) {
    float* srow = part + (size_t)i * E;
    for (int e = lane; e < E; e += 32) {
      const float sc = KP == 2 ? srow[e] + srow[kRmTok * E + e] : srow[e];
      srow[e] = sc;
      mykeys[e] = 1.0f / (1.0f + expf(-sc)) + (p.bias ? p.bias[e] : 0.0f);
    }
    __syncwarp();
    const int id = warp_topk_ids(mykeys, E, p.k);
    const float wv = warp_renorm(lane < p.k ? 1.0f / (1.0f + expf(-srow[id])) : 0.0f, p.k);
    if (lane < p.k) {
      const size_t t = (size_t)(t0 + i);
      p.ids[t * p.k + lane] = id;
      p.w[t * p.k + lane] = wv;
    }
    __syncwarp();
  }
}

namespace {
// Both caches below are process-wide, keyed by device, and guarded by one
// mutex (host threads may launch concurrently, on several devices).
std::mutex g_cluster_mu;

// Permits clusters of more than 8 CTAs for a kernel on the current device,
// once; an error means the device does not offer them and the caller falls
// back to 8.
cudaError_t allow_wide_clusters(const void* kernel) {
  static const void* done_k[32];
  static int done_dev[32];
  static int n = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cluster_mu);
  for (int i = 0; i < n; ++i)
    if (done_k[i] == kernel && done_dev[i] == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  if (n < 32) {
    done_k[n] = kernel;
    done_dev[n] = dev;
    ++n;
  }
  return cudaSuccess;
}
// Whether 16-CTA clusters can run for (device, token tile, shared memory
// size); -1 = not asked yet.
struct WideEntry {
  int dev, tt;
  size_t sm;
  int ok;
};
WideEntry g_wide[64];
int g_nwide = 0;
int wide_cluster_cache(int tt, size_t sm) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  std::lock_guard<std::mutex> lock(g_cluster_mu);
  for (int i = 0; i < g_nwide; ++i)
    if (g_wide[i].dev == dev && g_wide[i].tt == tt && g_wide[i].sm == sm) return g_wide[i].ok;
  return -1;
}
void wide_cluster_store(int tt, size_t sm, int ok) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return; }
  std::lock_guard<std::mutex> lock(g_cluster_mu);
  if (g_nwide < 64) g_wide[g_nwide++] = WideEntry{dev, tt, sm, ok};
}
}  // namespace

cudaError_t launch_route(const RouteParams& p, bool pdl, cudaStream_t stream) {
  // Chunks of 256 or more tokens: the tensor-core router (16-token tiles)
  if (p.T >= 256 && p.E <= 256 && p.H % 128 == 0 &&
      route_mma_smem(p.H, p.E) <= (size_t)200 * 1024) {
    const size_t sm = route_mma_smem(p.H, p.E);
    const cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(route_mma_kernel), sm);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.T + kRmTok - 1) / kRmTok));
    cfg.blockDim = dim3(kRmWarps * 32);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, route_mma_kernel, p);
  }
  // token tile: x tile <= 128 KB; cluster: split experts for small T
  int TT = 16;
  while (TT > 1 && (size_t)TT * p.H * 2 > 128 * 1024) TT >>= 1;
  if (p.T < TT) {
    int t = 1;
    while (t < p.T) t <<= 1;
    TT = t;
  }
  // Decode batches: 16-CTA clusters (a non-portable size where allowed, else
  // 8) split the experts, and the tokens go in tiles small enough to give
  // about 128 CTAs (each cluster reads the router rows from L2 once).
  const bool decode = p.T <= MOE_MAX_DECODE_TOKENS;
  if (decode)
    while (TT > 1 && (p.T + TT - 1) / TT * 16 < 128) TT >>= 1;
  // Longer chunks: tiles small enough for several CTAs per SM (about three
  // waves of CTAs on 152 SMs), so that the SIMT contraction has warps to
  // hide its latencies; every tile reads the router rows from L2.
  if (!decode)
    while (TT > 1 && (p.T + TT - 1) / TT < 448) TT >>= 1;
  const int ntiles = (p.T + TT - 1) / TT;
  // Longer chunks: split the experts of a tile over a cluster only when there
  // are few tiles.
  int C = decode ? 16 : (ntiles >= 32 ? 1 : (ntiles >= 8 ? 4 : 16));
  while (C > 1 && C > p.E) C >>= 1;
  const size_t sm = route_smem(p.H, p.E, C, TT);
  if (sm > 200 * 1024) return cudaErrorInvalidConfiguration;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntiles * C);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;

  cudaError_t e;
#define MOE_ROUTE_CASE(N)                                                                  \
  case N:                                                                                  \
    e = ensure_smem_attr(reinterpret_cast<const void*>(route_kernel<N>), sm);             \
    if (e != cudaSuccess) return e;                                                        \
    if (C > 8) {                                                                           \
      int ok16 = wide_cluster_cache(N, sm);                                                \
      if (ok16 < 0) {                                                                      \
        e = allow_wide_clusters(reinterpret_cast<const void*>(route_kernel<N>));           \
        int ncl = 0;                                                                       \
        if (e == cudaSuccess &&                                                            \
            cudaOccupancyMaxActiveClusters(&ncl, route_kernel<N>, &cfg) != cudaSuccess)    \
          ncl = 0;                                                                         \
        cudaGetLastError();                                                                \
        ok16 = (e == cudaSuccess && ncl >= 1) ? 1 : 0;                                     \
        wide_cluster_store(N, sm, ok16);                                                   \
      }                                                                                    \
      if (!ok16) C = 8;                                                                    \
      attr[0].val.clusterDim.x = C;                                                        \
      cfg.gridDim = dim3(ntiles * C);                                                      \
    }                                                                                      \
    return cudaLaunchKernelEx(&cfg, route_kernel<N>, p);
  switch (TT) {
    MOE_ROUTE_CASE(1)
    MOE_ROUTE_CASE(2)
    MOE_ROUTE_CASE(4)
    MOE_ROUTE_CASE(8)
    MOE_ROUTE_CASE(16)
    default:
      return cudaErrorInvalidConfiguration;
  }
#undef MOE_ROUTE_CASE
}

}  // namespace moe
