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

  // Scores: one warp per expert, lanes over H in 8-element chunks (many loads
  // in flight), then each score is stored straight into the shared memory of
  // the CTA that owns its token (token i of the tile belongs to rank i % C).
  const int h8 = H / 8;
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
    float psum = 0.0f;
    float psel = 0.0f;
    int isel = 0;
    for (int j = 0; j < p.k; ++j) {
      float best = -INFINITY;
      int bi = 0x7FFFFFFF;
      for (int e = lane; e < E; e += 32) {
        const float kv = mykeys[e];
        if (kv > best) { best = kv; bi = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
      }
      if (bi >= E) bi = 0;            // only with NaN keys
      const float pr = 1.0f / (1.0f + expf(-srow[bi]));
      psum += pr;
      if (lane == j) { psel = pr; isel = bi; }
      __syncwarp();
      if (lane == 0) mykeys[bi] = -INFINITY;
      __syncwarp();
    }
    if (lane < p.k) {
      const size_t t = (size_t)(t0 + i);
      p.ids[t * p.k + lane] = isel;
      p.w[t * p.k + lane] = psel / psum;
    }
    __syncwarp();
  }
}

namespace {
// Permits clusters of more than 8 CTAs for a kernel, once; an error means the
// device does not offer them and the caller falls back to 8.
cudaError_t allow_wide_clusters(const void* kernel) {
  static const void* done[8];
  static int n = 0;
  for (int i = 0; i < n; ++i)
    if (done[i] == kernel) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  if (n < 8) done[n++] = kernel;
  return cudaSuccess;
}
// Whether 16-CTA clusters can run for (token tile, shared memory size); -1 = not asked yet.
struct WideEntry {
  int tt;
  size_t sm;
  int ok;
};
WideEntry g_wide[32];
int g_nwide = 0;
int wide_cluster_cache(int tt, size_t sm) {
  for (int i = 0; i < g_nwide; ++i)
    if (g_wide[i].tt == tt && g_wide[i].sm == sm) return g_wide[i].ok;
  return -1;
}
void wide_cluster_store(int tt, size_t sm, int ok) {
  if (g_nwide < 32) g_wide[g_nwide++] = WideEntry{tt, sm, ok};
}
}  // namespace

cudaError_t launch_route(const RouteParams& p, bool pdl, cudaStream_t stream) {
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
