// The C ABI of libmoe (include/moe.h): host-side validation and launches.
//
// Every argument is checked before anything is launched; a bad argument is
// refused with a status code rather than ignored (the option table of the
// PocketLLM "Xing4.0-29B-A4B" page refuses flags it cannot honour).
#include <atomic>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "decode.cuh"
#include "moe.h"
#include "prefill.cuh"
#include "route.cuh"
#include "util_kernels.cuh"

namespace {

std::atomic<int> g_pdl{1};
constexpr uint64_t kDefaultBarrierWaitNs = 2000000000ull;   // 2 s
std::atomic<uint64_t> g_barrier_wait_ns{kDefaultBarrierWaitNs};

int num_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  int v = cache[dev].load();
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(v);
  }
  return v;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool dim_ok(int32_t v) { return v >= 64 && v <= 8192 && v % 64 == 0; }

moe_status check_shape(const moe_shape* s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (!dim_ok(s->hidden) || !dim_ok(s->ffn)) {
    const bool fmt_ok = s->hidden > 0 && s->ffn > 0 && s->hidden % 32 == 0 && s->ffn % 32 == 0;
    return fmt_ok ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID_ARG;
  }
  if (s->n_experts < 1 || s->n_experts > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
  if (s->top_k < 1 || s->top_k > s->n_experts || s->top_k > MOE_MAX_TOP_K)
    return MOE_ERR_INVALID_ARG;
  if (s->n_shared != 0 && s->n_shared != 1) return MOE_ERR_INVALID_ARG;
  if (s->n_shared && !dim_ok(s->ffn_shared)) {
    const bool fmt_ok = s->ffn_shared > 0 && s->ffn_shared % 32 == 0;
    return fmt_ok ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

moe_status check_weights(const moe_shape* s, const moe_expert_weights* w) {
  if (!w || !w->gate || !w->up || !w->down) return MOE_ERR_INVALID_ARG;
  if (s->n_shared && (!w->sh_gate || !w->sh_up || !w->sh_down)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[6] = {w->gate, w->up, w->down, w->sh_gate, w->sh_up, w->sh_down};
  for (int i = 0; i < (s->n_shared ? 6 : 3); ++i)
    if (!aligned(ptrs[i], 16)) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

moe_status layer_args(const moe_shape* s, const moe_expert_weights* w, const uint16_t* x,
                      int32_t T, int32_t Tmax, const int32_t* ids, const float* wts, float* y,
                      void* ws, uint32_t* status) {
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  if (T < 0 || T > Tmax) return MOE_ERR_INVALID_ARG;
  st = check_weights(s, w);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!x || !ids || !wts || !y || !ws) return ws ? MOE_ERR_INVALID_ARG : MOE_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ids, 4) || !aligned(wts, 4) ||
      !aligned(ws, 256) || (status && !aligned(status, 4)))
    return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

moe::DecodeParams decode_params(const moe_shape* shape, const moe_expert_weights* w,
                                const uint16_t* x, int32_t T, const int32_t* ids,
                                const float* weights, float* y, void* ws,
                                const moe::DecodeLayout& L, uint32_t* status) {
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  moe::DecodeParams p{};
  p.H = shape->hidden;
  p.F = shape->ffn;
  p.Fs = shape->n_shared ? shape->ffn_shared : 0;
  p.E = shape->n_experts;
  p.k = shape->top_k;
  p.n_shared = shape->n_shared;
  p.T = T;
  p.gate = reinterpret_cast<const uint8_t*>(w->gate);
  p.up = reinterpret_cast<const uint8_t*>(w->up);
  p.down = reinterpret_cast<const uint8_t*>(w->down);
  p.sh_gate = reinterpret_cast<const uint8_t*>(w->sh_gate);
  p.sh_up = reinterpret_cast<const uint8_t*>(w->sh_up);
  p.sh_down = reinterpret_cast<const uint8_t*>(w->sh_down);
  p.x = x;
  p.ids = ids;
  p.weights = weights;
  p.y = y;
  p.h_r = reinterpret_cast<float*>(base + L.h_r);
  p.h_s = reinterpret_cast<float*>(base + L.h_s);
  p.rec_r = reinterpret_cast<uint32_t*>(base + L.rec_r);
  p.rec_s = reinterpret_cast<uint32_t*>(base + L.rec_s);
  p.sync = reinterpret_cast<uint32_t*>(base + L.sync);
  p.xrec = reinterpret_cast<uint32_t*>(base + L.xrec);
  p.part = reinterpret_cast<float*>(base + L.part);
  p.status = status;
  p.wait_ns = g_barrier_wait_ns.load();
  return p;
}

}  // namespace

extern "C" {

moe_status moe_route_topk(const moe_shape* shape, const uint16_t* router_w,
                          const float* router_bias, const uint16_t* x, int32_t T,
                          int32_t* ids, float* weights, void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (T < 0 || T > (1 << 20)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!router_w || !x || !ids || !weights) return MOE_ERR_INVALID_ARG;
  if (!aligned(router_w, 16) || !aligned(x, 16) || !aligned(ids, 4) || !aligned(weights, 4) ||
      (router_bias && !aligned(router_bias, 4)))
    return MOE_ERR_MISALIGNED;
  moe::RouteParams p{shape->hidden, shape->n_experts, shape->top_k, T, router_w, router_bias,
                     x, ids, weights};
  const cudaError_t e = moe::launch_route(p, g_pdl.load() != 0,
                                          reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_workspace_bytes(const moe_shape* shape, int32_t max_tokens, int32_t mode) {
  if (check_shape(shape) != MOE_OK) return 0;
  if (mode == 0) {
    if (max_tokens < 1 || max_tokens > MOE_MAX_DECODE_TOKENS) return 0;
    return (size_t)moe::decode_layout(*shape, max_tokens).total;
  }
  if (mode == 1) {
    if (max_tokens < 1 || max_tokens > moe::kPrefillMaxTokens) return 0;
    return (size_t)moe::prefill_layout(*shape, max_tokens).total;
  }
  if (mode == 2) {
    if (max_tokens < 1 || max_tokens > moe::kPrefillMaxTokens) return 0;
    return (size_t)moe::prefill_layout(*shape, max_tokens, true).total;
  }
  return 0;
}

moe_status moe_iq4nl_decode(const moe_shape* shape, const moe_expert_weights* w,
                            const uint16_t* x, int32_t T, const int32_t* ids,
                            const float* weights, float* y, void* ws, size_t ws_bytes,
                            uint32_t* status, void* stream) {
  moe_status st = layer_args(shape, w, x, T, MOE_MAX_DECODE_TOKENS, ids, weights, y, ws, status);
  if (st != MOE_OK || T == 0) return st;
  const moe::DecodeLayout L = moe::decode_layout(*shape, T);
  if (ws_bytes < (size_t)L.total) return MOE_ERR_WORKSPACE;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  moe::DecodeParams p = decode_params(shape, w, x, T, ids, weights, y, ws, L, status);
  const cudaError_t e = moe::launch_decode(p, sms, g_pdl.load() != 0,
                                           reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_iq4nl_decode_routed(const moe_shape* shape, const uint16_t* router_w,
                                   const float* router_bias, const moe_expert_weights* w,
                                   const uint16_t* x, int32_t T, int32_t* ids, float* weights,
                                   float* y, void* ws, size_t ws_bytes, uint32_t* status,
                                   void* stream) {
  moe_status st = layer_args(shape, w, x, T, MOE_MAX_DECODE_TOKENS, ids, weights, y, ws, status);
  if (st != MOE_OK || T == 0) return st;
  if (!router_w) return MOE_ERR_INVALID_ARG;
  if (!aligned(router_w, 16) || (router_bias && !aligned(router_bias, 4)))
    return MOE_ERR_MISALIGNED;
  const moe::DecodeLayout L = moe::decode_layout(*shape, T);
  if (ws_bytes < (size_t)L.total) return MOE_ERR_WORKSPACE;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  moe::DecodeParams p = decode_params(shape, w, x, T, ids, weights, y, ws, L, status);
  p.Wr = router_w;
  p.bias = router_bias;
  p.ids_out = ids;
  p.w_out = weights;
  p.scores = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + L.scores);
  const cudaError_t e = moe::launch_decode_routed(p, sms, g_pdl.load() != 0,
                                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_iq4nl_decode_layers(const moe_shape* shape, int32_t n_layers,
                                   const moe_layer_weights* layers, const uint16_t* x,
                                   int32_t T, int32_t chained, int32_t* ids, float* weights,
                                   float* y, void* ws, size_t ws_bytes, uint32_t* status,
                                   void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (n_layers < 1 || n_layers > MOE_MAX_LAYERS || !layers) return MOE_ERR_INVALID_ARG;
  if (chained != 0 && chained != 1) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > MOE_MAX_DECODE_TOKENS) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    st = check_weights(shape, &layers[l].experts);
    if (st != MOE_OK) return st;
    if (!layers[l].router_w) return MOE_ERR_INVALID_ARG;
    if (!aligned(layers[l].router_w, 16) ||
        (layers[l].router_bias && !aligned(layers[l].router_bias, 4)))
      return MOE_ERR_MISALIGNED;
  }
  if (T == 0) return MOE_OK;
  if (!x || !ids || !weights || !y) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ids, 4) || !aligned(weights, 4) ||
      !aligned(ws, 256) || (status && !aligned(status, 4)))
    return MOE_ERR_MISALIGNED;
  const moe::DecodeLayout L = moe::decode_layout(*shape, T);
  if (ws_bytes < (size_t)L.total) return MOE_ERR_WORKSPACE;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  moe::DecodeParams p =
      decode_params(shape, &layers[0].experts, x, T, ids, weights, y, ws, L, status);
  p.route = 1;
  p.ids_out = ids;
  p.w_out = weights;
  p.L = n_layers;
  p.chained = chained;
  p.tscores = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ws) + L.tscores);
  p.xc = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(ws) + L.xc);
  p.scores = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + L.scores);
  static_assert(sizeof(moe::LayerTable) <= 16 * 1024, "layer table fits the launch parameters");
  moe::LayerTable lt;
  std::memset(&lt, 0, sizeof(lt));
  for (int l = 0; l < n_layers; ++l) {
    const moe_expert_weights& e = layers[l].experts;
    lt.layer[l] = moe::LayerPtrs{
        reinterpret_cast<const uint8_t*>(e.gate),    reinterpret_cast<const uint8_t*>(e.up),
        reinterpret_cast<const uint8_t*>(e.down),    reinterpret_cast<const uint8_t*>(e.sh_gate),
        reinterpret_cast<const uint8_t*>(e.sh_up),   reinterpret_cast<const uint8_t*>(e.sh_down),
        layers[l].router_w, layers[l].router_bias};
  }
  const cudaError_t e = moe::launch_decode_layers(p, lt, sms, g_pdl.load() != 0,
                                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_iq4nl_prefill_grouped(const moe_shape* shape, const moe_expert_weights* w,
                                     const uint16_t* x, int32_t T, const int32_t* ids,
                                     const float* weights, float* y, void* ws,
                                     size_t ws_bytes, uint32_t* status, void* stream) {
  moe_status st = layer_args(shape, w, x, T, moe::kPrefillMaxTokens, ids, weights, y, ws, status);
  if (st != MOE_OK || T == 0) return st;
  const moe::PrefillLayout L = moe::prefill_layout(*shape, T);
  if (ws_bytes < (size_t)L.total) return MOE_ERR_WORKSPACE;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  const cudaError_t e = moe::launch_prefill(*shape, *w, x, T, ids, weights, y,
                                            reinterpret_cast<uint8_t*>(ws), L, status, sms,
                                            g_pdl.load() != 0,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_iq4nl_prefill_grouped_fp8(const moe_shape* shape, const moe_expert_weights* w,
                                         const int8_t* row_exp, const uint16_t* x, int32_t T,
                                         const int32_t* ids, const float* weights, float* y,
                                         void* ws, size_t ws_bytes, uint32_t* status,
                                         void* stream) {
  moe_status st = layer_args(shape, w, x, T, moe::kPrefillMaxTokens, ids, weights, y, ws, status);
  if (st != MOE_OK || T == 0) return st;
  if (!row_exp) return MOE_ERR_INVALID_ARG;
  if (!moe::prefill_fp8_supported(*shape)) return MOE_ERR_UNSUPPORTED;
  const moe::PrefillLayout L = moe::prefill_layout(*shape, T, true);
  if (ws_bytes < (size_t)L.total) return MOE_ERR_WORKSPACE;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  const cudaError_t e = moe::launch_prefill_fp8(*shape, *w, row_exp, x, T, ids, weights, y,
                                                reinterpret_cast<uint8_t*>(ws), L, status, sms,
                                                g_pdl.load() != 0,
                                                reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int64_t moe_fp8_row_exponent_count(const moe_shape* shape) {
  if (check_shape(shape) != MOE_OK) return 0;
  return moe::fp8_row_exponent_count(*shape);
}

moe_status moe_iq4nl_fp8_row_exponents(const moe_shape* shape, const moe_expert_weights* w,
                                       int8_t* row_exp, void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!w || !row_exp) return MOE_ERR_INVALID_ARG;
  st = check_weights(shape, w);
  if (st != MOE_OK) return st;
  const cudaError_t e = moe::launch_fp8_row_exponents(*shape, *w, row_exp,
                                                      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_iq4nl_dequantize_e4m3(const void* mat, int64_t rows, int32_t K, int8_t* row_exp,
                                     uint8_t* out, void* stream) {
  if (rows < 0 || K < 32 || K % 32) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!mat || !row_exp || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(mat, 2) || !aligned(out, 4)) return MOE_ERR_MISALIGNED;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  const cudaError_t e = moe::launch_dequant_e4m3(mat, rows, K, row_exp, out, sms,
                                                 reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_iq4nl_dequantize(const void* blocks, int64_t n_blocks, int32_t mode,
                                void* out, void* stream) {
  if (n_blocks < 0 || (mode != MOE_DEQUANT_FP32 && mode != MOE_DEQUANT_FP16 &&
                       mode != MOE_DEQUANT_FP32_ONE_TOKEN))
    return MOE_ERR_INVALID_ARG;
  if (n_blocks == 0) return MOE_OK;
  if (!blocks || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(blocks, 2) || !aligned(out, 4)) return MOE_ERR_MISALIGNED;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  const cudaError_t e = moe::launch_dequant(blocks, n_blocks, mode, out, sms,
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_sanitize_routes(const int32_t* ids, const float* weights, int64_t n,
                               int32_t n_experts, int32_t* ids_out, float* weights_out,
                               uint32_t* status, void* stream) {
  if (n < 0 || n_experts < 1) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!ids || !weights || !ids_out || !weights_out) return MOE_ERR_INVALID_ARG;
  if (!aligned(ids, 4) || !aligned(weights, 4) || !aligned(ids_out, 4) ||
      !aligned(weights_out, 4) || (status && !aligned(status, 4)))
    return MOE_ERR_MISALIGNED;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  const cudaError_t e = moe::launch_sanitize(ids, weights, n, n_experts, ids_out, weights_out,
                                             status, sms, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int32_t moe_launches_per_call(const moe_shape* shape, int32_t T, int32_t call) {
  const moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return 0;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  if (call == 0) return 1;
  if (call == 1 || call == 2) {
    if (T > MOE_MAX_DECODE_TOKENS) return MOE_ERR_INVALID_ARG;
    moe::DecodeParams p{};
    p.H = shape->hidden;
    p.F = shape->ffn;
    p.Fs = shape->n_shared ? shape->ffn_shared : 0;
    p.E = shape->n_experts;
    p.k = shape->top_k;
    p.n_shared = shape->n_shared;
    p.T = T;
    p.route = call == 2 ? 1 : 0;
    size_t sm = 0;
    int rg = 0, rmax = 0;
    if (moe::fused_decode_supported(p, sms, &sm, &rg, &rmax)) return 1;
    p.route = 0;                     // otherwise the router runs first, then the layer
    const int n = moe::decode_launches(p, sms);
    return call == 2 ? n + 1 : n;
  }
  if (call == 3) return moe::prefill_launches(*shape, T);
  if (call == 5) return moe::prefill_fp8_supported(*shape) ? 6 : 0;
  if (call >= 6) {                           // 4 + 2 * n_layers + chained
    const int n_layers = (call - 4) / 2, chained = (call - 4) % 2;
    if (n_layers < 1 || n_layers > MOE_MAX_LAYERS || T > MOE_MAX_DECODE_TOKENS)
      return MOE_ERR_INVALID_ARG;
    moe::DecodeParams p{};
    p.H = shape->hidden;
    p.F = shape->ffn;
    p.Fs = shape->n_shared ? shape->ffn_shared : 0;
    p.E = shape->n_experts;
    p.k = shape->top_k;
    p.n_shared = shape->n_shared;
    p.T = T;
    p.route = 1;
    p.L = n_layers;
    p.chained = chained;
    return moe::layers_launches(p, sms);
  }
  return MOE_ERR_INVALID_ARG;
}

int32_t moe_set_pdl(int32_t enable) { return g_pdl.exchange(enable ? 1 : 0); }

uint64_t moe_set_barrier_wait_ns(uint64_t ns) { return g_barrier_wait_ns.exchange(ns); }

const char* moe_status_string(int32_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported by this build";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_MISALIGNED: return "misaligned pointer";
    case MOE_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char* moe_version(void) { return "libmoe 0.1 sm_103a"; }

}  // extern "C"
