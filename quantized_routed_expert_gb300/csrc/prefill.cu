// Prefill path of libmoe (sm_103a).
#include "prefill.cuh"

namespace moe {

namespace {
int64_t up256(int64_t v) { return (v + 255) / 256 * 256; }
}  // namespace

PrefillLayout prefill_layout(const moe_shape& s, int64_t T) {
  PrefillLayout L{};
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off = up256(off + bytes);
    return o;
  };
  const int64_t E = s.n_experts, k = s.top_k, H = s.hidden, F = s.ffn;
  const int64_t Fs = s.n_shared ? s.ffn_shared : 0;
  const int64_t rows = T * k + (s.n_shared ? T : 0);
  const int64_t fmax = F > Fs ? F : Fs;
  L.counts = take((E + 2) * 4);
  L.offsets = take((E + 2) * 4);
  L.perm = take(T * k * 4);
  L.x16 = take(T * H * 2);
  L.h16 = take(rows * fmax * 2);
  L.o = take(rows * H * 4);
  L.sched = take(64 * 1024);
  L.total = off;
  return L;
}

int prefill_launches(const moe_shape&, int) { return 0; }

cudaError_t launch_prefill(const moe_shape&, const moe_expert_weights&, const uint16_t*, int,
                           const int32_t*, const float*, float*, uint8_t*, const PrefillLayout&,
                           uint32_t*, int, bool, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace moe
