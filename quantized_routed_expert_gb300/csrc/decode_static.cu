// Decode without a caller-provided workspace (moe_iq4nl_decode_static).
//
// Some callers cannot allocate device memory when they need to run the layer:
// code that executes while another component is capturing its stream into a
// CUDA graph with a private memory pool, hosts that embed the library behind
// an allocator they do not control, and runtimes whose device memory is fully
// planned up front. For them this entry point runs moe_iq4nl_decode on a fixed
// scratch area that is part of the library itself: a file-scope device array
// of kStaticScratchBytes, which every GPU that loads the library holds until
// the process exits. The call allocates and frees nothing.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "decode.cuh"
#include "moe.h"

namespace {

constexpr size_t kStaticScratchBytes = MOE_STATIC_SCRATCH_BYTES;   // 8 MiB

// The scratch itself. Device code could name it directly; host code must
// obtain its device address with cudaGetSymbolAddress (the host-side name is
// only a stand-in, not a device address).
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Set-up, once per device, with that device current: the scratch's address.
// It is kept for the life of the process and never looked up again, so it goes
// stale if the device's context is destroyed (cudaDeviceReset); moe.h rules
// out calls after a reset.
moe_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

namespace {
inline bool aligned_to(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}
}  // namespace

extern "C" moe_status moe_iq4nl_decode_static(const moe_shape* shape,
                                              const moe_expert_weights* w, const uint16_t* x,
                                              int32_t T, const int32_t* ids,
                                              const float* weights, float* y, uint32_t* status,
                                              void* stream) {
  if (!shape || T < 0 || T > MOE_MAX_DECODE_TOKENS) return MOE_ERR_INVALID_ARG;
  if (T == 0) return moe_iq4nl_decode(shape, w, x, 0, ids, weights, y, nullptr, 0, status, stream);
  // Every argument is checked before anything is enqueued: the same rules as
  // moe_iq4nl_decode, which checks them again.
  const size_t need = moe_workspace_bytes(shape, T, 0);
  if (need == 0) return MOE_ERR_INVALID_ARG;                   // shape rule broken
  if (need > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch
  if (!w || !x || !ids || !weights || !y) return MOE_ERR_INVALID_ARG;
  const int nw = shape->n_shared ? 6 : 3;
  const void* wp[6] = {w->gate, w->up, w->down, w->sh_gate, w->sh_up, w->sh_down};
  for (int i = 0; i < nw; ++i) {
    if (!wp[i]) return MOE_ERR_INVALID_ARG;
    if (!aligned_to(wp[i], 16)) return MOE_ERR_MISALIGNED;
  }
  if (!aligned_to(x, 16) || !aligned_to(y, 16) || !aligned_to(ids, 4) ||
      !aligned_to(weights, 4) || (status && !aligned_to(status, 4)))
    return MOE_ERR_MISALIGNED;
  void* scratch = nullptr;
  const moe_status st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  // The scratch keeps whatever the previous call left (a call that timed out
  // may leave its counters non-zero). The fused decode kernel needs its
  // grid-barrier counters at zero when it starts, so clear exactly those words
  // on the stream first: a stream-ordered memset, not an allocation.
  // Everything else in the scratch is written before it is read within a call.
  const moe::DecodeLayout L = moe::decode_layout(*shape, T);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(reinterpret_cast<uint8_t*>(scratch) + L.sync, 0, 64, s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return moe_iq4nl_decode(shape, w, x, T, ids, weights, y, scratch, kStaticScratchBytes, status,
                          stream);
}
