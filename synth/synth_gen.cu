// Device fill of synthetic IQ4_NL expert tensors (input generation only).
//
// The same counter-based generator as synth/__init__.py, written from the
// same definition (SplitMix64 by Vigna; "draw i" = splitmix64(key + i)):
//   block b of expert e uses draws 3b, 3b+1, 3b+2 of key(seed, layer, tensor, e);
//   d = fp16_rne(1e-4 + 3e-4 * U), U = (draw >> 11) * 2^-53,
//   index bytes = draws 3b+1 and 3b+2, little-endian.
// The arithmetic for d is IEEE double multiply-then-add (no contraction) and a
// direct double->half RNE conversion, so host and device agree bit for bit.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace {

__host__ __device__ inline uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ inline uint64_t gen_key(uint64_t seed, uint64_t layer, uint64_t tensor,
                                            uint64_t sub) {
  uint64_t k = splitmix64(seed);
  k = splitmix64(k ^ layer);
  k = splitmix64(k ^ tensor);
  return splitmix64(k ^ sub);
}

__global__ void fill_iq4nl_kernel(uint16_t* __restrict__ dst, int64_t n_experts,
                                  int64_t blocks_per_expert, uint64_t seed, uint64_t layer,
                                  uint64_t tensor, int64_t expert0) {
  const int64_t total = n_experts * blocks_per_expert;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i / blocks_per_expert;
    const int64_t b = i - e * blocks_per_expert;
    const uint64_t k = gen_key(seed, layer, tensor, (uint64_t)(expert0 + e));
    const uint64_t h0 = splitmix64(k + 3ull * (uint64_t)b);
    const uint64_t h1 = splitmix64(k + 3ull * (uint64_t)b + 1ull);
    const uint64_t h2 = splitmix64(k + 3ull * (uint64_t)b + 2ull);
    const double u = (double)(h0 >> 11) * 0x1.0p-53;
    const double s = __dadd_rn(1e-4, __dmul_rn(3e-4, u));
    const uint16_t dbits = __half_as_ushort(__double2half(s));
    uint16_t* o = dst + i * 9;                    // 18-byte blocks, 2-byte aligned
    o[0] = dbits;
#pragma unroll
    for (int j = 0; j < 4; ++j) o[1 + j] = (uint16_t)(h1 >> (16 * j));
#pragma unroll
    for (int j = 0; j < 4; ++j) o[5 + j] = (uint16_t)(h2 >> (16 * j));
  }
}

}  // namespace

extern "C" int synth_fill_iq4nl(void* dst, int64_t n_experts, int64_t blocks_per_expert,
                                uint64_t seed, uint64_t layer, uint64_t tensor, int64_t expert0,
                                void* stream) {
  if (!dst || n_experts < 0 || blocks_per_expert < 0 || ((uintptr_t)dst & 1)) return -1;
  const int64_t total = n_experts * blocks_per_expert;
  if (total == 0) return 0;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 152 * 32) blocks = 152 * 32;
  fill_iq4nl_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(
      (uint16_t*)dst, n_experts, blocks_per_expert, seed, layer, tensor, expert0);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
