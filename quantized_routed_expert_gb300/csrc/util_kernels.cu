// Small kernels of libmoe: the IQ4_NL dequantiser and the route sanitiser.
#include "common.cuh"
#include "tc.cuh"
#include "util_kernels.cuh"

#include <mutex>

namespace moe {

cudaError_t ensure_smem_attr(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static const void* keys[256];
  static int devs[256];
  static size_t vals[256];
  static int n = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (keys[i] == kernel && devs[i] == dev && vals[i] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n; ++i)
    if (keys[i] == kernel && devs[i] == dev) { vals[i] = bytes; return cudaSuccess; }
  if (n < 256) { keys[n] = kernel; devs[n] = dev; vals[n] = bytes; ++n; }
  return cudaSuccess;
}

// The block decoder on its own, run through the very device functions the
// layer kernels use, one mode per decoder, so that a bit-exact comparison of
// its output covers the code that runs:
//   MOE_DEQUANT_FP32: split_pair + iq4_lookup8 + iq4_dot_block (decode, an
//     expert with several tokens);
//   MOE_DEQUANT_FP16: dequant_block_half (the prefill producers);
//   MOE_DEQUANT_FP32_ONE_TOKEN: pair_scales + iq4_pair_dot1 (decode, an expert
//     with one token: the split table, no merge).
// The dot-product decoders give a table value as the dot product of the block
// with a one-hot activation vector in the pair layout (word j holds the 16-bit
// values of positions j and j + 16), scaled by d exactly as the kernels scale
// a block's integer sum (fmaf of the integer, as float, by d times a unit
// activation scale, onto -0). One thread takes one pair of consecutive blocks (36
// bytes, the unit every layer kernel reads); a last odd block is paired with
// a zero block.
__device__ __forceinline__ void load_pair_bytes(const uint8_t* b, bool two, uint32_t (&w)[9]) {
#pragma unroll
  for (int i = 0; i < 9; ++i) {
    uint32_t v = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int o = 4 * i + j;
      const uint32_t byte = (o < kBlockB || two) ? b[o] : 0u;
      v |= byte << (8 * j);
    }
    w[i] = v;
  }
}

__global__ void dequant_kernel(const uint8_t* __restrict__ blocks, int64_t n_blocks, int mode,
                               void* __restrict__ out) {
  const int64_t n_pairs = (n_blocks + 1) / 2;
  for (int64_t pi = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; pi < n_pairs;
       pi += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b0 = 2 * pi;
    const bool two = b0 + 1 < n_blocks;
    uint32_t w[9];
    load_pair_bytes(blocks + b0 * kBlockB, two, w);
    const int nb = two ? 2 : 1;
    if (mode == MOE_DEQUANT_FP16) {
      uint32_t q0[4], q1[4], h[2][16];
#pragma unroll
      for (int i = 0; i < 4; ++i) q0[i] = prmt(w[i], w[i + 1], 0x5432u);
#pragma unroll
      for (int i = 0; i < 4; ++i) q1[i] = w[5 + i];
      dequant_block_half(q0, (uint16_t)(w[0] & 0xFFFFu), h[0]);
      dequant_block_half(q1, (uint16_t)(w[4] >> 16), h[1]);
      uint32_t* o = reinterpret_cast<uint32_t*>(out) + b0 * 16;
      for (int b = 0; b < nb; ++b)
#pragma unroll
        for (int i = 0; i < 16; ++i) o[16 * b + i] = h[b][i];
      continue;
    }
    float* o = reinterpret_cast<float*>(out) + b0 * 32;
    float d0, d1;
    uint32_t t0[8], t1[8];
    if (mode == MOE_DEQUANT_FP32) {
      uint32_t a0[4], a1[4];
      split_pair(w, d0, d1, a0, a1);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        iq4_lookup8(a0[i], t0[2 * i], t0[2 * i + 1]);
        iq4_lookup8(a1[i], t1[2 * i], t1[2 * i + 1]);
      }
    } else {
      pair_scales(w, d0, d1);
    }
#pragma unroll 1
    for (int pos = 0; pos < 32; ++pos) {
      // one-hot at position pos of both blocks: word pos % 16, half pos / 16
      uint32_t v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0u;
      const uint32_t one = pos < 16 ? 1u : 0x10000u;
      v[pos & 15] = one;
      v[16 + (pos & 15)] = one;
      int i0, i1;
      if (mode == MOE_DEQUANT_FP32) {
        i0 = iq4_dot_block(t0, v);
        i1 = iq4_dot_block(t1, v + 16);
      } else {
        iq4_pair_dot1(w, v, i0, i1);
      }
      // (an addend of -0 keeps the sign of a zero product, as d*T has it)
      o[pos] = fmaf((float)i0, d0 * 1.0f, -0.0f);
      if (two) o[32 + pos] = fmaf((float)i1, d1 * 1.0f, -0.0f);
    }
  }
}

__global__ void sanitize_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w,
                                int64_t n, int E, int32_t* ids_out, float* w_out,
                                uint32_t* status) {
  int bad = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t id = ids[i];
    const float wi = w[i];
    const bool ok = id >= 0 && id < E;
    ids_out[i] = ok ? id : 0;
    w_out[i] = ok ? wi : 0.0f;
    bad += ok ? 0 : 1;
  }
  if (status) {
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xFFFFFFFFu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(status, (uint32_t)(bad < 0xFFFF ? bad : 0xFFFF));
  }
}

cudaError_t launch_dequant(const void* blocks, int64_t n_blocks, int mode, void* out,
                           int num_sms, cudaStream_t stream) {
  const int64_t n = (n_blocks + 1) / 2;
  int64_t grid = (n + 127) / 128;
  if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
  if (grid < 1) grid = 1;
  dequant_kernel<<<(int)grid, 128, 0, stream>>>(reinterpret_cast<const uint8_t*>(blocks),
                                                 n_blocks, mode, out);
  return cudaGetLastError();
}

cudaError_t launch_sanitize(const int32_t* ids, const float* w, int64_t n, int E,
                            int32_t* ids_out, float* w_out, uint32_t* status, int num_sms,
                            cudaStream_t stream) {
  int64_t grid = (n + 255) / 256;
  if (grid > (int64_t)num_sms * 8) grid = (int64_t)num_sms * 8;
  if (grid < 1) grid = 1;
  sanitize_kernel<<<(int)grid, 256, 0, stream>>>(ids, w, n, E, ids_out, w_out, status);
  return cudaGetLastError();
}

}  // namespace moe
