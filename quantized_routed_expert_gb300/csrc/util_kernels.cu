// Small kernels of libmoe: the IQ4_NL dequantiser and the route sanitiser.
#include "common.cuh"
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

// One thread per output pair of weights (j, j+16) of a block: the block's
// index byte j holds both codes. Exact fp32 product d*T[q], or the fp16
// round-to-nearest-even of it (an fp16 multiply of two fp16 values whose exact
// product is rounded once).
__global__ void dequant_kernel(const uint8_t* __restrict__ blocks, int64_t n_blocks, int fp16,
                               void* __restrict__ out) {
  const int64_t n = n_blocks * 16;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i >> 4;
    const int j = (int)(i & 15);
    const uint8_t* blk = blocks + b * kBlockB;
    const uint16_t dbits = (uint16_t)blk[0] | ((uint16_t)blk[1] << 8);
    const uint8_t qb = blk[2 + j];
    // table value via the same byte_perm lookup the kernels use
    uint32_t r0, r1;
    iq4_lookup8((uint32_t)qb, r0, r1);
    const int t_lo = (int)(int8_t)(r0 & 0xFF);
    const int t_hi = (int)(int8_t)((r0 >> 8) & 0xFF);
    const int64_t o = b * 32;
    if (fp16) {
      const __half d = __ushort_as_half(dbits);
      __half* oh = reinterpret_cast<__half*>(out);
      oh[o + j] = __hmul(d, __int2half_rn(t_lo));
      oh[o + j + 16] = __hmul(d, __int2half_rn(t_hi));
    } else {
      const float d = __half2float(__ushort_as_half(dbits));
      float* of = reinterpret_cast<float*>(out);
      of[o + j] = d * (float)t_lo;
      of[o + j + 16] = d * (float)t_hi;
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

cudaError_t launch_dequant(const void* blocks, int64_t n_blocks, int fp16, void* out,
                           int num_sms, cudaStream_t stream) {
  const int64_t n = n_blocks * 16;
  int64_t grid = (n + 255) / 256;
  if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
  if (grid < 1) grid = 1;
  dequant_kernel<<<(int)grid, 256, 0, stream>>>(reinterpret_cast<const uint8_t*>(blocks),
                                                 n_blocks, fp16, out);
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
