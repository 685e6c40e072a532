// Device helpers shared by the libmoe kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

constexpr int kBlockW = 32;       // weights per IQ4_NL block
constexpr int kBlockB = 18;       // bytes per IQ4_NL block
constexpr int kPairB = 36;        // bytes per pair of consecutive blocks

// ---------------------------------------------------------------------------
// The IQ4_NL table as packed int8 (bytes T[0..3], T[4..7], T[8..11], T[12..15]).
// T = {-127,-104,-83,-65,-49,-35,-22,-10,1,13,25,38,53,69,89,113}.
constexpr uint32_t kTab0 = 0xBFAD9881u;
constexpr uint32_t kTab1 = 0xF6EADDCFu;
constexpr uint32_t kTab2 = 0x26190D01u;
constexpr uint32_t kTab3 = 0x71594535u;

// Eight 4-bit codes (one 32-bit word of a block's index bytes) to eight int8
// table values. Bytes of r0: T[c0], T[c1], T[c2], T[c3]; r1: T[c4..c7], where c
// are the nibbles from least significant up. One prmt picks from the lower half
// of the table (T[0..7]) and one from the upper half (T[8..15]) by the low three
// bits of each code; a third keeps, per byte, the half that bit 3 names. The
// selector nibbles handed to prmt have bit 3 clear (prmt's sign-replicate mode
// stays off).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ void iq4_lookup8(uint32_t q, uint32_t& r0, uint32_t& r1) {
  const uint32_t qm = q & 0x77777777u;
  const uint32_t sel = 0x32103210u | ((q >> 1) & 0x44444444u);
  r0 = prmt(prmt(kTab0, kTab1, qm), prmt(kTab2, kTab3, qm), sel);
  const uint32_t qm1 = qm >> 16;
  r1 = prmt(prmt(kTab0, kTab1, qm1), prmt(kTab2, kTab3, qm1), sel >> 16);
}

// The table split for single-token dot products, with no per-byte merge:
// prmt over the lower half T[0..7] with the raw code gives T[c] for c < 8 and
// -1 for c >= 8 (prmt's sign-replicate mode on a negative entry); prmt over
// the upper half stored as T[8..15] + 1, with bit 3 of each code flipped, gives
// T[c] + 1 for c >= 8 and 0 for c < 8 (sign of a positive entry). The two
// signed bytes sum to T[c] for every code, so a dot product may take both.
constexpr uint32_t kTabP2 = 0x271A0E02u;   // T[8..11] + 1 = 2, 14, 26, 39
constexpr uint32_t kTabP3 = 0x725A4636u;   // T[12..15] + 1 = 54, 70, 90, 114
__device__ __forceinline__ uint32_t iq4_lo4(uint32_t codes) {      // low 16 bits used
  return prmt(kTab0, kTab1, codes);
}
__device__ __forceinline__ uint32_t iq4_hi4(uint32_t flipped) {    // codes ^ 0x8888
  return prmt(kTabP2, kTabP3, flipped);
}

// Exact integer dot products of both blocks of a pair (its 36 bytes as nine
// words, straight from shared memory) with one token's pair-layout vector v[32]
// (words 0..15 for block 0, 16..31 for block 1), on the split table: no byte
// realignment and no merge step; each code's value enters as its two parts.
// Block 0's index bytes are pair bytes 2..17 (aligned word i: the high half of
// w[i], then the low half of w[i+1]); block 1's are w[5..8].
__device__ __forceinline__ void iq4_pair_dot1(const uint32_t (&w)[9], const uint32_t* v,
                                              int& dot0, int& dot1) {
  int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo0 = w[i] >> 16, hi0 = w[i + 1];
    const uint32_t f0 = lo0 ^ 0x8888u, f1 = hi0 ^ 0x8888u;
    const uint32_t l0 = iq4_lo4(lo0), l1 = iq4_lo4(hi0);
    const uint32_t h0 = iq4_hi4(f0), h1 = iq4_hi4(f1);
    a0 = __dp2a_lo((int)v[4 * i + 0], (int)l0, a0);
    a1 = __dp2a_hi((int)v[4 * i + 1], (int)l0, a1);
    a2 = __dp2a_lo((int)v[4 * i + 0], (int)h0, a2);
    a3 = __dp2a_hi((int)v[4 * i + 1], (int)h0, a3);
    a0 = __dp2a_lo((int)v[4 * i + 2], (int)l1, a0);
    a1 = __dp2a_hi((int)v[4 * i + 3], (int)l1, a1);
    a2 = __dp2a_lo((int)v[4 * i + 2], (int)h1, a2);
    a3 = __dp2a_hi((int)v[4 * i + 3], (int)h1, a3);
  }
  dot0 = (a0 + a1) + (a2 + a3);
  a0 = a1 = a2 = a3 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t q = w[5 + i];
    const uint32_t qf = q ^ 0x88888888u;
    const uint32_t l0 = iq4_lo4(q), l1 = iq4_lo4(q >> 16);
    const uint32_t h0 = iq4_hi4(qf), h1 = iq4_hi4(qf >> 16);
    a0 = __dp2a_lo((int)v[16 + 4 * i + 0], (int)l0, a0);
    a1 = __dp2a_hi((int)v[16 + 4 * i + 1], (int)l0, a1);
    a2 = __dp2a_lo((int)v[16 + 4 * i + 0], (int)h0, a2);
    a3 = __dp2a_hi((int)v[16 + 4 * i + 1], (int)h0, a3);
    a0 = __dp2a_lo((int)v[16 + 4 * i + 2], (int)l1, a0);
    a1 = __dp2a_hi((int)v[16 + 4 * i + 3], (int)l1, a1);
    a2 = __dp2a_lo((int)v[16 + 4 * i + 2], (int)h1, a2);
    a3 = __dp2a_hi((int)v[16 + 4 * i + 3], (int)h1, a3);
  }
  dot1 = (a0 + a1) + (a2 + a3);
}
// The two fp16 scales of a pair (as fp32).
__device__ __forceinline__ void pair_scales(const uint32_t (&w)[9], float& d0, float& d1) {
  d0 = __half2float(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu)));
  d1 = __half2float(__ushort_as_half((unsigned short)(w[4] >> 16)));
}

// Exact integer dot product of one block's 32 table values (8 words from
// iq4_lookup8 over the 4 index words) with a 32-vector in "pair" layout:
// word j holds (v_j, v_{j+16}) as two int16. Byte order of the looked-up words
// is (c_j, c_{j+16}, c_{j+1}, c_{j+17}), which dp2a.lo/.hi consume in place.
__device__ __forceinline__ int iq4_dot_block(const uint32_t (&t)[8], const uint32_t* v) {
  int a0 = 0, a1 = 0;                  // two chains: half the dependent dp2a depth
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a0 = __dp2a_lo((int)v[4 * i + 0], (int)t[2 * i], a0);
    a1 = __dp2a_hi((int)v[4 * i + 1], (int)t[2 * i], a1);
    a0 = __dp2a_lo((int)v[4 * i + 2], (int)t[2 * i + 1], a0);
    a1 = __dp2a_hi((int)v[4 * i + 3], (int)t[2 * i + 1], a1);
  }
  return a0 + a1;
}

// Decode one block pair (36 bytes, 4-byte aligned, as 9 words) into two fp16
// scales and the 8 index words of each block.
__device__ __forceinline__ void split_pair(const uint32_t (&w)[9], float& d0, float& d1,
                                           uint32_t (&q0)[4], uint32_t (&q1)[4]) {
  d0 = __half2float(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu)));
#pragma unroll
  for (int i = 0; i < 4; ++i) q0[i] = __byte_perm(w[i], w[i + 1], 0x5432);
  d1 = __half2float(__ushort_as_half((unsigned short)(w[4] >> 16)));
#pragma unroll
  for (int i = 0; i < 4; ++i) q1[i] = w[5 + i];
}

__device__ __forceinline__ void load_pair_smem(const uint8_t* p, uint32_t (&w)[9]) {
  const uint32_t* p32 = reinterpret_cast<const uint32_t*>(p);
#pragma unroll
  for (int i = 0; i < 9; ++i) w[i] = p32[i];
}

// ---------------------------------------------------------------------------
// Top-k of one token by one warp (router, sigmoid + bias selection). keys[e],
// e < E, are sigmoid(score) + bias. The choice: the largest key first, ties to
// the lower index; NaN and -inf keys are never chosen, and once no key is left
// every further choice is expert 0.
// A key becomes an order-preserving integer (larger key, larger integer; -0
// and +0 equal; 0 for a key never chosen). Lane l holds keys l, l + 32, ... in
// NPL registers. Each round takes the warp's largest integer by one reduction
// and the lowest index holding it by a second, and the owning lane clears that
// register: no shared memory, no divergent branch.
__device__ __forceinline__ uint32_t ordered_key_bits(float k) {
  const uint32_t u = __float_as_uint(k + 0.0f);       // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The selection itself, on the order-preserving integers v[i] of keys
// lane + 32 i (0 for a key never chosen); v is consumed.
template <int NPL>
__device__ __forceinline__ int warp_topk_bits(uint32_t (&v)[NPL], int k) {
  const int lane = threadIdx.x & 31;
  int id = 0;
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
    // with mx == 0 (no key left) every lane offers its first slot: expert 0
    uint32_t hit = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) hit |= (v[i] == mx ? 1u : 0u) << i;
    const uint32_t cand = hit ? (uint32_t)(lane + 32 * (__ffs(hit) - 1)) : 0xFFFFFFFFu;
    const uint32_t bi = __reduce_min_sync(0xFFFFFFFFu, cand);
    if (lane == j) id = (int)bi;
    const bool mine = (int)(bi & 31u) == lane;
    const int ri = (int)(bi >> 5);
#pragma unroll
    for (int i = 0; i < NPL; ++i) v[i] = (mine && i == ri) ? 0u : v[i];
  }
  return id;
}
// Keys in registers: lane l holds keys l, l + 32, ... (-inf beyond E).
template <int NPL>
__device__ __forceinline__ int warp_topk_regs(const float (&kv)[NPL], int k) {
  uint32_t v[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) v[i] = kv[i] > -INFINITY ? ordered_key_bits(kv[i]) : 0u;
  return warp_topk_bits<NPL>(v, k);
}
template <int NPL>
__device__ __forceinline__ int warp_topk_ids_t(const float* keys, int E, int k) {
  const int lane = threadIdx.x & 31;
  float kv[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    kv[i] = e < E ? keys[e] : -INFINITY;                  // NaN and -inf: never chosen
  }
  return warp_topk_regs<NPL>(kv, k);
}
// Lane j < k returns the j-th chosen expert id. Two widths only (E <= 64 and
// E <= 512), for kernels whose code size matters.
__device__ __forceinline__ int warp_topk_ids_512(const float* keys, int E, int k) {
  return E <= 64 ? warp_topk_ids_t<2>(keys, E, k) : warp_topk_ids_t<16>(keys, E, k);
}
// Lane j < k returns the j-th chosen expert id (E <= 1024).
__device__ __forceinline__ int warp_topk_ids(const float* keys, int E, int k) {
  const int n = (E + 31) >> 5;
  if (n <= 2) return warp_topk_ids_t<2>(keys, E, k);
  if (n <= 4) return warp_topk_ids_t<4>(keys, E, k);
  if (n <= 8) return warp_topk_ids_t<8>(keys, E, k);
  if (n <= 16) return warp_topk_ids_t<16>(keys, E, k);
  return warp_topk_ids_t<32>(keys, E, k);
}
// Renormalised weights: lane j < k holds the j-th choice's sigmoid p and gets
// p over the sum of the k chosen sigmoids, added in choice order.
__device__ __forceinline__ float warp_renorm(float p, int k) {
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, p, j);
  return p / sum;
}

// ---------------------------------------------------------------------------
// 16-bit block quantisation of an activation vector (x or h).
// For 32 values with largest biased fp32 exponent e: M_i = rint(v_i 2^(141-e))
// clamped to 32767 (so |M_i| <= 2^15 - 1), scale = 2^(e-141). Blocks whose
// largest exponent is <= 14 (|v| < 2^-112) are zero; an inf/NaN gives a NaN
// scale so that it propagates to the output.
__device__ __forceinline__ float quant_factor(uint32_t emax) {
  return __uint_as_float((268u - emax) << 23);
}
__device__ __forceinline__ float quant_scale(uint32_t emax) {
  if (emax <= 14u) return 0.0f;
  if (emax >= 255u) return __uint_as_float(0x7FC00000u);
  return __uint_as_float((emax - 14u) << 23);
}
// Round to nearest even by adding 1.5 * 2^23: |v * factor| <= 2^15, so the sum
// lies in [2^23, 2^24), where the float spacing is 1 (an FMA and an integer
// subtract instead of a float-to-int conversion; the same value). v * factor
// is exact (factor is a power of two), so fusing the multiply changes nothing.
__device__ __forceinline__ int quant_one(float v, uint32_t emax) {
  if (emax <= 14u || emax >= 255u) return 0;
  const int m = __float_as_int(fmaf(v, quant_factor(emax), 12582912.0f)) - 0x4B400000;
  return m > 32767 ? 32767 : m;
}

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, 1D bulk copy (TMA), programmatic dependent launch.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// The suspend-time hint lets the hardware park the waiting thread until the
// phase completes (or the hint's time passes) instead of returning at once,
// so waiting warps do not spin and take issue slots from computing warps.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
// Whether the phase of parity `parity` of an mbarrier has completed (no wait).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: gives up after ~kWaitLimitNs, records MOE_STATUS_TIMEOUT and
// returns false. Nothing in libmoe waits without a limit.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      if (status) atomicOr(status, MOE_STATUS_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait, by the whole warp, until a shared-memory counter that other
// warps of the CTA raise reaches `target` (acquire at CTA scope: what they
// wrote before raising it is visible after). false after ~kWaitLimitNs.
__device__ __forceinline__ uint32_t ld_acquire_cta_shared(const uint32_t* a) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(a)) : "memory");
  return v;
}
__device__ __forceinline__ bool wait_count_cta(const uint32_t* a, uint32_t target,
                                               uint32_t* status) {
  if (ld_acquire_cta_shared(a) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (ld_acquire_cta_shared(a) >= target) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      if (status) atomicOr(status, MOE_STATUS_TIMEOUT);
      return false;
    }
  }
}

// Global -> shared bulk copy that completes `bytes` of transaction on `bar`.
// src and dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// An L2 policy that marks lines evict-first: for data read once per call
// (streamed expert weights), so that it does not push out what is reused (the
// kernel's own instructions, activations, routes, h).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// bulk_g2s with an L2 cache policy on the global reads.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Host: raise a kernel's dynamic shared memory limit once per (kernel, device),
// so that launches made during stream capture issue nothing but the launch.
cudaError_t ensure_smem_attr(const void* kernel, size_t bytes);

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + expf(-g)) * u;
}

}  // namespace moe
