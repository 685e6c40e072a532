// tcgen05 (5th-generation tensor core), TMEM and tensor-map TMA wrappers (sm_100 family).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "common.cuh"

namespace moe {

// Shared-memory matrix descriptor for a K-major operand stored in the 128-byte
// swizzled canonical layout: 8-row atoms of 8 x 128 B, atoms 1024 B apart
// (stride byte offset), the 16-byte chunk c of row r stored at chunk c ^ (r % 8).
// The tile base is 1024-byte aligned. Advancing K by 16 fp16 elements adds 32 B
// to the start address.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address, 16-byte units
  d |= (uint64_t)1 << 16;                     // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset: 8-row atoms
  d |= (uint64_t)1 << 46;                     // descriptor version (sm_100)
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with E4M3 A and B (kind::f8f6f4; the instruction descriptor's A and
// B format fields hold 0, E4M3, as for fp16 above).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole warp: allocate `ncols` TMEM columns, address written to *dst (shared).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets TMEM lane
// (lane base + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
// 8 columns (32-bit) of this warp's 32 TMEM lanes: lane i gets lane i's
// columns taddr .. taddr + 7.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                 "=r"(v[6]), "=r"(v[7])
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 2D tiled TMA load (box given by the tensor map) completing on `bar`.
// x (innermost coordinate, elements) must make x * elsize a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Offset table for fp16 dequantisation: byte j holds T[j] + 128 (1..241), so
// that the half with bits 0x6400 | byte is exactly 1024 + T + 128.
constexpr uint32_t kTabU0 = 0x3F2D1801u;   // T[0..3]+128  = 1, 24, 45, 63
constexpr uint32_t kTabU1 = 0x766A5D4Fu;   // T[4..7]+128  = 79, 93, 106, 118
constexpr uint32_t kTabU2 = 0xA6998D81u;   // T[8..11]+128 = 129, 141, 153, 166
constexpr uint32_t kTabU3 = 0xF1D9C5B5u;   // T[12..15]+128 = 181, 197, 217, 241

// Eight codes (4 index bytes) -> the 8 offset table values in K order:
// lo = (U[lo nibble of byte 0..3]), hi = (U[hi nibble of byte 0..3]).
// prmt with selector nibbles whose bit 3 is clear (one instruction; the
// __byte_perm intrinsic masks a run-time selector itself).
__device__ __forceinline__ void iq4_lookup8_split(uint32_t q, uint32_t& lo, uint32_t& hi) {
  const uint32_t qm = q & 0x77777777u;
  const uint32_t sel = 0x32103210u | ((q >> 1) & 0x44444444u);
  const uint32_t r0 = prmt(prmt(kTabU0, kTabU1, qm), prmt(kTabU2, kTabU3, qm), sel);  // L0 H0 L1 H1
  const uint32_t qm1 = qm >> 16;
  const uint32_t r1 =
      prmt(prmt(kTabU0, kTabU1, qm1), prmt(kTabU2, kTabU3, qm1), sel >> 16);         // L2 H2 L3 H3
  lo = prmt(r0, r1, 0x6420u);
  hi = prmt(r0, r1, 0x7531u);
}

// Four offset-table bytes -> four fp16 d*T, each the round-to-nearest-even of
// the exact product (T is exact in fp16; one multiply rounds once).
__device__ __forceinline__ void offsets_to_half4(uint32_t u, __half2 d2, uint32_t& o01,
                                                 uint32_t& o23) {
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  uint32_t h01 = prmt(u, 0x64646464u, 0x4140u);
  uint32_t h23 = prmt(u, 0x64646464u, 0x4342u);
  __half2 t01 = __hsub2(*reinterpret_cast<__half2*>(&h01), bias);
  __half2 t23 = __hsub2(*reinterpret_cast<__half2*>(&h23), bias);
  __half2 w01 = __hmul2(t01, d2);
  __half2 w23 = __hmul2(t23, d2);
  o01 = *reinterpret_cast<uint32_t*>(&w01);
  o23 = *reinterpret_cast<uint32_t*>(&w23);
}

// One 32-weight block (its 4 index words, fp16 scale bits) to 32 fp16 weights
// d*T[q] in K order, two to a word: words 0..7 hold weights 0..15 (low
// nibbles), words 8..15 weights 16..31 (high nibbles). The prefill producers
// call this for every block they put into an A tile.
__device__ __forceinline__ void dequant_block_half(const uint32_t (&q)[4], uint16_t dbits,
                                                   uint32_t (&w)[16]) {
  const __half dh = __ushort_as_half(dbits);
  const __half2 d2 = __halves2half2(dh, dh);
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) iq4_lookup8_split(q[i], lo[i], hi[i]);
#pragma unroll
  for (int i = 0; i < 4; ++i) offsets_to_half4(lo[i], d2, w[2 * i], w[2 * i + 1]);     // 0..15
#pragma unroll
  for (int i = 0; i < 4; ++i) offsets_to_half4(hi[i], d2, w[8 + 2 * i], w[8 + 2 * i + 1]);  // 16..31
}

// ---------------------------------------------------------------------------
// E4M3 (OCP 8-bit float: bias 7, largest finite 448, no infinities) operands.

// Two fp32 values to two E4M3 codes, round to nearest even, finite overflow
// saturated to +-448: the first operand goes to the upper byte.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^e as an fp32 (e in [-126, 127]).
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// v 2^a 2^b for an E4M3 accumulator v (zero, or of magnitude in [2^-18, 2^30]:
// sums of products of E4M3 codes) and the exponents of its row (a, in
// [-14, 15]) and token (b). v 2^a is exact and normal, so one rounding at most,
// as in ldexpf(v, a + b), which serves when 2^b is not a normal fp32.
// v 2^e, with s = 2^e precomputed when e is in [-126, 127] (then the product
// is exact unless it falls below the normal range, where it rounds once, as
// ldexpf does); ldexpf otherwise.
__device__ __forceinline__ float pow2_scale(float v, int e, float s) {
  return (e >= -126 && e <= 127) ? v * s : ldexpf(v, e);
}
__device__ __forceinline__ float pow2_of(int e) {
  return exp2i(e < -126 ? -126 : (e > 127 ? 127 : e));
}

__device__ __forceinline__ float scale_acc(float v, float sa, int b, float sb) {
  return (b >= -126 && b <= 127) ? (v * sa) * sb : ldexpf(v * sa, b);
}

// The 16 E4M3 codes of one block's table, e4m3(d T[i] 2^-E) for the block's
// fp16 scale d and its row's exponent E: byte i of t[j] is code 4j + i. d T is
// exact in fp32 (11 by 7 significant bits) and the power of two is exact, so
// each code is the round-to-nearest-even of the exact scaled weight.
__device__ __forceinline__ void e4m3_block_table(uint16_t dbits, int E, uint32_t (&t)[4]) {
  const float ds = __half2float(__ushort_as_half(dbits)) * exp2i(-E);
  const float T0 = -127.f, T1 = -104.f, T2 = -83.f, T3 = -65.f, T4 = -49.f, T5 = -35.f,
              T6 = -22.f, T7 = -10.f, T8 = 1.f, T9 = 13.f, T10 = 25.f, T11 = 38.f, T12 = 53.f,
              T13 = 69.f, T14 = 89.f, T15 = 113.f;
  auto pack = [&](float a, float b, float c, float d) {
    return (uint32_t)cvt_e4m3x2(b * ds, a * ds) | ((uint32_t)cvt_e4m3x2(d * ds, c * ds) << 16);
  };
  t[0] = pack(T0, T1, T2, T3);
  t[1] = pack(T4, T5, T6, T7);
  t[2] = pack(T8, T9, T10, T11);
  t[3] = pack(T12, T13, T14, T15);
}

// Eight codes (one index word) through a 16-byte table t (as above), in the
// order of the word's nibbles: r0 = codes of index byte 0's low and high
// nibble, then byte 1's, r1 = the same for bytes 2 and 3 (three prmt per four
// codes, on a table held in registers).
__device__ __forceinline__ void lookup16_nibbles(uint32_t q, const uint32_t (&t)[4], uint32_t& r0,
                                                 uint32_t& r1) {
  const uint32_t qm = q & 0x77777777u;
  const uint32_t sel = 0x32103210u | ((q >> 1) & 0x44444444u);
  r0 = prmt(prmt(t[0], t[1], qm), prmt(t[2], t[3], qm), sel);
  const uint32_t qm1 = qm >> 16;
  r1 = prmt(prmt(t[0], t[1], qm1), prmt(t[2], t[3], qm1), sel >> 16);
}

// The E4M3 operands' order of K inside each 32-value block: position p holds
// value 4 (p / 8) + (p / 2) % 4 + 16 (p % 2), i.e. values j and j + 16 side by
// side, the order in which a block's index bytes hold them (low nibble j, high
// nibble j + 16). A and B of the contraction share it, so the sums are the
// same; the weight producers then store the lookups as they come out.
__host__ __device__ constexpr int e4m3_block_pos_value(int p) {
  return 4 * (p >> 3) + ((p >> 1) & 3) + 16 * (p & 1);
}

// One 32-weight block (its 4 index words, fp16 scale bits) of a row with
// exponent E to its 32 E4M3 codes in the block order above: byte p of
// w[p / 4]. The fp8 prefill producers call this for every block they put into
// an A tile.
__device__ __forceinline__ void dequant_block_e4m3(const uint32_t (&q)[4], uint16_t dbits, int E,
                                                   uint32_t (&w)[8]) {
  uint32_t t[4];
  e4m3_block_table(dbits, E, t);
#pragma unroll
  for (int i = 0; i < 4; ++i) lookup16_nibbles(q[i], t, w[2 * i], w[2 * i + 1]);
}

// floor(log2 |v|) - 6 from an fp32 bit pattern of |v| (0 for zero), the
// exponent that puts a vector's largest magnitude in [64, 128).
__device__ __forceinline__ int vec_exponent_bits(uint32_t mbits) {
  if (mbits == 0u) return 0;
  const int f = (int)(mbits >> 23);
  if (f == 0) return (31 - __clz(mbits)) - 149 - 6;    // subnormal: value = m 2^-149
  return (f - 127) - 6;
}

}  // namespace moe
