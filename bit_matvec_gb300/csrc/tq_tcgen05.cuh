// tq_tcgen05.cuh -- small wrappers over the 5th-generation tensor-core
// instructions (tcgen05.*) and the exact f16 conversions used by both
// tensor-core kernels. Internal to the library.
#pragma once

#include <cuda_fp8.h>

#include "tq_internal.cuh"

namespace tq {
namespace tc {

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B f16
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t idesc_f16(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with A and B e4m3 (format code 0 in
// bits 7-9 and 10-12) and D f32: the same fields as idesc_f16, read under the
// other kind.
constexpr uint32_t idesc_e4m3(int m, int n) { return idesc_f16(m, n); }

// Shared-memory matrix descriptor: start >> 4 (bits 0-13), LBO >> 4 (16-29),
// SBO >> 4 (32-45), the constant 0b001 at bits 46-48, no swizzle (61-63 = 0).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem], kind::f16.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f8f6f4 (K = 32): each 32-bit column of
// A holds four consecutive k as bytes 0..3.
__device__ __forceinline__ void mma_e4m3_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}

// ---------------------------------------------------------------- CTA pairs
//
// With .cta_group::2 the two CTAs of a cluster of 2 (ranks 0 and 1) act as one
// MMA unit: one MMA of M = 256 takes rows 0..127 of A and D from the tensor
// memory of rank 0 and rows 128..255 from that of rank 1 (the same column
// addresses in both), and N/2 columns of B from the shared memory of each CTA
// (the same shared-memory offsets in both); rank 0 issues it. Tensor memory is
// allocated, released and freed by one warp in each CTA of the pair, with the
// same column count.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of both CTAs of the cluster: a release-acquire barrier.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  if (CG == 2)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(slot_smem), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(slot_smem), "r"(ncols) : "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_relinquish() {
  if (CG == 2)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if (CG == 2)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f8f6f4, on the CTA pair (M = 256).
__device__ __forceinline__ void mma_e4m3_tmem_a_pair(uint32_t d_tmem, uint32_t a_tmem,
                                                     uint64_t b_desc, uint32_t idesc,
                                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at the same shared-memory offset in both CTAs of the
// pair when the pair MMAs this thread issued so far are complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(bar), "h"((uint16_t)3) : "memory");
}

// Arrive on the mbarrier at shared offset `bar` of the cluster CTA `rank`
// (this CTA's own when rank is its own rank), with the default semantics. The
// data it hands over is in tensor memory (A written, an accumulator read),
// ordered by the tcgen05 fences on either side of the barrier; a release at
// cluster scope here measured about 1,500 cycles per arrival on GB300.
__device__ __forceinline__ void mbarrier_arrive_rank(uint32_t bar, uint32_t rank) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
      "mbarrier.arrive.shared::cluster.b64 _, [ra];\n\t}"
      ::"r"(bar), "r"(rank) : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane -> registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// registers -> 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
        "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
        "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
        "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// registers -> 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
        "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
        "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// ---------------------------------------------------------------- e4m3 operands
//
// The e4m3 paths split an int8 activation q exactly into lo = q & 15 (0..15)
// and 16 * hi with hi = q >> 4 (-8..7); both parts, and both divided by 4,
// have at most four significant bits, so they are exact in e4m3. A weight
// code u at bits 2s..2s+1 of a byte, masked in place, is the e4m3 byte of
// u * 2^-9 (s = 0) or u * 4 * 2^-9 (s = 1; u = 2 sets the lowest exponent
// bit, 2^-6); after a right shift by 4 the same holds for s = 2, 3. Where A
// carries the factor 4 (odd s) the activation part is divided by 4, so every
// product is u * lo * 2^-9 or u * 16 hi * 2^-9 exactly, and f32 sums of up
// to 2^15 such products are exact.

// Two e4m3 bytes (x in the low byte); the values passed are exact in e4m3.
__device__ __forceinline__ uint32_t e4m3x2(float x, float y) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x, y), __NV_SATFINITE, __NV_E4M3);
}

// Four int8 activations (bytes of v) -> their lo and 16 * hi parts as e4m3
// bytes, both multiplied by m (1 or 1/4).
__device__ __forceinline__ void split_e4m3(uint32_t v, float m, uint32_t& lo, uint32_t& hi) {
  float l[4], h[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int q = (int)(int8_t)(v >> (8 * j));
    l[j] = (float)(q & 15) * m;
    h[j] = (float)((q >> 4) * 16) * m;
  }
  lo = e4m3x2(l[0], l[1]) | (e4m3x2(l[2], l[3]) << 16);
  hi = e4m3x2(h[0], h[1]) | (e4m3x2(h[2], h[3]) << 16);
}

// Codes of slot s (bits 2s..2s+1 of two bytes, placed in the low byte of each
// 16-bit half) -> f16 pair of w = u - 1. OR-ing 0x6400 (1024.0) makes the half
// 1024 + u * 4^s exactly; one FMA by 4^-s plus -(1024 * 4^-s + 1) gives u - 1.
// The two constants are written as f16x2 bit patterns so that no conversion
// runs on the device.
template <int s> struct WConst;
template <> struct WConst<0> { static constexpr uint32_t m = 0x3C003C00u, b = 0xE401E401u; };  // 1, -1025
template <> struct WConst<1> { static constexpr uint32_t m = 0x34003400u, b = 0xDC04DC04u; };  // 1/4, -257
template <> struct WConst<2> { static constexpr uint32_t m = 0x2C002C00u, b = 0xD410D410u; };  // 1/16, -65
template <> struct WConst<3> { static constexpr uint32_t m = 0x24002400u, b = 0xCC40CC40u; };  // 1/64, -17

template <int s>
__device__ __forceinline__ uint32_t codes_to_w(uint32_t x) {
  const uint32_t v = (x & (0x00030003u << (2 * s))) | 0x64006400u;
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(WConst<s>::m), "r"(WConst<s>::b));
  return r;
}

// int8 x4 -> two f16 pairs (exact): bias to u8, place under exponent 0x64
// (1024 + byte), subtract 1152 (f16x2 bits 0x64806480).
__device__ __forceinline__ void s8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x5150);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x5352);
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// 16 consecutive 32-bit columns of this thread's TMEM lane -> registers,
// without waiting: the caller issues tcgen05.wait::ld before reading r.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Packed pairs of f32 (f32x2 arithmetic, one instruction per pair).
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ uint64_t f2_packf(float lo, float hi) {
  return f2_pack(__float_as_uint(lo), __float_as_uint(hi));
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
  return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace tc
}  // namespace tq
