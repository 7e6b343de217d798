// Inline-PTX wrappers for the 5th-generation tensor cores (tcgen05): TMEM
// fences and loads, the shared-memory matrix descriptor, the kind::f16
// instruction descriptor, MMA issue and commit for one CTA or a CTA pair, and
// the epilogue activations shared by the grouped GEMM kernels.
#pragma once
#include <math.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 at bits 46-47, and the
// 128-byte swizzle mode (2) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, 10-12 = 1), A K-major (bit 15 = 0), B N-major (bit 16
// = 1), N >> 3 in bits 17-22, M >> 4 in bits 24-28.  For a CTA pair M is the
// pair's (256): each CTA holds M/2 rows of A and N/2 columns of B.
constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (format code 0 in
// bits 7-9 and 10-12), fp32 accumulator, both operands K-major.
constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | (0u << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

template <uint32_t IDESC>
__device__ __forceinline__ void mma_bf16_cta1(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
      : "memory");
}
// Issued by one thread of the pair's even CTA; reads A and B from both CTAs'
// shared memory at the descriptors' offsets and accumulates into both CTAs' TMEM.
template <uint32_t IDESC>
__device__ __forceinline__ void mma_bf16_cta2(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
      : "memory");
}
// FP8 pair MMA: K = 32 codes (32 bytes) per instruction.
template <uint32_t IDESC>
__device__ __forceinline__ void mma_f8_cta2(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
      : "memory");
}
// The mbarrier gets one arrival once every MMA this thread issued so far is done.
__device__ __forceinline__ void mma_commit_cta1(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// Same for pair MMAs; the arrival goes to the mbarrier at local offset `bar` in
// every CTA of `cta_mask` (an mbarrier signal, no data moves).
__device__ __forceinline__ void mma_commit_cta2(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Epilogue activations: the erf GELU x Phi(x), and SiLU for the SwiGLU gate.
// Phi comes from the erf approximation of Abramowitz and Stegun, Handbook of
// Mathematical Functions, eq. 7.1.26 (after Hastings): for z >= 0,
// erf(z) = 1 - (a1 t + a2 t^2 + ... + a5 t^5) exp(-z^2), t = 1 / (1 + p z),
// with |error| <= 1.5e-7.  With z = |x| / sqrt 2 and h = (1/2) (a1 t + ... +
// a5 t^5) exp(-x^2 / 2): Phi(x) = 1 - h for x >= 0 and h for x < 0.  The
// approximate reciprocal and exponential add a few ulp of h; all of it is far
// below the bf16 rounding of the stored activation (2^-9 relative), and it
// costs about half the instructions of erff in an epilogue that is bound by
// instruction issue when the contraction is short.
__device__ __forceinline__ float gelu_erf(float x) {
  constexpr float kP = 0.3275911f * 0.70710678118654752f;   // p / sqrt 2
  constexpr float kA1 = 0.5f * 0.254829592f, kA2 = 0.5f * -0.284496736f, kA3 = 0.5f * 1.421413741f,
                  kA4 = 0.5f * -1.453152027f, kA5 = 0.5f * 1.061405429f;
  const float t = __fdividef(1.f, fmaf(kP, fabsf(x), 1.f));
  const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, kA5, kA4), kA3), kA2), kA1);
  const float h = poly * __expf(-0.5f * x * x);
  return x * (x >= 0.f ? 1.f - h : h);
}
__device__ __forceinline__ float silu(float v) { return v / (1.f + __expf(-v)); }

}  // namespace moe
