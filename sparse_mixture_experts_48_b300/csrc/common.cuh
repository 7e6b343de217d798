// Shared device helpers and the workspace layout of the MoE-FFN forward path.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---- status bits recorded by kernels in the workspace header ----------------
enum : uint32_t { kErrTimeout = 1u, kErrDevice = 2u };

// Router tile: tokens per router CTA.  A CTA's local ranks fit in uint8.
constexpr int kRouterBM = 64;
// The bf16 router with E a multiple of 64 runs its logits on tcgen05 MMAs
// (M = 128 tokens, N = E) and takes 128 tokens per CTA.
constexpr int kRouterBMTc = 128;
__host__ __device__ inline int router_tile_tokens(int dtype, int E) {
  return (dtype == MOE_DT_BF16 && E % 64 == 0) ? kRouterBMTc : kRouterBM;
}
// Expert GEMM tile rows (the M of one tcgen05 MMA with cta_group::1).
constexpr int kGemmBM = 128;
// Most groups the standalone grouped GEMM takes.
constexpr int kGroupedGemmMaxGroups = 264;
// Limit of every device-side wait unless the caller sets one (2 s).
constexpr int64_t kDefaultTimeoutNs = 2000000000LL;

struct WsHeader {
  uint32_t err;          // OR of kErr* bits
  uint32_t err_where;    // first site that set a bit (diagnostic)
  uint32_t router_done;  // router CTAs finished (the last one runs the dispatch scan)
  uint32_t pad[61];
};

// Byte offsets of the regions inside the caller's workspace.
struct WsLayout {
  size_t hdr, hist, psum, base, lrank, npre, offsets, seg, slot, xperm, h, o;
  size_t ec_scores, ec_bits, ec_tokrow, ec_wrow, ec_perm;   // expert choice only
  size_t xs_perm, xq, xs_tok, hq, hs;                       // FP8 experts only
  size_t total;
  int64_t nblk;      // router CTAs
  int64_t rows_tk;   // rows of routed assignments: T * k, or E * C for expert choice
  int64_t rows_all;  // rows_tk + S * T
  int64_t ec_C;      // expert choice: tokens per expert; -1 for token choice
  int EW;            // words of the per-token expert mask
  int G;             // E + S weight slabs / segments
};

// Segment table for the grouped GEMMs (device arrays of G entries, + G+1 prefix).
struct SegTable {
  int* rows;         // rows of segment g
  int* w;            // weight slab of segment g
  int* out_row;      // first row of segment g in H / O
  int* a_row;        // first row of segment g in the GEMM-1 A source
  int* a_src;        // GEMM-1 A source: 0 = expert-grouped copy of x, 1 = x itself
  int* mtile_start;  // [G+1] prefix sum of ceil(rows / kGemmBM)
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

__device__ __forceinline__ void record_error(uint32_t* err, uint32_t bit, uint32_t where) {
  if (atomicOr(err, bit) == 0u) atomicExch(err + 1, where);
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before its predecessor has finished; it waits here,
// before its first read of the predecessor's results, until that grid has
// completed and its writes are visible.  Without the launch attribute this
// returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

// fp32 -> bf16 bits, round to nearest even (the hardware conversion).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&h);
}

// 32 consecutive bf16 at p (64 bytes, 16-byte aligned) -> fp32, four 16-byte loads.
__device__ __forceinline__ void load_bf16x32(const uint16_t* p, float (&f)[32]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = q[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      f[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
}

// ---- E4M3 (8-bit float: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
// largest finite 448) --------------------------------------------------------------
constexpr float kE4M3Max = 448.f;

// Scale pair of a vector whose largest magnitude is amax: encoding factor
// r = 448 / a and decoding scale s = a / 448, a = max(amax, 2^-60), both
// rounded once to fp32.
__device__ __forceinline__ void e4m3_scales(float amax, float& r, float& s) {
  const float a = fmaxf(amax, 0x1p-60f);
  r = __fdiv_rn(kE4M3Max, a);
  s = __fdiv_rn(a, kE4M3Max);
}

// Four fp32 values (already multiplied by r) -> four E4M3 codes, nearest with
// ties to even, saturating at +-448; v0 in the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
  uint16_t lo, hi;
  // The first source lands in the upper byte of the 16-bit result.
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v1), "f"(v0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v3), "f"(v2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// 8 bf16 (one 16-byte word) -> 8 E4M3 codes (8 bytes) with encoding factor r.
__device__ __forceinline__ uint2 e4m3x8_from_bf16(const uint4 v, float r) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float f[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __fmul_rn(__uint_as_float(w[j] << 16), r);
    f[2 * j + 1] = __fmul_rn(__uint_as_float(w[j] & 0xffff0000u), r);
  }
  return make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
}

// Largest |bf16| of one 16-byte word.
__device__ __forceinline__ float amax_bf16x8(const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
    m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
  }
  return m;
}

}  // namespace moe
