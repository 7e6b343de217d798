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
// Expert GEMM tile rows (the M of one tcgen05 MMA with cta_group::1).
constexpr int kGemmBM = 128;

struct WsHeader {
  uint32_t err;        // OR of kErr* bits
  uint32_t err_where;  // first site that set a bit (diagnostic)
  uint32_t pad[62];
};

// Byte offsets of the regions inside the caller's workspace.
struct WsLayout {
  size_t hdr, hist, psum, base, lrank, npre, offsets, seg, slot, xperm, h, o;
  size_t ec_scores, ec_bits, ec_tokrow, ec_wrow, ec_perm;   // expert choice only
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

__device__ __forceinline__ void record_error(uint32_t* err, uint32_t bit, uint32_t where) {
  if (atomicOr(err, bit) == 0u) atomicExch(err + 1, where);
}

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

}  // namespace moe
