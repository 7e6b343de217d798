// K4 -- combine: y[t] = sum_{j<k, kept} w_j O[slot(t, j)] + sum_{s<S} O[T k + s T + t]
// accumulated in fp32 in exactly that order (routed choices by rank, then the
// shared experts), one warp per token, 16-byte loads of the expert outputs.
// A dropped assignment adds nothing; the kept weights are not renormalised.
// No atomics: every y row is produced by one warp, so the result is bitwise
// reproducible.
//
// Sources: "MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现" §1.3 (weighted
// sum of the chosen experts' outputs); "手撕一个极简 MoE-FFN" §五/§六 (output +=
// weight * expert_out); "MoE架构解析" §三 关键技术① (dropped tokens skip the
// layer), §四 技术飞跃② (shared experts are always active).
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void fma8_bf16(float* acc, float w, uint4 v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] = fmaf(w, __uint_as_float(u[q] << 16), acc[2 * q]);
    acc[2 * q + 1] = fmaf(w, __uint_as_float(u[q] & 0xffff0000u), acc[2 * q + 1]);
  }
}

__device__ __forceinline__ void add8_bf16(float* acc, uint4 v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] += __uint_as_float(u[q] << 16);
    acc[2 * q + 1] += __uint_as_float(u[q] & 0xffff0000u);
  }
}

__global__ void __launch_bounds__(kWarps * 32) combine_bf16_kernel(CombineArgs a) {
  const int lane = threadIdx.x % 32;
  const int64_t t = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  if (t >= a.T) return;
  const int k = a.k;
  const int my_slot = lane < k ? a.slot[t * k + lane] : -1;
  const float my_w = lane < k ? a.topk_w[t * k + lane] : 0.f;
  int slots[8];
  float w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    slots[j] = __shfl_sync(0xffffffffu, my_slot, j);
    w[j] = __shfl_sync(0xffffffffu, my_w, j);
  }
  const int64_t chunks = a.d / 8;   // 8 bf16 per 16-byte chunk
  const uint4* O = (const uint4*)a.o;
  uint4* y = (uint4*)a.y + t * chunks;
  for (int64_t c = lane; c < chunks; c += 32) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k && slots[j] >= 0) v[j] = ld_stream(O + (int64_t)slots[j] * chunks + c);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k && slots[j] >= 0) fma8_bf16(acc, w[j], v[j]);
    for (int s = 0; s < a.S; ++s)
      add8_bf16(acc, ld_stream(O + (a.rows_tk + (int64_t)s * a.T + t) * chunks + c));
    uint4 out;
    out.x = pack_bf16x2(acc[0], acc[1]);
    out.y = pack_bf16x2(acc[2], acc[3]);
    out.z = pack_bf16x2(acc[4], acc[5]);
    out.w = pack_bf16x2(acc[6], acc[7]);
    y[c] = out;
  }
}

__global__ void __launch_bounds__(kWarps * 32) combine_f32_kernel(CombineArgs a) {
  const int lane = threadIdx.x % 32;
  const int64_t t = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  if (t >= a.T) return;
  const int k = a.k;
  const int my_slot = lane < k ? a.slot[t * k + lane] : -1;
  const float my_w = lane < k ? a.topk_w[t * k + lane] : 0.f;
  int slots[8];
  float w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    slots[j] = __shfl_sync(0xffffffffu, my_slot, j);
    w[j] = __shfl_sync(0xffffffffu, my_w, j);
  }
  const int64_t chunks = a.d / 4;   // 4 fp32 per 16-byte chunk
  const float4* O = (const float4*)a.o;
  float4* y = (float4*)a.y + t * chunks;
  for (int64_t c = lane; c < chunks; c += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k && slots[j] >= 0) {
        const float4 v = O[(int64_t)slots[j] * chunks + c];
        acc.x = fmaf(w[j], v.x, acc.x);
        acc.y = fmaf(w[j], v.y, acc.y);
        acc.z = fmaf(w[j], v.z, acc.z);
        acc.w = fmaf(w[j], v.w, acc.w);
      }
    }
    for (int s = 0; s < a.S; ++s) {
      const float4 v = O[(a.rows_tk + (int64_t)s * a.T + t) * chunks + c];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    y[c] = acc;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const int64_t blocks = (a.T + kWarps - 1) / kWarps;
  if (a.dtype == MOE_DT_BF16)
    combine_bf16_kernel<<<(unsigned)blocks, kWarps * 32, 0, s>>>(a);
  else
    combine_f32_kernel<<<(unsigned)blocks, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
