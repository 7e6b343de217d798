// K4 -- combine: y[t] = sum_{j<k, kept} w_j O[slot(t, j)] + sum_{s<S} O[T k + s T + t]
// accumulated in fp32 in exactly that order (routed choices by rank, then the
// shared experts), one warp per token, 16-byte loads of the fp32 expert outputs.
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

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// The expert outputs O are fp32 whatever the layer's storage dtype, so the only
// rounding after the expert GEMMs is the final store of y.
template <bool Y_F32>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(CombineArgs a) {
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
  for (int64_t c = lane; c < chunks; c += 32) {
    float4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k && slots[j] >= 0) v[j] = ld_stream(O + (int64_t)slots[j] * chunks + c);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k && slots[j] >= 0) {
        acc.x = fmaf(w[j], v[j].x, acc.x);
        acc.y = fmaf(w[j], v[j].y, acc.y);
        acc.z = fmaf(w[j], v[j].z, acc.z);
        acc.w = fmaf(w[j], v[j].w, acc.w);
      }
    }
    for (int s = 0; s < a.S; ++s) {
      const float4 u = ld_stream(O + (a.rows_tk + (int64_t)s * a.T + t) * chunks + c);
      acc.x += u.x; acc.y += u.y; acc.z += u.z; acc.w += u.w;
    }
    if (Y_F32) {
      reinterpret_cast<float4*>(a.y)[t * chunks + c] = acc;
    } else {
      uint2 out;
      out.x = pack_bf16x2(acc.x, acc.y);
      out.y = pack_bf16x2(acc.z, acc.w);
      reinterpret_cast<uint2*>(a.y)[t * chunks + c] = out;
    }
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const int64_t blocks = (a.T + kWarps - 1) / kWarps;
  if (a.y_f32)
    combine_kernel<true><<<(unsigned)blocks, kWarps * 32, 0, s>>>(a);
  else
    combine_kernel<false><<<(unsigned)blocks, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
