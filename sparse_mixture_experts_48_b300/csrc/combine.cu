// K4 -- combine: y[t] = sum_{j<k, kept} w_j O[slot(t, j)] + sum_{s<S} O[T k + s T + t]
// accumulated in fp32 in exactly that order (routed choices by rank, then the
// shared experts), one warp per token, streaming 16-byte loads of the fp32
// expert outputs with up to 8 of them in flight per lane.
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
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kWarps = 4;

// The expert outputs are read once: L1 bypassed, L2 evict-first.
__device__ __forceinline__ float4 ld_stream(const float4* p, uint64_t policy) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

// One warp per token.  The token's sources are its k routed choices (weight
// w_j, skipped when dropped) followed by the S shared experts (weight 1, rows
// T k + s T + t of O), NJ >= k + S of them padded to a power of two.  Each lane
// first issues every 16-byte load of U chunks (NJ * U <= 8 loads in flight per
// lane), then sums them in source order.  The expert outputs O are fp32
// whatever the storage dtype, so y is rounded once, at the store.
template <int NJ, bool Y_F32>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(CombineArgs a) {
  pdl_wait();
  constexpr int U = NJ >= 8 ? 1 : 8 / NJ;
  const int lane = threadIdx.x % 32;
  const int64_t t = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  if (t >= a.T || *(volatile const uint32_t*)a.err != 0u) return;
  const int k = a.k, nj = a.k + a.S;
  int64_t my_row = -1;
  float my_w = 0.f;
  if (lane < k) {
    my_row = a.slot[t * k + lane];
    my_w = a.topk_w[t * k + lane];
  } else if (lane < nj) {
    my_row = a.rows_tk + (int64_t)(lane - k) * a.T + t;
    my_w = 1.f;
  }
  int64_t row[NJ];
  float w[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    row[j] = __shfl_sync(0xffffffffu, my_row, j);
    w[j] = __shfl_sync(0xffffffffu, my_w, j);
  }
  const int64_t chunks = a.d / 4;   // 4 fp32 per 16-byte chunk
  const float4* O = (const float4*)a.o;
  const uint64_t policy = l2_policy_evict_first();
  for (int64_t c0 = lane; c0 < chunks; c0 += 32 * U) {
    float4 v[NJ][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + 32 * u;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if (row[j] >= 0 && c < chunks) v[j][u] = ld_stream(O + row[j] * chunks + c, policy);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + 32 * u;
      if (c >= chunks) break;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        if (row[j] >= 0) {
          // fma with weight 1 rounds exactly like a plain add
          acc.x = fmaf(w[j], v[j][u].x, acc.x);
          acc.y = fmaf(w[j], v[j][u].y, acc.y);
          acc.z = fmaf(w[j], v[j][u].z, acc.z);
          acc.w = fmaf(w[j], v[j][u].w, acc.w);
        }
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
}

template <int NJ>
cudaError_t launch_nj(const CombineArgs& a, int64_t blocks, cudaStream_t s) {
  if (a.y_f32) return launch_maybe_pdl(a.pdl, combine_kernel<NJ, true>, dim3((unsigned)blocks), dim3(kWarps * 32), 0, s, a);
  return launch_maybe_pdl(a.pdl, combine_kernel<NJ, false>, dim3((unsigned)blocks), dim3(kWarps * 32), 0, s, a);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const int64_t blocks = (a.T + kWarps - 1) / kWarps;
  const int nj = a.k + a.S;
  if (nj > 16) return cudaErrorInvalidValue;   // k <= 8 and S <= 8
  if (nj <= 1) return launch_nj<1>(a, blocks, s);
  if (nj <= 2) return launch_nj<2>(a, blocks, s);
  if (nj <= 4) return launch_nj<4>(a, blocks, s);
  if (nj <= 8) return launch_nj<8>(a, blocks, s);
  return launch_nj<16>(a, blocks, s);
}

}  // namespace moe
