// K3f -- grouped expert GEMM for fp32 storage, on the CUDA cores.
//
// tcgen05 takes no fp32 operands (its nearest kind, tf32, keeps 10 mantissa
// bits, too coarse for a 1e-4 relative bound on y), so fp32 layers run this
// FFMA kernel.  One CTA computes a 128 x 64 tile of one segment; the bias and
// the activation (or the SwiGLU product of the two accumulators) are applied
// before the single store.  fp32 layers are the small configurations, where
// this kernel is latency-bound, not throughput-bound.
//
// Sources: "手撕一个极简 MoE-FFN" §四 (Expert = w2(relu(w1 x))), §六 (one expert
// runs once on all of its tokens); "术业有专攻：learn-minimind MoE混合专家模型架构
// 入门指南" §二 (SwiGLU experts).
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int BM = kGemmBM;   // 128 rows: the tile grid of the segment table
constexpr int BN = 64;
constexpr int BK = 16;
constexpr int kThreads = 256; // 16 x 16 threads, each 8 rows x 4 columns
static_assert(BM * BK % kThreads == 0 && BK * BN % kThreads == 0, "whole slices per thread");

__device__ __forceinline__ float act_f32(int act, float v) {
  if (act == MOE_ACT_RELU) return v > 0.f ? v : 0.f;
  if (act == MOE_ACT_GELU) return 0.5f * v * (1.f + erff(v * 0.70710678118654752f));
  return v;
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads) gemm_f32_kernel(GemmArgs a) {
  pdl_wait();
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN];
  __shared__ float B3s[SWIGLU ? BK : 1][BN];
  const int* mt = a.seg.mtile_start;
  for (int tile = blockIdx.y; tile < mt[a.G]; tile += gridDim.y) {
  int g = 0;
  {
    int lo = 0, hi = a.G - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (mt[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    g = lo;
  }
  const int m0 = (tile - mt[g]) * BM;
  const int rows = a.seg.rows[g];
  const int w = a.seg.w[g];
  const int orow = a.seg.out_row[g];
  const int arow = a.a_from_out_rows ? orow : a.seg.a_row[g];
  const float* A = (const float*)((a.a_from_out_rows || a.seg.a_src[g] == 0) ? a.A0 : a.A1);
  const int K = a.K, N = a.N;
  const int n0 = blockIdx.x * BN;
  const float* B = (const float*)a.B + (int64_t)w * K * N;
  const float* B3 = SWIGLU ? (const float*)a.B3 + (int64_t)w * K * N : nullptr;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;

  float acc[8][4], acc3[SWIGLU ? 8 : 1][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[i][j] = 0.f;
      if (SWIGLU) acc3[i][j] = 0.f;
    }

  // Software pipelined over k: the next k-slice's A and B elements are
  // loaded into registers while the current slice in shared memory is
  // multiplied, so a k-step costs its FMAs rather than a load round trip.
  constexpr int AE = BM * BK / kThreads;   // A elements per thread per slice (8)
  constexpr int BE = BK * BN / kThreads;   // B elements per thread per slice (4)
  float ra[AE], rb[BE], rb3[SWIGLU ? BE : 1];
  auto load_slice = [&](int k0) {
#pragma unroll
    for (int u = 0; u < AE; ++u) {
      const int i = threadIdx.x + u * kThreads;
      const int r = i / BK, c = i % BK;
      const bool ok = m0 + r < rows && k0 + c < K;
      ra[u] = ok ? A[(int64_t)(arow + m0 + r) * K + k0 + c] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < BE; ++u) {
      const int i = threadIdx.x + u * kThreads;
      const int r = i / BN, c = i % BN;
      const bool ok = k0 + r < K && n0 + c < N;
      rb[u] = ok ? B[(int64_t)(k0 + r) * N + n0 + c] : 0.f;
      if (SWIGLU) rb3[u] = ok ? B3[(int64_t)(k0 + r) * N + n0 + c] : 0.f;
    }
  };
  load_slice(0);
  for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
    for (int u = 0; u < AE; ++u) {
      const int i = threadIdx.x + u * kThreads;
      As[i % BK][i / BK] = ra[u];
    }
#pragma unroll
    for (int u = 0; u < BE; ++u) {
      const int i = threadIdx.x + u * kThreads;
      Bs[i / BN][i % BN] = rb[u];
      if (SWIGLU) B3s[i / BN][i % BN] = rb3[u];
    }
    __syncthreads();
    if (k0 + BK < K) load_slice(k0 + BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[8], bv[4], b3v[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) av[i] = As[kk][ty * 8 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bv[j] = Bs[kk][tx * 4 + j];
        if (SWIGLU) b3v[j] = B3s[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
          if (SWIGLU) acc3[i][j] = fmaf(av[i], b3v[j], acc3[i][j]);
        }
    }
    __syncthreads();
  }
  const float* bias = (const float*)a.bias;
  float* C = (float*)a.C;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = m0 + ty * 8 + i;
    if (r >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + tx * 4 + j;
      if (c >= N) continue;
      float v = acc[i][j];
      if (SWIGLU) {
        v = (v / (1.f + expf(-v))) * acc3[i][j];
      } else {
        if (bias) v += bias[(int64_t)w * N + c];
        v = act_f32(a.act, v);
      }
      C[(int64_t)(orow + r) * N + c] = v;
    }
  }
  __syncthreads();
  }
}

}  // namespace

cudaError_t launch_grouped_gemm_f32(const GemmArgs& a, cudaStream_t s) {
  if (a.max_mtiles <= 0) return cudaSuccess;
  dim3 grid((unsigned)((a.N + BN - 1) / BN), (unsigned)(a.max_mtiles < 65535 ? a.max_mtiles : 65535));
  if (a.act == MOE_ACT_SWIGLU) return launch_maybe_pdl(a.pdl, gemm_f32_kernel<true>, grid, dim3(kThreads), 0, s, a);
  return launch_maybe_pdl(a.pdl, gemm_f32_kernel<false>, grid, dim3(kThreads), 0, s, a);
}

}  // namespace moe
