// Backward pass with expert-choice routing: the two kernels that differ from
// token choice.  The scalar is L = sum_t <dy_t, y_t> + dL_aux * L_aux with
//   y_t = sum over the experts e that chose t of p_te o_e(x_t) + shared experts,
// p the gate probabilities over all E, the choice itself piecewise constant.
//
//   ec_combine_bwd  one warp per grouped row (expert e, token t):
//                   dO_row = p_te dy_t (bf16) and dw_row = <dy_t, O_row> (fp32).
//   ec_router_bwd   one warp per token, lane l owning experts l, l + 32, ...:
//                   dp_te = dw_row(t, e) where e chose t, plus the load-balance
//                   term dL_aux alpha E f_e / T with f_e = 1/E; then through the
//                   gating over all E (softmax: dl = p (dp - <p, dp>); normalised
//                   sigmoid p = s / sum s: dl = (dp - <p, dp>) / sum s s (1 - s)).
// The expert GEMMs, dx, dW_g and the bias sums are those of token choice.
// Every sum runs in a fixed order (a lane's strided terms, then a fixed xor
// tree), so gradients are bitwise reproducible.
//
// Sources: "MoE架构解析" §2.2 (expert choice); "MoE混合专家模型：Transformer稀疏前馈
// 网络原理与PyTorch实现" §4.3 (main and aux loss in one backward), §2.3 (the
// load-balance loss); "MoE架构解析" §四 技术飞跃③ (normalised sigmoid gating).
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kWarps = 4;

__global__ void __launch_bounds__(kWarps * 32) ec_combine_bwd_kernel(EcCombineBwdArgs a) {
  const int lane = threadIdx.x % 32;
  const int64_t r = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  if (r >= a.rows || *(volatile const uint32_t*)a.err != 0u || r % a.Cs >= a.C) return;
  const int d = a.d;
  const int64_t t = a.perm[r];
  const float w = a.w_row[r];
  const uint16_t* dy = (const uint16_t*)a.dy + t * d;
  const float* o = a.o + r * d;
  uint16_t* dO = (uint16_t*)a.dO + r * d;
  float dot = 0.f;
  for (int c = lane * 2; c < d; c += 64) {
    const uint32_t yy = *(const uint32_t*)(dy + c);
    const float y0 = bf16_bits_to_f32((uint16_t)(yy & 0xffffu)), y1 = bf16_bits_to_f32((uint16_t)(yy >> 16));
    const float2 ov = *(const float2*)(o + c);
    dot = fmaf(y0, ov.x, dot);
    dot = fmaf(y1, ov.y, dot);
    *(uint32_t*)(dO + c) = pack_bf16x2(w * y0, w * y1);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  if (lane == 0) a.dw_row[r] = dot;
}

constexpr int kMaxE = 256;
constexpr int kPerLane = kMaxE / 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__global__ void __launch_bounds__(kWarps * 32) ec_router_bwd_kernel(EcRouterBwdArgs a) {
  const int lane = threadIdx.x % 32;
  const int64_t t = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  if (t >= a.T || *(volatile const uint32_t*)a.err != 0u) return;
  const int E = a.E;
  const bool soft = a.gating == MOE_GATE_SOFTMAX;
  const float* lt = a.logits + t * E;
  float g[kPerLane], dp[kPerLane];
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    const int e = lane + 32 * j;
    g[j] = e < E ? lt[e] : -INFINITY;
    mx = fmaxf(mx, g[j]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  // the gating's numerators (exp(l - max), or the sigmoids) and their total
  float z = 0.f;
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    const int e = lane + 32 * j;
    if (e < E) {
      g[j] = soft ? expf(g[j] - mx) : 1.f / (1.f + expf(-g[j]));
      z += g[j];
    } else {
      g[j] = 0.f;
    }
  }
  z = warp_sum(z);
  const float rz = 1.f / z;
  // dp: the chosen pairs' <dy, o>, plus the aux term (f_e = 1/E)
  const float aux = (float)((double)a.dL_aux * a.alpha / (double)a.T);
  float pdp = 0.f;
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    const int e = lane + 32 * j;
    dp[j] = 0.f;
    if (e < E) {
      dp[j] = aux;
      if ((a.bits[t * a.EW + j] >> lane) & 1u) dp[j] += a.dw_row[a.tok_row[t * E + e]];
      pdp += g[j] * rz * dp[j];
    }
  }
  pdp = warp_sum(pdp);
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    const int e = lane + 32 * j;
    if (e < E) {
      const float pe = g[j] * rz;
      a.dl[t * E + e] = soft ? pe * (dp[j] - pdp) : (dp[j] - pdp) * rz * g[j] * (1.f - g[j]);
    }
  }
}

}  // namespace

cudaError_t launch_ec_combine_bwd(const EcCombineBwdArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  if (a.C <= 0 || a.Cs < a.C || a.d % 64 != 0) return cudaErrorInvalidValue;
  ec_combine_bwd_kernel<<<(unsigned)((a.rows + kWarps - 1) / kWarps), kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ec_router_bwd(const EcRouterBwdArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (a.E > kMaxE) return cudaErrorInvalidValue;
  ec_router_bwd_kernel<<<(unsigned)((a.T + kWarps - 1) / kWarps), kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
