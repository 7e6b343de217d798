// E4M3 quantisation for the FP8 expert path.
//
//   quantize_rows     one CTA per bf16 row: its largest magnitude a, then codes
//                     q_i = e4m3(fl32(v_i * fl32(448 / a))) and the row's decoding
//                     scale fl32(a / 448) (a floored at 2^-60).  Used on the hidden
//                     activations between the two expert GEMMs, and on its own.
//   quantize_weights  one CTA per 32 columns of a [K, N] weight slab: the same
//                     rule per column (one scale per output unit), written
//                     transposed as [N, K] so that the GEMM reads both operands
//                     K-major.
//
// Source: "MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现" §5.2 (expert
// parameters quantised from 16-bit to 8-bit floats to halve their memory).  The
// format is E4M3; rounding is to nearest with ties to even, saturating at 448.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kQThreads = 256;

__device__ __forceinline__ float block_max(float m, float* s_part) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) s_part[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < kQThreads / 32 ? s_part[lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) s_part[kQThreads / 32] = m;
  }
  __syncthreads();
  return s_part[kQThreads / 32];
}

__global__ void __launch_bounds__(kQThreads) quantize_rows_kernel(QuantRowsArgs a) {
  __shared__ float s_part[kQThreads / 32 + 1];
  if (a.err && *(volatile const uint32_t*)a.err != 0u) return;
  int64_t r = blockIdx.x;
  if (r < a.rows0) {
    if (a.live0 && r >= (int64_t)*a.live0) return;
  } else {
    r = a.row1 + (r - a.rows0);
  }
  const int64_t words = a.cols / 8;
  const uint4* src = (const uint4*)a.X + r * words;
  float m = 0.f;
  for (int64_t c = threadIdx.x; c < words; c += kQThreads) m = fmaxf(m, amax_bf16x8(src[c]));
  m = block_max(m, s_part);
  float rr, sc;
  e4m3_scales(m, rr, sc);
  const int64_t ow = a.cols / 16;
  uint4* dst = (uint4*)(a.Q + r * a.cols);
  for (int64_t c = threadIdx.x; c < ow; c += kQThreads) {
    const uint2 lo = e4m3x8_from_bf16(src[2 * c], rr);
    const uint2 hi = e4m3x8_from_bf16(src[2 * c + 1], rr);
    dst[c] = make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  if (threadIdx.x == 0) a.scale[r] = sc;
}

constexpr int kWN = 32;    // columns per CTA
constexpr int kWK = 64;    // k rows per transposed tile

__global__ void __launch_bounds__(kQThreads) quantize_weights_kernel(QuantWeightsArgs a) {
  __shared__ float s_part[kQThreads / 32][kWN];
  __shared__ float s_r[kWN];
  __shared__ __align__(16) uint8_t s_tile[kWN][kWK + 8];
  const int64_t g = blockIdx.y, n0 = (int64_t)blockIdx.x * kWN;
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  const uint16_t* W = (const uint16_t*)a.W + g * a.K * a.N;
  const int64_t n = n0 + tx;
  float m = 0.f;
  if (n < a.N)
    for (int64_t k = ty; k < a.K; k += kQThreads / 32) m = fmaxf(m, fabsf(bf16_bits_to_f32(W[k * a.N + n])));
  s_part[ty][tx] = m;
  __syncthreads();
  if (ty == 0) {
    float mm = s_part[0][tx];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) mm = fmaxf(mm, s_part[i][tx]);
    float r, sc;
    e4m3_scales(mm, r, sc);
    s_r[tx] = r;
    if (n < a.N) a.scale[g * a.N + n] = sc;
  }
  __syncthreads();
  const float r = s_r[tx];
  uint8_t* Q = a.Q + g * a.N * a.K;
  const int wrow = threadIdx.x / 8, wch = threadIdx.x % 8;   // write: 32 rows x 8 chunks of 8 codes
  for (int64_t k0 = 0; k0 < a.K; k0 += kWK) {
    for (int i = ty; i < kWK; i += kQThreads / 32) {
      const int64_t k = k0 + i;
      uint8_t q = 0;
      if (n < a.N && k < a.K) q = (uint8_t)(e4m3x4(__fmul_rn(bf16_bits_to_f32(W[k * a.N + n]), r), 0.f, 0.f, 0.f) & 0xffu);
      s_tile[tx][i] = q;
    }
    __syncthreads();
    if (n0 + wrow < a.N && k0 + wch * 8 < a.K)
      *reinterpret_cast<uint2*>(Q + (n0 + wrow) * a.K + k0 + wch * 8) =
          *reinterpret_cast<const uint2*>(&s_tile[wrow][wch * 8]);
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_quantize_rows(const QuantRowsArgs& a, cudaStream_t s) {
  const int64_t blocks = a.rows0 + a.rows1;
  if (blocks <= 0) return cudaSuccess;
  if (a.cols % 16 != 0 || blocks >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  quantize_rows_kernel<<<(unsigned)blocks, kQThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_weights(const QuantWeightsArgs& a, cudaStream_t s) {
  if (a.G <= 0 || a.K <= 0 || a.N <= 0) return cudaSuccess;
  if (a.K % 16 != 0 || a.G > 65535) return cudaErrorInvalidValue;
  dim3 grid((unsigned)((a.N + kWN - 1) / kWN), (unsigned)a.G);
  quantize_weights_kernel<<<grid, kQThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
