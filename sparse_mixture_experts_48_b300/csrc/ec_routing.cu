// Expert-choice routing: each expert chooses its C highest-scoring tokens
// (instead of each token choosing k experts), so every expert gets the same
// load; a token may be chosen by several experts or by none.
//
//   ec_select   one CTA per expert: 4-pass radix select (8 bits a pass) of the
//               C-th largest score in the expert's column of the scores
//               (expert-major [E, T], written by the router), then the chosen
//               tokens in token order: scores above the threshold, and of the
//               scores equal to it the lowest token indices.  Writes the grouped
//               order perm[e*C + i], each row's gate weight, each (token,
//               expert)'s row, and a per-token bit mask of the choosing experts.
//   ec_gather   one warp per grouped row: copies its token's row of x.
//   ec_combine  one warp per token: sum over the experts that chose it, in
//               ascending expert order, of weight x expert output, then the
//               shared experts.  No atomics: bitwise reproducible.
//
// Source: "MoE架构解析" §2.2 (expert choice: balanced expert load, tokens that
// several experts choose, tokens no expert chooses).  Scores are the gate
// probabilities; equal scores go to the lower token index.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxCachedT = 32768;   // keys kept in shared memory up to this T (128 KB)

// Block-wide exclusive scan of one int per thread; returns the block total.
__device__ int block_excl_scan(int v, int* s_warp, int* excl) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kSelWarps ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += n;
    }
    if (lane < kSelWarps) s_warp[lane] = wi - w;   // exclusive warp offsets
    if (lane == 31) s_warp[32] = wi;               // block total
  }
  __syncthreads();
  *excl = s_warp[warp] + incl - v;
  const int total = s_warp[32];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kSelThreads) ec_select_kernel(EcSelectArgs a) {
  extern __shared__ uint32_t s_keys[];            // cached keys (T <= kMaxCachedT)
  __shared__ int s_hist[256];
  __shared__ int s_warp[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int e = blockIdx.x;
  const int64_t T = a.T;
  const int64_t C = a.C;
  const float* col = a.scores_em + (int64_t)e * T;
  const bool cached = T <= kMaxCachedT;
  if (*(volatile const uint32_t*)a.err != 0u) return;
  // Scores are probabilities >= 0: their fp32 bit patterns order like the values.
  auto key = [&](int64_t t) -> uint32_t { return cached ? s_keys[t] : __float_as_uint(col[t]); };
  if (cached)
    for (int64_t t = threadIdx.x; t < T; t += kSelThreads) s_keys[t] = __float_as_uint(col[t]);
  if (threadIdx.x == 0) {
    s_prefix = 0u;
    s_remaining = (int)C;
  }
  __syncthreads();

  // Radix select, most significant byte first: after the four passes
  // s_prefix is the C-th largest key and s_remaining the number of tokens
  // with exactly that key still to take (the lowest token indices).
  uint32_t mask = 0u;
  if (C > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = threadIdx.x; i < 256; i += kSelThreads) s_hist[i] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      for (int64_t t = threadIdx.x; t < T; t += kSelThreads) {
        const uint32_t k = key(t);
        if ((k & mask) == prefix) atomicAdd(&s_hist[(k >> shift) & 255u], 1);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int rem = s_remaining, cum = 0, b = 255;
        for (; b > 0; --b) {
          if (cum + s_hist[b] >= rem) break;
          cum += s_hist[b];
        }
        s_remaining = rem - cum;
        s_prefix = prefix | ((uint32_t)b << shift);
      }
      mask |= 255u << shift;
      __syncthreads();
    }
  }
  const uint32_t thr = s_prefix;
  const int need_eq = C > 0 ? s_remaining : 0;

  // Chosen tokens in token order: key > thr, or key == thr among the first
  // need_eq such tokens.  Two running block scans (equal keys, chosen).
  int eq_base = 0, pos_base = 0;
  for (int64_t t0 = 0; t0 < T; t0 += kSelThreads) {
    const int64_t t = t0 + threadIdx.x;
    const uint32_t k = t < T ? key(t) : 0u;
    const bool gt = C > 0 && t < T && k > thr;
    const bool eq = C > 0 && t < T && k == thr;
    int eq_ex;
    const int eq_tot = block_excl_scan(eq ? 1 : 0, s_warp, &eq_ex);
    const bool take = gt || (eq && eq_base + eq_ex < need_eq);
    int pos_ex;
    const int pos_tot = block_excl_scan(take ? 1 : 0, s_warp, &pos_ex);
    if (take) {
      const int64_t row = (int64_t)e * C + pos_base + pos_ex;
      a.perm[row] = (int32_t)t;
      a.w_row[row] = __uint_as_float(k);
      a.tok_row[t * a.E + e] = (int32_t)row;
      atomicOr(&a.bits[t * a.EW + e / 32], 1u << (e % 32));
    }
    eq_base += eq_tot;
    pos_base += pos_tot;
  }
}

constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32) ec_gather_kernel(EcGatherArgs a) {
  const int lane = threadIdx.x % 32;
  const int64_t r = (int64_t)blockIdx.x * kGatherWarps + threadIdx.x / 32;
  if (r >= a.rows || *(volatile const uint32_t*)a.err != 0u) return;
  const int64_t t = a.perm[r];
  const int64_t chunks = (int64_t)a.d * a.esz / 16;
  const uint4* src = (const uint4*)((const uint8_t*)a.x + t * chunks * 16);
  uint4* dst = (uint4*)((uint8_t*)a.xperm + r * chunks * 16);
  const uint64_t policy = l2_policy_evict_first();
  constexpr int U = 4;
  for (int64_t c0 = lane; c0 < chunks; c0 += 32 * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c0 + 32 * u < chunks) v[u] = ld_stream_u4(src + c0 + 32 * u, policy);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c0 + 32 * u < chunks) st_stream_u4(dst + c0 + 32 * u, v[u], policy);
  }
}

constexpr int kCombineWarps = 4;
constexpr int kMaxSources = 256 + 8;   // E + S

__global__ void __launch_bounds__(kCombineWarps * 32) ec_combine_kernel(EcCombineArgs a) {
  __shared__ int64_t s_row[kCombineWarps][kMaxSources];
  __shared__ float s_w[kCombineWarps][kMaxSources];
  const int lane = threadIdx.x % 32, wl = threadIdx.x / 32;
  const int64_t t = (int64_t)blockIdx.x * kCombineWarps + wl;
  if (t >= a.T || *(volatile const uint32_t*)a.err != 0u) return;
  // The token's sources in order: choosing experts ascending, then the shared experts.
  int n = 0;
  for (int w = 0; w < a.EW; ++w) {
    uint32_t bits = a.bits[t * a.EW + w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      if (lane == 0) {
        const int64_t row = a.tok_row[t * a.E + w * 32 + b];
        s_row[wl][n] = row;
        s_w[wl][n] = a.w_row[row];
      }
      ++n;
    }
  }
  if (lane == 0)
    for (int s = 0; s < a.S; ++s) {
      s_row[wl][n + s] = a.rows_routed + (int64_t)s * a.T + t;
      s_w[wl][n + s] = 1.f;
    }
  n += a.S;
  __syncwarp();
  const int64_t chunks = a.d / 4;
  const float4* O = (const float4*)a.o;
  const uint64_t policy = l2_policy_evict_first();
  for (int64_t c = lane; c < chunks; c += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < n; ++j) {
      const uint4 u = ld_stream_u4(O + s_row[wl][j] * chunks + c, policy);
      const float4 v = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                   __uint_as_float(u.w));
      const float w = s_w[wl][j];
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    if (a.y_f32) {
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

cudaError_t launch_ec_select(const EcSelectArgs& a, cudaStream_t s) {
  if (a.E <= 0) return cudaSuccess;
  const size_t smem = a.T <= kMaxCachedT ? (size_t)(a.T > 0 ? a.T : 1) * 4 : 0;
  cudaError_t e = cudaFuncSetAttribute(ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 1024);
  if (e != cudaSuccess) return e;
  ec_select_kernel<<<a.E, kSelThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ec_gather(const EcGatherArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  ec_gather_kernel<<<(unsigned)((a.rows + kGatherWarps - 1) / kGatherWarps), kGatherWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ec_combine(const EcCombineArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (a.E + a.S > kMaxSources) return cudaErrorInvalidValue;
  ec_combine_kernel<<<(unsigned)((a.T + kCombineWarps - 1) / kCombineWarps), kCombineWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
