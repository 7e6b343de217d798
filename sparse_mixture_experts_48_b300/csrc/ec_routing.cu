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
// Each expert's rows start Cs >= C apart (Cs = C in the forward; the backward
// pads them to whole blocks of its weight-gradient GEMMs).
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

// Histogram privatised per group of kHistWarps warps: the top bytes of
// probabilities fall into a handful of bins, and 1024 threads adding into one
// histogram would serialise on them.
constexpr int kHistGroups = 8;
constexpr int kHistWarps = kSelWarps / kHistGroups;

__global__ void __launch_bounds__(kSelThreads) ec_select_kernel(EcSelectArgs a) {
  extern __shared__ uint32_t s_keys[];            // cached keys (T <= kMaxCachedT)
  __shared__ int s_hist[256];
  __shared__ int s_hpart[kHistGroups][256];
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
      for (int i = threadIdx.x; i < kHistGroups * 256; i += kSelThreads) (&s_hpart[0][0])[i] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      int* hp = s_hpart[(threadIdx.x / 32) / kHistWarps];
      for (int64_t t = threadIdx.x; t < T; t += kSelThreads) {
        const uint32_t k = key(t);
        if ((k & mask) == prefix) atomicAdd(&hp[(k >> shift) & 255u], 1);
      }
      __syncthreads();
      for (int i = threadIdx.x; i < 256; i += kSelThreads) {
        int h = 0;
#pragma unroll
        for (int g = 0; g < kHistGroups; ++g) h += s_hpart[g][i];
        s_hist[i] = h;
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // The bin holding the rem-th largest key, searched from the top: lane
        // l owns bins 255 - 8l .. 248 - 8l; a scan over the lanes gives the
        // keys in the higher bins, and the first lane whose bins reach rem
        // names the bin (and the keys of that bin still to take).
        const int ln = threadIdx.x;
        const int rem = s_remaining;
        int cnt[8], local = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = s_hist[255 - (8 * ln + j)];
          local += cnt[j];
        }
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, off);
          if (ln >= off) incl += v;
        }
        int cum = incl - local, bin = -1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (bin < 0) {
            if (cum + cnt[j] >= rem) bin = 255 - (8 * ln + j);
            else cum += cnt[j];
          }
        }
        const uint32_t found = __ballot_sync(0xffffffffu, bin >= 0);
        // the keys that match the prefix always number at least rem: bin 0 at the latest
        if (found != 0u && ln == __ffs(found) - 1) {
          s_remaining = rem - cum;
          s_prefix = prefix | ((uint32_t)bin << shift);
        }
      }
      mask |= 255u << shift;
      __syncthreads();
    }
  }
  const uint32_t thr = s_prefix;
  const int need_eq = C > 0 ? s_remaining : 0;

  // Chosen tokens in token order: key > thr, or key == thr among the first
  // need_eq such tokens.  Warp w owns the contiguous tokens [w B, (w + 1) B):
  // it counts its keys above and equal to the threshold, one scan over the 32
  // warps places every warp's equal keys and chosen tokens, and each warp then
  // walks its block again in order, ranking with ballots.
  const int lane = threadIdx.x % 32, wid = threadIdx.x / 32;
  const int64_t B = ((T + kSelWarps - 1) / kSelWarps + 31) / 32 * 32;
  const int64_t wb = (int64_t)wid * B;
  int gt = 0, eq = 0;
  if (C > 0)
    for (int64_t t = wb + lane; t < wb + B && t < T; t += 32) {
      const uint32_t k = key(t);
      gt += k > thr;
      eq += k == thr;
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, off);
    eq += __shfl_xor_sync(0xffffffffu, eq, off);
  }
  __shared__ int s_eq[kSelWarps], s_take[kSelWarps];
  if (lane == 0) s_eq[wid] = eq;
  __syncthreads();
  if (wid == 0) {
    // equal keys before each warp, then how many of its own it takes, then
    // the chosen tokens before each warp
    const int ne = lane < kSelWarps ? s_eq[lane] : 0;
    int ni = ne;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, ni, off);
      if (lane >= off) ni += v;
    }
    const int eq_before = ni - ne;
    int take_eq = need_eq - eq_before;
    take_eq = take_eq < 0 ? 0 : (take_eq > ne ? ne : take_eq);
    if (lane < kSelWarps) s_take[lane] = take_eq;
  }
  __syncthreads();
  const int my_take_eq = s_take[wid];
  const int my_count = gt + my_take_eq;
  __shared__ int s_pos[kSelWarps];
  if (lane == 0) s_pos[wid] = my_count;
  __syncthreads();
  if (wid == 0) {
    int v = lane < kSelWarps ? s_pos[lane] : 0;
    int vi = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, vi, off);
      if (lane >= off) vi += u;
    }
    __syncwarp();
    if (lane < kSelWarps) s_pos[lane] = vi - v;
  }
  __syncthreads();
  int pos = s_pos[wid];
  int eq_seen = 0;
  const uint32_t lt = (1u << lane) - 1u;
  if (C > 0)
    for (int64_t t0 = wb; t0 < wb + B && t0 < T; t0 += 32) {
      const int64_t t = t0 + lane;
      const uint32_t k = t < T && t < wb + B ? key(t) : 0u;
      const bool in = t < T && t < wb + B;
      const bool g = in && k > thr, q = in && k == thr;
      const uint32_t qb = __ballot_sync(0xffffffffu, q);
      const bool take = g || (q && eq_seen + __popc(qb & lt) < my_take_eq);
      const uint32_t tb = __ballot_sync(0xffffffffu, take);
      if (take) {
        const int64_t row = (int64_t)e * a.Cs + pos + __popc(tb & lt);
        a.perm[row] = (int32_t)t;
        a.w_row[row] = __uint_as_float(k);
        a.tok_row[t * a.E + e] = (int32_t)row;
        atomicOr(&a.bits[t * a.EW + e / 32], 1u << (e % 32));
      }
      eq_seen += __popc(qb);
      pos += __popc(tb);
    }
}

constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32) ec_gather_kernel(EcGatherArgs a) {
  const int lane = threadIdx.x % 32;
  const int64_t r = (int64_t)blockIdx.x * kGatherWarps + threadIdx.x / 32;
  if (r >= a.rows || *(volatile const uint32_t*)a.err != 0u || r % a.Cs >= a.C) return;
  const int64_t t = a.perm[r];
  if (a.xs_perm && lane == 0) a.xs_perm[r] = a.xs_tok[t];
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
  // The token's sources in order: choosing experts ascending, then the shared
  // experts.  Lane l looks at expert w * 32 + l of mask word w; a ballot
  // places the chosen ones in expert order.
  int n = 0;
  const uint32_t lt = (1u << lane) - 1u;
  for (int w = 0; w < a.EW; ++w) {
    const uint32_t word = a.bits[t * a.EW + w];
    const bool chosen = (word >> lane) & 1u;
    if (chosen) {
      const int64_t row = a.tok_row[t * a.E + w * 32 + lane];
      const int at = n + __popc(word & lt);
      s_row[wl][at] = row;
      s_w[wl][at] = a.w_row[row];
    }
    n += __popc(word);
  }
  if (lane < a.S) {
    s_row[wl][n + lane] = a.rows_routed + (int64_t)lane * a.T + t;
    s_w[wl][n + lane] = 1.f;
  }
  n += a.S;
  __syncwarp();
  const int64_t chunks = a.d / 4;
  const float4* O = (const float4*)a.o;
  const uint64_t policy = l2_policy_evict_first();
  constexpr int kBatch = 4;   // sources whose loads are in flight together
  constexpr int U = 2;        // 16-byte chunks per lane per pass
  for (int64_t c0 = lane; c0 < chunks; c0 += 32 * U) {
    float4 acc[U];
#pragma unroll
    for (int v = 0; v < U; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < n; j0 += kBatch) {
      uint4 u[kBatch][U];
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
#pragma unroll
        for (int v = 0; v < U; ++v)
          if (j0 + b < n && c0 + 32 * v < chunks)
            u[b][v] = ld_stream_u4(O + s_row[wl][j0 + b] * chunks + c0 + 32 * v, policy);
      // accumulated in source order, as one load at a time would
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (j0 + b < n) {
          const float w = s_w[wl][j0 + b];
#pragma unroll
          for (int v = 0; v < U; ++v) {
            if (c0 + 32 * v < chunks) {
              acc[v].x = fmaf(w, __uint_as_float(u[b][v].x), acc[v].x);
              acc[v].y = fmaf(w, __uint_as_float(u[b][v].y), acc[v].y);
              acc[v].z = fmaf(w, __uint_as_float(u[b][v].z), acc[v].z);
              acc[v].w = fmaf(w, __uint_as_float(u[b][v].w), acc[v].w);
            }
          }
        }
      }
    }
#pragma unroll
    for (int v = 0; v < U; ++v) {
      const int64_t c = c0 + 32 * v;
      if (c >= chunks) continue;
      if (a.y_f32) {
        reinterpret_cast<float4*>(a.y)[t * chunks + c] = acc[v];
      } else {
        uint2 out;
        out.x = pack_bf16x2(acc[v].x, acc[v].y);
        out.y = pack_bf16x2(acc[v].z, acc[v].w);
        reinterpret_cast<uint2*>(a.y)[t * chunks + c] = out;
      }
    }
  }
}

}  // namespace

cudaError_t launch_ec_select(const EcSelectArgs& a, cudaStream_t s) {
  if (a.E <= 0) return cudaSuccess;
  if (a.Cs < a.C) return cudaErrorInvalidValue;
  const size_t smem = a.T <= kMaxCachedT ? (size_t)(a.T > 0 ? a.T : 1) * 4 : 0;
  cudaError_t e = cudaFuncSetAttribute(ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 1024);
  if (e != cudaSuccess) return e;
  ec_select_kernel<<<a.E, kSelThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ec_gather(const EcGatherArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  if (a.C <= 0 || a.Cs < a.C) return cudaErrorInvalidValue;
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
