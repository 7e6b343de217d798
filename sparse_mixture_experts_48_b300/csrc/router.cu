// K1 -- router: logits l = x W_g + b_g, softmax or normalised-sigmoid gating,
// top-k with the lower expert index winning ties, renormalised weights, and
// per-CTA routing partials (selection histogram, local ranks, sums of p).
//
// The logit contraction has N = E <= 256 and K = d: per token it does 2 d E
// flops on d * 2 bytes of x, so for E >= 16 plain FP32 FMA would fall below the
// HBM rate.  The bf16 path therefore runs the contraction on the tensor cores
// with warp-level mma.sync (m16n8k16, fp32 accumulate); x and W_g tiles are
// staged in shared memory by a 3-stage cp.async pipeline.  Nothing here is a
// large GEMM worth a TMEM pipeline: the kernel streams x once and is bound by
// HBM.  The gating, selection and partial sums run on one thread per token.
//
// Sources: "MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现" §2.1 (linear +
// softmax router, top-k, renormalise); "手撕一个极简 MoE-FFN" §三 (Router,
// top_k_routing and its worked example); "MoE架构解析" §四 技术飞跃③ (normalised
// sigmoid gating); "Mixture of Experts混合专家模型架构原理与路由策略实现",
// 门控网络的数学原理 (W_g is [d_model, num_experts]).
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kBK = 64;        // bf16 k-tile (128 bytes per x row)
constexpr int kStages = 3;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool full) {
  int n = full ? 16 : 0;   // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---- the per-token tail shared by both dtypes ----------------------------------
// sl: [kRouterBM][ldl] fp32 logits without bias, rows of this CTA's tokens.
// bits: [E][1 + kRouterBM/32] scratch words.
__device__ void router_finalize(float* sl, int ldl, uint32_t* bits, const RouterArgs& a, int64_t blk) {
  constexpr int NW = (kRouterBM + 31) / 32;
  const int tid = threadIdx.x;
  const int E = a.E, k = a.k;
  const int64_t t0 = blk * kRouterBM;
  for (int i = tid; i < E * NW; i += blockDim.x) bits[i] = 0u;
  __syncthreads();

  const int64_t t = t0 + tid;
  const bool valid = tid < kRouterBM && t < a.T;
  float val[8];
  int idx[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) { val[j] = 0.f; idx[j] = -1; }
  if (valid) {
    float* l = sl + tid * ldl;
    const bool bf = a.dtype == MOE_DT_BF16;
    for (int e = 0; e < E; ++e) {
      float b = 0.f;
      if (a.bg) b = bf ? bf16_bits_to_f32(((const uint16_t*)a.bg)[e]) : ((const float*)a.bg)[e];
      l[e] += b;
    }
    if (a.logits_out)
      for (int e = 0; e < E; ++e) a.logits_out[t * E + e] = l[e];
    // Top-k by insertion: larger logit first, equal logits by lower index.
    for (int e = 0; e < E; ++e) {
      float cv = l[e];
      int ci = e;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < k) {
          bool better = idx[j] < 0 || cv > val[j] || (cv == val[j] && ci < idx[j]);
          if (better) {
            float tv = val[j]; int ti = idx[j];
            val[j] = cv; idx[j] = ci;
            cv = tv; ci = ti;
          }
        }
      }
    }
    // Gating over all E (these p feed P), and the renormalised top-k weights.
    float z = 0.f, zsel = 0.f;
    float g[8];
    if (a.gating == MOE_GATE_SOFTMAX) {
      const float m = val[0];
      for (int e = 0; e < E; ++e) { float v = expf(l[e] - m); l[e] = v; z += v; }
#pragma unroll
      for (int j = 0; j < 8; ++j) if (j < k) { g[j] = expf(val[j] - m); zsel += g[j]; }
    } else {
      for (int e = 0; e < E; ++e) { float v = 1.f / (1.f + expf(-l[e])); l[e] = v; z += v; }
#pragma unroll
      for (int j = 0; j < 8; ++j) if (j < k) { g[j] = 1.f / (1.f + expf(-val[j])); zsel += g[j]; }
    }
    const float rz = 1.f / z;
    for (int e = 0; e < E; ++e) l[e] *= rz;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        a.topk_idx[t * k + j] = idx[j];
        a.topk_w[t * k + j] = g[j] / zsel;
        atomicOr(&bits[idx[j] * NW + tid / 32], 1u << (tid % 32));
      }
    }
  }
  __syncthreads();
  if (valid) {
    const int w = tid / 32;
    const uint32_t below = (1u << (tid % 32)) - 1u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        const uint32_t* be = bits + idx[j] * NW;
        int r = __popc(be[w] & below);
        for (int q = 0; q < w; ++q) r += __popc(be[q]);
        a.lrank[t * k + j] = (uint8_t)r;
      }
    }
  }
  const int nvalid = (int)(a.T - t0 < kRouterBM ? a.T - t0 : kRouterBM);
  for (int e = tid; e < E; e += blockDim.x) {
    int h = 0;
    for (int q = 0; q < NW; ++q) h += __popc(bits[e * NW + q]);
    a.hist[blk * E + e] = h;
    float s = 0.f;
    for (int r = 0; r < nvalid; ++r) s += sl[r * ldl + e];   // fixed order
    a.psum[blk * E + e] = s;
  }
}

// ---- bf16: tensor-core logits ---------------------------------------------------
// Shared memory: the cp.async pipeline, later reused for the fp32 logits
// [kRouterBM][EP + 1]; the selection bit masks sit after the larger of the two.
__host__ __device__ constexpr size_t bf16_bits_offset(int NT) {
  return (size_t)kStages * (kRouterBM * kBK * 2 + kBK * 8 * NT * 2) > (size_t)kRouterBM * (8 * NT + 1) * 4
             ? (size_t)kStages * (kRouterBM * kBK * 2 + kBK * 8 * NT * 2)
             : (size_t)kRouterBM * (8 * NT + 1) * 4;
}
__host__ __device__ constexpr size_t bf16_smem_bytes(int NT) {
  return bf16_bits_offset(NT) + (size_t)8 * NT * ((kRouterBM + 31) / 32) * 4;
}

// NT n-tiles of 8 experts; EP = 8 NT >= E.  Warp w computes tokens 16w..16w+15.
template <int NT>
__global__ void __launch_bounds__(kThreads) router_bf16_kernel(RouterArgs a) {
  constexpr int EP = 8 * NT;
  constexpr int RW = EP / 8;                  // 16-byte chunks per W_g row
  constexpr int XS = kRouterBM * kBK * 2;     // bytes of one x stage
  constexpr int WS = kBK * EP * 2;            // bytes of one W stage
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* xs = smem;
  uint8_t* ws = smem + kStages * XS;
  uint32_t* bits = (uint32_t*)(smem + bf16_bits_offset(NT));

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int64_t blk = blockIdx.x;
  const int64_t t0 = blk * kRouterBM;
  const int d = a.d, E = a.E;
  const uint16_t* x = (const uint16_t*)a.x;
  const uint16_t* W = (const uint16_t*)a.Wg;
  const int nk = d / kBK;
  const bool wvec = (E % 8) == 0;

  auto xswz = [](int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); };
  auto wswz = [](int r, int c) { return r * (EP * 2) + ((RW >= 8 ? (c ^ (r & 7)) : c) << 4); };

  auto load_stage = [&](int kt, int st) {
    const uint32_t xb = smem_u32(xs + st * XS);
    for (int i = tid; i < kRouterBM * 8; i += kThreads) {
      int r = i >> 3, c = i & 7;
      int64_t t = t0 + r;
      bool ok = t < a.T;
      const uint16_t* src = x + (ok ? t : 0) * d + kt * kBK + c * 8;
      cp_async16(xb + xswz(r, c), src, ok);
    }
    const uint32_t wb = smem_u32(ws + st * WS);
    if (wvec) {
      for (int i = tid; i < kBK * RW; i += kThreads) {
        int r = i / RW, c = i % RW;
        bool ok = c * 8 < E;
        const uint16_t* src = W + (int64_t)(kt * kBK + r) * E + (ok ? c * 8 : 0);
        cp_async16(wb + wswz(r, c), src, ok);
      }
    } else {
      for (int i = tid; i < kBK * EP; i += kThreads) {
        int r = i / EP, e = i % EP;
        uint16_t v = e < E ? W[(int64_t)(kt * kBK + r) * E + e] : (uint16_t)0;
        *(uint16_t*)(ws + st * WS + wswz(r, e / 8) + (e % 8) * 2) = v;
      }
    }
  };

  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[n][q] = 0.f;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nk) load_stage(s, s);
    cp_async_commit();
  }
  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {
      int nxt = kt + kStages - 1;
      if (nxt < nk) load_stage(nxt, nxt % kStages);
      cp_async_commit();
    }
    const int st = kt % kStages;
    const uint32_t xb = smem_u32(xs + st * XS);
    const uint32_t wb = smem_u32(ws + st * WS);
#pragma unroll
    for (int ks = 0; ks < kBK / 16; ++ks) {
      uint32_t af[4];
      {
        int r = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        int c = ks * 2 + (lane >> 4);
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(af[0]), "=r"(af[1]), "=r"(af[2]), "=r"(af[3])
                     : "r"(xb + xswz(r, c)));
      }
#pragma unroll
      for (int np = 0; np < (NT + 1) / 2; ++np) {
        uint32_t bf[4];
        const int i = lane >> 3;
        const int kr = ks * 16 + (lane & 7) + 8 * (i & 1);
        if (NT == 1) {
          asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                       : "=r"(bf[0]), "=r"(bf[1])
                       : "r"(wb + wswz(kr, 0)));
        } else {
          const int nc = 2 * np + (i >> 1);
          asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                       : "=r"(bf[0]), "=r"(bf[1]), "=r"(bf[2]), "=r"(bf[3])
                       : "r"(wb + wswz(kr, nc)));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = 2 * np + h;
          if (n < NT) {
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+f"(acc[n][0]), "+f"(acc[n][1]), "+f"(acc[n][2]), "+f"(acc[n][3])
                : "r"(af[0]), "r"(af[1]), "r"(af[2]), "r"(af[3]), "r"(bf[2 * h]), "r"(bf[2 * h + 1]));
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  // Logits to shared memory (reusing the pipeline buffers).
  float* sl = (float*)smem;
  const int ldl = EP + 1;
  {
    const int r0 = warp * 16 + (lane >> 2);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int c = n * 8 + 2 * (lane & 3);
      sl[r0 * ldl + c] = acc[n][0];
      sl[r0 * ldl + c + 1] = acc[n][1];
      sl[(r0 + 8) * ldl + c] = acc[n][2];
      sl[(r0 + 8) * ldl + c + 1] = acc[n][3];
    }
  }
  __syncthreads();
  router_finalize(sl, ldl, bits, a, blk);
}

// ---- fp32: CUDA-core logits ------------------------------------------------------
constexpr int kBK32 = 32;
__global__ void __launch_bounds__(kThreads) router_f32_kernel(RouterArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int E = a.E, d = a.d;
  const int ldl = E + 1;
  float* sl = (float*)smem;                        // [64][E+1] accumulators
  float* xs = sl + kRouterBM * ldl;                // [64][33]
  float* wsm = xs + kRouterBM * (kBK32 + 1);       // [32][E]
  uint32_t* bits = (uint32_t*)(wsm + kBK32 * E);
  const int tid = threadIdx.x;
  const int64_t blk = blockIdx.x, t0 = blk * kRouterBM;
  const float* x = (const float*)a.x;
  const float* W = (const float*)a.Wg;
  for (int i = tid; i < kRouterBM * ldl; i += kThreads) sl[i] = 0.f;
  for (int kt = 0; kt < d; kt += kBK32) {
    __syncthreads();
    for (int i = tid; i < kRouterBM * kBK32; i += kThreads) {
      int r = i / kBK32, c = i % kBK32;
      int64_t t = t0 + r;
      xs[r * (kBK32 + 1) + c] = (t < a.T && kt + c < d) ? x[t * d + kt + c] : 0.f;
    }
    for (int i = tid; i < kBK32 * E; i += kThreads) {
      int r = i / E, e = i % E;
      wsm[i] = (kt + r < d) ? W[(int64_t)(kt + r) * E + e] : 0.f;
    }
    __syncthreads();
    for (int o = tid; o < kRouterBM * E; o += kThreads) {
      int r = o / E, e = o % E;
      float s = sl[r * ldl + e];
      for (int c = 0; c < kBK32; ++c) s = fmaf(xs[r * (kBK32 + 1) + c], wsm[c * E + e], s);
      sl[r * ldl + e] = s;
    }
  }
  __syncthreads();
  router_finalize(sl, ldl, bits, a, blk);
}

template <int NT>
cudaError_t launch_bf16(const RouterArgs& a, int64_t nblk, cudaStream_t s) {
  const size_t bytes = bf16_smem_bytes(NT);
  cudaError_t e = cudaFuncSetAttribute(router_bf16_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)bytes);
  if (e != cudaSuccess) return e;
  router_bf16_kernel<NT><<<(unsigned)nblk, kThreads, bytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
  const int64_t nblk = (a.T + kRouterBM - 1) / kRouterBM;
  if (nblk == 0) return cudaSuccess;
  if (a.dtype == MOE_DT_F32) {
    size_t bytes = (size_t)kRouterBM * (a.E + 1) * 4 + (size_t)kRouterBM * (kBK32 + 1) * 4 +
                   (size_t)kBK32 * a.E * 4 + (size_t)a.E * ((kRouterBM + 31) / 32) * 4;
    cudaError_t e = cudaFuncSetAttribute(router_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    router_f32_kernel<<<(unsigned)nblk, kThreads, bytes, s>>>(a);
    return cudaGetLastError();
  }
  const int ep = (a.E + 7) / 8;
  if (ep <= 1) return launch_bf16<1>(a, nblk, s);
  if (ep <= 2) return launch_bf16<2>(a, nblk, s);
  if (ep <= 4) return launch_bf16<4>(a, nblk, s);
  if (ep <= 8) return launch_bf16<8>(a, nblk, s);
  if (ep <= 16) return launch_bf16<16>(a, nblk, s);
  return launch_bf16<32>(a, nblk, s);
}

}  // namespace moe
