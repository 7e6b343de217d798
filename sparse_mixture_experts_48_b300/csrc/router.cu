// K1 -- router: logits l = x W_g + b_g, softmax or normalised-sigmoid gating,
// top-k with the lower expert index winning ties, renormalised weights, and
// per-CTA routing partials (selection histogram, local ranks, sums of p).
//
// The logit contraction has N = E <= 256 and K = d: per token it does 2 d E
// flops on d * 2 bytes of x, so for E >= 16 plain FP32 FMA would fall below the
// HBM rate.  The bf16 path therefore runs the contraction on the tensor cores
// with warp-level mma.sync (m16n8k16, fp32 accumulate); x tiles are staged in
// shared memory by TMA into a deep ring, W_g tiles (small, L2-resident) by
// cp.async.  Nothing here is a large GEMM worth a TMEM pipeline: the kernel
// streams x once and is bound by HBM.  The gating, selection and partial sums
// run on one thread per token.
//
// Sources: "MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现" §2.1 (linear +
// softmax router, top-k, renormalise); "手撕一个极简 MoE-FFN" §三 (Router,
// top_k_routing and its worked example); "MoE架构解析" §四 技术飞跃③ (normalised
// sigmoid gating); "Mixture of Experts混合专家模型架构原理与路由策略实现",
// 门控网络的数学原理 (W_g is [d_model, num_experts]).
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kBK = 64;        // bf16 k-tile (128 bytes per x row)

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
// A CTA owns kRouterBM = 64 tokens and walks d in k-tiles of 64.  Per k-tile a
// ring stage holds the x tile [64 tokens][64 k] (8 KB, brought by one TMA copy
// with the 128-byte swizzle, rows past T zero-filled) and the W_g tile
// [64 k][EP experts] (cp.async, same swizzle for EP >= 64).  The ring is deep
// (up to 8 stages, about 64 KB of x in flight per CTA) because the kernel
// only streams x once: its speed is the number of bytes it keeps in flight.
// After the ring the same shared memory holds the fp32 logits [64][EP + 1].
template <int NT>
struct RouterBf16 {
  static constexpr int EP = 8 * NT;
  static constexpr int XS = kRouterBM * kBK * 2;   // 8 KB, a multiple of 1 KB (swizzle atom)
  static constexpr int WS = kBK * EP * 2;           // 1 KB * NT
  static constexpr int STAGE = XS + WS;
  static constexpr int STAGES = (96 * 1024 / STAGE) > 8 ? 8 : ((96 * 1024 / STAGE) < 2 ? 2 : 96 * 1024 / STAGE);
  static constexpr size_t RING = (size_t)STAGES * STAGE;
  static constexpr size_t LOGITS = (size_t)kRouterBM * (EP + 1) * 4;
  static constexpr size_t BITS_OFF = RING > LOGITS ? RING : LOGITS;
  static constexpr size_t BITS = (size_t)EP * ((kRouterBM + 31) / 32) * 4;
  static constexpr size_t BAR_OFF = BITS_OFF + BITS;
  static constexpr size_t SMEM = 1024 + BAR_OFF + STAGES * 8 + 16;   // + 1 KB to align the ring
};

constexpr uint32_t kWhereRouter = 0x300;

// NT n-tiles of 8 experts; EP = 8 NT >= E.  Warp w computes tokens 16w..16w+15.
template <int NT>
__global__ void __launch_bounds__(kThreads) router_bf16_kernel(const __grid_constant__ CUtensorMap tmX,
                                                               RouterArgs a) {
  using L = RouterBf16<NT>;
  constexpr int EP = L::EP, RW = EP / 8, STAGES = L::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint32_t* bits = (uint32_t*)(smem + L::BITS_OFF);
  uint64_t* full = (uint64_t*)(smem + L::BAR_OFF);
  uint32_t* abort_flag = (uint32_t*)(full + STAGES);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int64_t blk = blockIdx.x;
  const int64_t t0 = blk * kRouterBM;
  const int d = a.d, E = a.E;
  const uint16_t* W = (const uint16_t*)a.Wg;
  const int nk = d / kBK;
  const bool wvec = (E % 8) == 0;
  const uint64_t limit = (uint64_t)a.timeout_ns;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(smem_u32(&full[s]), 1);
    *abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
  }
  __syncthreads();

  auto wswz = [](int r, int c) { return r * (EP * 2) + ((RW >= 8 ? (c ^ (r & 7)) : c) << 4); };
  auto xs = [&](int st) { return smem + st * L::STAGE; };
  auto ws = [&](int st) { return smem + st * L::STAGE + L::XS; };

  auto issue = [&](int kt, int st) {
    if (tid == 0) {
      // The slot was last read (ldmatrix) before the barrier this thread passed.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const uint32_t fb = smem_u32(&full[st]);
      mbar_expect_tx(fb, (uint32_t)L::XS);
      tma_load_2d(smem_u32(xs(st)), &tmX, kt * kBK, (int)t0, fb);
    }
    const uint32_t wb = smem_u32(ws(st));
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
        *(uint16_t*)(ws(st) + wswz(r, e / 8) + (e % 8) * 2) = v;
      }
    }
  };

  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[n][q] = 0.f;

  int issued = 0;
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nk) { issue(s, s); ++issued; }
    cp_async_commit();
  }
  int stop = -1;   // k-tile at which the CTA gave up, or -1
  for (int kt = 0; kt < nk; ++kt) {
    const int st = kt % STAGES;
    cp_async_wait<STAGES - 2>();
    const bool ok = mbar_wait(smem_u32(&full[st]), (uint32_t)(kt / STAGES) & 1u, abort_flag, limit, a.err,
                              kWhereRouter + 1);
    if (__syncthreads_or(!ok)) { stop = kt; break; }
    {
      const int nxt = kt + STAGES - 1;
      if (nxt < nk) { issue(nxt, nxt % STAGES); ++issued; }
      cp_async_commit();
    }
    const uint32_t xb = smem_u32(xs(st));
    const uint32_t wb = smem_u32(ws(st));
#pragma unroll
    for (int ks = 0; ks < kBK / 16; ++ks) {
      uint32_t af[4];
      {
        // x tile row r, 16-byte chunk c sits at r * 128 + ((c ^ (r & 7)) << 4).
        int r = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        int c = ks * 2 + (lane >> 4);
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(af[0]), "=r"(af[1]), "=r"(af[2]), "=r"(af[3])
                     : "r"(xb + r * 128 + ((c ^ (r & 7)) << 4)));
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
  if (stop >= 0) {
    // Stop cleanly: every TMA copy this CTA started lands before it exits.
    // Tiles before `stop` were consumed; tiles stop..issued-1 (at most
    // STAGES - 1, one per slot) may still be in flight.  The error word is
    // set, so the later stages of the layer skip their work.
    if (tid == 0)
      for (int kt = stop; kt < issued; ++kt)
        mbar_drain(smem_u32(&full[kt % STAGES]), (uint32_t)(kt / STAGES) & 1u,
                   limit > 2000000000ull ? limit : 2000000000ull);
    __syncthreads();
    return;
  }
  __syncthreads();
  // Logits to shared memory (reusing the ring: every copy has been consumed).
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
  const size_t bytes = RouterBf16<NT>::SMEM;
  CUtensorMap tmX;
  if (!tmap_bf16_2d(&tmX, a.x, a.T, a.d, kBK, kRouterBM)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(router_bf16_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)bytes);
  if (e != cudaSuccess) return e;
  router_bf16_kernel<NT><<<(unsigned)nblk, kThreads, bytes, s>>>(tmX, a);
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
