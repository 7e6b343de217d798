// K3 -- grouped expert GEMM on the 5th-generation tensor cores (tcgen05).
//
//   C[r, :] = epilogue( A[r, :] B[w(g)] )   for each row r of each segment g
//
// One persistent CTA per SM walks the tiles of all segments (segment-major,
// then 256-column block, then 128-row block, so the CTAs running together
// share one weight slab through L2).  Warp roles inside a CTA:
//   warp 0      TMA producer: A tile 128 x 64 (K-major, 128-byte swizzle) and
//               four B boxes 64(N) x 64(K) (N-major, 128-byte swizzle) per stage
//               into a 4-stage shared-memory ring (48 KB per stage);
//   warp 1      TMEM owner; one elected lane issues tcgen05.mma
//               (kind::f16, bf16 x bf16 -> fp32, M = 128, N = 256, K = 16) into
//               one of two 256-column TMEM accumulators, and tcgen05.commit
//               releases ring slots and hands finished accumulators over;
//   warps 2-9   epilogue: tcgen05.ld 32 lanes x 32 columns at a time, bias +
//               ReLU / exact-erf GELU, or the SwiGLU product silu(a) * b of the
//               two halves of the accumulator (columns 0-127 = x W1, 128-255 =
//               x W3 of the same 128 hidden units), round to bf16, store.
// While the epilogue drains one accumulator the MMA fills the other.
//
// Rows past a segment's end in its last 128-row block are computed (they read
// the next segment's rows, or the zero fill past the tensor) but never stored.
// Every wait is bounded in time; a wait that runs out sets a CTA-wide abort
// flag and the workspace error word, every role stops, outstanding TMA loads
// and MMAs are waited for (again bounded), TMEM is freed and the CTA returns.
//
// Sources: "手撕一个极简 MoE-FFN" §四 (Expert = w2(act(w1 x))), §六 (group the
// tokens of each expert and run it once on the batch); "MoE混合专家模型：
// Transformer稀疏前馈网络原理与PyTorch实现" §4.1 (GELU expert); "术业有专攻：
// learn-minimind MoE混合专家模型架构入门指南" §二 (SwiGLU experts).
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace moe {
cudaError_t launch_grouped_gemm_f32(const GemmArgs& a, cudaStream_t s);

namespace {

constexpr int BM = kGemmBM;          // 128
constexpr int BK = 64;               // 128 bytes of bf16: one swizzle row
constexpr int MMA_N = 256;
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;     // 8 KB: 64 columns x 64 k
constexpr int B_BYTES = 4 * B_BOX_BYTES;     // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr int TMEM_COLS = 512;               // two 256-column accumulators
constexpr int MAX_G = 264;
constexpr uint32_t kWhereGemm = 0x100;

struct Ctl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t done;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t skip;      // an earlier stage failed: compute nothing
  int mt[MAX_G + 1];
  int rows[MAX_G];
  int w[MAX_G];
  int orow[MAX_G];
  int arow[MAX_G];
  int asrc[MAX_G];
};

constexpr size_t kSmemBytes = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(Ctl);

__device__ __forceinline__ void map_tile(const Ctl& c, int G, int n_tiles, int tile, int& g, int& m, int& n) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c.mt[mid] * n_tiles <= tile) lo = mid; else hi = mid - 1;
  }
  g = lo;
  const int local = tile - c.mt[g] * n_tiles;
  const int mtg = c.mt[g + 1] - c.mt[g];
  n = local / mtg;
  m = local - n * mtg;
}

template <bool SWIGLU, bool OUT_F32>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB3,
                        GemmArgs a) {
  constexpr int BN_OUT = SWIGLU ? 128 : 256;   // output columns per tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;            // 1 KB aligned ring for the 128-byte swizzle
  uint8_t* ring = smem_raw + (base - raw);
  Ctl& c = *reinterpret_cast<Ctl*>(ring + STAGES * STAGE_BYTES);
  volatile uint32_t* abort = &c.abort;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = a.G;
  const int n_tiles = (a.N + BN_OUT - 1) / BN_OUT;
  const int nkb = a.K / BK;
  const uint64_t limit = (uint64_t)a.timeout_ns;
  // Tear-down waits for copies and MMAs this CTA started; they finish on their
  // own, so they get a generous limit whatever the caller's wait limit is.
  const uint64_t drain_limit = limit > 2000000000ull ? limit : 2000000000ull;

  // ---- set-up ----
  for (int i = threadIdx.x; i <= G; i += blockDim.x) c.mt[i] = a.seg.mtile_start[i];
  for (int i = threadIdx.x; i < G; i += blockDim.x) {
    c.rows[i] = a.seg.rows[i];
    c.w[i] = a.seg.w[i];
    c.orow[i] = a.seg.out_row[i];
    c.arow[i] = a.a_from_out_rows ? a.seg.out_row[i] : a.seg.a_row[i];
    c.asrc[i] = a.a_from_out_rows ? 0 : a.seg.a_src[i];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&c.full[s]), 1);
      mbar_init(smem_u32(&c.empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&c.tfull[s]), 1);
      mbar_init(smem_u32(&c.tempty[s]), EPI_WARPS);
    }
    mbar_init(smem_u32(&c.done), 1);
    c.abort = 0u;
    c.skip = *(volatile const uint32_t*)a.err;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA0) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA1) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    if (SWIGLU) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB3) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&c.tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const int total = c.skip ? 0 : c.mt[G] * n_tiles;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[STAGES];
      bool issued[STAGES];
      for (int s = 0; s < STAGES; ++s) { issued[s] = false; issued_phase[s] = 0; }
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int g, m, n;
        map_tile(c, G, n_tiles, tile, g, m, n);
        const int arow = c.arow[g] + m * BM;
        const CUtensorMap* amap = c.asrc[g] ? &tmA1 : &tmA0;
        const int wslab = c.w[g];
        const int n0 = n * BN_OUT;
        const int cols_left = a.N - n0;
        int nbox_half = SWIGLU ? (cols_left >= 128 ? 2 : 1) : 0;
        int nbox = SWIGLU ? 2 * nbox_half : (cols_left >= 256 ? 4 : cols_left / 64);
        const uint32_t bytes = (uint32_t)(A_BYTES + nbox * B_BOX_BYTES);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&c.empty[stage]), phase ^ 1u, abort, limit, a.err, kWhereGemm + 1)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&c.full[stage]);
          mbar_expect_tx(fb, bytes);
          const uint32_t sa = base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          tma_load_2d(sa, amap, kb * BK, arow, fb);
          if (SWIGLU) {
            for (int h = 0; h < nbox_half; ++h) {
              tma_load_3d(sb + h * B_BOX_BYTES, &tmB, n0 + 64 * h, kb * BK, wslab, fb);
              tma_load_3d(sb + (2 + h) * B_BOX_BYTES, &tmB3, n0 + 64 * h, kb * BK, wslab, fb);
            }
          } else {
            for (int bx = 0; bx < nbox; ++bx) tma_load_3d(sb + bx * B_BOX_BYTES, &tmB, n0 + 64 * bx, kb * BK, wslab, fb);
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // Every load this thread issued has landed before the CTA may exit.
      for (int s = 0; s < STAGES; ++s)
        if (issued[s]) mbar_drain(smem_u32(&c.full[s]), issued_phase[s], drain_limit);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t aphase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(smem_u32(&c.tempty[acc]), aphase ^ 1u, abort, limit, a.err, kWhereGemm + 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * MMA_N);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&c.full[stage]), phase, abort, limit, a.err, kWhereGemm + 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // A: K-major, 8-row groups 1024 B apart; a K step of 16 is 32 bytes.
            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
            // B: N-major, 64-column boxes 8 KB apart (LBO), 8-row k groups 1024 B
            // apart (SBO); a K step of 16 rows is 2048 bytes.
            const uint64_t bd = smem_desc(sb + kk * 2048, B_BOX_BYTES, 1024);
            mma_bf16_cta1<idesc_bf16(BM, MMA_N)>(d_tmem, ad, bd, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit_cta1(smem_u32(&c.empty[stage]));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit_cta1(smem_u32(&c.tfull[acc]));
      }
      // All MMAs issued by this thread complete before TMEM is released.
      mma_commit_cta1(smem_u32(&c.done));
      mbar_drain(smem_u32(&c.done), 0u, drain_limit);
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;       // which half of the tile's columns
    const int row = q * 32 + lane;
    int it = 0;
    const uint16_t* bias = (const uint16_t*)a.bias;
    uint16_t* C = (uint16_t*)a.C;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      int g, m, n;
      map_tile(c, G, n_tiles, tile, g, m, n);
      const int acc = it & 1;
      const uint32_t aphase = (uint32_t)(it >> 1) & 1u;
      bool ok = mbar_wait(smem_u32(&c.tfull[acc]), aphase, abort, limit, a.err, kWhereGemm + 4);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int grow = m * BM + row;
      const bool valid = grow < c.rows[g];
      const int64_t orow = (int64_t)c.orow[g] + grow;
      const int wslab = c.w[g];
      const int n0 = n * BN_OUT;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * MMA_N);
      constexpr int CHUNKS = BN_OUT / 32;   // 32-column chunks per tile
      for (int ch = half * (CHUNKS / 2); ch < (half + 1) * (CHUNKS / 2); ++ch) {
        const int col0 = n0 + ch * 32;
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)(ch * 32), v);
        if (SWIGLU) {
          uint32_t u[32];
          tmem_ld32(tbase + 128u + (uint32_t)(ch * 32), u);
          tmem_wait_ld();
          if (valid && col0 < a.N) {
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = silu(__uint_as_float(v[2 * i])) * __uint_as_float(u[2 * i]);
              const float h1 = silu(__uint_as_float(v[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
              p[i] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(C + orow * a.N + col0);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
          }
        } else {
          tmem_wait_ld();
          if (valid && col0 < a.N) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
            if (bias) {
              float bv[32];
              load_bf16x32(bias + (int64_t)wslab * a.N + col0, bv);
#pragma unroll
              for (int i = 0; i < 32; ++i) f[i] += bv[i];
            }
            if (a.act == MOE_ACT_RELU) {
#pragma unroll
              for (int i = 0; i < 32; ++i) f[i] = f[i] > 0.f ? f[i] : 0.f;
            } else if (a.act == MOE_ACT_GELU) {
#pragma unroll
              for (int i = 0; i < 32; ++i) f[i] = gelu_erf(f[i]);
            }
            if (OUT_F32) {
              float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.C) + orow * a.N + col0);
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
            } else {
              uint32_t p[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
              uint4* dst = reinterpret_cast<uint4*>(C + orow * a.N + col0);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c.tempty[acc]));
    }
  }

  // ---- tear-down: everyone here, nothing in flight, then free TMEM ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---- host: tensor maps --------------------------------------------------------
// Row-major [rows, K] bf16, box 64 (K) x 128 (rows).
bool map_rows(CUtensorMap* m, const void* ptr, int64_t rows, int K) { return tmap_bf16_2d(m, ptr, rows, K, BK, BM); }

// Stacked weights [G, K, N] bf16, box 64 (N) x 64 (K) x 1.
bool map_weights(CUtensorMap* m, const void* ptr, int G, int K, int N) {
  return tmap_bf16_3d(m, ptr, G, K, N, 64, BK);
}

}  // namespace

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t s) {
  if (a.dtype == MOE_DT_F32) return launch_grouped_gemm_f32(a, s);
  if (!a.single_cta || a.fp8) return launch_grouped_gemm_pair(a, s);
  if (a.max_mtiles <= 0) return cudaSuccess;
  if (a.G > MAX_G || a.K % BK != 0 || a.N % 64 != 0) return cudaErrorInvalidValue;
  if (a.out_f32 && a.act == MOE_ACT_SWIGLU) return cudaErrorInvalidValue;
  CUtensorMap mA0, mA1, mB, mB3;
  const bool swiglu = a.act == MOE_ACT_SWIGLU;
  if (!map_rows(&mA0, a.A0, a.rows_A0, a.K)) return cudaErrorInvalidValue;
  if (a.A1) {
    if (!map_rows(&mA1, a.A1, a.rows_A1, a.K)) return cudaErrorInvalidValue;
  } else {
    mA1 = mA0;
  }
  if (!map_weights(&mB, a.B, a.Gw, a.K, a.N)) return cudaErrorInvalidValue;
  if (swiglu) {
    if (!map_weights(&mB3, a.B3, a.Gw, a.K, a.N)) return cudaErrorInvalidValue;
  } else {
    mB3 = mB;
  }
  const int bn = swiglu ? 128 : 256;
  const int64_t max_tiles = a.max_mtiles * ((a.N + bn - 1) / bn);
  const int grid = (int)(max_tiles < sm_count() ? max_tiles : sm_count());
  auto go = [&](auto kernel) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    kernel<<<grid, THREADS, kSmemBytes, s>>>(mA0, mA1, mB, mB3, a);
    return cudaSuccess;
  };
  cudaError_t e;
  if (swiglu)
    e = go(gemm_tcgen05_kernel<true, false>);
  else if (a.out_f32)
    e = go(gemm_tcgen05_kernel<false, true>);
  else
    e = go(gemm_tcgen05_kernel<false, false>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
