// Expert GEMMs of the backward pass, on CTA pairs (cta_group::2 tcgen05 MMAs,
// 256 x 256 pair tiles, the same pipeline as the forward kernel).
//
//   dgrad  C[r, :] = epi( A[r, :] W[g]^T (+ A2[r, :] W2[g]^T) )
//          for each row r of segment g: the activation gradient through a
//          weight slab.  A (dO, or dA then dU) is read K-major as in the
//          forward; the weights are read K-major too: W[g] is stored [N, K]
//          (the forward's [in, out] slab of the layer it differentiates), so a
//          B tile is a 128-row x 64-k TMA box, like an A tile.  With a second
//          phase (SwiGLU: dA W1^T + dU W3^T) the k-loop runs on into the
//          second pair of tensors and accumulates into the same TMEM.
//          Epilogues: fp32 store (dx of the grouped rows), or the activation
//          backward from the saved pre-activations (dH -> dA, dU in bf16).
//   wgrad  dW[g] = X_g^T D_g: the weight gradient of segment g, summed over
//          its rows.  X (activations, [rows, M]) is read MN-major: a tile is
//          two 64-column x 64-row TMA boxes, the layout of the forward's B
//          tiles; D ([rows, N]) N-major as in the forward.  The k-loop runs
//          over the segment's rows, which the backward pass pads to whole
//          64-row blocks with zero rows, so no block crosses into the next
//          segment.  A segment without rows stores zeros.
// Every wait is bounded; a pair tears down at cluster barriers both CTAs reach.
//
// Sources: "手撕一个极简 MoE-FFN" §四 (Expert = w2(act(w1 x))), §七 (the aux loss
// trained jointly); "MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现" §4.3
// (one backward through the main and the aux loss).
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int BMP = 256;
constexpr int BMC = 128;
constexpr int BK = 64;
constexpr int MMA_N = 256;
constexpr int UMMA_K = 16;
constexpr int STAGES = 6;
constexpr int A_BYTES = BMC * BK * 2;          // 16 KB
constexpr int B_BYTES = 128 * BK * 2;          // 16 KB: this CTA's 128 columns
constexpr int BOX8 = 64 * BK * 2;              // 8 KB: one 64 x 64 box
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t kPairStageTx = 2u * STAGE_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int MAX_G = 264;
constexpr uint32_t kWhere = 0x500;

enum { kDgradF32 = 0, kDgradAct = 1, kWgrad = 2 };

// kind::f16, bf16 x bf16 -> fp32; a_mn / b_mn: operand stored MN-major.
constexpr uint32_t idesc(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(MMA_N >> 3) << 17) | ((uint32_t)(BMP >> 4) << 24);
}

struct Ctl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t done;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t skip;
  int mt[MAX_G + 1];     // dgrad: prefix of ceil(rows / 256); wgrad: g * tiles per slab
  int rows[MAX_G];
  int w[MAX_G];
  int orow[MAX_G];
  int asrc[MAX_G];
};
// fp32 outputs (dgrad of the grouped rows, weight gradients) leave through
// shared memory and TMA stores: a 4 KB 32 x 32 tile per epilogue warp, paid
// for with one ring stage.
constexpr int kStageTileBytes = 32 * 32 * 4;
// (The activation backward stages its two bf16 32 x 32 outputs, dA and dU, in
// the same 4 KB per warp.)
template <int MODE>
constexpr int ring_stages() { return STAGES - 1; }
template <int MODE>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)ring_stages<MODE>() * STAGE_BYTES + sizeof(Ctl) + 1024 + (size_t)EPI_WARPS * kStageTileBytes;
}
static_assert(smem_bytes<kDgradF32>() <= 227 * 1024 && smem_bytes<kDgradAct>() <= 227 * 1024,
              "shared memory per CTA");

// sigma(a) with the fast divide (0 for a below about -87, where 1 + e^-a
// leaves the divide's range; sigma is below 1e-37 there).
__device__ __forceinline__ float sigmoid_fast(float a) { return __fdividef(1.f, 1.f + __expf(-a)); }
__device__ __forceinline__ float gelu_grad(float z) {
  // d/dz [z Phi(z)] = Phi(z) + z phi(z)
  return 0.5f * (1.f + erff(z * 0.70710678118654752f)) + z * 0.39894228040143268f * __expf(-0.5f * z * z);
}

template <int MODE, bool TWO_PHASE>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_bwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                    const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2, BwdGemmArgs a,
                    int tma_store) {
  constexpr bool WGRAD = MODE == kWgrad;
  constexpr int NST = ring_stages<MODE>();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* ring = smem_raw + (base - raw);
  Ctl& c = *reinterpret_cast<Ctl*>(ring + NST * STAGE_BYTES);
  // fp32 outputs: the epilogue warps' TMA-store tiles, 1 KB aligned (128-byte swizzle)
  const uint32_t stg = (base + (uint32_t)(NST * STAGE_BYTES + sizeof(Ctl)) + 1023u) & ~1023u;
  volatile uint32_t* abort = &c.abort;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int G = a.G;
  // dgrad: output columns N, reduction K (per phase); wgrad: M x N per slab.
  const int n_tiles = (a.N + MMA_N - 1) / MMA_N;
  const int m_tiles_w = WGRAD ? (a.M + BMP - 1) / BMP : 0;
  const int nkb_phase = WGRAD ? 0 : a.K / BK;
  const uint64_t limit = (uint64_t)a.timeout_ns;
  const uint64_t drain_limit = limit > 2000000000ull ? limit : 2000000000ull;

  for (int i = threadIdx.x; i < G; i += blockDim.x) {
    c.rows[i] = a.seg.rows[i];
    c.w[i] = a.seg.w[i];
    c.orow[i] = a.seg.out_row[i];
    c.asrc[i] = a.x_from_asrc ? a.seg.a_src[i] : 0;
  }
  if (warp == 0) {
    const int PG = (G + 31) / 32;
    int local = 0;
    for (int i = 0; i < PG; ++i) {
      const int g = lane * PG + i;
      if (g < G) local += WGRAD ? m_tiles_w * n_tiles : (a.seg.rows[g] + BMP - 1) / BMP * n_tiles;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < PG; ++i) {
      const int g = lane * PG + i;
      if (g < G) {
        c.mt[g] = run;
        run += WGRAD ? m_tiles_w * n_tiles : (a.seg.rows[g] + BMP - 1) / BMP * n_tiles;
      }
    }
    if (lane == 31) c.mt[G] = incl;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&c.full[s]), 1);
      mbar_init(smem_u32(&c.empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&c.tfull[s]), 1);
      mbar_init(smem_u32(&c.tempty[s]), 2 * EPI_WARPS);
    }
    mbar_init(smem_u32(&c.done), 1);
    c.abort = 0u;
    c.skip = *(volatile const uint32_t*)a.err;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    if (TWO_PHASE || WGRAD) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA2) : "memory");
    if (TWO_PHASE) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB2) : "memory");
  }
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&c.tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const int total = c.skip ? 0 : c.mt[G];

  // tile -> (segment g, row block m, column block n); wgrad: m is a block of
  // the slab's M rows.
  auto map_tile = [&](int tile, int& g, int& m, int& n) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (c.mt[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    g = lo;
    const int local = tile - c.mt[g];
    if (WGRAD && a.M > a.N) {
      // Pairs running at the same time share the larger operand's column
      // block (X^T rows m) and sweep the smaller one's, which stays in L2.
      m = local / n_tiles;
      n = local - m * n_tiles;
      return;
    }
    const int mtg = WGRAD ? m_tiles_w : (c.mt[g + 1] - c.mt[g]) / n_tiles;
    n = local / mtg;
    m = local - n * mtg;
  };
  auto tile_kb = [&](int g) { return WGRAD ? c.rows[g] / BK : (TWO_PHASE ? 2 : 1) * nkb_phase; };

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      const uint32_t full_leader = mapa_shared(smem_u32(&c.full[0]), 0);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[NST];
      bool issued[NST];
      for (int s = 0; s < NST; ++s) { issued[s] = false; issued_phase[s] = 0; }
      for (int tile = pair; tile < total; tile += npairs) {
        int g, m, n;
        map_tile(tile, g, m, n);
        const int nkb = tile_kb(g);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_i(smem_u32(&c.empty[stage]), phase ^ 1u, abort, limit, a.err, kWhere + 1)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_expect_tx(smem_u32(&c.full[stage]), kPairStageTx);
          const uint32_t fb = full_leader + (uint32_t)(stage * 8);
          const uint32_t sa = base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          if (WGRAD) {
            // A' = X^T: columns m0.. of X rows of the k-block; X is the
            // segment's grouped activations, or x itself (a_src 1, from row 0).
            const CUtensorMap* xm = c.asrc[g] ? &tmA2 : &tmA;
            const int xrow = (c.asrc[g] ? 0 : c.orow[g]) + kb * BK;
            const int mcol = m * BMP + (int)rank * BMC;
            tma_load_2d_pair(sa, xm, mcol, xrow, fb);
            tma_load_2d_pair(sa + BOX8, xm, mcol + 64, xrow, fb);
            const int drow = c.orow[g] + kb * BK;
            const int ncol = n * MMA_N + (int)rank * 128;
            tma_load_2d_pair(sb, &tmB, ncol, drow, fb);
            tma_load_2d_pair(sb + BOX8, &tmB, ncol + 64, drow, fb);
          } else {
            const bool second = TWO_PHASE && kb >= nkb_phase;
            const int kk = (second ? kb - nkb_phase : kb) * BK;
            const int arow = c.orow[g] + m * BMP + (int)rank * BMC;
            tma_load_2d_pair(sa, second ? &tmA2 : &tmA, kk, arow, fb);
            // B' = W^T: 128 rows (output columns) of the slab, 64 k.
            const int brow = n * MMA_N + (int)rank * 128;
            tma_load_3d_pair(sb, second ? &tmB2 : &tmB, kk, brow, c.w[g], fb);
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      if (rank == 0)
        for (int s = 0; s < NST; ++s)
          if (issued[s]) mbar_drain(smem_u32(&c.full[s]), issued_phase[s], drain_limit);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader) ----------------
    if (lane == 0 && rank == 0) {
      constexpr uint32_t kId = WGRAD ? idesc(true, true) : idesc(false, false);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = pair; tile < total && ok; tile += npairs, ++it) {
        int g, m, n;
        map_tile(tile, g, m, n);
        const int nkb = tile_kb(g);
        const int acc = it & 1;
        const uint32_t aphase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_i(smem_u32(&c.tempty[acc]), aphase ^ 1u, abort, limit, a.err, kWhere + 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * MMA_N);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_i(smem_u32(&c.full[stage]), phase, abort, limit, a.err, kWhere + 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k4 = 0; k4 < BK / UMMA_K; ++k4) {
            uint64_t ad, bd;
            if (WGRAD) {
              // MN-major: 64-column boxes 8 KB apart, 8-row k groups 1024 B apart.
              ad = smem_desc(sa + k4 * 2048, BOX8, 1024);
              bd = smem_desc(sb + k4 * 2048, BOX8, 1024);
            } else {
              // K-major: 8-row groups 1024 B apart; a K step of 16 is 32 bytes.
              ad = smem_desc(sa + k4 * 32, 16, 1024);
              bd = smem_desc(sb + k4 * 32, 16, 1024);
            }
            mma_bf16_cta2<kId>(d_tmem, ad, bd, (kb | k4) != 0 ? 1u : 0u);
          }
          mma_commit_cta2(smem_u32(&c.empty[stage]), 0x3);
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit_cta2(smem_u32(&c.tfull[acc]), 0x3);
      }
      mma_commit_cta2(smem_u32(&c.done), 0x3);
    }
    if (lane == 0) mbar_drain(smem_u32(&c.done), 0u, drain_limit);
  } else {
    // ---------------- epilogue (both CTAs) ----------------
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const uint32_t tempty_leader = mapa_shared(smem_u32(&c.tempty[0]), 0);
    int it = 0;
    for (int tile = pair; tile < total; tile += npairs, ++it) {
      int g, m, n;
      map_tile(tile, g, m, n);
      const int nkb = tile_kb(g);
      const int acc = it & 1;
      const uint32_t aphase = (uint32_t)(it >> 1) & 1u;
      if (MODE == kDgradAct) {
        // While the tile's MMAs run, pull this thread's pre-activations (its
        // row, its half of the tile's columns) into L2 for the epilogue.
        const int grow = m * BMP + (int)rank * BMC + row;
        const int c0 = n * MMA_N + half * 128;
        const int ncols = a.N - c0 < 128 ? a.N - c0 : 128;
        if (grow < c.rows[g] && ncols > 0) {
          const size_t off = ((size_t)(c.orow[g] + grow) * a.N + c0) * 2;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"((const uint8_t*)a.pre_a + off),
                       "r"(ncols * 2)
                       : "memory");
          if (a.act == MOE_ACT_SWIGLU)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"((const uint8_t*)a.pre_u + off),
                         "r"(ncols * 2)
                         : "memory");
        }
      }
      bool ok = mbar_wait_i(smem_u32(&c.tfull[acc]), aphase, abort, limit, a.err, kWhere + 4);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int n0 = n * MMA_N;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * MMA_N);
      // Output row of this thread and whether it is stored.
      int64_t orow;
      bool valid;
      // First output row of this warp's 32 and whether all 32 are stored (then
      // an fp32 output leaves by TMA store, one 32 x 32 box per chunk).
      int64_t wrow0;
      bool wfull;
      if (WGRAD) {
        const int mr = m * BMP + (int)rank * BMC + row;
        valid = mr < a.M;
        orow = (int64_t)c.w[g] * a.M + mr;          // dW[g] is [M, N]
        wrow0 = (int64_t)c.w[g] * a.M + m * BMP + (int)rank * BMC + q * 32;
        wfull = m * BMP + (int)rank * BMC + q * 32 + 31 < a.M;
      } else {
        const int grow = m * BMP + (int)rank * BMC + row;
        valid = grow < c.rows[g];
        orow = (int64_t)c.orow[g] + grow;
        wrow0 = (int64_t)c.orow[g] + m * BMP + (int)rank * BMC + q * 32;
        wfull = m * BMP + (int)rank * BMC + q * 32 + 31 < c.rows[g];
      }
      const bool tma_st = tma_store && wfull;
      const uint32_t wbuf = stg + (uint32_t)((warp - 2) * kStageTileBytes);
      for (int ch = half * 4; ch < half * 4 + 4; ++ch) {
        const int col0 = n0 + ch * 32;
        uint32_t v[32];
        if (nkb > 0) {
          tmem_ld32(tbase + (uint32_t)(ch * 32), v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;      // no rows: a zero gradient
        }
        if (!valid || col0 >= a.N) continue;
        if (MODE == kDgradAct) {
          // dH -> dA (and dU) from the saved pre-activations.
          // Row offsets are multiples of N (a multiple of 64) and col0 of 32:
          // the 32 pre-activations are 64 aligned bytes, four vector loads.
          float av[32];
          load_bf16x32((const uint16_t*)a.pre_a + orow * a.N + col0, av);
          uint32_t da[32], du[32];
          if (a.act == MOE_ACT_SWIGLU) {
            float uv[32];
            load_bf16x32((const uint16_t*)a.pre_u + orow * a.N + col0, uv);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              // silu(a) = a s, silu'(a) = s (1 + a (1 - s)), s = sigma(a)
              const float dh = __uint_as_float(v[i]);
              const float sg = sigmoid_fast(av[i]);
              da[i] = __float_as_uint(dh * uv[i] * (sg * (1.f + av[i] * (1.f - sg))));
              du[i] = __float_as_uint(dh * (av[i] * sg));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float dh = __uint_as_float(v[i]);
              const float gr = a.act == MOE_ACT_RELU ? (av[i] > 0.f ? 1.f : 0.f) : gelu_grad(av[i]);
              da[i] = __float_as_uint(dh * gr);
            }
          }
          uint32_t p[16], pu[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(__uint_as_float(da[2 * i]), __uint_as_float(da[2 * i + 1]));
          const bool two = a.act == MOE_ACT_SWIGLU;
          if (two) {
#pragma unroll
            for (int i = 0; i < 16; ++i) pu[i] = pack_bf16x2(__uint_as_float(du[2 * i]), __uint_as_float(du[2 * i + 1]));
          }
          if (tma_st) {
            // 32 rows x 64 bytes per output, 16-byte chunk j of row `lane` at
            // lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4): the 64-byte swizzle.
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t at = (uint32_t)(lane * 64) + ((uint32_t)(j ^ ((lane >> 1) & 3)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(wbuf + at), "r"(p[4 * j]),
                           "r"(p[4 * j + 1]), "r"(p[4 * j + 2]), "r"(p[4 * j + 3])
                           : "memory");
              if (two)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(wbuf + 2048u + at), "r"(pu[4 * j]),
                             "r"(pu[4 * j + 1]), "r"(pu[4 * j + 2]), "r"(pu[4 * j + 3])
                             : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, wbuf, col0, (int)wrow0);
              if (two) tma_store_2d(&tmC2, wbuf + 2048u, col0, (int)wrow0);
              bulk_commit_group();
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>((uint16_t*)a.C + orow * a.N + col0);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
            if (two) {
              uint4* dst2 = reinterpret_cast<uint4*>((uint16_t*)a.C2 + orow * a.N + col0);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst2[i] = make_uint4(pu[4 * i], pu[4 * i + 1], pu[4 * i + 2], pu[4 * i + 3]);
            }
          }
        } else if (tma_st) {
          // Row `lane` of the warp's tile, 16-byte chunk i at lane * 128 + ((i ^ (lane & 7)) << 4)
          // (the tensor map's 128-byte swizzle); the buffer is reused once the
          // previous chunk's store has read it.
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t at = wbuf + (uint32_t)(lane * 128) + ((uint32_t)(i ^ (lane & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(at), "r"(v[4 * i]), "r"(v[4 * i + 1]),
                         "r"(v[4 * i + 2]), "r"(v[4 * i + 3])
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, wbuf, col0, (int)wrow0);
            bulk_commit_group();
          }
        } else {
          float4* dst = reinterpret_cast<float4*>((float*)a.C + orow * a.N + col0);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader + (uint32_t)(acc * 8));
    }
    // The tiles' TMA stores have completed before the CTA's shared memory goes.
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  abort_grace(a.err);
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

template <int MODE, bool TWO_PHASE>
cudaError_t launch_mode(const BwdGemmArgs& a, const CUtensorMap& mA, const CUtensorMap& mA2, const CUtensorMap& mB,
                        const CUtensorMap& mB2, int64_t max_tiles, cudaStream_t s) {
  auto kernel = gemm_bwd_kernel<MODE, TWO_PHASE>;
  constexpr size_t kSmemBytes = smem_bytes<MODE>();
  // fp32 output as a tensor map for the TMA-store epilogue: dgrad rows of the
  // grouped order, or the stacked weight gradients [Gw * M, N].
  // The activation backward's bf16 outputs dA (and dU) likewise, 32 x 32 boxes
  // of 64-byte rows.
  CUtensorMap mC = mA, mC2 = mA;
  int tma_store = 0;
  if (MODE != kDgradAct) {
    const int64_t rows_c = MODE == kWgrad ? (int64_t)a.Gw * a.M : a.rows_A;
    tma_store = tmap_f32_2d(&mC, a.C, rows_c, a.N, 32) ? 1 : 0;
  } else {
    tma_store = tmap_bf16_2d_swizzle(&mC, a.C, a.rows_A, a.N, 32, 32, 64) &&
                        (a.act != MOE_ACT_SWIGLU || tmap_bf16_2d_swizzle(&mC2, a.C2, a.rows_A, a.N, 32, 32, 64))
                    ? 1
                    : 0;
  }
  static int max_clusters = -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters < 0) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (sm_count() / 2), 1, 1);
    int nc = 0;
    e = cudaOccupancyMaxActiveClusters(&nc, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (nc <= 0) return cudaErrorInvalidConfiguration;
    max_clusters = nc;
  }
  const int64_t pairs = max_tiles < max_clusters ? max_tiles : max_clusters;
  if (pairs <= 0) return cudaSuccess;
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  return cudaLaunchKernelEx(&cfg, kernel, mA, mA2, mB, mB2, mC, mC2, a, tma_store);
}

}  // namespace

cudaError_t launch_gemm_dgrad(const BwdGemmArgs& a, cudaStream_t s) {
  if (a.G > MAX_G || a.K % BK != 0 || a.N % 64 != 0 || a.max_tiles <= 0) return a.max_tiles <= 0 ? cudaSuccess
                                                                                                  : cudaErrorInvalidValue;
  CUtensorMap mA, mA2, mB, mB2;
  const bool two = a.A2 != nullptr;
  // A: grouped activations [rows, K], box 64 (k) x 128 (rows).
  if (!tmap_bf16_2d(&mA, a.A, a.rows_A, a.K, BK, BMC)) return cudaErrorInvalidValue;
  if (two && !tmap_bf16_2d(&mA2, a.A2, a.rows_A, a.K, BK, BMC)) return cudaErrorInvalidValue;
  // B': the weight slabs [G, N, K] (K contiguous), box 64 (k) x 128 (rows).
  if (!tmap_bf16_3d(&mB, a.B, a.Gw, a.N, a.K, BK, 128)) return cudaErrorInvalidValue;
  if (two && !tmap_bf16_3d(&mB2, a.B2, a.Gw, a.N, a.K, BK, 128)) return cudaErrorInvalidValue;
  if (!two) { mA2 = mA; mB2 = mB; }
  cudaError_t e;
  if (a.act_bwd) {
    e = two ? launch_mode<kDgradAct, true>(a, mA, mA2, mB, mB2, a.max_tiles, s)
            : launch_mode<kDgradAct, false>(a, mA, mA2, mB, mB2, a.max_tiles, s);
  } else {
    e = two ? launch_mode<kDgradF32, true>(a, mA, mA2, mB, mB2, a.max_tiles, s)
            : launch_mode<kDgradF32, false>(a, mA, mA2, mB, mB2, a.max_tiles, s);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gemm_wgrad(const BwdGemmArgs& a, cudaStream_t s) {
  if (a.G > MAX_G || a.M % 64 != 0 || a.N % 64 != 0) return cudaErrorInvalidValue;
  if (a.max_tiles <= 0) return cudaSuccess;
  CUtensorMap mX, mX2, mD, mD2;
  // X: [rows, M] activations, box 64 (m columns) x 64 (rows); x itself for a_src 1.
  if (!tmap_bf16_2d(&mX, a.A, a.rows_A, a.M, 64, BK)) return cudaErrorInvalidValue;
  if (a.A2) {
    if (!tmap_bf16_2d(&mX2, a.A2, a.rows_A2, a.M, 64, BK)) return cudaErrorInvalidValue;
  } else {
    mX2 = mX;
  }
  // D: [rows, N], box 64 (n columns) x 64 (rows).
  if (!tmap_bf16_2d(&mD, a.B, a.rows_B, a.N, 64, BK)) return cudaErrorInvalidValue;
  mD2 = mD;
  cudaError_t e = launch_mode<kWgrad, false>(a, mX, mX2, mD, mD2, a.max_tiles, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
