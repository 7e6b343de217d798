// K3 on CTA pairs -- grouped expert GEMM with 2-CTA tcgen05 MMAs (cta_group::2).
//
//   C[r, :] = epilogue( A[r, :] B[w(g)] )   for each row r of each segment g
//
// A thread-block cluster of two CTAs on two SMs computes one 256 x 256 pair
// tile: CTA rank 0 (the leader) and rank 1 each stage their own 128 rows of A
// and their own half of the 256 B columns (for SwiGLU: the leader the 128 x W1
// columns, the peer the same 128 x W3 columns), and one leader thread issues
// M256 N256 K16 MMAs that read both CTAs' shared memory and accumulate into
// both CTAs' TMEM (128 lanes x 256 columns each).  Against the single-CTA
// 128 x 256 tile, every SM stages and feeds the tensor core 32 KB instead of
// 48 KB per 64-deep k-block for the same MMA work, so a 6-stage ring fits.
//
// Persistent: each pair walks the pair tiles (segment-major, then 256-column
// block, then 256-row block) with a stride of the number of pairs.  Roles:
//   warp 0      TMA producer of its CTA.  Its copies complete on the LEADER's
//               full barrier (.cta_group::2), which the leader's producer arms
//               with both CTAs' byte count (64 KB per stage).
//   warp 1      TMEM owner (both CTAs allocate collectively); in the leader one
//               lane issues the MMAs and commits to both CTAs' empty / tfull
//               barriers (an mbarrier signal multicast to the pair; no data is
//               multicast).
//   warps 2-9   epilogue of its CTA's 128 rows, as in the single-CTA kernel;
//               drained accumulators are released on the leader's tempty
//               barrier (16 arrivals: both CTAs' epilogue warps).
// Rows past a segment's end are computed but never stored; B boxes past N are
// zero-filled by TMA (their columns are never stored).
//
// FP8 instantiation: A and B hold E4M3 codes, both K-major (B stored [N, K] per
// slab), a k-block is 128 codes (128 bytes: the same 32 KB stage), and the
// leader issues M256 N256 K32 kind::f8f6f4 MMAs.  K needs only be a multiple
// of 64: TMA fills the codes past K with zeros.  The epilogue multiplies each
// accumulator by its row's and its column's decoding scales.  Every wait is bounded;
// set-up and tear-down meet at cluster barriers that both CTAs always reach.
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
namespace {

constexpr int BMP = 256;                        // rows of a pair tile
constexpr int BMC = 128;                        // rows per CTA
constexpr int BK = 64;                          // 128 bytes of bf16: one swizzle row
constexpr int MMA_N = 256;
constexpr int UMMA_K = 16;
constexpr int STAGES = 6;
constexpr int A_BYTES = BMC * BK * 2;           // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;        // 8 KB: 64 columns x 64 k
constexpr int B_BYTES = 2 * B_BOX_BYTES;        // 16 KB: this CTA's 128 columns
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB
constexpr uint32_t kPairStageTx = 2u * STAGE_BYTES;
constexpr int EPI_WARPS = 8;                   // epilogue warps (16 for wide-epilogue bf16 outputs)
constexpr int THREADS = 64 + EPI_WARPS * 32;
// bf16-output GEMMs with K up to this take 16 epilogue warps (5 ring stages):
// a short main loop per tile leaves the epilogue (bias, activation, store of
// 256 columns) as the longer half of the overlap, and twice the warps hide
// its latencies.  Longer K keep 8 epilogue warps and 6 stages.
#ifndef MOE_WIDE_EPI_MAX_K
#define MOE_WIDE_EPI_MAX_K 1024
#endif
constexpr int kWideEpiMaxK = MOE_WIDE_EPI_MAX_K;

constexpr int TMEM_COLS = 512;                  // two 256-column accumulators
constexpr int MAX_G = 264;
constexpr uint32_t kWhere = 0x400;
constexpr uint32_t kIdescPair = idesc_bf16(BMP, MMA_N);
constexpr uint32_t kIdescPairF8 = idesc_e4m3(BMP, MMA_N);
constexpr int BK8 = 128;                        // E4M3 codes per k-block (128 bytes)

struct Ctl {
  uint64_t full[STAGES];    // leader: both CTAs' copies of the stage have landed
  uint64_t empty[STAGES];   // each CTA: the MMAs reading the stage are done
  uint64_t tfull[2];        // each CTA: accumulator complete
  uint64_t tempty[2];       // leader: both CTAs' epilogues drained the accumulator
  uint64_t done;            // each CTA: every MMA of the pair is done
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t skip;
  int mt[MAX_G + 1];        // prefix of ceil(rows / 256) over the segments
  int rows[MAX_G];
  int w[MAX_G];
  int orow[MAX_G];
  int arow[MAX_G];
  int asrc[MAX_G];
};

// fp32 outputs (expert GEMM 2) stage each epilogue warp's 32 x 32 tile in
// shared memory for a TMA store: 4 KB per warp, paid for with one ring stage.
// bf16 outputs (expert GEMM 1: H) stage their 32 x 32 tile the same way (2 KB
// per warp, which still fits beside the six ring stages): per-thread 16-byte
// stores put 32 rows in one store instruction and stall the epilogue on the
// LSU queue, which costs time whenever the main loop of a tile is short.
// SAVE_PRE (the backward's recomputed GEMM 1) stages its three bf16 32 x 32
// tiles (H, pre_a, pre_u: 2 KB each).
#ifndef MOE_STAGE_BF16_OUT
#define MOE_STAGE_BF16_OUT 1
#endif
constexpr bool kStageBf16Out = MOE_STAGE_BF16_OUT != 0;
constexpr int kStageTileBytes = 32 * 32 * 4;
constexpr int kStageBf16Bytes = 32 * 32 * 2;
template <bool OUT_F32, bool SAVE_PRE, bool FP8>
constexpr int warp_stage_bytes() {
  return OUT_F32 ? kStageTileBytes
                 : SAVE_PRE ? 3 * kStageBf16Bytes : (FP8 || kStageBf16Out) ? kStageBf16Bytes : 0;
}
template <bool OUT_F32, bool SAVE_PRE, bool FP8, int EPI = EPI_WARPS>
constexpr size_t smem_for(int stages) {
  return 1024 + (size_t)stages * STAGE_BYTES + sizeof(Ctl) +
         (warp_stage_bytes<OUT_F32, SAVE_PRE, FP8>()
              ? 1024 + (size_t)EPI * warp_stage_bytes<OUT_F32, SAVE_PRE, FP8>()
              : 0);
}
// As many ring stages (up to STAGES) as fit beside the staging tiles.
template <bool OUT_F32, bool SAVE_PRE, bool FP8, int EPI = EPI_WARPS>
constexpr int ring_stages() {
  int s = STAGES;
  while (s > 2 && smem_for<OUT_F32, SAVE_PRE, FP8, EPI>(s) > 227 * 1024) --s;
  return s;
}
template <bool OUT_F32, bool SAVE_PRE, bool FP8, int EPI = EPI_WARPS>
constexpr size_t smem_bytes() {
  return smem_for<OUT_F32, SAVE_PRE, FP8, EPI>(ring_stages<OUT_F32, SAVE_PRE, FP8, EPI>());
}
static_assert(smem_bytes<false, false, false>() <= 227 * 1024 && smem_bytes<true, false, false>() <= 227 * 1024 &&
                  smem_bytes<false, true, false>() <= 227 * 1024 && smem_bytes<false, false, true>() <= 227 * 1024,
              "shared memory per CTA");
static_assert(!kStageBf16Out || ring_stages<false, false, false>() == STAGES, "bf16 staging keeps six stages");
static_assert(smem_bytes<false, false, false, 16>() <= 227 * 1024, "shared memory per CTA, 16 epilogue warps");


// 16 packed bf16 pairs (one thread's 32 columns) into row `lane` of a 32 x 32
// bf16 staging tile laid out with the 64-byte swizzle: 16-byte chunk j at
// lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4).
__device__ __forceinline__ void stage_bf16_row(uint32_t buf, int lane, const uint32_t (&p)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t at = buf + (uint32_t)(lane * 64) + ((uint32_t)(j ^ ((lane >> 1) & 3)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(at), "r"(p[4 * j]), "r"(p[4 * j + 1]),
                 "r"(p[4 * j + 2]), "r"(p[4 * j + 3])
                 : "memory");
  }
}
__device__ __forceinline__ void pack_row(const uint32_t (&v)[32], uint32_t (&p)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
}

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

// 32 fp32 values (as bits) -> 32 bf16 at dst (64 bytes, 16-byte aligned).
__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const uint32_t (&v)[32]) {
  uint32_t p[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d4[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
}

// v[i] <- v[i] * ra * s[i] for 32 consecutive column scales s (16-byte aligned).
__device__ __forceinline__ void scale_acc32(uint32_t (&v)[32], float ra, const float* s) {
  const float4* s4 = reinterpret_cast<const float4*>(s);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 q = s4[i];
    v[4 * i] = __float_as_uint(__uint_as_float(v[4 * i]) * (ra * q.x));
    v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) * (ra * q.y));
    v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) * (ra * q.z));
    v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) * (ra * q.w));
  }
}

// SAVE_PRE (expert GEMM 1 of the backward pass's forward recomputation): the
// pre-activations a = x W1 + b1 (and u = x W3 for SwiGLU) are also stored, in
// bf16, at the output's rows and columns (a.pre_a, a.pre_u).
template <bool SWIGLU, bool OUT_F32, bool SAVE_PRE, bool FP8 = false, int EPI = EPI_WARPS>
__global__ void __launch_bounds__(64 + EPI * 32, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB3,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmP,
                     const __grid_constant__ CUtensorMap tmU, GemmArgs a) {
  pdl_wait();   // launched after the previous kernel may start early: its results come first
  constexpr int BN_OUT = SWIGLU ? 128 : 256;   // output columns per pair tile
  constexpr int NST = ring_stages<OUT_F32, SAVE_PRE, FP8, EPI>();
  constexpr bool STAGE_H = !OUT_F32 && (SAVE_PRE || FP8 || kStageBf16Out);   // bf16 H leaves by TMA store
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;            // 1 KB aligned ring for the 128-byte swizzle
  uint8_t* ring = smem_raw + (base - raw);
  Ctl& c = *reinterpret_cast<Ctl*>(ring + NST * STAGE_BYTES);
  // OUT_F32: the epilogue warps' TMA-store tiles, 1 KB aligned (128-byte swizzle)
  const uint32_t stg = (base + (uint32_t)(NST * STAGE_BYTES + sizeof(Ctl)) + 1023u) & ~1023u;
  volatile uint32_t* abort = &c.abort;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();        // 0: leader, 1: peer
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int G = a.G;
  const int n_tiles = (a.N + BN_OUT - 1) / BN_OUT;
  const int nkb = FP8 ? (a.K + BK8 - 1) / BK8 : a.K / BK;
  const uint64_t limit = (uint64_t)a.timeout_ns;
  const uint64_t drain_limit = limit > 2000000000ull ? limit : 2000000000ull;

  // ---- set-up ----
  for (int i = threadIdx.x; i < G; i += blockDim.x) {
    c.rows[i] = a.seg.rows[i];
    c.w[i] = a.seg.w[i];
    c.orow[i] = a.seg.out_row[i];
    c.arow[i] = a.a_from_out_rows ? a.seg.out_row[i] : a.seg.a_row[i];
    c.asrc[i] = a.a_from_out_rows ? 0 : a.seg.a_src[i];
  }
  if (warp == 0) {
    // Pair m-tiles per segment: exclusive prefix of ceil(rows / 256), lane l
    // owning segments [l * PG, (l + 1) * PG).
    const int PG = (G + 31) / 32;
    int local = 0;
    for (int i = 0; i < PG; ++i) {
      const int g = lane * PG + i;
      if (g < G) local += (a.seg.rows[g] + BMP - 1) / BMP;
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
        run += (a.seg.rows[g] + BMP - 1) / BMP;
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
      mbar_init(smem_u32(&c.tempty[s]), 2 * EPI);
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
    __syncwarp();
    // Collective with the peer CTA's warp 1: the same columns in both TMEMs.
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&c.tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();     // both CTAs' barriers are initialised before either signals the other
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const int total = c.skip ? 0 : c.mt[G] * n_tiles;

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
        map_tile(c, G, n_tiles, tile, g, m, n);
        const int arow = c.arow[g] + m * BMP + (int)rank * BMC;
        const CUtensorMap* amap = c.asrc[g] ? &tmA1 : &tmA0;
        const int wslab = c.w[g];
        // B columns of this CTA: SwiGLU -> W1 (leader) or W3 (peer) columns
        // n0..n0+127; otherwise columns n0 + 128 rank .. + 127.
        const CUtensorMap* bmap = (SWIGLU && rank) ? &tmB3 : &tmB;
        const int bcol = SWIGLU ? n * BN_OUT : n * BN_OUT + (int)rank * 128;
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
          if (FP8) {
            // A: 128 rows x 128 codes; B: this CTA's 128 columns (rows of the
            // [N, K] slab) x 128 codes.
            tma_load_2d_pair(sa, amap, kb * BK8, arow, fb);
            tma_load_3d_pair(sb, bmap, kb * BK8, bcol, wslab, fb);
          } else {
            tma_load_2d_pair(sa, amap, kb * BK, arow, fb);
            tma_load_3d_pair(sb, bmap, bcol, kb * BK, wslab, fb);
            tma_load_3d_pair(sb + B_BOX_BYTES, bmap, bcol + 64, kb * BK, wslab, fb);
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // Both CTAs' copies complete on the leader's barriers: the leader
      // waits for every stage it armed before the pair may tear down.
      if (rank == 0)
        for (int s = 0; s < NST; ++s)
          if (issued[s]) mbar_drain(smem_u32(&c.full[s]), issued_phase[s], drain_limit);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader) ----------------
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = pair; tile < total && ok; tile += npairs, ++it) {
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
          if (FP8) {
#pragma unroll
            for (int kk = 0; kk < BK8 / 32; ++kk) {
              // A and B K-major, 8-row groups 1024 B apart; a K step of 32 codes is 32 bytes.
              const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
              const uint64_t bd = smem_desc(sb + kk * 32, 16, 1024);
              mma_f8_cta2<kIdescPairF8>(d_tmem, ad, bd, (kb | kk) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              // A: K-major, 8-row groups 1024 B apart; a K step of 16 is 32 bytes.
              const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
              // B: N-major, 64-column boxes 8 KB apart (LBO), 8-row k groups
              // 1024 B apart (SBO); a K step of 16 rows is 2048 bytes.
              const uint64_t bd = smem_desc(sb + kk * 2048, B_BOX_BYTES, 1024);
              mma_bf16_cta2<kIdescPair>(d_tmem, ad, bd, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          mma_commit_cta2(smem_u32(&c.empty[stage]), 0x3);
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit_cta2(smem_u32(&c.tfull[acc]), 0x3);
      }
      // Every MMA of the pair (it writes both TMEMs) completes before either
      // CTA releases its TMEM.
      mma_commit_cta2(smem_u32(&c.done), 0x3);
    }
    if (lane == 0) mbar_drain(smem_u32(&c.done), 0u, drain_limit);
  } else {
    // ---------------- epilogue (both CTAs) ----------------
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int part = (warp - 2) >> 2;       // which share of the tile's columns (EPI / 4 shares)
    const int row = q * 32 + lane;
    const uint32_t tempty_leader = mapa_shared(smem_u32(&c.tempty[0]), 0);
    int it = 0;
    const uint16_t* bias = (const uint16_t*)a.bias;
    uint16_t* C = (uint16_t*)a.C;
    for (int tile = pair; tile < total; tile += npairs, ++it) {
      int g, m, n;
      map_tile(c, G, n_tiles, tile, g, m, n);
      const int acc = it & 1;
      const uint32_t aphase = (uint32_t)(it >> 1) & 1u;
      bool ok = mbar_wait_i(smem_u32(&c.tfull[acc]), aphase, abort, limit, a.err, kWhere + 4);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int grow = m * BMP + (int)rank * BMC + row;
      const bool valid = grow < c.rows[g];
      const int64_t orow = (int64_t)c.orow[g] + grow;
      const int wslab = c.w[g];
      const int n0 = n * BN_OUT;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * MMA_N);
      float ra = 0.f;                       // FP8: this row's decoding scale
      if (FP8 && valid) ra = (c.asrc[g] ? a.a_scale1 : a.a_scale0)[c.arow[g] + grow];
      // fp32 output: a warp whose 32 rows all lie inside the segment stores
      // each 32 x 32 chunk with one TMA store (a partial warp stores its valid
      // rows itself, so no store reaches the next segment's rows).
      const int wrow0 = m * BMP + (int)rank * BMC + q * 32;
      const bool tma_st = (OUT_F32 || STAGE_H) && a.rows_C > 0 && wrow0 + 31 < c.rows[g];
      const uint32_t wbuf = stg + (uint32_t)((warp - 2) * warp_stage_bytes<OUT_F32, SAVE_PRE, FP8>());
      constexpr int CHUNKS = BN_OUT / 32;   // 32-column chunks per tile
      constexpr int PER = CHUNKS / (EPI / 4);
      for (int ch = part * PER; ch < (part + 1) * PER; ++ch) {
        const int col0 = n0 + ch * 32;
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)(ch * 32), v);
        if (SWIGLU) {
          uint32_t u[32];
          tmem_ld32(tbase + 128u + (uint32_t)(ch * 32), u);
          tmem_wait_ld();
          if (FP8 && valid && col0 < a.N) {
            scale_acc32(v, ra, a.b_scale + (int64_t)wslab * a.N + col0);
            scale_acc32(u, ra, a.b3_scale + (int64_t)wslab * a.N + col0);
          }
          if (SAVE_PRE && valid && col0 < a.N && !tma_st) {
            store_bf16x32((uint16_t*)a.pre_a + orow * a.N + col0, v);
            store_bf16x32((uint16_t*)a.pre_u + orow * a.N + col0, u);
          }
          if (valid && col0 < a.N) {
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = silu(__uint_as_float(v[2 * i])) * __uint_as_float(u[2 * i]);
              const float h1 = silu(__uint_as_float(v[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
              p[i] = pack_bf16x2(h0, h1);
            }
            if (STAGE_H && tma_st) {
              // H (and with SAVE_PRE pre_a, pre_u) of the warp's 32 rows leave by TMA stores.
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
              stage_bf16_row(wbuf, lane, p);
              if (SAVE_PRE) {
                uint32_t pa[16], pu[16];
                pack_row(v, pa);
                pack_row(u, pu);
                stage_bf16_row(wbuf + kStageBf16Bytes, lane, pa);
                stage_bf16_row(wbuf + 2 * kStageBf16Bytes, lane, pu);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                const int r0 = (int)(c.orow[g] + wrow0);
                tma_store_2d(&tmC, wbuf, col0, r0);
                if (SAVE_PRE) {
                  tma_store_2d(&tmP, wbuf + kStageBf16Bytes, col0, r0);
                  tma_store_2d(&tmU, wbuf + 2 * kStageBf16Bytes, col0, r0);
                }
                bulk_commit_group();
              }
            } else {
              uint4* dst = reinterpret_cast<uint4*>(C + orow * a.N + col0);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
            }
          }
        } else {
          tmem_wait_ld();
          if (valid && col0 < a.N) {
            if (FP8) scale_acc32(v, ra, a.b_scale + (int64_t)wslab * a.N + col0);
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
            if (bias) {
              float bv[32];
              load_bf16x32(bias + (int64_t)wslab * a.N + col0, bv);
#pragma unroll
              for (int i = 0; i < 32; ++i) f[i] += bv[i];
            }
            uint32_t pa[16];             // SAVE_PRE: the pre-activations, packed
            if (SAVE_PRE) {
              uint32_t fb[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) fb[i] = __float_as_uint(f[i]);
              if (tma_st)
                pack_row(fb, pa);
              else
                store_bf16x32((uint16_t*)a.pre_a + orow * a.N + col0, fb);
            }
            if (a.act == MOE_ACT_RELU) {
#pragma unroll
              for (int i = 0; i < 32; ++i) f[i] = f[i] > 0.f ? f[i] : 0.f;
            } else if (a.act == MOE_ACT_GELU) {
#pragma unroll
              for (int i = 0; i < 32; ++i) f[i] = gelu_erf(f[i]);
            }
            if (OUT_F32 && tma_st) {
              // Row `lane` of the warp's tile, 16-byte chunk i at lane * 128 + ((i ^ (lane & 7)) << 4):
              // the 128-byte swizzle the tensor map reads back.  The buffer is
              // reused once the previous chunk's store has read it.
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint32_t at = wbuf + (uint32_t)(lane * 128) + ((uint32_t)(i ^ (lane & 7)) << 4);
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(at), "f"(f[4 * i]), "f"(f[4 * i + 1]),
                             "f"(f[4 * i + 2]), "f"(f[4 * i + 3])
                             : "memory");
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmC, wbuf, col0, (int)(c.orow[g] + wrow0));
                bulk_commit_group();
              }
            } else if (OUT_F32) {
              float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.C) + orow * a.N + col0);
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
            } else if (STAGE_H && tma_st) {
              uint32_t p[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
              stage_bf16_row(wbuf, lane, p);
              if (SAVE_PRE) stage_bf16_row(wbuf + kStageBf16Bytes, lane, pa);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                const int r0 = (int)(c.orow[g] + wrow0);
                tma_store_2d(&tmC, wbuf, col0, r0);
                if (SAVE_PRE) tma_store_2d(&tmP, wbuf + kStageBf16Bytes, col0, r0);
                bulk_commit_group();
              }
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
      if (lane == 0) mbar_arrive_cluster(tempty_leader + (uint32_t)(acc * 8));
    }
    // The tiles' TMA stores have completed before the CTA's shared memory goes.
    if ((OUT_F32 || STAGE_H) && lane == 0) bulk_wait_all();
  }

  // ---- tear-down: both CTAs here, nothing in flight, then free TMEM ----
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  abort_grace(a.err);
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

bool map_rows(CUtensorMap* m, const void* ptr, int64_t rows, int K) { return tmap_bf16_2d(m, ptr, rows, K, BK, BMC); }
bool map_weights(CUtensorMap* m, const void* ptr, int G, int K, int N) {
  return tmap_bf16_3d(m, ptr, G, K, N, 64, BK);
}

template <bool SWIGLU, bool OUT_F32, bool SAVE_PRE = false, bool FP8 = false, int EPI = EPI_WARPS>
cudaError_t launch_pair(const GemmArgs& a, const CUtensorMap& mA0, const CUtensorMap& mA1, const CUtensorMap& mB,
                        const CUtensorMap& mB3, int64_t max_pair_tiles, cudaStream_t s) {
  auto kernel = gemm_pair_kernel<SWIGLU, OUT_F32, SAVE_PRE, FP8, EPI>;
  constexpr size_t kSmemBytes = smem_bytes<OUT_F32, SAVE_PRE, FP8, EPI>();
  // C (fp32), or H and the pre-activations (bf16, 64-byte rows), as tensor maps
  // for the TMA-store epilogue (else unused copies of A's)
  CUtensorMap mC = mA0, mP = mA0, mU = mA0;
  GemmArgs args = a;
  bool ok_maps = a.rows_C > 0;
  if (OUT_F32) {
    ok_maps = ok_maps && tmap_f32_2d(&mC, a.C, a.rows_C, a.N, 32);
  } else if (SAVE_PRE) {
    ok_maps = ok_maps && tmap_bf16_2d_swizzle(&mC, a.C, a.rows_C, a.N, 32, 32, 64) &&
              tmap_bf16_2d_swizzle(&mP, a.pre_a, a.rows_C, a.N, 32, 32, 64) &&
              (!SWIGLU || tmap_bf16_2d_swizzle(&mU, a.pre_u, a.rows_C, a.N, 32, 32, 64));
  } else if (FP8 || kStageBf16Out) {
    ok_maps = ok_maps && tmap_bf16_2d_swizzle(&mC, a.C, a.rows_C, a.N, 32, 32, 64);
  } else {
    ok_maps = false;
  }
  if (!ok_maps) args.rows_C = 0;
  static int max_clusters = -1;   // per kernel instantiation, per process (one device type)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(64 + EPI * 32, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters < 0) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (sm_count() / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    max_clusters = n;
  }
  const int64_t pairs = max_pair_tiles < max_clusters ? max_pair_tiles : max_clusters;
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  if (a.pdl) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kernel, mA0, mA1, mB, mB3, mC, mP, mU, args);
}

}  // namespace

// FP8 experts: E4M3 codes, A [rows, K], B [Gw, N, K].
static cudaError_t launch_pair_fp8(const GemmArgs& a, cudaStream_t s) {
  if (a.G > MAX_G || a.K % 64 != 0 || a.N % 64 != 0) return cudaErrorInvalidValue;
  if (a.out_f32 && a.act == MOE_ACT_SWIGLU) return cudaErrorInvalidValue;
  if (a.pre_a || !a.a_scale0 || !a.b_scale || (a.A1 && !a.a_scale1)) return cudaErrorInvalidValue;
  const bool swiglu = a.act == MOE_ACT_SWIGLU;
  if (swiglu && (!a.B3 || !a.b3_scale)) return cudaErrorInvalidValue;
  CUtensorMap mA0, mA1, mB, mB3;
  if (!tmap_u8_2d(&mA0, a.A0, a.rows_A0, a.K, BMC)) return cudaErrorInvalidValue;
  if (a.A1) {
    if (!tmap_u8_2d(&mA1, a.A1, a.rows_A1, a.K, BMC)) return cudaErrorInvalidValue;
  } else {
    mA1 = mA0;
  }
  if (!tmap_u8_3d(&mB, a.B, a.Gw, a.N, a.K, 128)) return cudaErrorInvalidValue;
  if (swiglu) {
    if (!tmap_u8_3d(&mB3, a.B3, a.Gw, a.N, a.K, 128)) return cudaErrorInvalidValue;
  } else {
    mB3 = mB;
  }
  const int bn = swiglu ? 128 : 256;
  const int64_t max_pair_tiles = a.max_mtiles * ((a.N + bn - 1) / bn);
  cudaError_t e;
  if (swiglu)
    e = launch_pair<true, false, false, true>(a, mA0, mA1, mB, mB3, max_pair_tiles, s);
  else if (a.out_f32)
    e = launch_pair<false, true, false, true>(a, mA0, mA1, mB, mB3, max_pair_tiles, s);
  else
    e = launch_pair<false, false, false, true>(a, mA0, mA1, mB, mB3, max_pair_tiles, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm_pair(const GemmArgs& a, cudaStream_t s) {
  if (a.max_mtiles <= 0) return cudaSuccess;
  if (a.fp8) return launch_pair_fp8(a, s);
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
  // a.max_mtiles bounds the 128-row tiles, hence also the 256-row pair tiles.
  const int64_t max_pair_tiles = a.max_mtiles * ((a.N + bn - 1) / bn);
  cudaError_t e;
  if (a.pre_a && swiglu)
    e = launch_pair<true, false, true>(a, mA0, mA1, mB, mB3, max_pair_tiles, s);
  else if (a.pre_a)
    e = launch_pair<false, false, true>(a, mA0, mA1, mB, mB3, max_pair_tiles, s);
  else if (swiglu && a.K <= kWideEpiMaxK)
    e = launch_pair<true, false, false, false, 16>(a, mA0, mA1, mB, mB3, max_pair_tiles, s);
  else if (swiglu)
    e = launch_pair<true, false>(a, mA0, mA1, mB, mB3, max_pair_tiles, s);
  else if (a.out_f32)
    e = launch_pair<false, true>(a, mA0, mA1, mB, mB3, max_pair_tiles, s);
  else if (a.K <= kWideEpiMaxK)
    e = launch_pair<false, false, false, false, 16>(a, mA0, mA1, mB, mB3, max_pair_tiles, s);
  else
    e = launch_pair<false, false>(a, mA0, mA1, mB, mB3, max_pair_tiles, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
