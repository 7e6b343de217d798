// K1 -- router: logits l = x W_g + b_g, softmax or normalised-sigmoid gating,
// top-k with the lower expert index winning ties, renormalised weights, and
// per-CTA routing partials (selection histogram, local ranks, sums of p).
//
// The logit contraction has N = E <= 256 and K = d: per token it does 2 d E
// flops on d * 2 bytes of x, so for E >= 16 plain FP32 FMA would fall below the
// HBM rate.  The bf16 path therefore runs the contraction on the tensor cores
// with warp-level mma.sync (m16n8k16, fp32 accumulate).  One producer warp
// streams x (and W_g when E is 8, 16, 32, 64, 128 or 256) by TMA into a deep
// shared-memory ring; eight MMA warps (four 16-token row blocks x two k-groups
// taking the even and odd k-tiles) consume it, each at its own pace (full /
// empty mbarriers per stage, no block-wide barrier in the loop).  Nothing here
// is a large GEMM worth a TMEM pipeline: the kernel streams x once, and its
// speed is set by how many bytes and independent instructions are in flight.
// The gating and selection tail runs on four threads per token.
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
#include "scan.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int kRowBlocks = 4;                         // m16 row blocks of a CTA's 64 tokens
constexpr int kMmaWarps = 2 * kRowBlocks;             // x 2 k-groups (even / odd k-tiles)
constexpr int kWarmTailWarp = kMmaWarps + 1;          // after the producer warp: dry tail pass
constexpr int kWarmScanWarp = kMmaWarps + 2;          // dry scan pass
constexpr int kThreadsBf16 = (kMmaWarps + 3) * 32;    // MMA warps, producer, two warm-up warps
constexpr int kTailThreadsBf16 = kThreadsBf16 - 32;   // all but the scan warm-up warp (the last)
constexpr int kDryTokens = 8;                         // tokens of a dry tail pass (one warp)
constexpr int kThreadsF32 = 256;
constexpr int kTPT = 4;                               // threads per token in the tail
constexpr int kBK = 64;                               // bf16 k-tile (128 bytes per x row)
constexpr uint32_t kWhereRouter = 0x300;
static_assert(kRouterBM == 16 * kRowBlocks, "one m16 row block per MMA warp of a k-group");

// Named barrier 1 over the `count` threads running the tail (a multiple of 32;
// the whole CTA except, in the mma.sync router, its scan warm-up warp).
__device__ __forceinline__ void tail_sync(int count) { asm volatile("bar.sync 1, %0;" ::"r"(count) : "memory"); }
__device__ __forceinline__ bool tail_sync_or(int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(count)
      : "memory");
  return r != 0u;
}

// ---- the per-token tail shared by both dtypes ----------------------------------
// sl: [BM][ldl] fp32 logits without bias, rows of this CTA's BM tokens.
// bits: [E][BM / 32] scratch words.  Threads with virtual ids 4i..4i+3 (one
// warp) own token i; thread q holds the experts e = q + 4 j, j < EPT, in
// registers.  Top-k is k rounds of a quad argmax: each thread's largest
// not-yet-taken logit (lower index on a tie), merged over the quad with two
// shuffle rounds, so all four threads pick the same expert in the same round.
//
// vt / nvt: this thread's id among the nvt threads running the tail (threads
// 0 .. nvt - 1 of the CTA, nvt >= 4 BM, synchronised by tail_sync).
// dry: one warp (vt = lane, nvt = 32) runs the same code on the first 8
// tokens while the CTA still streams x, writing only its own scratch (sl,
// bits) and nothing in global memory.  The tail runs once per
// CTA, so on a cold instruction cache its time is the fetch of its code (the
// expert GEMMs' weights have pushed it out of L2 since the previous call);
// the dry pass fetches it in the shadow of the stream.  Each kernel calls it
// from one place only, inside a two-pass loop (dry, then real), so that both
// passes run the same instructions.
template <int BM, int EPT>
__device__ __forceinline__ void router_finalize(float* sl, int ldl, uint32_t* bits, const RouterArgs& a,
                                             int64_t blk, int vt, int nvt, bool dry) {
  static_assert(BM % 32 == 0 && BM <= 256, "local ranks are uint8");
  static_assert(EPT >= 1 && EPT <= 64, "taken bits are one uint64_t");
  constexpr int NW = BM / 32;
  const int E = a.E, k = a.k;
  const int64_t t0 = blk * BM;
  for (int i = vt; i < E * NW; i += nvt) bits[i] = 0u;
  if (dry) __syncwarp(); else tail_sync(nvt);

  const int tok = vt / kTPT, q = vt % kTPT;
  const int64_t t = t0 + tok;
  const bool valid = vt < kTPT * BM && t < a.T && (!dry || tok < 8);
  const bool wr = valid && !dry;   // global writes
  float val[8];
  int idx[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) { val[j] = 0.f; idx[j] = -1; }
  if (vt < kTPT * BM) {            // whole warps: the shuffles see every thread of each quad
    float* l = sl + tok * ldl;
    const bool bf = a.dtype == MOE_DT_BF16;
    float v[EPT];
    if constexpr (EPT <= 32) {
      // Loads first, stores after: with a store between two loads the compiler
      // has to keep them in order (the pointers may alias), and every load then
      // waits out the previous one.
#pragma unroll
      for (int i = 0; i < EPT; ++i) {
        const int e = q + kTPT * i;
        v[i] = 0.f;
        if (valid && e < E) {
          v[i] = l[e];
          if (dry) v[i] = 0.f;   // the dry pass's scratch rows hold no logits
        }
      }
      if (a.bg) {
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
          const int e = q + kTPT * i;
          if (valid && e < E) v[i] += bf ? bf16_bits_to_f32(((const uint16_t*)a.bg)[e]) : ((const float*)a.bg)[e];
        }
      }
      if (a.noise) {   // noisy scores: everything below uses them
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
          const int e = q + kTPT * i;
          if (valid && e < E) v[i] += a.noise[t * E + e];
        }
      }
      if (wr && (a.raw_logits || (a.logits_out && !a.scores_em))) {
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
          const int e = q + kTPT * i;
          if (e < E) {
            if (a.logits_out && !a.scores_em) a.logits_out[t * E + e] = v[i];
            if (a.raw_logits) a.raw_logits[t * E + e] = v[i];
          }
        }
      }
    } else {   // 64 logits a thread: one pass, so that they fit in registers
#pragma unroll
      for (int i = 0; i < EPT; ++i) {
        const int e = q + kTPT * i;
        v[i] = 0.f;
        if (valid && e < E) {
          float x = l[e];
          if (dry) x = 0.f;
          if (a.bg) x += bf ? bf16_bits_to_f32(((const uint16_t*)a.bg)[e]) : ((const float*)a.bg)[e];
          if (a.noise) x += a.noise[t * E + e];
          v[i] = x;
          if (wr && a.logits_out && !a.scores_em) a.logits_out[t * E + e] = x;
          if (wr && a.raw_logits) a.raw_logits[t * E + e] = x;
        }
      }
    }
    // k rounds of the quad argmax (expert choice uses only the maximum, val[0]).
    const int kr = a.scores_em ? 1 : k;
    if constexpr (EPT >= 8 && EPT <= 32) {
      // Each thread's logits as order-preserving unsigned keys: the IEEE bits
      // with the sign folded, -0 read as +0 (so that it ties with +0), 1 for
      // NaN (below every number), 0 for an expert past E.  A round takes the
      // thread's largest key not yet chosen by a pairwise tree (depth log2 EPT
      // instead of a chain of EPT compares), whose left operand always holds
      // the lower experts, so that a tie keeps the lower index.
      uint32_t key[EPT];
#pragma unroll
      for (int i = 0; i < EPT; ++i) {
        uint32_t b = __float_as_uint(v[i]);
        b = b == 0x80000000u ? 0u : b;
        const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
        key[i] = (!valid || q + kTPT * i >= E) ? 0u : ((b & 0x7fffffffu) > 0x7f800000u ? 1u : ord);
      }
      uint32_t taken = 0;           // bit i: expert q + 4 i already chosen
#pragma unroll 1
      for (int j = 0; j < kr; ++j) {
        uint32_t kk[EPT];
        int ss[EPT];
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
          kk[i] = ((taken >> i) & 1u) ? 0u : key[i];
          ss[i] = i;
        }
#pragma unroll
        for (int st = 1; st < EPT; st <<= 1) {
#pragma unroll
          for (int i = 0; i + st < EPT; i += 2 * st) {
            const bool r = kk[i + st] > kk[i];
            kk[i] = r ? kk[i + st] : kk[i];
            ss[i] = r ? ss[i + st] : ss[i];
          }
        }
        uint32_t bk = kk[0];
        int bi = bk != 0u ? q + kTPT * ss[0] : 0x7fffffff;
#pragma unroll
        for (int m = 1; m < kTPT; m <<= 1) {
          const uint32_t pk = __shfl_xor_sync(0xffffffffu, bk, m);
          const int pi = __shfl_xor_sync(0xffffffffu, bi, m);
          // The larger key, the lower index on equal keys; key 0 (no candidate
          // left) loses to every candidate.
          if (pk > bk || (pk == bk && pi < bi)) { bk = pk; bi = pi; }
        }
        const float bv = bk >= 0x80000000u ? __uint_as_float(bk & 0x7fffffffu)
                         : bk > 1u         ? __uint_as_float(~bk)
                         : bk == 1u        ? __uint_as_float(0x7fc00000u)
                                           : -INFINITY;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
          if (jj == j) { val[jj] = bv; idx[jj] = bi; }
        if (bk != 0u && (bi % kTPT) == q) taken |= 1u << (bi / kTPT);
      }
    } else {   // a few logits a thread (a short chain), or 64 (registers)
      uint64_t taken = 0;           // bit i: expert q + 4 i already chosen
#pragma unroll 1
      for (int j = 0; j < kr; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        if (valid) {
#pragma unroll
          for (int i = 0; i < EPT; ++i) {
            const int e = q + kTPT * i;
            // experts ascend within the thread: a strict > keeps the lower index
            if (e < E && !((taken >> i) & 1ull) && (v[i] > bv || bi == 0x7fffffff)) { bv = v[i]; bi = e; }
          }
        }
#pragma unroll
        for (int m = 1; m < kTPT; m <<= 1) {
          const float pv = __shfl_xor_sync(0xffffffffu, bv, m);
          const int pi = __shfl_xor_sync(0xffffffffu, bi, m);
          // A thread with no candidate left (bi unset) takes its partner's; a
          // NaN logit never replaces a candidate nor leaves an index unset.
          if (bi == 0x7fffffff || (pi != 0x7fffffff && (pv > bv || (pv == bv && pi < bi)))) { bv = pv; bi = pi; }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
          if (jj == j) { val[jj] = bv; idx[jj] = bi; }
        if (valid && (bi % kTPT) == q) taken |= 1ull << (bi / kTPT);
      }
    }
    // Gating over all E (these p feed P), and the renormalised top-k weights.
    float z = 0.f;
    if (valid) {
      const bool sm = a.gating == MOE_GATE_SOFTMAX;
      const float mx = val[0];
#pragma unroll
      for (int i = 0; i < EPT; ++i) {
        if (q + kTPT * i < E) {
          const float p = sm ? expf(v[i] - mx) : 1.f / (1.f + expf(-v[i]));
          v[i] = p;
          z += p;
        }
      }
    }
    // The same total on every thread of the quad: (z0 + z1) + (z2 + z3), each
    // pair summed lower thread first.
#pragma unroll
    for (int m = 1; m < kTPT; m <<= 1) {
      const float zp = __shfl_xor_sync(0xffffffffu, z, m);
      z = (q & m) ? zp + z : z + zp;
    }
    if (valid) {
      const float rz = 1.f / z;
#pragma unroll
      for (int i = 0; i < EPT; ++i) {
        const int e = q + kTPT * i;
        if (e < E) {
          const float p = v[i] * rz;
          l[e] = p;
          if (wr && a.scores_em) {
            // Expert choice: the experts choose on these gate probabilities.
            a.scores_em[(int64_t)e * a.T + t] = p;
            if (a.logits_out) a.logits_out[t * E + e] = p;
          }
        }
      }
      if (!a.scores_em && q == 0) {
        float g[8], zsel = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j < k) {
            g[j] = a.gating == MOE_GATE_SOFTMAX ? expf(val[j] - val[0]) : 1.f / (1.f + expf(-val[j]));
            zsel += g[j];
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < k) g[j] = g[j] / zsel;
        if (wr) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j < k) {
              a.topk_idx[t * k + j] = idx[j];
              a.topk_w[t * k + j] = g[j];
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < k) atomicOr(&bits[idx[j] * NW + tok / 32], 1u << (tok % 32));
      }
    }
  }
  if (dry) __syncwarp(); else tail_sync(nvt);
  if (valid && q == 0 && !a.scores_em) {
    const int w = tok / 32;
    const uint32_t below = (1u << (tok % 32)) - 1u;
    int rk[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      rk[j] = 0;
      if (j < k) {
        const uint32_t* be = bits + idx[j] * NW;
        rk[j] = __popc(be[w] & below);
#pragma unroll
        for (int qq = 0; qq < NW - 1; ++qq)
          if (qq < w) rk[j] += __popc(be[qq]);
      }
    }
    if (wr) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < k) a.lrank[t * k + j] = (uint8_t)rk[j];
    }
  }
  // Per expert: selections (popc of the bit masks) and the sum of gate
  // probabilities over the CTA's tokens, one warp per expert: lane l adds
  // rows l, l + 32, ..., then a fixed xor-tree over the lanes.  With many
  // experts a warp takes four of its experts at a time, so that their chains
  // overlap.
  const int nvalid = dry ? 8 : (int)(a.T - t0 < BM ? a.T - t0 : BM);
  const int lane = vt % 32, nwarps = nvt / 32;
  const int Ep = dry ? 1 : E;
  constexpr int EU = EPT >= 8 ? 4 : 1;
  for (int e0 = vt / 32; e0 < Ep; e0 += EU * nwarps) {
    float s[EU];
#pragma unroll
    for (int u = 0; u < EU; ++u) s[u] = 0.f;
    for (int r = lane; r < nvalid; r += 32) {
#pragma unroll
      for (int u = 0; u < EU; ++u)
        if (e0 + u * nwarps < Ep) s[u] += sl[r * ldl + e0 + u * nwarps];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
      for (int u = 0; u < EU; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
    }
    if (lane == 0 && !dry) {
      int h[EU];
#pragma unroll
      for (int u = 0; u < EU; ++u) {
        const int e = e0 + u * nwarps;
        h[u] = 0;
        if (e < E) {
#pragma unroll
          for (int qq = 0; qq < NW; ++qq) h[u] += __popc(bits[e * NW + qq]);
        }
      }
#pragma unroll
      for (int u = 0; u < EU; ++u) {
        const int e = e0 + u * nwarps;
        if (e < E) {
          a.hist[e * a.nblk + blk] = h[u];
          a.psum[e * a.nblk + blk] = s[u];
        }
      }
    }
  }
}

// Every router CTA ends here, also one that stopped early.  With the scan
// fused, each CTA publishes its partials (fence), takes a ticket, and the CTA
// that takes the last one runs the dispatch scan over all CTAs' partials; a
// stopped CTA still takes its ticket, so the scan always runs (and, seeing the
// status word set, publishes empty segments).  `scratch`: shared memory no
// longer in use, at least 2 KB.
// dry: the warm-up warps run the scan's dry pass instead (no ticket, no
// global writes; `scratch` their own 2 KB), fetching the scan's code while x
// streams: any CTA may be the last to finish.  Each kernel calls this from
// one place.
// warp / nwarps: this warp's part of the scan (the real pass: every warp of
// the CTA; a dry pass: its warm-up warps).
template <int kScanE, int kScanU>
__device__ __forceinline__ void router_retire(const RouterArgs& a, uint8_t* scratch, bool dry, int warp,
                                              int nwarps) {
  if (!a.fused_scan) return;
  __shared__ uint32_t s_last;
  if (!dry) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(a.done, 1u) == (uint32_t)(a.nblk - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }
  int* s_npre = reinterpret_cast<int*>(scratch);
  float* s_psum = reinterpret_cast<float*>(s_npre + scan_detail::kMaxE);
  scan_detail::scan_body<kScanE, kScanU>(a.scan, s_npre, s_psum, warp, nwarps, dry);
}

// ---- bf16: tensor-core logits ---------------------------------------------------
// A CTA owns kRouterBM = 64 tokens and walks d in k-tiles of 64.  Per k-tile a
// ring stage holds KSUB consecutive x tiles [64 tokens][64 k] (8 KB each, one
// TMA copy each, 128-byte swizzle, rows past T zero-filled) and the matching
// W_g tiles [64 k][EP experts], kept as boxes of at most 64 experts whose rows
// are swizzled like the TMA copy writes them.  The ring holds about 100 KB:
// the kernel's speed is the number of bytes it keeps in flight.
// After the ring the same shared memory holds the fp32 logits [64][EP + 1].
template <int NT, int KSUB_, int STAGES_>
struct RouterBf16 {
  static constexpr int EP = 8 * NT;
  static constexpr int KSUB = KSUB_;                // k-tiles per ring stage
  static constexpr int STAGES = STAGES_;
  static constexpr int WCOLS = EP < 64 ? EP : 64;   // experts per W box
  static constexpr int WRB = WCOLS * 2;             // bytes of one W box row: 16 .. 128
  static constexpr int XS = kRouterBM * kBK * 2;    // 8 KB per x k-tile, a multiple of 1 KB (swizzle atom)
  static constexpr int WS = kBK * EP * 2;           // 1 KB * NT per W k-tile
  static constexpr int STAGE = KSUB * (XS + WS);    // [KSUB x tiles][KSUB W tiles]
  static constexpr size_t RING = (size_t)STAGES * STAGE;
  static constexpr size_t LOGITS = (size_t)kRouterBM * (EP + 1) * 4;
  static constexpr size_t BITS_OFF = RING > LOGITS ? RING : LOGITS;
  static constexpr size_t BITS = (size_t)EP * (kRouterBM / 32) * 4;
  // Scratch of the warm-up warps: the dry tail's logit rows and bit masks, the
  // dry scan's totals.
  static constexpr size_t DRY_OFF = (BITS_OFF + BITS + 15) / 16 * 16;
  static constexpr size_t DRY_SL = (size_t)kDryTokens * (EP + 1) * 4;
  static constexpr size_t DRY_BITS = BITS;
  static constexpr size_t DRY_SCAN = 2 * scan_detail::kMaxE * 4;
  static constexpr size_t BAR_OFF = (DRY_OFF + DRY_SL + DRY_BITS + DRY_SCAN + 7) / 8 * 8;
  static constexpr size_t SMEM = 1024 + BAR_OFF + 2 * STAGES * 8 + 16;   // + 1 KB to align the ring

  // Byte offset in a W k-tile of 16-byte chunk c (experts 8c..8c+7) of k-row r:
  // box c / (WRB/16), and inside it the TMA swizzle of WRB-byte rows
  // (16-byte chunk index XOR address bits 7.. of the row start).
  __device__ static int woff(int r, int c) {
    constexpr int CPR = WRB / 16;
    const int box = c / CPR, cb = c % CPR;
    return box * (kBK * WRB) + r * WRB + ((cb ^ ((r * WRB / 128) & (CPR - 1))) << 4);
  }
};

// Ring shape per expert count: a stage spans KSUB consecutive k-tiles, so a
// token row is fetched KSUB * 128 contiguous bytes at a time (DRAM pages are
// opened for more than one 128-byte piece), and the ring stays near 108 KB so
// that two CTAs share an SM.  An even KSUB gives both k-groups of MMA warps
// the same share of every stage.
template <int NT> struct RouterShape;
template <> struct RouterShape<1> { static constexpr int KSUB = 4, STAGES = 3; };
template <> struct RouterShape<2> { static constexpr int KSUB = 2, STAGES = 5; };
template <> struct RouterShape<4> { static constexpr int KSUB = 2, STAGES = 4; };
template <> struct RouterShape<8> { static constexpr int KSUB = 2, STAGES = 3; };
template <> struct RouterShape<16> { static constexpr int KSUB = 2, STAGES = 2; };
template <> struct RouterShape<32> { static constexpr int KSUB = 1, STAGES = 2; };

// NT n-tiles of 8 experts; EP = 8 NT >= E.  Warps 0-7 compute (row block w %
// 4: tokens 16 (w % 4) .. + 15; k-tiles of parity w / 4); warp 8 is the
// producer; warps 9 and 10 make the dry passes of the tail and of the scan
// while x streams.  tma_w: W_g tiles come by TMA (E == EP); otherwise the
// producer warp copies them with plain loads.
template <int NT, int KSUB, int STAGES_>
__global__ void __launch_bounds__(kThreadsBf16) router_bf16_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                   const __grid_constant__ CUtensorMap tmW,
                                                                   RouterArgs a, int tma_w) {
  using L = RouterBf16<NT, KSUB, STAGES_>;
  constexpr int EP = L::EP, STAGES = L::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint32_t* bits = (uint32_t*)(smem + L::BITS_OFF);
  uint64_t* full = (uint64_t*)(smem + L::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint32_t* abort_flag = (uint32_t*)(empty + STAGES);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int64_t blk = blockIdx.x;
  const int64_t t0 = blk * kRouterBM;
  const int E = a.E;
  const int nk = a.d / kBK;                 // k-tiles
  const int ns = (nk + KSUB - 1) / KSUB;    // ring steps
  const uint64_t limit = (uint64_t)a.timeout_ns;
  const uint64_t drain_limit = limit > 2000000000ull ? limit : 2000000000ull;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), tma_w ? 1u : 33u);   // producer lane 0 (+ 32 lanes after plain copies)
      mbar_init(smem_u32(&empty[s]), kMmaWarps);
    }
    *abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  bool stopped = false;
  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[n][q] = 0.f;

  if (warp == kMmaWarps) {
    // ---------------- producer ----------------
    const uint16_t* W = (const uint16_t*)a.Wg;
    const uint64_t x_policy = l2_policy_evict_first();   // x is streamed once
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
      if (tma_w) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
    }
    int kt = 0;   // ring step
    for (; kt < ns; ++kt) {
      const int st = kt % STAGES;
      const int k0 = kt * KSUB;
      const int nsub = nk - k0 < KSUB ? nk - k0 : KSUB;
      bool ok = true;
      if (kt >= STAGES)
        ok = mbar_wait_i(smem_u32(&empty[st]), (uint32_t)((kt / STAGES) - 1) & 1u, abort_flag, limit, a.err,
                         kWhereRouter + 1);
      if (!__all_sync(0xffffffffu, ok)) { stopped = true; break; }
      uint8_t* xs = smem + st * L::STAGE;
      uint8_t* ws = xs + KSUB * L::XS;
      const uint32_t fb = smem_u32(&full[st]);
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(fb, (uint32_t)(nsub * (L::XS + (tma_w ? L::WS : 0))));
        for (int i = 0; i < nsub; ++i)
          tma_load_2d_hint(smem_u32(xs + i * L::XS), &tmX, (k0 + i) * kBK, (int)t0, fb, x_policy);
        if (tma_w)
          for (int i = 0; i < nsub; ++i)
            for (int b = 0; b < EP / L::WCOLS; ++b)
              tma_load_2d(smem_u32(ws + i * L::WS + b * (kBK * L::WRB)), &tmW, b * L::WCOLS, (k0 + i) * kBK, fb);
      }
      if (!tma_w) {
        // W_g rows are E * 2 bytes: not TMA-able unless E is a multiple of 8,
        // and E < EP leaves a zero tail.  Plain copies, then every lane arrives.
        const bool vec = (E % 8) == 0;
        for (int i = lane; i < nsub * kBK * (EP / 8); i += 32) {
          const int sub = i / (kBK * (EP / 8)), rem = i % (kBK * (EP / 8));
          const int r = rem / (EP / 8), c = rem % (EP / 8);
          const uint16_t* src = W + (int64_t)((k0 + sub) * kBK + r) * E;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (vec) {
            if (c * 8 < E) v = *reinterpret_cast<const uint4*>(src + c * 8);
          } else {
            uint32_t h[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) h[q] = (c * 8 + q < E) ? (uint32_t)src[c * 8 + q] : 0u;
            v = make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
          }
          *reinterpret_cast<uint4*>(ws + sub * L::WS + L::woff(r, c)) = v;
        }
        mbar_arrive(fb);
      }
    }
    if (stopped && lane == 0) {
      // Every TMA copy this CTA started lands before it exits: the last
      // STAGES ring steps issued, one per slot, may still be in flight.
      for (int j = kt - STAGES > 0 ? kt - STAGES : 0; j < kt; ++j)
        mbar_drain(smem_u32(&full[j % STAGES]), (uint32_t)(j / STAGES) & 1u, drain_limit);
    }
  } else if (warp < kMmaWarps) {
    // ---------------- MMA warps ----------------
    // Warp w: row block w % 4, k-group w / 4 (k-tiles of that parity).  Every
    // warp waits on and releases every stage, so the empty barrier's phases
    // stay in step even when a stage holds no k-tile of the warp's parity.
    const int rb = warp % kRowBlocks, kg = warp / kRowBlocks;
    for (int kt = 0; kt < ns; ++kt) {
      const int st = kt % STAGES;
      const int nsub = nk - kt * KSUB < KSUB ? nk - kt * KSUB : KSUB;
      bool ok = mbar_wait_i(smem_u32(&full[st]), (uint32_t)(kt / STAGES) & 1u, abort_flag, limit, a.err,
                            kWhereRouter + 2);
      if (!__all_sync(0xffffffffu, ok)) { stopped = true; break; }
      for (int sub = 0; sub < nsub; ++sub) {
      if (((kt * KSUB + sub) & 1) != kg) continue;
      const uint32_t xb = smem_u32(smem + st * L::STAGE) + sub * L::XS;
      const uint32_t wb = smem_u32(smem + st * L::STAGE) + KSUB * L::XS + sub * L::WS;
#pragma unroll
      for (int ks = 0; ks < kBK / 16; ++ks) {
        uint32_t af[4];
        {
          // x tile row r, 16-byte chunk c sits at r * 128 + ((c ^ (r & 7)) << 4).
          const int r = rb * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int c = ks * 2 + (lane >> 4);
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
                         : "r"(wb + L::woff(kr, 0)));
          } else {
            const int nc = 2 * np + (i >> 1);
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(bf[0]), "=r"(bf[1]), "=r"(bf[2]), "=r"(bf[3])
                         : "r"(wb + L::woff(kr, nc)));
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
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
    }
  }
  // The tail, in two passes through one copy of its code.  Pass 0 (dry) runs
  // only on the two warm-up warps, while the other warps still stream: the
  // tail on 8 tokens of scratch, and the scan.  Pass 1 runs the tail on every
  // warp but the scan warm-up warp (which may still be in its dry pass; the
  // tail's barriers leave it out), then the retirement on all.
  const int ldl = EP + 1;
  uint8_t* dry_area = smem + L::DRY_OFF;
#pragma unroll 1
  for (int pass = warp >= kWarmTailWarp ? 0 : 1; pass < 2; ++pass) {
    const bool dry = pass == 0;
    if (dry ? warp == kWarmTailWarp : warp != kWarmScanWarp) {
      bool stop = false;
      if (!dry) {
        // Every warp is past its last read of the ring before the logits overwrite it.
        stop = tail_sync_or(kTailThreadsBf16, stopped);
        if (!stop) {
          float* sl = (float*)smem;
          // logits = (even k-tiles) + (odd k-tiles): k-group 1 stores its partial, and
          // the k-group 0 warp of the same row block (same lane -> same elements) adds
          // its own in front.
          const int r0 = (warp % kRowBlocks) * 16 + (lane >> 2);
          if (warp >= kRowBlocks && warp < kMmaWarps) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              const int c = n * 8 + 2 * (lane & 3);
              sl[r0 * ldl + c] = acc[n][0];
              sl[r0 * ldl + c + 1] = acc[n][1];
              sl[(r0 + 8) * ldl + c] = acc[n][2];
              sl[(r0 + 8) * ldl + c + 1] = acc[n][3];
            }
          }
          tail_sync(kTailThreadsBf16);
          if (warp < kRowBlocks) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              const int c = n * 8 + 2 * (lane & 3);
              sl[r0 * ldl + c] = acc[n][0] + sl[r0 * ldl + c];
              sl[r0 * ldl + c + 1] = acc[n][1] + sl[r0 * ldl + c + 1];
              sl[(r0 + 8) * ldl + c] = acc[n][2] + sl[(r0 + 8) * ldl + c];
              sl[(r0 + 8) * ldl + c + 1] = acc[n][3] + sl[(r0 + 8) * ldl + c + 1];
            }
          }
          tail_sync(kTailThreadsBf16);
        }
      }
      if (!stop)
        router_finalize<kRouterBM, EP / kTPT>(dry ? (float*)dry_area : (float*)smem, ldl,
                                              dry ? (uint32_t*)(dry_area + L::DRY_SL) : bits, a, blk,
                                              dry ? lane : tid, dry ? 32 : kTailThreadsBf16, dry);
    }
    if (!dry || warp == kWarmScanWarp)
      // E <= 32: one expert per warp and round, 256 router CTAs per load
      // round (T = 16384 in one round); more experts: two per warp.
      router_retire<(NT <= 4 ? 1 : 2), (NT <= 4 ? 8 : 4)>(a, dry ? dry_area + L::DRY_SL + L::DRY_BITS : smem, dry, dry ? 0 : warp,
                          dry ? 1 : kThreadsBf16 / 32);
  }
}

// ---- fp32: CUDA-core logits ------------------------------------------------------
constexpr int kBK32 = 32;
// EPT: experts per tail thread, E <= 4 EPT.
template <int EPT>
__global__ void __launch_bounds__(kThreadsF32) router_f32_kernel(RouterArgs a) {
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
  for (int i = tid; i < kRouterBM * ldl; i += kThreadsF32) sl[i] = 0.f;
  for (int kt = 0; kt < d; kt += kBK32) {
    __syncthreads();
    for (int i = tid; i < kRouterBM * kBK32; i += kThreadsF32) {
      int r = i / kBK32, c = i % kBK32;
      int64_t t = t0 + r;
      xs[r * (kBK32 + 1) + c] = (t < a.T && kt + c < d) ? x[t * d + kt + c] : 0.f;
    }
    for (int i = tid; i < kBK32 * E; i += kThreadsF32) {
      int r = i / E, e = i % E;
      wsm[i] = (kt + r < d) ? W[(int64_t)(kt + r) * E + e] : 0.f;
    }
    __syncthreads();
    for (int o = tid; o < kRouterBM * E; o += kThreadsF32) {
      int r = o / E, e = o % E;
      float s = sl[r * ldl + e];
      for (int c = 0; c < kBK32; ++c) s = fmaf(xs[r * (kBK32 + 1) + c], wsm[c * E + e], s);
      sl[r * ldl + e] = s;
    }
  }
  __syncthreads();
  router_finalize<kRouterBM, EPT>(sl, ldl, bits, a, blk, tid, kThreadsF32, false);
  router_retire<2, 4>(a, smem, false, tid / 32, kThreadsF32 / 32);
}

template <int NT>
cudaError_t launch_bf16(const RouterArgs& a, int64_t nblk, cudaStream_t s) {
  constexpr int KSUB = RouterShape<NT>::KSUB, STAGES = RouterShape<NT>::STAGES;
  using L = RouterBf16<NT, KSUB, STAGES>;
  static_assert(L::SMEM <= 113 * 1024, "two router CTAs per SM");
  const size_t bytes = L::SMEM;
  CUtensorMap tmX, tmW;
  if (!tmap_bf16_2d(&tmX, a.x, a.T, a.d, kBK, kRouterBM)) return cudaErrorInvalidValue;
  int tma_w = 0;
  if (a.E == L::EP) {
    if (!tmap_bf16_2d_swizzle(&tmW, a.Wg, a.d, a.E, L::WCOLS, kBK, L::WRB)) return cudaErrorInvalidValue;
    tma_w = 1;
  } else {
    tmW = tmX;   // not read
  }
  auto kern = router_bf16_kernel<NT, KSUB, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)nblk, kThreadsBf16, bytes, s>>>(tmX, tmW, a, tma_w);
  return cudaGetLastError();
}


// ---- bf16 with E a multiple of 64: tcgen05 logits -------------------------------
// A CTA owns kRouterBMTc = 128 tokens.  The logit contraction of the tile is
// one tcgen05 MMA chain, M = 128 tokens x N = E experts x K = d, accumulated
// in TMEM:
//   warp 0      TMA producer: per 64-deep k-block the x tile [128 tokens][64 k]
//               (16 KB, K-major, 128-byte swizzle, rows past T zero-filled) and
//               the E / 64 W_g boxes [64 k][64 experts] (8 KB each, N-major,
//               128-byte swizzle) into a ring of about 192 KB;
//   warp 1      TMEM owner; one lane issues M128 N=E K16 kind::f16 MMAs and
//               commits ring slots back to the producer;
//   warps 4-7   read the accumulator (one TMEM lane quadrant each, a token per
//               lane) into fp32 logits in shared memory, over the drained ring;
//   warps 8-12 dry passes of the tail and of the scan (instruction warm-up);
// then all 16 warps run the gating / top-k tail and the per-CTA partials.
// Against the mma.sync router (64 tokens per CTA, W_g tiles beside every x
// tile in the ring), a CTA here reads each W_g tile once per 128 tokens and
// keeps 16 KB of x per stage in flight, and the MMA work is a handful of
// instructions per k-block.
namespace rtc {
constexpr int BM = kRouterBMTc;
constexpr int XS = BM * kBK * 2;           // 16 KB x tile per k-block
constexpr int WBOX = kBK * 64 * 2;         // 8 KB per 64-expert W_g box
constexpr int THREADS = 512;               // 16 warps: the tail runs 4 threads per token
constexpr int RING = 192 * 1024;
constexpr int EPI_WARP0 = 4;               // warps 4..7: TMEM lane quadrants 0..3
constexpr int WARM_TAIL_WARP = 8;          // idle until the tail: its dry pass
constexpr int WARM_SCAN_WARP0 = 9;         // warps 9..12: the scan's dry pass, a role each
constexpr uint32_t kWhere = kWhereRouter + 0x10;

template <int NB>   // E = 64 NB
struct Shape {
  static constexpr int E = 64 * NB;
  static constexpr int STAGE = XS + NB * WBOX;
  static constexpr int STAGES = RING / STAGE;          // 8, 6, 4, 4
  static constexpr int TCOLS = NB == 1 ? 64 : NB == 2 ? 128 : 256;   // TMEM columns (a power of 2)
  // Logit rows E + 4 floats apart: E + 4 is 4 mod 32 words, so the tail's
  // reads (8 tokens x 4 threads of a warp, experts q + 4 i) fall in 32
  // different banks, and a row starts on a 16-byte boundary for the vector
  // stores out of TMEM.
  static constexpr int LDL = E + 4;
  static constexpr size_t LOGITS = (size_t)BM * LDL * 4;
  static constexpr size_t BITS_OFF = (size_t)STAGES * STAGE;
  static constexpr size_t BITS = (size_t)E * (BM / 32) * 4;
  // Scratch of the warm-up warps (dry tail rows and masks, dry scan totals).
  static constexpr size_t DRY_OFF = (BITS_OFF + BITS + 15) / 16 * 16;
  static constexpr size_t DRY_SL = (size_t)kDryTokens * LDL * 4;
  static constexpr size_t DRY_BITS = BITS;
  static constexpr size_t DRY_SCAN = 2 * scan_detail::kMaxE * 4;
  static constexpr size_t BAR_OFF = (DRY_OFF + DRY_SL + DRY_BITS + DRY_SCAN + 7) / 8 * 8;
  static constexpr size_t SMEM = 1024 + BAR_OFF + (2 * STAGES + 2) * 8 + 16;
  static_assert(LOGITS <= BITS_OFF, "the logits fit in the drained ring");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};
}  // namespace rtc

template <int NB>
__global__ void __launch_bounds__(rtc::THREADS, 1) router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                    const __grid_constant__ CUtensorMap tmW,
                                                                    RouterArgs a) {
  using L = rtc::Shape<NB>;
  constexpr int E = L::E, STAGES = L::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t base = smem_u32(smem);
  uint32_t* bits = (uint32_t*)(smem + L::BITS_OFF);
  uint64_t* full = (uint64_t*)(smem + L::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* done = tfull + 1;
  uint32_t* tmem_slot = (uint32_t*)(done + 1);
  uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* abort = abort_flag;

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int64_t blk = blockIdx.x;
  const int t0 = (int)(blk * rtc::BM);
  const int nk = a.d / kBK;
  const uint64_t limit = (uint64_t)a.timeout_ns;
  const uint64_t drain_limit = limit > 2000000000ull ? limit : 2000000000ull;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1u);
      mbar_init(smem_u32(&empty[s]), 1u);
    }
    mbar_init(smem_u32(tfull), 1u);
    mbar_init(smem_u32(done), 1u);
    *abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(L::TCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool stopped = false;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
      const uint64_t x_policy = l2_policy_evict_first();   // x is streamed once
      int kb = 0;
      for (; kb < nk; ++kb) {
        const int st = kb % STAGES;
        if (kb >= STAGES &&
            !mbar_wait_i(smem_u32(&empty[st]), (uint32_t)((kb / STAGES) - 1) & 1u, abort, limit, a.err,
                         rtc::kWhere + 1)) {
          stopped = true;
          break;
        }
        const uint32_t fb = smem_u32(&full[st]);
        const uint32_t sa = base + (uint32_t)(st * L::STAGE);
        mbar_expect_tx(fb, (uint32_t)L::STAGE);
        tma_load_2d_hint(sa, &tmX, kb * kBK, t0, fb, x_policy);
#pragma unroll
        for (int b = 0; b < NB; ++b) tma_load_2d(sa + rtc::XS + b * rtc::WBOX, &tmW, 64 * b, kb * kBK, fb);
      }
      // Every copy this thread started lands before the CTA goes on: the last
      // STAGES k-blocks issued, one per slot, may still be in flight.
      for (int j = kb - STAGES > 0 ? kb - STAGES : 0; j < kb; ++j)
        mbar_drain(smem_u32(&full[j % STAGES]), (uint32_t)(j / STAGES) & 1u, drain_limit);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int kb = 0;
      for (; kb < nk; ++kb) {
        const int st = kb % STAGES;
        if (!mbar_wait_i(smem_u32(&full[st]), (uint32_t)(kb / STAGES) & 1u, abort, limit, a.err, rtc::kWhere + 2)) {
          stopped = true;
          break;
        }
        tc_fence_after();
        const uint32_t sa = base + (uint32_t)(st * L::STAGE);
        const uint32_t sb = sa + rtc::XS;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // A (x): K-major, 8-row groups 1024 B apart; a K step of 16 is 32 bytes.
          const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
          // B (W_g): N-major, 64-expert boxes 8 KB apart (LBO), 8-row k groups
          // 1024 B apart (SBO); a K step of 16 rows is 2048 bytes.
          const uint64_t bd = smem_desc(sb + kk * 2048, rtc::WBOX, 1024);
          mma_bf16_cta1<idesc_bf16(rtc::BM, E)>(tmem, ad, bd, (kb | kk) != 0 ? 1u : 0u);
        }
        mma_commit_cta1(smem_u32(&empty[st]));
      }
      if (!stopped) mma_commit_cta1(smem_u32(tfull));
      // Every MMA issued completes before TMEM or the ring is touched again.
      mma_commit_cta1(smem_u32(done));
      mbar_drain(smem_u32(done), 0u, drain_limit);
    }
  } else if (warp >= rtc::EPI_WARP0 && warp < rtc::EPI_WARP0 + 4) {
    // ---------------- accumulator -> shared-memory logits ----------------
    const bool ok = __all_sync(0xffffffffu, mbar_wait_i(smem_u32(tfull), 0u, abort, limit, a.err, rtc::kWhere + 3));
    if (!ok) {
      stopped = true;
    } else {
      tc_fence_after();
      const int q = warp & 3;                        // TMEM lanes 32 q .. 32 q + 31
      const int row = q * 32 + lane;                 // the CTA's token
      float* sl = (float*)smem;
#pragma unroll 1
      for (int c = 0; c < E / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(sl + row * L::LDL + c * 32 + i) =
              make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                          __uint_as_float(v[i + 3]));
      }
    }
    tc_fence_before();
  }
  // The tail in two passes through one copy of its code: pass 0 (dry) on the
  // warm-up warps while the stream runs (warp 8 the tail, warps 9-12 the scan's
  // four roles side by side), pass 1 on every warp (the tail needs all 512
  // threads, four per token).
  uint8_t* dry_area = smem + L::DRY_OFF;
  const bool warm_scan = warp >= rtc::WARM_SCAN_WARP0 && warp < rtc::WARM_SCAN_WARP0 + 4;
#pragma unroll 1
  for (int pass = (warp == rtc::WARM_TAIL_WARP || warm_scan) ? 0 : 1; pass < 2; ++pass) {
    const bool dry = pass == 0;
    bool stop = false;
    if (!dry) {
      // The ring is drained (every MMA done, every copy landed) and the logits are
      // in shared memory before the tail reads them; TMEM can go.
      stop = __syncthreads_or(stopped || *abort != 0u);
      if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(L::TCOLS) : "memory");
      }
    }
    if (!stop && (!dry || warp == rtc::WARM_TAIL_WARP))
      router_finalize<rtc::BM, E / kTPT>(dry ? (float*)dry_area : (float*)smem, L::LDL,
                                         dry ? (uint32_t*)(dry_area + L::DRY_SL) : bits, a, blk, dry ? lane : tid,
                                         dry ? 32 : rtc::THREADS, dry);
    if (!dry || warm_scan)
      router_retire<4, 4>(a, dry ? dry_area + L::DRY_SL + L::DRY_BITS : smem, dry,
                          dry ? warp - rtc::WARM_SCAN_WARP0 : warp, dry ? 4 : rtc::THREADS / 32);
  }
}

template <int NB>
cudaError_t launch_tc(const RouterArgs& a, int64_t nblk, cudaStream_t s) {
  using L = rtc::Shape<NB>;
  CUtensorMap tmX, tmW;
  if (!tmap_bf16_2d(&tmX, a.x, a.T, a.d, kBK, rtc::BM)) return cudaErrorInvalidValue;
  if (!tmap_bf16_2d(&tmW, a.Wg, a.d, a.E, 64, kBK)) return cudaErrorInvalidValue;
  auto kern = router_tc_kernel<NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)nblk, rtc::THREADS, L::SMEM, s>>>(tmX, tmW, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
  if (a.bm != router_tile_tokens(a.dtype, a.E)) return cudaErrorInvalidValue;
  const int64_t nblk = (a.T + a.bm - 1) / a.bm;
  if (nblk == 0) return cudaSuccess;
  if (a.bm == kRouterBMTc) {
    switch (a.E / 64) {
      case 1: return launch_tc<1>(a, nblk, s);
      case 2: return launch_tc<2>(a, nblk, s);
      case 3: return launch_tc<3>(a, nblk, s);
      case 4: return launch_tc<4>(a, nblk, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (a.dtype == MOE_DT_F32) {
    size_t bytes = (size_t)kRouterBM * (a.E + 1) * 4 + (size_t)kRouterBM * (kBK32 + 1) * 4 +
                   (size_t)kBK32 * a.E * 4 + (size_t)a.E * (kRouterBM / 32) * 4;
    auto kern = a.E <= 8 ? router_f32_kernel<2> : a.E <= 32 ? router_f32_kernel<8> : router_f32_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)nblk, kThreadsF32, bytes, s>>>(a);
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
