// The dispatch scan (step a4 and the statistics of step a9), as a device
// function run by one whole CTA: by the scan kernel, or by the last router CTA
// to finish (the router then needs no second launch).
//
// Per expert, an exclusive prefix over the router CTAs of their selection
// counts (every assignment's rank among earlier tokens choosing the same
// expert), the pre-capacity counts n_e, kept counts min(n_e, C), segment
// offsets, f, P, L_aux, the routing-health statistics and the segment / tile
// table of the grouped GEMMs.  Fixed reduction orders throughout.
//
// Sources: "MoE架构解析" §三 关键技术① (capacity = tokens / experts x capacity
// factor; overflow skips the layer); "手撕一个极简 MoE-FFN" §七 (f = counts /
// (T k), P = mean score, L = alpha N sum f P); "MoE混合专家模型：Transformer稀疏
// 前馈网络原理与PyTorch实现" §2.3 (Switch load-balance loss), §3.3 (routing health).
#pragma once
#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace scan_detail {

constexpr int kMaxE = 256;

// Exclusive prefix over 32 lanes of per-lane partial sums (lane order).
__device__ __forceinline__ int warp_excl_scan(int v, int lane, int* total) {
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  *total = __shfl_sync(0xffffffffu, incl, 31);
  return incl - v;
}

// Run by every thread of the CTA (warp = threadIdx.x / 32, nwarps = blockDim.x
// / 32, at least four warps; one barrier inside); s_npre and s_psum are
// shared arrays of kMaxE entries.  The router CTAs' partials are read with
// L1-bypassing loads: in the fused form they were written by other SMs during
// this same launch.
// kScanE experts per warp per round, kScanU 32-block chunks of each loaded per
// round: the standalone scan kernel takes <4, 8>, the last CTA of the
// mma.sync and fp32 routers a lighter <2, 4> (or <1, 8>) so that their kernels
// keep the registers of their own main loops, and that of the 512-thread
// tcgen05 router <4, 4> (64 experts over its 16 warps in one round).
// dry: the same code over one round of phase 1 and the roles of phase 2,
// writing only s_npre / s_psum (no barrier: one warp alone takes all four
// roles, or four warps one each): it brings the code into the instruction
// cache before the real pass, which runs once per launch and is otherwise
// bound by fetching its code (the caller runs both passes through one call
// site).
template <int kScanE, int kScanU>
__device__ __forceinline__ void scan_body(const ScanArgs& a, int* s_npre, float* s_psum, int warp, int nwarps,
                                       bool dry) {
  const int lane = threadIdx.x % 32;
  const int E = dry ? (a.E < 1 ? a.E : 1) : a.E;
  const int64_t nblk = dry ? (a.nblk < 32 * kScanU ? a.nblk : 32 * kScanU) : a.nblk;
  // An earlier stage gave up: its partials are not valid.  Publish empty
  // segments so that nothing later reads or writes through them.
  const bool failed = *(volatile const uint32_t*)a.err != 0u;

  // Phase 1, one warp per expert: exclusive prefix over the router CTAs of
  // their selection counts (the rank base of each CTA's tokens), the expert's
  // total selections n_e, and the sum of its gate probabilities (per lane in
  // block order, then a fixed xor tree).  A warp takes kScanE experts at a
  // time (e, e + nwarps, ...) and issues all their loads of a round (kScanU
  // 32-block chunks each) before any scan, so a round costs one load latency.
  const bool ec = a.ec_C >= 0;   // expert choice: n_e = C for every expert, no ranks
  for (int eb = warp; eb < E; eb += nwarps * kScanE) {
    int run[kScanE];
    float ps[kScanE];
#pragma unroll
    for (int j = 0; j < kScanE; ++j) { run[j] = 0; ps[j] = 0.f; }
    for (int64_t b0 = 0; b0 < nblk; b0 += 32 * kScanU) {
      int v[kScanE][kScanU];
      float p[kScanE][kScanU];
#pragma unroll
      for (int j = 0; j < kScanE; ++j) {
        const int e = eb + j * nwarps;
#pragma unroll
        for (int u = 0; u < kScanU; ++u) {
          const int64_t b = b0 + 32 * u + lane;
          const bool in = e < E && b < nblk;
          v[j][u] = (in && !ec) ? __ldcg(a.hist + e * a.nblk + b) : 0;
          p[j][u] = in ? __ldcg(a.psum + e * a.nblk + b) : 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < kScanE; ++j) {
        const int e = eb + j * nwarps;
#pragma unroll
        for (int u = 0; u < kScanU; ++u) {
          const int64_t b = b0 + 32 * u + lane;
          int tot;
          const int ex = warp_excl_scan(v[j][u], lane, &tot);
          if (e < E && b < nblk && !ec && !dry) a.base[e * a.nblk + b] = run[j] + ex;
          run[j] += tot;
          ps[j] += p[j][u];
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kScanE; ++j) {
      const int e = eb + j * nwarps;
      if (ec) run[j] = (int)a.ec_C;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps[j] += __shfl_xor_sync(0xffffffffu, ps[j], off);
      if (lane == 0 && e < E) {
        s_npre[e] = failed ? 0 : run[j];
        s_psum[e] = ps[j];
      }
    }
  }
  if (dry) __syncwarp(); else __syncthreads();

  // Phase 2: four warps at once, each from the shared totals, so the single-
  // warp chains run side by side: warp 0 counts and offsets (what the gather
  // needs), warp 1 f, P and L_aux, warp 2 the routing-health statistics, warp
  // 3 the segment / tile table.  Lane l owns experts [l PE, (l + 1) PE).
  // Every sum is a fixed tree, in fp32 (B300's fp64 rate is low); the
  // differences that could cancel are formed exactly in integers first.
  const int PE = (E + 31) / 32;
  const int e0 = lane * PE;
  // Rows a routed segment occupies: its kept count, padded to a.pad_rows.
  const int pad = a.pad_rows > 1 ? a.pad_rows : 1;
  auto kept = [&](int n) { return (a.capacity < 0 || n <= a.capacity) ? n : (int)a.capacity; };
  auto seg_rows = [&](int n) { return (kept(n) + pad - 1) / pad * pad; };
  // Selections in all: T k for token choice, E C for expert choice.
  const int64_t Tk = ec ? (int64_t)E * a.ec_C : a.T * (int64_t)a.k;

  // Warp w < 4 takes role w; a dry pass on one warp takes all four.
  const bool all_roles = dry && nwarps == 1;
  const int role_end = all_roles ? 4 : (warp < 4 ? warp + 1 : 0);
#pragma unroll 1
  for (int role = all_roles ? 0 : warp; role < role_end; ++role) {
  if (role == 0) {
    int cnt_local = 0;
    for (int i = 0; i < PE; ++i) {
      const int e = e0 + i;
      if (e < E) cnt_local += seg_rows(s_npre[e]);
    }
    int kept_total;
    int off = warp_excl_scan(cnt_local, lane, &kept_total);
    for (int i = 0; i < PE; ++i) {
      const int e = e0 + i;
      if (e < E) {
        const int n = s_npre[e];
        if (!dry) {
          a.n_pre[e] = n;
          a.counts[e] = kept(n);
          a.offsets[e] = off;
        }
        off += seg_rows(n);
      }
    }
    if (lane == 0 && !dry) a.offsets[E] = kept_total;
  } else if (role == 1) {
    // f = n / (T k) and P = (sum of p) / T, each one correctly rounded fp32
    // division; L_aux = alpha E sum f P (positive terms, fixed tree).
    float L = 0.f;
    for (int i = 0; i < PE; ++i) {
      const int e = e0 + i;
      if (e < E) {
        const float fe = a.T > 0 ? __fdiv_rn((float)s_npre[e], (float)Tk) : 0.f;
        const float Pe = a.T > 0 ? __fdiv_rn(s_psum[e], (float)a.T) : 0.f;
        if (!dry) {
          a.f[e] = fe;
          a.P[e] = Pe;
        }
        L = __fmaf_rn(fe, Pe, L);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);   // fixed tree order
    if (lane == 0 && !dry) *a.L_aux = (float)a.alpha * (float)E * L;
  } else if (role == 2) {
    if (a.route_stats) {
      // Routing health of the pre-capacity shares f_e = n_e / (T k): entropy
      // -sum f ln f, variance (1/E) sum (f - 1/E)^2 with f - 1/E = (n E - T k) /
      // (T k E) (the numerator exact), CV = E sqrt(variance).
      float H = 0.f, V = 0.f;
      for (int i = 0; i < PE; ++i) {
        const int e = e0 + i;
        if (e < E && a.T > 0) {
          const int n = s_npre[e];
          const float fe = __fdiv_rn((float)n, (float)Tk);
          if (n > 0) H -= fe * logf(fe);
          const float dv = __fdiv_rn((float)((int64_t)n * E - Tk), (float)Tk * (float)E);
          V = __fmaf_rn(dv, dv, V);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        H += __shfl_xor_sync(0xffffffffu, H, o);
        V += __shfl_xor_sync(0xffffffffu, V, o);
      }
      if (lane == 0 && !dry) {
        V = __fdiv_rn(V, (float)E);
        a.route_stats[0] = H;
        a.route_stats[1] = V;
        a.route_stats[2] = (float)E * sqrtf(V);
      }
    }
  } else if (role == 3) {
    // Segments of the grouped GEMMs: routed experts read the grouped copy of
    // x, shared experts read x itself and write rows T*k + s*T.
    const int G = E + a.S;
    const int PG = (G + 31) / 32;
    const int g0 = lane * PG;
    int mt_local = 0, row_local = 0;
    for (int i = 0; i < PG; ++i) {
      const int g = g0 + i;
      if (g < G) {
        int rows;
        if (g < E) {
          rows = seg_rows(s_npre[g]);
          row_local += rows;
        } else {
          rows = failed ? 0 : (int)(pad > 1 ? a.shared_stride : a.T);
        }
        mt_local += (rows + kGemmBM - 1) / kGemmBM;
      }
    }
    int mt_total, row_total;
    int mt = warp_excl_scan(mt_local, lane, &mt_total);
    int orow_r = warp_excl_scan(row_local, lane, &row_total);
    for (int i = 0; i < PG; ++i) {
      const int g = g0 + i;
      if (g < G) {
        int rows, orow, arow, asrc;
        if (g < E) {
          rows = seg_rows(s_npre[g]);
          orow = orow_r;
          orow_r += rows;
          arow = orow;
          asrc = 0;
        } else {
          rows = failed ? 0 : (int)(pad > 1 ? a.shared_stride : a.T);
          orow = (int)(a.rows_tk + (int64_t)(g - E) * a.shared_stride);
          arow = 0;
          asrc = 1;
        }
        if (!dry) {
          a.seg.rows[g] = rows;
          a.seg.w[g] = g;
          a.seg.out_row[g] = orow;
          a.seg.a_row[g] = arow;
          a.seg.a_src[g] = asrc;
          a.seg.mtile_start[g] = mt;
        }
        mt += (rows + kGemmBM - 1) / kGemmBM;
      }
    }
    if (lane == 0 && !dry) a.seg.mtile_start[G] = mt_total;
  }
  }   // roles
}

}  // namespace scan_detail
}  // namespace moe
