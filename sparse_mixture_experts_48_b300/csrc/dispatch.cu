// K2 -- dispatch: capacity slots in token order, drops, the expert-grouped
// order of the kept assignments, the balance statistics, and the gather of x
// rows into the expert-contiguous buffer the grouped GEMM reads.
//
// Two launches:
//   scan    one CTA: per expert, an exclusive prefix over the router CTAs of
//           their selection counts (so every assignment's rank among earlier
//           tokens choosing the same expert is known), the pre-capacity
//           counts n_e, kept counts min(n_e, C), segment offsets, f, P, L_aux
//           and the segment / tile table of the grouped GEMMs.
//   gather  one warp per token: rank = CTA prefix + local rank; kept iff
//           rank < C; slot = offset[e] + rank; then the token's row of x is
//           read once with 16-byte loads and written to each kept slot.
// All sums use a fixed order, so results are bitwise reproducible.
//
// Sources: "MoE架构解析" §三 关键技术① (capacity = tokens / experts x capacity
// factor; overflow skips the layer); "手撕一个极简 MoE-FFN" §六 (gather the
// tokens of one expert and run the expert once on the batch), §七 (f = counts /
// (T k), P = mean score, L = alpha N sum f P); "MoE混合专家模型：Transformer稀疏
// 前馈网络原理与PyTorch实现" §2.3 (Switch load-balance loss).
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kMaxE = 256;
constexpr int kScanU = 4;   // 32-block chunks loaded per round, per lane

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

__global__ void __launch_bounds__(kScanThreads) scan_kernel(ScanArgs a) {
  __shared__ int s_npre[kMaxE];
  __shared__ float s_psum[kMaxE];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = blockDim.x / 32;
  const int E = a.E;
  // An earlier stage gave up: its partials are not valid.  Publish empty
  // segments so that nothing later reads or writes through them.
  const bool failed = *(volatile const uint32_t*)a.err != 0u;

  // Phase 1, one warp per expert: exclusive prefix over the router CTAs of
  // their selection counts (the rank base of each CTA's tokens), the expert's
  // total selections n_e, and the sum of its gate probabilities.  Loads of
  // kScanU chunks are issued before their scans.
  const bool ec = a.ec_C >= 0;   // expert choice: n_e = C for every expert, no ranks
  for (int e = warp; e < E; e += nwarps) {
    int run = 0;
    float ps = 0.f;
    for (int64_t b0 = 0; b0 < a.nblk; b0 += 32 * kScanU) {
      int v[kScanU];
      float p[kScanU];
#pragma unroll
      for (int u = 0; u < kScanU; ++u) {
        const int64_t b = b0 + 32 * u + lane;
        v[u] = (b < a.nblk && !ec) ? a.hist[e * a.nblk + b] : 0;
        p[u] = b < a.nblk ? a.psum[e * a.nblk + b] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kScanU; ++u) {
        const int64_t b = b0 + 32 * u + lane;
        int tot;
        const int ex = warp_excl_scan(v[u], lane, &tot);
        if (b < a.nblk && !ec) a.base[e * a.nblk + b] = run + ex;
        run += tot;
        ps += p[u];
      }
    }
    if (ec) run = (int)a.ec_C;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    if (lane == 0) {
      s_npre[e] = failed ? 0 : run;
      s_psum[e] = ps;
    }
  }
  __syncthreads();
  if (warp != 0) return;

  // Phase 2, one warp: lane l owns experts [l * PE, (l + 1) * PE).
  const int PE = (E + 31) / 32;
  const int e0 = lane * PE;
  // Rows a routed segment occupies: its kept count, padded to a.pad_rows.
  const int pad = a.pad_rows > 1 ? a.pad_rows : 1;
  auto seg_rows = [&](int n) {
    const int c = (a.capacity < 0 || n <= a.capacity) ? n : (int)a.capacity;
    return (c + pad - 1) / pad * pad;
  };
  int cnt_local = 0;
  for (int i = 0; i < PE; ++i) {
    const int e = e0 + i;
    if (e < E) cnt_local += seg_rows(s_npre[e]);
  }
  int kept_total;
  int off = warp_excl_scan(cnt_local, lane, &kept_total);
  // f divides by all selections: T k for token choice, E C for expert choice.
  const double Tk = ec ? (double)E * (double)a.ec_C : (double)a.T * (double)a.k;
  double L = 0.0;
  for (int i = 0; i < PE; ++i) {
    const int e = e0 + i;
    if (e < E) {
      const int n = s_npre[e];
      const int c = (a.capacity < 0 || n <= a.capacity) ? n : (int)a.capacity;
      a.n_pre[e] = n;
      a.counts[e] = c;
      a.offsets[e] = off;
      off += seg_rows(n);
      const float fe = a.T > 0 ? __fdiv_rn((float)n, (float)Tk) : 0.f;
      const float Pe = a.T > 0 ? __fdiv_rn(s_psum[e], (float)a.T) : 0.f;
      a.f[e] = fe;
      a.P[e] = Pe;
      L += (double)fe * (double)Pe;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);   // fixed tree order
  if (lane == 0) {
    a.offsets[E] = kept_total;
    *a.L_aux = (float)(a.alpha * (double)E * L);
  }
  if (a.route_stats) {
    // Routing health of the pre-capacity shares f_e = n_e / (T k): entropy
    // -sum f ln f, variance (1/E) sum (f - 1/E)^2, CV = E sqrt(variance).
    double H = 0.0, V = 0.0;
    for (int i = 0; i < PE; ++i) {
      const int e = e0 + i;
      if (e < E && a.T > 0) {
        const double fe = (double)s_npre[e] / Tk;
        if (fe > 0.0) H -= fe * log(fe);
        V += (fe - 1.0 / E) * (fe - 1.0 / E);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      H += __shfl_xor_sync(0xffffffffu, H, o);
      V += __shfl_xor_sync(0xffffffffu, V, o);
    }
    if (lane == 0) {
      V /= (double)E;
      a.route_stats[0] = (float)H;
      a.route_stats[1] = (float)V;
      a.route_stats[2] = (float)((double)E * sqrt(V));
    }
  }
  // Segments of the grouped GEMMs: routed experts read the grouped copy of x,
  // shared experts read x itself and write rows T*k + s*T.  The offsets of
  // the routed segments are this warp's own (in registers / recomputed), so
  // nothing is read back from global memory.
  const int G = E + a.S;
  const int PG = (G + 31) / 32;
  const int g0 = lane * PG;
  int mt_local = 0;
  for (int i = 0; i < PG; ++i) {
    const int g = g0 + i;
    if (g < G) {
      int rows;
      if (g < E) {
        rows = seg_rows(s_npre[g]);
      } else {
        rows = failed ? 0 : (int)(pad > 1 ? a.shared_stride : a.T);
      }
      mt_local += (rows + kGemmBM - 1) / kGemmBM;
    }
  }
  int mt_total;
  int mt = warp_excl_scan(mt_local, lane, &mt_total);
  // Row offsets of routed segments: exclusive prefix of kept counts over g < E.
  int row_local = 0;
  for (int i = 0; i < PG; ++i) {
    const int g = g0 + i;
    if (g < E) row_local += seg_rows(s_npre[g]);
  }
  int row_total;
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
      a.seg.rows[g] = rows;
      a.seg.w[g] = g;
      a.seg.out_row[g] = orow;
      a.seg.a_row[g] = arow;
      a.seg.a_src[g] = asrc;
      a.seg.mtile_start[g] = mt;
      mt += (rows + kGemmBM - 1) / kGemmBM;
    }
  }
  if (lane == 0) a.seg.mtile_start[G] = mt_total;
}

constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32) gather_kernel(GatherArgs a) {
  const int lane = threadIdx.x % 32;
  const int64_t t = (int64_t)blockIdx.x * kGatherWarps + threadIdx.x / 32;
  if (t >= a.T || *(volatile const uint32_t*)a.err != 0u) return;
  const int k = a.k, E = a.E;
  int my_slot = -1;
  if (lane < k) {
    const int e = a.topk_idx[t * k + lane];
    const int64_t b = t / kRouterBM;
    const int r = a.base[e * a.nblk + b] + (int)a.lrank[t * k + lane];
    const bool kept = a.capacity < 0 || r < a.capacity;
    my_slot = kept ? a.offsets[e] + r : -1;
    a.slot[t * k + lane] = my_slot;
    a.dropped[t * k + lane] = kept ? 0 : 1;
    if (kept && a.perm_token) a.perm_token[my_slot] = (int32_t)t;
  }
  int slots[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) slots[j] = __shfl_sync(0xffffffffu, my_slot, j);
  if (a.fp8) {
    // FP8 experts: quantise the bf16 row on the way.  Pass 1 finds its largest
    // magnitude; pass 2 re-reads the row (now in L1 / L2) and writes 16 codes
    // per 16-byte store to every kept slot (and to the token-order copy that
    // the shared experts read).
    const int64_t words = a.d / 8;
    const uint4* src = (const uint4*)a.x + t * words;
    float m = 0.f;
    for (int64_t c = lane; c < words; c += 32) m = fmaxf(m, amax_bf16x8(src[c]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float r, sc;
    e4m3_scales(m, r, sc);
    const int64_t ow = a.d / 16;
    uint4* dst = (uint4*)a.xperm;
    for (int64_t c = lane; c < ow; c += 32) {
      const uint2 lo = e4m3x8_from_bf16(src[2 * c], r);
      const uint2 hi = e4m3x8_from_bf16(src[2 * c + 1], r);
      const uint4 q = make_uint4(lo.x, lo.y, hi.x, hi.y);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < k && slots[j] >= 0) dst[(int64_t)slots[j] * ow + c] = q;
      if (a.xq) reinterpret_cast<uint4*>(a.xq)[t * ow + c] = q;
    }
    if (lane < k && my_slot >= 0) a.xs_perm[my_slot] = sc;
    if (lane == 0 && a.xs_tok) a.xs_tok[t] = sc;
    return;
  }
  const int esz = a.dtype == MOE_DT_BF16 ? 2 : 4;
  const int64_t chunks = (int64_t)a.d * esz / 16;
  const uint64_t policy = l2_policy_evict_first();   // x read once, the grouped copy written once
  const uint4* src = (const uint4*)((const uint8_t*)a.x + t * chunks * 16);
  uint4* dst = (uint4*)a.xperm;
  constexpr int U = 4;
  for (int64_t c0 = lane; c0 < chunks; c0 += 32 * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + u * 32;
      if (c < chunks) v[u] = ld_stream_u4(src + c, policy);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k && slots[j] >= 0) {
        uint4* drow = dst + (int64_t)slots[j] * chunks;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t c = c0 + u * 32;
          if (c < chunks) st_stream_u4(drow + c, v[u], policy);
        }
      }
    }
  }
}

// Segment table of the standalone grouped GEMM from caller row offsets.  The
// offsets are checked on the device: if any segment is not inside [0, M] or
// they decrease, no segment gets rows (nothing is computed or written) and the
// error word records it.
__global__ void segments_kernel(const int32_t* off, int G, int64_t M, SegTable seg, uint32_t* err) {
  if (threadIdx.x != 0) return;
  bool bad = false;
  for (int g = 0; g < G; ++g) {
    const int64_t lo = off[g], hi = off[g + 1];
    if (lo < 0 || hi < lo || hi > M) bad = true;
  }
  int mt = 0;
  for (int g = 0; g < G; ++g) {
    const int rows = bad ? 0 : off[g + 1] - off[g];
    seg.rows[g] = rows;
    seg.w[g] = g;
    seg.out_row[g] = bad ? 0 : off[g];
    seg.a_row[g] = seg.out_row[g];
    seg.a_src[g] = 0;
    seg.mtile_start[g] = mt;
    mt += (rows + kGemmBM - 1) / kGemmBM;
  }
  seg.mtile_start[G] = mt;
  if (bad) record_error(err, kErrDevice, 0x200);
}

}  // namespace

cudaError_t launch_segments_from_offsets(const int32_t* offsets, int G, int64_t M, SegTable seg, uint32_t* err,
                                         cudaStream_t s) {
  segments_kernel<<<1, 32, 0, s>>>(offsets, G, M, seg, err);
  return cudaGetLastError();
}

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s) {
  scan_kernel<<<1, kScanThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const int64_t blocks = (a.T + kGatherWarps - 1) / kGatherWarps;
  gather_kernel<<<(unsigned)blocks, kGatherWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
