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
#include "scan.cuh"

namespace moe {
namespace {

constexpr int kScanThreads = 256;

__global__ void __launch_bounds__(kScanThreads) scan_kernel(ScanArgs a) {
  __shared__ int s_npre[scan_detail::kMaxE];
  __shared__ float s_psum[scan_detail::kMaxE];
  scan_detail::scan_body<4, 8>(a, s_npre, s_psum, threadIdx.x / 32, blockDim.x / 32, false);
}

constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32) gather_kernel(GatherArgs a) {
  pdl_wait();
  const int lane = threadIdx.x % 32;
  const int64_t t = (int64_t)blockIdx.x * kGatherWarps + threadIdx.x / 32;
  if (t >= a.T || *(volatile const uint32_t*)a.err != 0u) return;
  const int k = a.k, E = a.E;
  int my_slot = -1;
  if (lane < k) {
    const int e = a.topk_idx[t * k + lane];
    const int64_t b = t / a.bm;
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
  return launch_maybe_pdl(a.pdl, gather_kernel, dim3((unsigned)blocks), dim3(kGatherWarps * 32), 0, s, a);
}

}  // namespace moe
