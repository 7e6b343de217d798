// Host-side launchers of the MoE-FFN kernels (one per pipeline stage).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "common.cuh"

namespace moe {

struct ScanArgs {
  int64_t T;
  int E, k, S;
  int64_t capacity;    // -1: unlimited
  double alpha;
  int64_t nblk;
  const int32_t* hist;
  const float* psum;
  int32_t* base;       // [E, nblk] rank of each router CTA's first selection of e
  int32_t* n_pre;      // [E]
  int32_t* counts;     // [E] kept
  int32_t* offsets;    // [E+1]
  float* f;
  float* P;
  float* L_aux;
  float* route_stats;  // [3] entropy, variance, CV of the selection shares, or null
  SegTable seg;
  int64_t rows_tk;     // T * k (E * C for expert choice): first H / O row of the shared experts
  const uint32_t* err; // workspace status word: non-zero = an earlier stage failed
  int64_t ec_C;        // expert choice: every expert has exactly this many selections; -1 otherwise
  int pad_rows;        // routed segments padded to multiples of this many rows (1: packed)
  int64_t shared_stride;  // rows between shared segments (T, or T padded)
};
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s);

struct RouterArgs {
  const void* x;    // [T, d]
  const void* Wg;   // [d, E]
  const void* bg;   // [E] or null
  const float* noise;  // [T, E] fp32 added to the logits before gating, or null
  int64_t T;
  int d, E, k, gating, dtype;
  float* logits_out;   // [T, E] or null
  int32_t* topk_idx;   // [T, k]
  float* topk_w;       // [T, k]
  uint8_t* lrank;      // [T, k] rank among the CTA's earlier tokens choosing the same expert
  int bm;              // tokens per router CTA: router_tile_tokens(dtype, E)
  int64_t nblk;        // router CTAs (bm tokens each)
  int32_t* hist;       // [E, nblk] selections per router CTA (expert-major: the scan reads rows)
  float* psum;         // [E, nblk] sum of gate probabilities per router CTA
  uint32_t* err;       // workspace status word
  int64_t timeout_ns;  // limit of every device-side wait
  float* scores_em;    // expert choice: gate probabilities [E, T] (no top-k), else null
  float* raw_logits;   // [T, E] the (noisy) logits before gating, or null (the backward's copy)
  // When fused_scan is set, the last router CTA to finish runs the dispatch
  // scan with `scan` (its hist / psum are this launch's partials); `done`
  // counts finished router CTAs and is zero when the launch starts.
  bool fused_scan;
  ScanArgs scan;
  uint32_t* done;
};
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);


struct GatherArgs {
  const void* x;
  int64_t T;
  int d, E, k, dtype;
  int64_t capacity;
  const int32_t* topk_idx;
  const uint8_t* lrank;
  const int32_t* base;  // [E, nblk]
  int bm;               // tokens per router CTA
  int64_t nblk;
  const int32_t* offsets;
  int32_t* slot;        // [T, k]
  uint8_t* dropped;     // [T, k]
  int32_t* perm_token;  // [T*k] or null
  void* xperm;          // [T*k, d]
  const uint32_t* err;  // non-zero: skip (the ranks are not valid)
  // FP8 experts: x (bf16) is quantised per token row on the way; xperm holds
  // E4M3 codes, xs_perm [T*k] each grouped row's decoding scale, and (shared
  // experts) xq [T, d] / xs_tok [T] the quantised rows in token order.
  bool fp8;
  float* xs_perm;
  uint8_t* xq;
  float* xs_tok;
  bool pdl;             // launch with programmatic serialization after the previous kernel
};
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s);

// Launch `kern` on `s`, with programmatic stream serialization when `pdl`: the
// kernel may then be scheduled while the stream's previous kernel finishes,
// and it calls pdl_wait() before reading that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Per-row E4M3 quantisation of bf16 rows (fp8.cu): row r of X -> codes Q[r]
// and decoding scale scale[r].  Rows [0, rows0) are live only below *live0
// (when live0 is set: the kept routed rows of H); rows [row1, row1 + rows1)
// follow (the shared experts' rows of H).
struct QuantRowsArgs {
  const void* X;        // [., cols] bf16
  uint8_t* Q;           // [., cols]
  float* scale;         // [.]
  int64_t cols;
  int64_t rows0;
  const int32_t* live0; // or null: all rows0 rows
  int64_t row1, rows1;
  const uint32_t* err;  // or null
};
cudaError_t launch_quantize_rows(const QuantRowsArgs& a, cudaStream_t s);

// Weight slabs W [G, K, N] bf16 -> Q [G, N, K] E4M3 with one scale per (g, n).
struct QuantWeightsArgs {
  const void* W;
  uint8_t* Q;
  float* scale;
  int64_t G, K, N;
};
cudaError_t launch_quantize_weights(const QuantWeightsArgs& a, cudaStream_t s);

struct CombineArgs {
  const float* o;       // [rows_all, d] expert outputs, fp32
  int64_t T;
  int d, k, S;
  bool y_f32;           // y is fp32 (else bf16)
  int64_t rows_tk;
  const int32_t* slot;
  const float* topk_w;
  void* y;              // [T, d]
  const uint32_t* err;  // non-zero: skip (an earlier stage failed)
  bool pdl;             // launch with programmatic serialization after the previous kernel
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);

// Expert-choice routing (ec_routing.cu).
struct EcSelectArgs {
  const float* scores_em;  // [E, T] gate probabilities
  int64_t T, C;
  int64_t Cs;              // rows reserved per expert in the grouped order (>= C; padding after C)
  int E, EW;               // EW = ceil(E / 32) words of the per-token expert mask
  int32_t* perm;           // [E * Cs] chosen tokens, grouped by expert, tokens ascending
  float* w_row;            // [E * Cs] gate weight of each grouped row
  int32_t* tok_row;        // [T, E] grouped row of (token, expert) where chosen
  uint32_t* bits;          // [T, EW] choosing experts of each token (zeroed by the caller)
  const uint32_t* err;
};
cudaError_t launch_ec_select(const EcSelectArgs& a, cudaStream_t s);

struct EcGatherArgs {
  const void* x;            // [T, d]: x, or with FP8 experts its E4M3 codes
  const int32_t* perm;
  int64_t rows;             // E * Cs; the rows c >= C of each expert's Cs are skipped
  int64_t C, Cs;
  int d, esz;
  void* xperm;
  const uint32_t* err;
  const float* xs_tok;      // FP8: each token row's decoding scale [T], or null
  float* xs_perm;           // FP8: copied to each grouped row [rows]
};
cudaError_t launch_ec_gather(const EcGatherArgs& a, cudaStream_t s);

struct EcCombineArgs {
  const float* o;          // expert outputs, fp32
  const uint32_t* bits;
  const int32_t* tok_row;
  const float* w_row;
  int64_t T;
  int E, EW, S, d;
  int64_t rows_routed;     // E * C: first row of the shared experts
  bool y_f32;
  void* y;
  const uint32_t* err;
};
cudaError_t launch_ec_combine(const EcCombineArgs& a, cudaStream_t s);

// Grouped GEMM over the segment table.
struct GemmArgs {
  int dtype;
  int act;              // MOE_ACT_*
  int G;
  int K, N;
  bool a_from_out_rows; // A row of segment g = seg.out_row[g] (else seg.a_row / seg.a_src)
  SegTable seg;
  const void* A0;       // [rows_A0, K]
  int64_t rows_A0;
  const void* A1;       // [rows_A1, K] (second A source) or null
  int64_t rows_A1;
  const void* B;        // [Gw, K, N]
  const void* B3;       // [Gw, K, N] or null (SwiGLU)
  int Gw;               // weight slabs
  const void* bias;     // [Gw, N] or null
  void* C;              // [rows, N]
  bool out_f32;         // C is fp32 (else the dtype of A and B)
  int64_t max_mtiles;   // upper bound of seg.mtile_start[G]
  uint32_t* err;
  int64_t timeout_ns;
  bool single_cta;      // bf16: the one-CTA 128 x 256 tile kernel instead of the CTA-pair kernel
  void* pre_a;          // if set (pair kernel, bf16 out): pre-activations a = A B + bias, [rows, N] bf16
  void* pre_u;          // SwiGLU with pre_a: u = A B3, [rows, N] bf16
  // FP8 experts (pair kernel): A0 / A1 hold E4M3 codes with one decoding scale
  // per row (a_scale0 / a_scale1, indexed like the A rows); B / B3 hold E4M3
  // codes stored [Gw, N, K] (K-major) with one scale per (slab, column)
  // (b_scale / b3_scale, [Gw, N]).  The epilogue multiplies the accumulator by
  // both scales before the bias and the activation.
  int64_t rows_C;       // rows of C; > 0 with out_f32 lets the pair kernel store whole 32-row
                        // warp tiles by TMA (0: per-thread stores only)
  bool fp8;
  const float* a_scale0;
  const float* a_scale1;
  const float* b_scale;
  const float* b3_scale;
  bool pdl;             // launch with programmatic serialization after the previous kernel
};
cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_grouped_gemm_pair(const GemmArgs& a, cudaStream_t s);

// Expert GEMMs of the backward pass (grouped_gemm_bwd.cu).
struct BwdGemmArgs {
  int G, Gw;               // segments, weight slabs
  SegTable seg;            // rows (padded to 64-row multiples), w, out_row, a_src
  int M, N, K;             // dgrad: reduction K, output columns N; wgrad: slab M x N
  const void* A;           // dgrad: [rows_A, K] (dO, or dA); wgrad: X [rows_A, M]
  const void* A2;          // dgrad second phase (dU), or wgrad: x [rows_A2, M] for a_src 1
  int64_t rows_A, rows_A2;
  const void* B;           // dgrad: weight slabs [Gw, N, K]; wgrad: D [rows_B, N]
  int64_t rows_B;
  const void* B2;          // dgrad second phase (W3)
  void* C;                 // dgrad: fp32 [rows, N] or dA bf16; wgrad: fp32 [Gw, M, N]
  void* C2;                // dgrad SwiGLU: dU bf16
  const void* pre_a;       // dgrad with act_bwd: saved pre-activations [rows, N] bf16
  const void* pre_u;
  int act;
  bool act_bwd;            // dgrad epilogue: activation backward (dH -> dA, dU)
  bool x_from_asrc;        // wgrad: segments with a_src 1 read X rows from A2 starting at row 0
  int64_t max_tiles;       // upper bound of the pair tiles
  uint32_t* err;
  int64_t timeout_ns;
};
cudaError_t launch_gemm_dgrad(const BwdGemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_wgrad(const BwdGemmArgs& a, cudaStream_t s);

// Backward-pass kernels around the GEMMs (moe_backward.cu).
struct PadZeroArgs {
  void* buf;               // grouped buffer
  int64_t row_bytes;       // multiple of 16
  int G, E;
  int64_t T;
  const int32_t* counts;   // kept rows of the routed segments
  SegTable seg;            // rows = padded rows, out_row
};
cudaError_t launch_pad_zero(const PadZeroArgs& a, cudaStream_t s);

struct CombineBwdArgs {
  const void* dy;          // [T, d] bf16
  const float* o;          // expert outputs [rows, d] fp32
  const int32_t* slot;     // [T, k]
  const float* topk_w;
  int64_t T;
  int d, k, S;
  int64_t rows_routed, shared_stride;   // shared expert s, token t: row rows_routed + s * shared_stride + t
  void* dO;                // [rows, d] bf16
  float* dw;               // [T, k]
  const uint32_t* err;
};
cudaError_t launch_combine_bwd(const CombineBwdArgs& a, cudaStream_t s);

struct RouterBwdArgs {
  const float* logits;     // [T, E] (noisy) router logits
  const int32_t* topk_idx;
  const float* topk_w;
  const float* dw;
  const int32_t* n_pre;    // [E] selections before the capacity cut
  int64_t T;
  int E, k, gating;
  double alpha;
  float dL_aux;
  float* dl;               // [T, E]
  const uint32_t* err;
};
cudaError_t launch_router_bwd(const RouterBwdArgs& a, cudaStream_t s);

struct DxArgs {
  const float* dxp;        // [rows, d] gradients of the grouped rows
  const int32_t* slot;
  const float* dl;
  const void* Wg;          // [d, E] bf16
  int64_t T;
  int d, k, E, S;
  int64_t rows_routed, shared_stride;
  float* dx;               // [T, d]
  const uint32_t* err;
  // expert choice (k = 0, slot unused): the chosen rows of token t are
  // tok_row[t, e] for the experts e set in bits[t]; else null
  const uint32_t* ec_bits;
  const int32_t* ec_tok_row;
  int EW;
};
cudaError_t launch_dx(const DxArgs& a, cudaStream_t s);

// Expert-choice backward: grouped rows e * Cs + c (c < C), tok_row / bits as
// written by ec_select.
struct EcCombineBwdArgs {
  const void* dy;          // [T, d] bf16
  const float* o;          // expert outputs [rows, d] fp32
  const int32_t* perm;     // [E * Cs]
  const float* w_row;      // [E * Cs]
  int64_t rows, C, Cs;     // rows = E * Cs
  int d;
  void* dO;                // [rows, d] bf16
  float* dw_row;           // [E * Cs] <dy_t, o_row>
  const uint32_t* err;
};
cudaError_t launch_ec_combine_bwd(const EcCombineBwdArgs& a, cudaStream_t s);

struct EcRouterBwdArgs {
  const float* logits;     // [T, E] (noisy) router logits
  const uint32_t* bits;    // [T, EW] choosing experts of each token
  const int32_t* tok_row;  // [T, E]
  const float* dw_row;     // [E * Cs]
  int64_t T;
  int E, EW, gating;
  double alpha;
  float dL_aux;
  float* dl;               // [T, E]
  const uint32_t* err;
};
cudaError_t launch_ec_router_bwd(const EcRouterBwdArgs& a, cudaStream_t s);

struct DwgArgs {
  const void* x;           // [T, d] bf16
  const float* dl;         // [T, E]
  int64_t T;
  int d, E;
  int64_t nchunk;
  float* part;             // [nchunk, d, E]
  float* bpart;            // [nchunk, E]
  float* dWg;              // [d, E]
  float* dbg;              // [E] or null
};
int64_t dwg_chunks(int64_t T);
cudaError_t launch_dwg(const DwgArgs& a, cudaStream_t s);

struct ColsumArgs {
  const void* buf;         // grouped [rows, N] bf16
  SegTable seg;
  int G;
  int64_t N;
  float* out;              // [Gw, N]
};
cudaError_t launch_colsum(const ColsumArgs& a, cudaStream_t s);

// The standalone grouped GEMM (moe_grouped_gemm and its variant without a
// workspace): argument checks, and the launches on a scratch area of
// moe_grouped_gemm_workspace_size(G) bytes (status word, then the tile table).
moe_status check_grouped_gemm_args(int32_t dtype, int32_t act, int32_t G, const int32_t* seg_offsets, int64_t M,
                                   int32_t K, int32_t N, const void* A, const void* B, const void* B3,
                                   const void* bias, const void* C);
moe_status launch_grouped_gemm_on_scratch(int32_t dtype, int32_t act, int32_t G, const int32_t* seg_offsets,
                                          int64_t M, int32_t K, int32_t N, const void* A, const void* B,
                                          const void* B3, const void* bias, void* C, uint8_t* scratch,
                                          moe_stream stream, const moe_launch_opts* opts);

// Builds a segment table from row offsets (standalone grouped GEMM entry point).
cudaError_t launch_segments_from_offsets(const int32_t* offsets, int G, int64_t M, SegTable seg, uint32_t* err,
                                         cudaStream_t s);

int sm_count();

}  // namespace moe
