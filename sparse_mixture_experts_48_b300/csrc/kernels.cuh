// Host-side launchers of the MoE-FFN kernels (one per pipeline stage).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

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
  int64_t nblk;        // router CTAs (kRouterBM tokens each)
  int32_t* hist;       // [E, nblk] selections per router CTA (expert-major: the scan reads rows)
  float* psum;         // [E, nblk] sum of gate probabilities per router CTA
  uint32_t* err;       // workspace status word
  int64_t timeout_ns;  // limit of every device-side wait
  float* scores_em;    // expert choice: gate probabilities [E, T] (no top-k), else null
};
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);

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
};
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s);

struct GatherArgs {
  const void* x;
  int64_t T;
  int d, E, k, dtype;
  int64_t capacity;
  const int32_t* topk_idx;
  const uint8_t* lrank;
  const int32_t* base;  // [E, nblk]
  int64_t nblk;
  const int32_t* offsets;
  int32_t* slot;        // [T, k]
  uint8_t* dropped;     // [T, k]
  int32_t* perm_token;  // [T*k] or null
  void* xperm;          // [T*k, d]
  const uint32_t* err;  // non-zero: skip (the ranks are not valid)
};
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t s);

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
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);

// Expert-choice routing (ec_routing.cu).
struct EcSelectArgs {
  const float* scores_em;  // [E, T] gate probabilities
  int64_t T, C;
  int E, EW;               // EW = ceil(E / 32) words of the per-token expert mask
  int32_t* perm;           // [E * C] chosen tokens, grouped by expert, tokens ascending
  float* w_row;            // [E * C] gate weight of each grouped row
  int32_t* tok_row;        // [T, E] grouped row of (token, expert) where chosen
  uint32_t* bits;          // [T, EW] choosing experts of each token (zeroed by the caller)
  const uint32_t* err;
};
cudaError_t launch_ec_select(const EcSelectArgs& a, cudaStream_t s);

struct EcGatherArgs {
  const void* x;
  const int32_t* perm;
  int64_t rows;
  int d, esz;
  void* xperm;
  const uint32_t* err;
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
};
cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_grouped_gemm_pair(const GemmArgs& a, cudaStream_t s);

// Builds a segment table from row offsets (standalone grouped GEMM entry point).
cudaError_t launch_segments_from_offsets(const int32_t* offsets, int G, int64_t M, SegTable seg, uint32_t* err,
                                         cudaStream_t s);

int sm_count();

}  // namespace moe
