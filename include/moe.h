/*
 * moe.h -- C ABI of libmoe.so: a Mixture-of-Experts feed-forward layer on one
 * NVIDIA B300 (sm_103a).  The forward pass (token-choice routing below, or
 * expert choice: MOE_FLAG_EXPERT_CHOICE), with bf16 / fp32 experts or E4M3
 * experts (moe_forward_fp8), and its backward pass (moe_backward).
 *
 * The token-choice layer, per token t of x [T, d]:
 *   1. router logits    l[t,e] = b_g[e] + sum_i x[t,i] W_g[i,e]
 *        ("MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现" §2.1;
 *         "Mixture of Experts混合专家模型架构原理与路由策略实现", 门控网络的数学原理:
 *         W_g has shape [d_model, num_experts])
 *   2. gating           softmax over the E experts ("手撕一个极简 MoE-FFN" §三), or
 *                       normalised sigmoid: sigmoid per expert, then normalised
 *                       ("MoE架构解析" §四 技术飞跃③)
 *   3. top-k            the k largest logits (descending; equal logits: lower
 *                       expert index first), weights renormalised to sum 1
 *                       ("手撕一个极简 MoE-FFN" §三, worked example: scores
 *                       [0.1,0.5,0.3,0.1], k=2 -> experts [1,2], weights
 *                       [0.625,0.375]); sigmoid gating divides the selected
 *                       sigmoids by their sum
 *   4. capacity         C = ceil(T * capacity_factor / E); each expert keeps its
 *                       first C assignments in token order (token t before t+1,
 *                       a token's choices in rank order), the rest are dropped:
 *                       they add nothing to y (they reach the next layer through
 *                       the residual, which is outside this layer)
 *                       ("MoE架构解析" §三 关键技术①)
 *   5. experts          ReLU/GELU: o = act(x W1[e] + b1[e]) W2[e] + b2[e]
 *                       ("手撕一个极简 MoE-FFN" §四; GELU is the exact erf form);
 *                       SwiGLU: o = (silu(x W1[e]) * (x W3[e])) W2[e]
 *                       ("术业有专攻：learn-minimind MoE混合专家模型架构入门指南" §二)
 *   6. combine          y[t] = sum_{j<k, kept} w_j o_{idx_j}(t) + sum_{s<S} o_{E+s}(t),
 *                       accumulated in fp32 in exactly that order; shared experts
 *                       are always active with weight 1 ("MoE架构解析" §四 技术飞跃②)
 *   7. balance stats    f_i = (selections of i before the capacity cut) / (T k),
 *                       P_i = mean_t p[t,i], L_aux = alpha * E * sum_i f_i P_i
 *                       ("手撕一个极简 MoE-FFN" §七; "MoE混合专家模型..." §2.3)
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers (cudaMalloc'd or torch-owned),
 *    owned by the caller.  The library never allocates, frees or keeps them.
 *  - Layouts are dense row-major; weights are stored [in, out]:
 *      x [T, d]; W_g [d, E]; b_g [E]; W1, W3 [E+S, d, f]; W2 [E+S, f, d];
 *      b1 [E+S, f]; b2 [E+S, d]; y [T, d].  Experts 0..E-1 are routed,
 *      E..E+S-1 are the shared experts.
 *    x, W_g, b_g, W*, b*, y have the config's dtype (fp32, or bf16 bits);
 *    topk_w, f, P, L_aux, router_logits are always fp32.
 *  - Work is enqueued on `stream` and returns without synchronising.  Host
 *    checks happen before anything is enqueued; on a non-OK status nothing was
 *    launched.  Device-side failures (a bounded wait that ran out) are
 *    recorded in the workspace and reported by moe_check_device_errors().
 *  - Calls are deterministic: the same inputs give bitwise the same outputs.
 *  - Calls sharing one workspace must be ordered on the GPU (same stream, or
 *    synchronised); concurrent calls need separate workspaces.
 */
#ifndef MOE_B300_MOE_H
#define MOE_B300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream; /* a cudaStream_t; NULL = the legacy default stream */
typedef struct CUevent_st* moe_event;   /* a cudaEvent_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* NULL where a tensor is required, bad sizes, aliasing, misalignment */
  MOE_ERR_UNSUPPORTED = 2, /* a valid layer this library does not run (e.g. k > 8, d % 64 for bf16) */
  MOE_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch error, sticky error) */
  MOE_ERR_TIMEOUT = 5,     /* a device-side wait exceeded its limit; outputs are not valid */
  MOE_ERR_DEVICE = 6       /* a device-side consistency check failed; outputs are not valid */
} moe_status;

enum { MOE_GATE_SOFTMAX = 0, MOE_GATE_SIGMOID_NORM = 1 };
enum { MOE_ACT_RELU = 0, MOE_ACT_GELU = 1, MOE_ACT_SWIGLU = 2, MOE_ACT_NONE = 3 };
enum { MOE_DT_F32 = 0, MOE_DT_BF16 = 1 };

/* Stages of moe_forward that stage events bracket: router, select, gather,
 * expert GEMM 1, expert GEMM 2, combine.  The router stage includes the
 * dispatch scan (ranks, capacity, offsets, statistics), which its last CTA
 * runs; the select stage holds the per-expert selection with expert choice
 * and is empty otherwise; with FP8 experts the gather stage also holds the
 * per-token quantisation of x. */
#define MOE_NUM_STAGES 6

/* The layer.  64 bytes, natural alignment. */
typedef struct {
  int64_t T;              /* tokens, >= 0 */
  int32_t d_model;        /* d */
  int32_t d_ff;           /* f, hidden width of every expert */
  int32_t E;              /* routed experts, 1..256 */
  int32_t k;              /* experts per token, 1..min(E, 8) */
  int32_t n_shared;       /* always-on shared experts S, 0..8 */
  int32_t act;            /* MOE_ACT_RELU / _GELU / _SWIGLU */
  int32_t gating;         /* MOE_GATE_SOFTMAX / _SIGMOID_NORM */
  int32_t dtype;          /* MOE_DT_F32 / _BF16: storage of x, weights, biases and y */
  double capacity_factor; /* <= 0: no capacity limit */
  double alpha;           /* coefficient of L_aux (the pages use 0.01) */
  int64_t flags;          /* OR of MOE_FLAG_*; other bits must be 0 */
} moe_config;

/* y is written in fp32 whatever `dtype` is (e.g. for an fp32 residual stream).
 * Without it y has the storage dtype and carries that dtype's final rounding. */
#define MOE_FLAG_Y_F32 1
/* Expert-choice routing ("MoE架构解析" §2.2): instead of each token choosing
 * its top-k experts, each expert chooses the C tokens with the largest gate
 * probability s[t,e] (softmax, or normalised sigmoid, over the experts; equal
 * probabilities: lower token index first), C = min(T, ceil(T cf / E)) with a
 * capacity factor cf > 0, else min(T, ceil(T k / E)).  Every expert gets the
 * same load; a token may be chosen by several experts or by none.
 *   y[t] = sum over the experts e that chose t, ascending, of s[t,e] o_e(t),
 *          plus the shared experts; a token no expert chose gets only those.
 * Outputs: expert_counts = C for every expert; f_e = 1/E; P and L_aux as for
 * token choice; route_stats of the shares; perm_token [E*C]: the chosen tokens
 * of each expert, ascending; router_logits: the probabilities s[t,e] the
 * experts chose on.  topk_idx, topk_w, dropped_mask and slot are not used
 * (may be NULL). */
#define MOE_FLAG_EXPERT_CHOICE 2
/* FP8 experts: the expert weights are E4M3 codes with scales (moe_fp8_experts,
 * made by moe_quantize_weights_fp8) and the layer runs through
 * moe_forward_fp8; moe_workspace_size then sizes that call's workspace.
 * Needs dtype == MOE_DT_BF16 (x, y, W_g, b1, b2 stay bf16).  With
 * MOE_FLAG_EXPERT_CHOICE x is quantised once per token and the chosen rows
 * take their token's codes and scale. */
#define MOE_FLAG_FP8_EXPERTS 4

/* Launch options; pass NULL for defaults. */
typedef struct {
  /* If non-NULL: created events recorded on `stream` around the kernels.
   * moe_forward: MOE_NUM_STAGES + 1 events; event i just before stage i,
   * event MOE_NUM_STAGES after the last.  moe_forward_fp8: MOE_NUM_STAGES + 2
   * events; the extra one (index MOE_NUM_STAGES + 1) is recorded after the
   * hidden activations' quantisation, between events 4 and 5 (so [4, 7) is
   * that kernel and [7, 5) the second expert GEMM).  moe_grouped_gemm: 2
   * events, before and after the GEMM kernel. */
  moe_event* stage_events;
  /* Limit of every device-side wait in nanoseconds; 0 = 2 s.  A wait that
   * runs out makes the kernel stop cleanly and records MOE_ERR_TIMEOUT. */
  int64_t wait_timeout_ns;
  /* OR of MOE_OPT_*; 0 = defaults. */
  int64_t flags;
} moe_launch_opts;

/* bf16 expert GEMMs: run the one-CTA 128 x 256 tile kernel instead of the
 * default CTA-pair (2-SM) 256 x 256 tile kernel.  Same results up to fp32
 * summation order inside the tensor core; kept for comparison and testing. */
#define MOE_OPT_GEMM_SINGLE_CTA 1

/* Human-readable name of a status.  Never NULL. */
const char* moe_status_string(moe_status s);

/* MOE_OK if the config describes a layer this library runs, else the reason. */
moe_status moe_validate_config(const moe_config* cfg);

/* Device workspace bytes moe_forward needs for `cfg` (0 if cfg is invalid).
 * It holds the routing scratch, the expert-grouped copy of x [T*k, d], the
 * hidden activations [T*k + S*T, f] (dtype) and the expert outputs
 * [T*k + S*T, d] (fp32, so that the gate-weighted sum rounds only once). */
size_t moe_workspace_size(const moe_config* cfg);

/* Expert capacity C = ceil(T * capacity_factor / E) computed in double, or -1
 * when capacity_factor <= 0 (no limit) ("MoE架构解析" §三 关键技术①).  With
 * MOE_FLAG_EXPERT_CHOICE: the tokens each expert chooses (see that flag). */
int64_t moe_capacity(const moe_config* cfg);

/* The layer's forward pass (steps 1-7 above).
 * Inputs (device, read only):
 *   x, W_g, W1, W2 required; b_g, b1, b2 optional (NULL = no bias; biases are
 *   not used with SwiGLU); W3 required iff act == MOE_ACT_SWIGLU.
 *   router_noise: optional fp32 [T, E], added to the router logits before
 *   gating and top-k (Gaussian noise to encourage exploration, "Mixture of
 *   Experts混合专家模型架构原理与路由策略实现", 门控网络的数学原理); the caller
 *   draws and scales it.  Selection, weights, P and router_logits then all
 *   use the noisy logits.  NULL = no noise.
 * Outputs (device, written):
 *   y [T, d] in dtype, or fp32 with MOE_FLAG_Y_F32 (must not overlap x),
 *   topk_idx int32 [T, k] (descending logit),
 *   topk_w fp32 [T, k], expert_counts int32 [E] (kept assignments per expert),
 *   dropped_mask uint8 [T, k] (1 = cut by capacity), f fp32 [E], P fp32 [E],
 *   L_aux fp32 [1].
 * Optional outputs (NULL = not written):
 *   route_stats fp32 [3]: routing health of the pre-capacity selection shares
 *   f_e = n_e / (T k) ("MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现"
 *   §3.3): entropy -sum f ln f (ln E when uniform), variance (1/E) sum (f -
 *   1/E)^2, and the coefficient of variation of the counts, E sqrt(variance);
 *   router_logits fp32 [T, E]; perm_token int32 [T*k]: token of each row of
 *   the expert-grouped order (experts ascending, tokens ascending inside an
 *   expert; entries past sum(expert_counts) are not written); slot int32 [T, k]:
 *   row of assignment (t, j) in that order, -1 if dropped.
 * workspace: device, 256-byte aligned, >= moe_workspace_size(cfg) bytes,
 *   owned by the caller, contents need not be initialised.
 * All device pointers must be 16-byte aligned.  T == 0 is valid: it writes
 * expert_counts = f = P = 0 and L_aux = 0, and the per-token tensors (x, y,
 * topk_idx, topk_w, dropped_mask and the optional ones) may then be NULL. */
moe_status moe_forward(const moe_config* cfg, const void* x, const void* W_g, const void* b_g,
                       const float* router_noise, const void* W1, const void* b1, const void* W2, const void* b2,
                       const void* W3, void* y, int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                       uint8_t* dropped_mask, float* f, float* P, float* L_aux, float* route_stats,
                       float* router_logits, int32_t* perm_token, int32_t* slot, void* workspace,
                       size_t workspace_bytes, moe_stream stream, const moe_launch_opts* opts);

/* The same forward pass with HOST buffers: x_host, router_noise_host (or
 * NULL) and the outputs (route_stats_host may be NULL) are host
 * memory (page-locked, e.g. cudaHostAlloc, for the copies to run
 * asynchronously; pageable memory works but its copies block the host).
 * Enqueued on `stream`: one host->device copy of x into the workspace,
 * moe_forward on device copies of every tensor, then one device->host copy per
 * output.  The weights (W_g .. W3) stay device pointers.  The host outputs are
 * complete once `stream` is synchronised.
 * workspace: >= moe_forward_host_workspace_size(cfg) bytes (moe_forward's
 * workspace followed by the device copies of x and the outputs).
 * Two calls on two streams with two workspaces overlap one call's copies
 * with the other's kernels; calls sharing a workspace must be ordered. */
size_t moe_forward_host_workspace_size(const moe_config* cfg);
moe_status moe_forward_host(const moe_config* cfg, const void* x_host, const void* W_g, const void* b_g,
                            const float* router_noise_host, const void* W1, const void* b1, const void* W2,
                            const void* b2, const void* W3, void* y_host, int32_t* topk_idx_host, float* topk_w_host,
                            int32_t* expert_counts_host, uint8_t* dropped_mask_host, float* f_host, float* P_host,
                            float* L_aux_host, float* route_stats_host, void* workspace, size_t workspace_bytes,
                            moe_stream stream, const moe_launch_opts* opts);

/* Backward pass of the layer (bf16; token or expert choice): gradients of
 *   L = sum_t <dy_t, y_t> + dL_aux * L_aux
 * (the load-balance loss joins the main loss before one backward, "MoE混合专家
 * 模型：Transformer稀疏前馈网络原理与PyTorch实现" §4.3) with respect to x, W_g,
 * b_g, W1, b1, W2, b2 and W3.  The forward pass is recomputed inside (nothing
 * is kept between calls); routing, the capacity cut and f carry no gradient;
 * the renormalised top-k weights and L_aux (through P) carry the router's.
 * Inputs: as moe_forward (device), plus dy [T, d] bf16 and the scalar dL_aux
 * (1.0 when L_aux is added to the loss as is).
 * Outputs (device, fp32, overwritten): dx [T, d], dW_g [d, E], db_g [E] (iff
 * b_g), dW1 [E+S, d, f], db1 [E+S, f] (iff b1), dW2 [E+S, f, d], db2 [E+S, d]
 * (iff b2), dW3 [E+S, d, f] (iff SwiGLU).
 * With MOE_FLAG_EXPERT_CHOICE the choice of tokens carries no gradient, the
 * gate probabilities s[t,e] weighting the chosen experts' outputs carry the
 * router's, and L_aux (constant alpha there: f_e = 1/E and sum_e P_e = 1)
 * carries none beyond rounding.
 * workspace: >= moe_backward_workspace_size(cfg) bytes, 256-byte aligned.
 * MOE_ERR_UNSUPPORTED for fp32 layers and for MOE_FLAG_FP8_EXPERTS.
 * Deterministic: bitwise the same gradients for the same inputs. */
size_t moe_backward_workspace_size(const moe_config* cfg);
moe_status moe_backward(const moe_config* cfg, const void* x, const void* W_g, const void* b_g,
                        const float* router_noise, const void* W1, const void* b1, const void* W2, const void* b2,
                        const void* W3, const void* dy, float dL_aux, float* dx, float* dW_g, float* db_g,
                        float* dW1, float* db1, float* dW2, float* db2, float* dW3, void* workspace,
                        size_t workspace_bytes, moe_stream stream, const moe_launch_opts* opts);

/* ---- FP8 (E4M3) experts ---------------------------------------------------------
 * "MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现" §5.2: expert parameters
 * quantised from 16-bit to 8-bit floats halve their memory at a usually
 * acceptable loss of quality.  Format E4M3 (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; largest finite 448).  A vector v is quantised with one scale
 * pair: a = max(max_i |v_i|, 2^-60), encoding factor r = fl32(448 / a), decoding
 * scale s = fl32(a / 448), codes q_i = e4m3(fl32(v_i r)) rounded to nearest with
 * ties to even and saturating at +-448; v_i ~ s value(q_i).
 *
 * Quantise weight slabs W [G, K, N] (bf16, the layer's [in, out] layout), one
 * vector per (slab, output column n): codes Wq [G, N, K] (transposed: K-major)
 * and decoding scales [G, N] fp32.  Device pointers, Wq 16-byte aligned;
 * K a multiple of 16; G <= 65535.  Asynchronous on `stream`. */
moe_status moe_quantize_weights_fp8(const void* W, int64_t G, int64_t K, int64_t N, uint8_t* Wq, float* scale,
                                    moe_stream stream);

/* Quantise the rows of X [rows, cols] (bf16), one vector per row: codes
 * Q [rows, cols] and decoding scales [rows] fp32.  cols a multiple of 16;
 * device pointers, 16-byte aligned.  The layer applies this to the hidden
 * activations between its two expert GEMMs, and to x while grouping it. */
moe_status moe_quantize_rows_fp8(const void* X, int64_t rows, int64_t cols, uint8_t* Q, float* scale,
                                 moe_stream stream);

/* FP8 expert weights, all device pointers (slabs: E routed, then S shared). */
typedef struct {
  const uint8_t* W1;  /* [E+S, f, d] codes of W1 (moe_quantize_weights_fp8 of [E+S, d, f]) */
  const float* s1;    /* [E+S, f] */
  const uint8_t* W3;  /* SwiGLU only, as W1; else NULL */
  const float* s3;
  const uint8_t* W2;  /* [E+S, d, f] codes of W2 ([E+S, f, d]) */
  const float* s2;    /* [E+S, d] */
} moe_fp8_experts;

/* The layer with FP8 experts (cfg->flags must include MOE_FLAG_FP8_EXPERTS).
 * Routing, statistics and gate weights are moe_forward's, on the bf16 x and
 * W_g.  Each token row of x is quantised (one scale per row) while it is
 * grouped; expert GEMM 1 multiplies E4M3 codes on the tensor cores (fp32
 * accumulation), scales by the row's and the output unit's decoding scales,
 * adds b1 (bf16, not with SwiGLU) and applies the activation; the hidden
 * activations are held in bf16, then quantised per row; expert GEMM 2 the
 * same with W2 and b2; the combine is moe_forward's (fp32 expert outputs).
 * Arguments as moe_forward, with the expert weights in `w`.  d and f
 * multiples of 64. */
moe_status moe_forward_fp8(const moe_config* cfg, const void* x, const void* W_g, const void* b_g,
                           const float* router_noise, const moe_fp8_experts* w, const void* b1, const void* b2,
                           void* y, int32_t* topk_idx, float* topk_w, int32_t* expert_counts, uint8_t* dropped_mask,
                           float* f, float* P, float* L_aux, float* route_stats, float* router_logits,
                           int32_t* perm_token, int32_t* slot, void* workspace, size_t workspace_bytes,
                           moe_stream stream, const moe_launch_opts* opts);

/* moe_forward_fp8 with HOST buffers, as moe_forward_host is moe_forward
 * with host buffers (the FP8 expert weights stay device pointers);
 * workspace: >= moe_forward_host_workspace_size(cfg) bytes. */
moe_status moe_forward_fp8_host(const moe_config* cfg, const void* x_host, const void* W_g, const void* b_g,
                                const float* router_noise_host, const moe_fp8_experts* w, const void* b1,
                                const void* b2, void* y_host, int32_t* topk_idx_host, float* topk_w_host,
                                int32_t* expert_counts_host, uint8_t* dropped_mask_host, float* f_host, float* P_host,
                                float* L_aux_host, float* route_stats_host, void* workspace, size_t workspace_bytes,
                                moe_stream stream, const moe_launch_opts* opts);

/* Where an intermediate of moe_forward / moe_forward_fp8 lies in the
 * workspace after a call (for inspection and tests): *offset and *bytes of
 * region `region` for `cfg`.  MOE_ERR_INVALID_ARG for an invalid cfg or a
 * region the cfg does not have.  Rows are those of the expert-grouped order
 * (T*k routed rows, then S*T shared rows). */
#define MOE_REGION_XPERM 1     /* grouped copy of x [T*k, d]: dtype, or E4M3 codes */
#define MOE_REGION_X_SCALE 2   /* FP8: decoding scale of each grouped row [T*k] fp32 */
#define MOE_REGION_H 3         /* hidden activations [T*k + S*T, f] (bf16 with FP8) */
#define MOE_REGION_H_CODES 4   /* FP8: E4M3 codes of H [T*k + S*T, f] */
#define MOE_REGION_H_SCALE 5   /* FP8: decoding scale of each row of H [T*k + S*T] fp32 */
#define MOE_REGION_O 6         /* expert outputs [T*k + S*T, d] fp32 */
moe_status moe_workspace_region(const moe_config* cfg, int32_t region, size_t* offset, size_t* bytes);

/* Waits for `stream`, then reports the device-side status of the last call
 * that used `workspace`: MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE, or
 * MOE_ERR_CUDA if the stream itself reports an error.  Synchronising. */
moe_status moe_check_device_errors(const void* workspace, moe_stream stream);

/* The expert grouped GEMM on its own (the layer's step 5 for one weight set):
 *   for every group g and row r in [seg_offsets[g], seg_offsets[g+1]):
 *     act == MOE_ACT_NONE:    C[r, :] = A[r, :] B[g] (+ bias[g])
 *     act == MOE_ACT_RELU/GELU: C[r, :] = act(A[r, :] B[g] + bias[g])
 *     act == MOE_ACT_SWIGLU:  C[r, :] = silu(A[r, :] B[g]) * (A[r, :] B3[g])
 * A [M, K], B and B3 [G, K, N], bias [G, N] or NULL, C [M, N]; rows of C
 * outside every group are not written.  seg_offsets: DEVICE int32 [G+1],
 * non-decreasing, seg_offsets[0] >= 0, seg_offsets[G] <= M.  fp32
 * accumulation; C is rounded to dtype.  bf16 needs K, N multiples of 64.
 * workspace: >= moe_grouped_gemm_workspace_size(G) bytes, 256-byte aligned. */
size_t moe_grouped_gemm_workspace_size(int32_t G);
moe_status moe_grouped_gemm(int32_t dtype, int32_t act, int32_t G, const int32_t* seg_offsets, int64_t M,
                            int32_t K, int32_t N, const void* A, const void* B, const void* B3,
                            const void* bias, void* C, void* workspace, size_t workspace_bytes,
                            moe_stream stream, const moe_launch_opts* opts);

/* moe_grouped_gemm without a workspace, for callers that cannot allocate
 * device memory when they call (memory planned once at start-up, a plugin
 * inside a framework that owns every allocation, or a loop that must not call
 * cudaMalloc, which can synchronise the device).  The pages have no
 * counterpart: this is a calling convention of this library, not a step of the
 * layer.  Same arguments, options and results as moe_grouped_gemm minus the
 * workspace.  Its scratch (6656 bytes: a status word and the tile table) is a
 * fixed device array inside the library, held by every GPU that loads it until
 * the process exits, so G <= 264 (else MOE_ERR_UNSUPPORTED).  The first call
 * in a CUDA context, with that context's device current, looks up the array's
 * address and keeps it for that context; make it before any stream capture.
 * A context that is destroyed and made again (cudaDeviceReset) gets a new
 * address, looked up again by its own first call.  All calls on a device share
 * the array (each clears what it needs first), so calls that may overlap on
 * the GPU race: order them.  Device-side failures are not reported (use
 * moe_grouped_gemm with moe_check_device_errors to detect them); invalid
 * seg_offsets leave C as it was.  It calls no cudaMalloc, cudaFree or other
 * allocating routine. */
moe_status moe_grouped_gemm_noalloc(int32_t dtype, int32_t act, int32_t G, const int32_t* seg_offsets, int64_t M,
                                    int32_t K, int32_t N, const void* A, const void* B, const void* B3,
                                    const void* bias, void* C, moe_stream stream, const moe_launch_opts* opts);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_MOE_H */
