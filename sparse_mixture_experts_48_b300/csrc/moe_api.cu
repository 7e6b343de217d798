// The C ABI of libmoe.so (declared in include/moe.h): argument checks,
// workspace layout, and the launch sequence of the layer's kernels.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"
#include "kernels.cuh"

using namespace moe;

namespace {

constexpr int kMaxE = 256;
constexpr int kMaxK = 8;
constexpr int kMaxShared = 8;


// Expert choice: tokens per expert, min(T, ceil(T cf / E)), or min(T, ceil(T k / E))
// without a capacity factor (the compute of top-k token choice).
int64_t ec_capacity_of(const moe_config* c) {
  const double v = c->capacity_factor > 0.0 ? ceil((double)c->T * c->capacity_factor / (double)c->E)
                                            : ceil((double)c->T * (double)c->k / (double)c->E);
  return (int64_t)v < c->T ? (int64_t)v : c->T;
}

moe_status check_cfg(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d_model <= 0 || c->d_ff <= 0 || c->E <= 0 || c->k <= 0 || c->n_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->k > c->E) return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_ACT_RELU && c->act != MOE_ACT_GELU && c->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (c->gating != MOE_GATE_SOFTMAX && c->gating != MOE_GATE_SIGMOID_NORM) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_DT_F32 && c->dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (c->flags & ~(int64_t)(MOE_FLAG_Y_F32 | MOE_FLAG_EXPERT_CHOICE | MOE_FLAG_FP8_EXPERTS)) return MOE_ERR_INVALID_ARG;
  if ((c->flags & MOE_FLAG_FP8_EXPERTS) && c->dtype != MOE_DT_BF16) return MOE_ERR_UNSUPPORTED;
  if (!isfinite(c->capacity_factor) || !isfinite(c->alpha)) return MOE_ERR_INVALID_ARG;
  if (c->E > kMaxE || c->k > kMaxK || c->n_shared > kMaxShared) return MOE_ERR_UNSUPPORTED;
  if (c->dtype == MOE_DT_BF16 && (c->d_model % 64 != 0 || c->d_ff % 64 != 0)) return MOE_ERR_UNSUPPORTED;
  if (c->dtype == MOE_DT_F32 && (c->d_model % 4 != 0 || c->d_ff % 4 != 0)) return MOE_ERR_UNSUPPORTED;
  // Row indices of the grouped buffers are int32 (and TMA coordinates).
  const int64_t routed = (c->flags & MOE_FLAG_EXPERT_CHOICE) ? (int64_t)c->E * ec_capacity_of(c) : c->T * (int64_t)c->k;
  const int64_t rows_all = routed + (int64_t)c->n_shared * c->T;
  if (rows_all >= ((int64_t)1 << 31) - 2 * kGemmBM) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

WsLayout layout(const moe_config* c) {
  WsLayout L;
  const size_t esz = c->dtype == MOE_DT_BF16 ? 2 : 4;
  const bool ec = (c->flags & MOE_FLAG_EXPERT_CHOICE) != 0;
  const int bm = router_tile_tokens(c->dtype, c->E);
  L.nblk = (c->T + bm - 1) / bm;
  L.ec_C = ec ? ec_capacity_of(c) : -1;
  L.EW = (c->E + 31) / 32;
  L.rows_tk = ec ? (int64_t)c->E * L.ec_C : c->T * (int64_t)c->k;
  L.rows_all = L.rows_tk + (int64_t)c->n_shared * c->T;
  L.G = c->E + c->n_shared;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + (bytes ? bytes : 1), 256);
    return at;
  };
  L.hdr = take(sizeof(WsHeader));
  L.hist = take((size_t)L.nblk * c->E * 4);
  L.psum = take((size_t)L.nblk * c->E * 4);
  L.base = take((size_t)L.nblk * c->E * 4);
  L.lrank = take((size_t)L.rows_tk);
  L.npre = take((size_t)c->E * 4);
  L.offsets = take((size_t)(c->E + 1) * 4);
  L.seg = take((size_t)(6 * L.G + 1) * 4);
  L.slot = take((size_t)L.rows_tk * 4);
  const bool fp8 = (c->flags & MOE_FLAG_FP8_EXPERTS) != 0;
  L.xperm = take((size_t)L.rows_tk * c->d_model * (fp8 ? 1 : esz));
  L.h = take((size_t)L.rows_all * c->d_ff * esz);
  L.o = take((size_t)L.rows_all * c->d_model * 4);
  L.ec_scores = take(ec ? (size_t)c->E * c->T * 4 : 0);
  L.ec_bits = take(ec ? (size_t)c->T * L.EW * 4 : 0);
  L.ec_tokrow = take(ec ? (size_t)c->T * c->E * 4 : 0);
  L.ec_wrow = take(ec ? (size_t)L.rows_tk * 4 : 0);
  L.ec_perm = take(ec ? (size_t)L.rows_tk * 4 : 0);
  // FP8: the token-order codes of x serve the shared experts, and with expert
  // choice also the grouped copy (gathered from them)
  const bool sh8 = fp8 && (c->n_shared > 0 || ec);
  L.xs_perm = take(fp8 ? (size_t)L.rows_tk * 4 : 0);
  L.xq = take(sh8 ? (size_t)c->T * c->d_model : 0);
  L.xs_tok = take(sh8 ? (size_t)c->T * 4 : 0);
  L.hq = take(fp8 ? (size_t)L.rows_all * c->d_ff : 0);
  L.hs = take(fp8 ? (size_t)L.rows_all * 4 : 0);
  L.total = off;
  return L;
}

SegTable seg_table(uint8_t* ws, size_t off, int G) {
  int* p = (int*)(ws + off);
  SegTable s;
  s.rows = p;
  s.w = p + G;
  s.out_row = p + 2 * G;
  s.a_row = p + 3 * G;
  s.a_src = p + 4 * G;
  s.mtile_start = p + 5 * G;
  return s;
}

int64_t capacity_of(const moe_config* c) {
  if (c->capacity_factor <= 0.0) return -1;
  // ceil(T * cf / E) in double, the expert-capacity formula.
  return (int64_t)ceil((double)c->T * c->capacity_factor / (double)c->E);
}

// Device staging of moe_forward_host, placed after the moe_forward workspace.
struct HostStage {
  size_t x, y, idx, w, cnt, drop, f, P, L, noise, stats, total;
};

HostStage host_stage(const moe_config* c, size_t base) {
  HostStage h;
  const size_t esz = c->dtype == MOE_DT_BF16 ? 2 : 4;
  const bool y_f32 = (c->flags & MOE_FLAG_Y_F32) != 0 || c->dtype == MOE_DT_F32;
  const size_t tk = (size_t)c->T * c->k;
  size_t off = align_up(base, 256);
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + (bytes ? bytes : 1), 256);
    return at;
  };
  h.x = take((size_t)c->T * c->d_model * esz);
  h.y = take((size_t)c->T * c->d_model * (y_f32 ? 4 : 2));
  h.idx = take(tk * 4);
  h.w = take(tk * 4);
  h.cnt = take((size_t)c->E * 4);
  h.drop = take(tk);
  h.f = take((size_t)c->E * 4);
  h.P = take((size_t)c->E * 4);
  h.L = take(4);
  h.noise = take((size_t)c->T * c->E * 4);
  h.stats = take(3 * 4);
  h.total = off;
  return h;
}

// Workspace of moe_backward: the forward recomputation in a padded grouped
// layout (every routed segment padded to whole 128-row blocks, the shared
// segments to T rounded up to 128, padding rows zero) and the gradients.
struct BwdLayout {
  size_t hdr, hist, psum, base, lrank, npre, offsets, seg, slot, idx, w, drop, cnt, f, P, L, logits;
  size_t xperm, pre_a, pre_u, h, o, dO, dA, dU, dxp, dw, dl, part, bpart, total;
  size_t ec_scores, ec_bits, ec_tokrow, ec_wrow, ec_perm, ec_dw;   // expert choice
  int64_t nblk, Tpad, rows_routed, rows_all, nchunk;
  int64_t ec_C, ec_Cs;   // expert choice: tokens per expert, rows reserved per expert (C padded)
  int G, EW;
};

BwdLayout bwd_layout(const moe_config* c) {
  BwdLayout L;
  const bool swiglu = c->act == MOE_ACT_SWIGLU;
  const int64_t T = c->T;
  L.G = c->E + c->n_shared;
  const int bm = router_tile_tokens(c->dtype, c->E);
  L.nblk = (T + bm - 1) / bm;
  L.Tpad = (T + 127) / 128 * 128;
  const bool ec = (c->flags & MOE_FLAG_EXPERT_CHOICE) != 0;
  L.ec_C = ec ? ec_capacity_of(c) : -1;
  L.ec_Cs = ec ? (L.ec_C + 127) / 128 * 128 : 0;
  L.EW = (c->E + 31) / 32;
  L.rows_routed = ec ? (int64_t)c->E * L.ec_Cs
                     : (T * c->k + 127) / 128 * 128 + 128 * (int64_t)c->E;   // >= sum of padded segments
  L.rows_all = L.rows_routed + (int64_t)c->n_shared * L.Tpad;
  L.nchunk = dwg_chunks(T);
  const size_t d = c->d_model, f = c->d_ff, tk = (size_t)T * c->k, ra = (size_t)L.rows_all;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + (bytes ? bytes : 1), 256);
    return at;
  };
  L.hdr = take(sizeof(WsHeader));
  L.hist = take((size_t)L.nblk * c->E * 4);
  L.psum = take((size_t)L.nblk * c->E * 4);
  L.base = take((size_t)L.nblk * c->E * 4);
  L.lrank = take(tk);
  L.npre = take((size_t)c->E * 4);
  L.offsets = take((size_t)(c->E + 1) * 4);
  L.seg = take((size_t)(6 * L.G + 1) * 4);
  L.slot = take(tk * 4);
  L.idx = take(tk * 4);
  L.w = take(tk * 4);
  L.drop = take(tk);
  L.cnt = take((size_t)c->E * 4);
  L.f = take((size_t)c->E * 4);
  L.P = take((size_t)c->E * 4);
  L.L = take(4);
  L.logits = take((size_t)T * c->E * 4);
  L.xperm = take((size_t)L.rows_routed * d * 2);
  L.pre_a = take(ra * f * 2);
  L.pre_u = take(swiglu ? ra * f * 2 : 0);
  L.h = take(ra * f * 2);
  L.o = take(ra * d * 4);
  L.dO = take(ra * d * 2);
  L.dA = take(ra * f * 2);
  L.dU = take(swiglu ? ra * f * 2 : 0);
  L.dxp = take(ra * d * 4);
  L.dw = take(tk * 4);
  L.dl = take((size_t)T * c->E * 4);
  L.part = take((size_t)L.nchunk * d * c->E * 4);
  L.bpart = take((size_t)L.nchunk * c->E * 4);
  const size_t ecr = ec ? (size_t)L.rows_routed : 0;
  L.ec_scores = take(ec ? (size_t)c->E * T * 4 : 0);
  L.ec_bits = take(ec ? (size_t)T * L.EW * 4 : 0);
  L.ec_tokrow = take(ec ? (size_t)T * c->E * 4 : 0);
  L.ec_wrow = take(ecr * 4);
  L.ec_perm = take(ecr * 4);
  L.ec_dw = take(ecr * 4);
  L.total = off;
  return L;
}

moe_status check_bwd_cfg(const moe_config* c) {
  moe_status st = check_cfg(c);
  if (st != MOE_OK) return st;
  if (c->dtype != MOE_DT_BF16 || (c->flags & MOE_FLAG_FP8_EXPERTS)) return MOE_ERR_UNSUPPORTED;
  const BwdLayout L = bwd_layout(c);
  if (L.rows_all >= ((int64_t)1 << 31) - 2 * kGemmBM) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

struct StageClock {
  const moe_launch_opts* o;
  cudaStream_t s;
  cudaError_t mark(int i) const {
    if (o && o->stage_events) return cudaEventRecord((cudaEvent_t)o->stage_events[i], s);
    return cudaSuccess;
  }
};

}  // namespace

namespace moe {

moe_status check_grouped_gemm_args(int32_t dtype, int32_t act, int32_t G, const int32_t* seg_offsets, int64_t M,
                                   int32_t K, int32_t N, const void* A, const void* B, const void* B3,
                                   const void* bias, const void* C) {
  if (dtype != MOE_DT_F32 && dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (act != MOE_ACT_NONE && act != MOE_ACT_RELU && act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU)
    return MOE_ERR_INVALID_ARG;
  if (G <= 0 || M < 0 || K <= 0 || N <= 0 || !seg_offsets || !A || !B || !C) return MOE_ERR_INVALID_ARG;
  if ((act == MOE_ACT_SWIGLU) != (B3 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (G > kGroupedGemmMaxGroups) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_DT_BF16 && (K % 64 != 0 || N % 64 != 0)) return MOE_ERR_UNSUPPORTED;
  if (M >= ((int64_t)1 << 31) - 2 * kGemmBM) return MOE_ERR_UNSUPPORTED;
  const void* all[] = {seg_offsets, A, B, B3, bias, C};
  for (const void* p : all)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status launch_grouped_gemm_on_scratch(int32_t dtype, int32_t act, int32_t G, const int32_t* seg_offsets,
                                          int64_t M, int32_t K, int32_t N, const void* A, const void* B,
                                          const void* B3, const void* bias, void* C, uint8_t* scratch,
                                          moe_stream stream, const moe_launch_opts* opts) {
  cudaStream_t s = (cudaStream_t)stream;
  WsHeader* hdr = (WsHeader*)scratch;
  const SegTable seg = seg_table(scratch, align_up(sizeof(WsHeader), 256), G);
  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_segments_from_offsets(seg_offsets, G, M, seg, &hdr->err, s) != cudaSuccess) return MOE_ERR_CUDA;
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.dtype = dtype; g.act = act; g.G = G; g.K = K; g.N = N; g.a_from_out_rows = true; g.seg = seg;
  g.A0 = A; g.rows_A0 = M > 0 ? M : 1; g.A1 = nullptr; g.B = B; g.B3 = B3; g.Gw = G; g.bias = bias; g.C = C;
  g.max_mtiles = M > 0 ? (M + kGemmBM - 1) / kGemmBM + G : 0;
  g.rows_C = M;               // whole 32-row warp tiles inside a group leave by TMA store
  g.err = &hdr->err;
  g.timeout_ns = (opts && opts->wait_timeout_ns > 0) ? opts->wait_timeout_ns : kDefaultTimeoutNs;
  g.single_cta = opts && (opts->flags & MOE_OPT_GEMM_SINGLE_CTA);
  if (opts && opts->stage_events && cudaEventRecord((cudaEvent_t)opts->stage_events[0], s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_grouped_gemm(g, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (opts && opts->stage_events && cudaEventRecord((cudaEvent_t)opts->stage_events[1], s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace moe

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_validate_config(const moe_config* cfg) { return check_cfg(cfg); }

size_t moe_workspace_size(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return layout(cfg).total;
}

int64_t moe_capacity(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK) return -1;
  if (cfg->flags & MOE_FLAG_EXPERT_CHOICE) return ec_capacity_of(cfg);
  return capacity_of(cfg);
}

// The layer; q8 != NULL: FP8 experts (W1, W2, W3 are then q8's codes).
static moe_status forward_impl(const moe_config* cfg, const void* x, const void* W_g, const void* b_g,
                               const float* router_noise, const void* W1, const void* b1, const void* W2,
                               const void* b2, const void* W3, const moe_fp8_experts* q8, void* y,
                               int32_t* topk_idx, float* topk_w, int32_t* expert_counts, uint8_t* dropped_mask,
                               float* f, float* P, float* L_aux, float* route_stats, float* router_logits,
                               int32_t* perm_token, int32_t* slot, void* workspace, size_t workspace_bytes,
                               moe_stream stream, const moe_launch_opts* opts) {
  moe_status st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  const bool fp8 = (c.flags & MOE_FLAG_FP8_EXPERTS) != 0;
  if (fp8 != (q8 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (fp8) {
    if (!q8->s1 || !q8->s2 || (q8->W3 != nullptr) != (q8->s3 != nullptr)) return MOE_ERR_INVALID_ARG;
    const void* sc[] = {q8->s1, q8->s2, q8->s3};
    for (const void* p : sc)
      if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  // Required tensors.  With T == 0 the per-token tensors hold no elements and
  // may be NULL (allocators hand out NULL for empty buffers).
  const bool empty = c.T == 0;
  const bool ec = (c.flags & MOE_FLAG_EXPERT_CHOICE) != 0;   // topk_idx, topk_w, dropped_mask unused
  if (!W_g || !W1 || !W2 || !expert_counts || !f || !P || !L_aux) return MOE_ERR_INVALID_ARG;
  if (!empty && (!x || !y)) return MOE_ERR_INVALID_ARG;
  if (!empty && !ec && (!topk_idx || !topk_w || !dropped_mask)) return MOE_ERR_INVALID_ARG;
  if (swiglu != (W3 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (swiglu && (b1 || b2)) return MOE_ERR_INVALID_ARG;
  const void* all[] = {x, W_g, b_g, W1, b1, W2, b2, W3, y, topk_idx, topk_w, expert_counts, dropped_mask,
                       f, P, L_aux, router_logits, perm_token, slot, router_noise, route_stats};
  for (const void* p : all)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  // y must not overlap x.
  const size_t esz = c.dtype == MOE_DT_BF16 ? 2 : 4;
  const bool y_f32 = (c.flags & MOE_FLAG_Y_F32) != 0 || c.dtype == MOE_DT_F32;
  const size_t xbytes = (size_t)c.T * c.d_model * esz;
  const size_t ybytes = (size_t)c.T * c.d_model * (y_f32 ? 4 : 2);
  if (xbytes && (const uint8_t*)y < (const uint8_t*)x + xbytes && (const uint8_t*)x < (const uint8_t*)y + ybytes)
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(&c);
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  const int64_t timeout = (opts && opts->wait_timeout_ns > 0) ? opts->wait_timeout_ns : kDefaultTimeoutNs;

  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  WsHeader* hdr = (WsHeader*)(ws + L.hdr);
  const SegTable seg = seg_table(ws, L.seg, L.G);
  int32_t* slot_buf = slot ? slot : (int32_t*)(ws + L.slot);
  const int64_t C = capacity_of(&c);
  StageClock clk{opts, s};

  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (ec && c.T > 0 && cudaMemsetAsync(ws + L.ec_bits, 0, (size_t)c.T * L.EW * 4, s) != cudaSuccess)
    return MOE_ERR_CUDA;

  // 1. router, and (in its last CTA) the scan: ranks, capacity, offsets,
  //    statistics, segment table
  if (clk.mark(0) != cudaSuccess) return MOE_ERR_CUDA;
  RouterArgs ra;
  memset(&ra, 0, sizeof(ra));
  ra.x = x; ra.Wg = W_g; ra.bg = b_g; ra.noise = router_noise; ra.T = c.T; ra.d = c.d_model; ra.E = c.E; ra.k = c.k;
  ra.gating = c.gating; ra.dtype = c.dtype; ra.logits_out = router_logits; ra.topk_idx = topk_idx;
  ra.topk_w = topk_w; ra.lrank = ws + L.lrank; ra.hist = (int32_t*)(ws + L.hist); ra.psum = (float*)(ws + L.psum);
  ra.err = &hdr->err; ra.timeout_ns = timeout; ra.nblk = L.nblk;
  ra.bm = router_tile_tokens(c.dtype, c.E);
  ra.scores_em = ec ? (float*)(ws + L.ec_scores) : nullptr; ra.raw_logits = nullptr;
  ScanArgs sa;
  memset(&sa, 0, sizeof(sa));
  sa.T = c.T; sa.E = c.E; sa.k = c.k; sa.S = c.n_shared; sa.capacity = ec ? -1 : C; sa.alpha = c.alpha;
  sa.nblk = L.nblk; sa.ec_C = L.ec_C; sa.pad_rows = 1; sa.shared_stride = c.T;
  sa.hist = ra.hist; sa.psum = ra.psum; sa.base = (int32_t*)(ws + L.base); sa.n_pre = (int32_t*)(ws + L.npre);
  sa.counts = expert_counts; sa.offsets = (int32_t*)(ws + L.offsets); sa.f = f; sa.P = P; sa.L_aux = L_aux;
  sa.route_stats = route_stats;
  sa.seg = seg; sa.rows_tk = L.rows_tk; sa.err = &hdr->err;
  ra.fused_scan = L.nblk > 0;
  ra.scan = sa;
  ra.done = &hdr->router_done;
  if (launch_router(ra, s) != cudaSuccess) return MOE_ERR_CUDA;
  // No router CTA (T = 0): the scan on its own writes the empty statistics.
  if (!ra.fused_scan && launch_scan(sa, s) != cudaSuccess) return MOE_ERR_CUDA;

  // 2. expert choice: each expert's choice of tokens
  if (clk.mark(1) != cudaSuccess) return MOE_ERR_CUDA;
  if (ec) {
    EcSelectArgs ea;
    ea.scores_em = (const float*)(ws + L.ec_scores); ea.T = c.T; ea.C = L.ec_C; ea.Cs = L.ec_C; ea.E = c.E; ea.EW = L.EW;
    ea.perm = (int32_t*)(ws + L.ec_perm); ea.w_row = (float*)(ws + L.ec_wrow); ea.tok_row = (int32_t*)(ws + L.ec_tokrow);
    ea.bits = (uint32_t*)(ws + L.ec_bits); ea.err = &hdr->err;
    if (c.T > 0 && launch_ec_select(ea, s) != cudaSuccess) return MOE_ERR_CUDA;
  }

  // 3. gather into the expert-grouped buffer
  if (clk.mark(2) != cudaSuccess) return MOE_ERR_CUDA;
  if (ec) {
    EcGatherArgs eg;
    eg.x = x; eg.perm = (const int32_t*)(ws + L.ec_perm); eg.rows = c.T > 0 ? L.rows_tk : 0; eg.d = c.d_model;
    eg.esz = (int)esz; eg.xperm = ws + L.xperm; eg.err = &hdr->err; eg.xs_tok = nullptr; eg.xs_perm = nullptr;
    eg.C = L.ec_C; eg.Cs = L.ec_C;
    if (fp8) {
      // quantise x once per token, then gather the codes and their scales
      QuantRowsArgs qx;
      qx.X = x; qx.Q = ws + L.xq; qx.scale = (float*)(ws + L.xs_tok); qx.cols = c.d_model; qx.rows0 = c.T;
      qx.live0 = nullptr; qx.row1 = c.T; qx.rows1 = 0; qx.err = &hdr->err;
      if (launch_quantize_rows(qx, s) != cudaSuccess) return MOE_ERR_CUDA;
      eg.x = ws + L.xq; eg.esz = 1; eg.xs_tok = (const float*)(ws + L.xs_tok); eg.xs_perm = (float*)(ws + L.xs_perm);
    }
    if (launch_ec_gather(eg, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (perm_token && L.rows_tk > 0 &&
        cudaMemcpyAsync(perm_token, ws + L.ec_perm, (size_t)L.rows_tk * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  GatherArgs ga;
  memset(&ga, 0, sizeof(ga));
  ga.x = x; ga.T = c.T; ga.d = c.d_model; ga.E = c.E; ga.k = c.k; ga.dtype = c.dtype; ga.capacity = C;
  ga.topk_idx = topk_idx; ga.lrank = ra.lrank; ga.base = sa.base; ga.offsets = sa.offsets; ga.slot = slot_buf;
  ga.dropped = dropped_mask; ga.perm_token = perm_token; ga.xperm = ws + L.xperm; ga.err = &hdr->err;
  ga.nblk = L.nblk; ga.bm = ra.bm;
  // Without stage events between them, the gather, the GEMMs and the combine
  // of a token-choice bf16 / fp32 forward launch with programmatic stream
  // serialization: each may be scheduled while its predecessor finishes, and
  // waits in the kernel for that predecessor's results.
  const bool pdl = !ec && !fp8 && !(opts && opts->stage_events);
  ga.pdl = pdl;
  const bool sh8 = fp8 && c.n_shared > 0;
  if (fp8) {
    ga.fp8 = true;
    ga.xs_perm = (float*)(ws + L.xs_perm);
    ga.xq = sh8 ? ws + L.xq : nullptr;
    ga.xs_tok = sh8 ? (float*)(ws + L.xs_tok) : nullptr;
  }
  if (!ec && launch_gather(ga, s) != cudaSuccess) return MOE_ERR_CUDA;

  // 4./5. expert GEMMs
  const int64_t max_mtiles = (L.rows_tk + kGemmBM - 1) / kGemmBM + c.E +
                             (int64_t)c.n_shared * ((c.T + kGemmBM - 1) / kGemmBM);
  GemmArgs g1;
  memset(&g1, 0, sizeof(g1));
  g1.dtype = c.dtype; g1.act = c.act; g1.G = L.G; g1.K = c.d_model; g1.N = c.d_ff; g1.a_from_out_rows = false;
  g1.seg = seg; g1.A0 = ws + L.xperm; g1.rows_A0 = L.rows_tk > 0 ? L.rows_tk : 1;
  g1.A1 = c.n_shared > 0 ? x : nullptr; g1.rows_A1 = c.T;
  g1.B = W1; g1.B3 = W3; g1.Gw = L.G; g1.bias = b1; g1.C = ws + L.h; g1.max_mtiles = c.T > 0 ? max_mtiles : 0;
  g1.err = &hdr->err; g1.timeout_ns = timeout;
  g1.single_cta = opts && (opts->flags & MOE_OPT_GEMM_SINGLE_CTA);
  g1.rows_C = L.rows_all;     // H leaves by TMA store (whole 32-row warp tiles)
  g1.pdl = pdl;
  if (fp8) {
    g1.fp8 = true;
    g1.A1 = sh8 ? ws + L.xq : nullptr;
    g1.a_scale0 = (const float*)(ws + L.xs_perm); g1.a_scale1 = sh8 ? (const float*)(ws + L.xs_tok) : nullptr;
    g1.B = q8->W1; g1.B3 = q8->W3; g1.b_scale = q8->s1; g1.b3_scale = q8->s3;
  }
  if (clk.mark(3) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_grouped_gemm(g1, s) != cudaSuccess) return MOE_ERR_CUDA;

  GemmArgs g2 = g1;
  g2.act = MOE_ACT_NONE; g2.K = c.d_ff; g2.N = c.d_model; g2.a_from_out_rows = true;
  g2.A0 = ws + L.h; g2.rows_A0 = L.rows_all > 0 ? L.rows_all : 1; g2.A1 = nullptr; g2.rows_A1 = 0;
  g2.B = W2; g2.B3 = nullptr; g2.bias = b2; g2.C = ws + L.o; g2.out_f32 = true; g2.rows_C = L.rows_all;
  if (clk.mark(4) != cudaSuccess) return MOE_ERR_CUDA;
  if (fp8) {
    // H (bf16) -> E4M3 codes with one scale per row: the kept routed rows and the shared rows.
    QuantRowsArgs qa;
    qa.X = ws + L.h; qa.Q = ws + L.hq; qa.scale = (float*)(ws + L.hs); qa.cols = c.d_ff;
    qa.rows0 = c.T > 0 ? L.rows_tk : 0; qa.live0 = sa.offsets + c.E;
    qa.row1 = L.rows_tk; qa.rows1 = (int64_t)c.n_shared * c.T; qa.err = &hdr->err;
    if (launch_quantize_rows(qa, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (opts && opts->stage_events && cudaEventRecord((cudaEvent_t)opts->stage_events[MOE_NUM_STAGES + 1], s) !=
                                          cudaSuccess)
      return MOE_ERR_CUDA;
    g2.A0 = ws + L.hq; g2.a_scale0 = (const float*)(ws + L.hs); g2.a_scale1 = nullptr;
    g2.B = q8->W2; g2.b_scale = q8->s2; g2.b3_scale = nullptr;
  }
  if (launch_grouped_gemm(g2, s) != cudaSuccess) return MOE_ERR_CUDA;

  // 6. combine
  if (clk.mark(5) != cudaSuccess) return MOE_ERR_CUDA;
  CombineArgs ca;
  ca.o = (const float*)(ws + L.o); ca.T = c.T; ca.d = c.d_model; ca.k = c.k; ca.S = c.n_shared; ca.y_f32 = y_f32;
  ca.rows_tk = L.rows_tk; ca.slot = slot_buf; ca.topk_w = topk_w; ca.y = y; ca.err = &hdr->err;
  ca.pdl = pdl;
  if (ec) {
    EcCombineArgs ek;
    ek.o = (const float*)(ws + L.o); ek.bits = (const uint32_t*)(ws + L.ec_bits);
    ek.tok_row = (const int32_t*)(ws + L.ec_tokrow); ek.w_row = (const float*)(ws + L.ec_wrow); ek.T = c.T;
    ek.E = c.E; ek.EW = L.EW; ek.S = c.n_shared; ek.d = c.d_model; ek.rows_routed = L.rows_tk; ek.y_f32 = y_f32;
    ek.y = y; ek.err = &hdr->err;
    if (launch_ec_combine(ek, s) != cudaSuccess) return MOE_ERR_CUDA;
  } else if (launch_combine(ca, s) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  if (clk.mark(6) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_forward(const moe_config* cfg, const void* x, const void* W_g, const void* b_g,
                       const float* router_noise, const void* W1, const void* b1, const void* W2, const void* b2,
                       const void* W3, void* y, int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                       uint8_t* dropped_mask, float* f, float* P, float* L_aux, float* route_stats,
                       float* router_logits, int32_t* perm_token, int32_t* slot, void* workspace,
                       size_t workspace_bytes, moe_stream stream, const moe_launch_opts* opts) {
  if (cfg && (cfg->flags & MOE_FLAG_FP8_EXPERTS)) return MOE_ERR_INVALID_ARG;   // moe_forward_fp8
  return forward_impl(cfg, x, W_g, b_g, router_noise, W1, b1, W2, b2, W3, nullptr, y, topk_idx, topk_w,
                      expert_counts, dropped_mask, f, P, L_aux, route_stats, router_logits, perm_token, slot,
                      workspace, workspace_bytes, stream, opts);
}

moe_status moe_forward_fp8(const moe_config* cfg, const void* x, const void* W_g, const void* b_g,
                           const float* router_noise, const moe_fp8_experts* w, const void* b1, const void* b2,
                           void* y, int32_t* topk_idx, float* topk_w, int32_t* expert_counts, uint8_t* dropped_mask,
                           float* f, float* P, float* L_aux, float* route_stats, float* router_logits,
                           int32_t* perm_token, int32_t* slot, void* workspace, size_t workspace_bytes,
                           moe_stream stream, const moe_launch_opts* opts) {
  if (!cfg || !(cfg->flags & MOE_FLAG_FP8_EXPERTS) || !w) return MOE_ERR_INVALID_ARG;
  return forward_impl(cfg, x, W_g, b_g, router_noise, w->W1, b1, w->W2, b2, w->W3, w, y, topk_idx, topk_w,
                      expert_counts, dropped_mask, f, P, L_aux, route_stats, router_logits, perm_token, slot,
                      workspace, workspace_bytes, stream, opts);
}

moe_status moe_quantize_weights_fp8(const void* W, int64_t G, int64_t K, int64_t N, uint8_t* Wq, float* scale,
                                    moe_stream stream) {
  if (G < 0 || K < 0 || N < 0) return MOE_ERR_INVALID_ARG;
  if (G == 0 || K == 0 || N == 0) return MOE_OK;
  if (!W || !Wq || !scale || !aligned16(W) || !aligned16(Wq) || !aligned16(scale)) return MOE_ERR_INVALID_ARG;
  if (K % 16 != 0 || G > 65535) return MOE_ERR_UNSUPPORTED;
  QuantWeightsArgs a;
  a.W = W; a.Q = Wq; a.scale = scale; a.G = G; a.K = K; a.N = N;
  return launch_quantize_weights(a, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_quantize_rows_fp8(const void* X, int64_t rows, int64_t cols, uint8_t* Q, float* scale,
                                 moe_stream stream) {
  if (rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MOE_OK;
  if (!X || !Q || !scale || !aligned16(X) || !aligned16(Q) || !aligned16(scale)) return MOE_ERR_INVALID_ARG;
  if (cols % 16 != 0 || rows >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  QuantRowsArgs a;
  a.X = X; a.Q = Q; a.scale = scale; a.cols = cols; a.rows0 = rows; a.live0 = nullptr; a.row1 = rows;
  a.rows1 = 0; a.err = nullptr;
  return launch_quantize_rows(a, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_workspace_region(const moe_config* cfg, int32_t region, size_t* offset, size_t* bytes) {
  if (check_cfg(cfg) != MOE_OK || !offset || !bytes) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(cfg);
  const bool fp8 = (cfg->flags & MOE_FLAG_FP8_EXPERTS) != 0;
  const size_t esz = cfg->dtype == MOE_DT_BF16 ? 2 : 4;
  const size_t d = cfg->d_model, f = cfg->d_ff, tk = (size_t)L.rows_tk, ra = (size_t)L.rows_all;
  switch (region) {
    case MOE_REGION_XPERM: *offset = L.xperm; *bytes = tk * d * (fp8 ? 1 : esz); return MOE_OK;
    case MOE_REGION_H: *offset = L.h; *bytes = ra * f * esz; return MOE_OK;
    case MOE_REGION_O: *offset = L.o; *bytes = ra * d * 4; return MOE_OK;
    default: break;
  }
  if (!fp8) return MOE_ERR_INVALID_ARG;
  switch (region) {
    case MOE_REGION_X_SCALE: *offset = L.xs_perm; *bytes = tk * 4; return MOE_OK;
    case MOE_REGION_H_CODES: *offset = L.hq; *bytes = ra * f; return MOE_OK;
    case MOE_REGION_H_SCALE: *offset = L.hs; *bytes = ra * 4; return MOE_OK;
    default: return MOE_ERR_INVALID_ARG;
  }
}

size_t moe_forward_host_workspace_size(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return host_stage(cfg, layout(cfg).total).total;
}

// moe_forward_host / moe_forward_fp8_host (q8 != NULL).
static moe_status forward_host_impl(const moe_config* cfg, const void* x_host, const void* W_g, const void* b_g,
                                    const float* router_noise_host, const void* W1, const void* b1, const void* W2,
                                    const void* b2, const void* W3, const moe_fp8_experts* q8, void* y_host,
                                    int32_t* topk_idx_host, float* topk_w_host, int32_t* expert_counts_host,
                                    uint8_t* dropped_mask_host, float* f_host, float* P_host, float* L_aux_host,
                                    float* route_stats_host, void* workspace, size_t workspace_bytes,
                                    moe_stream stream, const moe_launch_opts* opts) {
  moe_status st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (((cfg->flags & MOE_FLAG_FP8_EXPERTS) != 0) != (q8 != nullptr)) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *cfg;
  const bool empty = c.T == 0;
  const bool ec = (c.flags & MOE_FLAG_EXPERT_CHOICE) != 0;
  if (!expert_counts_host || !f_host || !P_host || !L_aux_host) return MOE_ERR_INVALID_ARG;
  if (!empty && (!x_host || !y_host)) return MOE_ERR_INVALID_ARG;
  if (!empty && !ec && (!topk_idx_host || !topk_w_host || !dropped_mask_host)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(&c);
  const HostStage h = host_stage(&c, L.total);
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < h.total) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  const size_t esz = c.dtype == MOE_DT_BF16 ? 2 : 4;
  const bool y_f32 = (c.flags & MOE_FLAG_Y_F32) != 0 || c.dtype == MOE_DT_F32;
  const size_t tk = (size_t)c.T * c.k;
  const size_t xbytes = (size_t)c.T * c.d_model * esz, ybytes = (size_t)c.T * c.d_model * (y_f32 ? 4 : 2);
  if (xbytes && cudaMemcpyAsync(ws + h.x, x_host, xbytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  const size_t nbytes = (size_t)c.T * c.E * 4;
  if (router_noise_host && nbytes &&
      cudaMemcpyAsync(ws + h.noise, router_noise_host, nbytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  st = forward_impl(cfg, ws + h.x, W_g, b_g, router_noise_host ? (const float*)(ws + h.noise) : nullptr, W1, b1,
                    W2, b2, W3, q8, ws + h.y, (int32_t*)(ws + h.idx), (float*)(ws + h.w), (int32_t*)(ws + h.cnt),
                    ws + h.drop, (float*)(ws + h.f), (float*)(ws + h.P), (float*)(ws + h.L),
                    route_stats_host ? (float*)(ws + h.stats) : nullptr, nullptr, nullptr, nullptr, workspace,
                    L.total, stream, opts);
  if (st != MOE_OK) return st;
  struct Copy { void* dst; size_t off, bytes; } copies[] = {
      {y_host, h.y, ybytes},          {topk_idx_host, h.idx, tk * 4}, {topk_w_host, h.w, tk * 4},
      {expert_counts_host, h.cnt, (size_t)c.E * 4}, {dropped_mask_host, h.drop, tk},
      {f_host, h.f, (size_t)c.E * 4}, {P_host, h.P, (size_t)c.E * 4}, {L_aux_host, h.L, 4},
      {route_stats_host, h.stats, route_stats_host ? (size_t)12 : 0}};
  for (const Copy& cp : copies)
    if (cp.dst && cp.bytes && cudaMemcpyAsync(cp.dst, ws + cp.off, cp.bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_forward_host(const moe_config* cfg, const void* x_host, const void* W_g, const void* b_g,
                            const float* router_noise_host, const void* W1, const void* b1, const void* W2,
                            const void* b2, const void* W3, void* y_host, int32_t* topk_idx_host, float* topk_w_host,
                            int32_t* expert_counts_host, uint8_t* dropped_mask_host, float* f_host, float* P_host,
                            float* L_aux_host, float* route_stats_host, void* workspace, size_t workspace_bytes,
                            moe_stream stream, const moe_launch_opts* opts) {
  if (cfg && (cfg->flags & MOE_FLAG_FP8_EXPERTS)) return MOE_ERR_INVALID_ARG;   // moe_forward_fp8_host
  return forward_host_impl(cfg, x_host, W_g, b_g, router_noise_host, W1, b1, W2, b2, W3, nullptr, y_host,
                           topk_idx_host, topk_w_host, expert_counts_host, dropped_mask_host, f_host, P_host,
                           L_aux_host, route_stats_host, workspace, workspace_bytes, stream, opts);
}

moe_status moe_forward_fp8_host(const moe_config* cfg, const void* x_host, const void* W_g, const void* b_g,
                                const float* router_noise_host, const moe_fp8_experts* w, const void* b1,
                                const void* b2, void* y_host, int32_t* topk_idx_host, float* topk_w_host,
                                int32_t* expert_counts_host, uint8_t* dropped_mask_host, float* f_host, float* P_host,
                                float* L_aux_host, float* route_stats_host, void* workspace, size_t workspace_bytes,
                                moe_stream stream, const moe_launch_opts* opts) {
  if (!cfg || !(cfg->flags & MOE_FLAG_FP8_EXPERTS) || !w) return MOE_ERR_INVALID_ARG;
  return forward_host_impl(cfg, x_host, W_g, b_g, router_noise_host, w->W1, b1, w->W2, b2, w->W3, w, y_host,
                           topk_idx_host, topk_w_host, expert_counts_host, dropped_mask_host, f_host, P_host,
                           L_aux_host, route_stats_host, workspace, workspace_bytes, stream, opts);
}

size_t moe_backward_workspace_size(const moe_config* cfg) {
  if (check_bwd_cfg(cfg) != MOE_OK) return 0;
  return bwd_layout(cfg).total;
}

moe_status moe_backward(const moe_config* cfg, const void* x, const void* W_g, const void* b_g,
                        const float* router_noise, const void* W1, const void* b1, const void* W2, const void* b2,
                        const void* W3, const void* dy, float dL_aux, float* dx, float* dW_g, float* db_g,
                        float* dW1, float* db1, float* dW2, float* db2, float* dW3, void* workspace,
                        size_t workspace_bytes, moe_stream stream, const moe_launch_opts* opts) {
  moe_status st = check_bwd_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  const bool ec = (c.flags & MOE_FLAG_EXPERT_CHOICE) != 0;
  const bool empty = c.T == 0;
  if (!W_g || !W1 || !W2 || !dW_g || !dW1 || !dW2) return MOE_ERR_INVALID_ARG;
  if (!empty && (!x || !dy || !dx)) return MOE_ERR_INVALID_ARG;
  if (swiglu != (W3 != nullptr) || swiglu != (dW3 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (swiglu && (b1 || b2)) return MOE_ERR_INVALID_ARG;
  if ((b_g != nullptr) != (db_g != nullptr) || (b1 != nullptr) != (db1 != nullptr) ||
      (b2 != nullptr) != (db2 != nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!isfinite(dL_aux)) return MOE_ERR_INVALID_ARG;
  const void* all[] = {x, W_g, b_g, router_noise, W1, b1, W2, b2, W3, dy, dx, dW_g, db_g, dW1, db1, dW2, db2, dW3};
  for (const void* p : all)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  const BwdLayout L = bwd_layout(&c);
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  const int64_t timeout = (opts && opts->wait_timeout_ns > 0) ? opts->wait_timeout_ns : kDefaultTimeoutNs;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  WsHeader* hdr = (WsHeader*)(ws + L.hdr);
  const SegTable seg = seg_table(ws, L.seg, L.G);
  const int64_t C = capacity_of(&c);
  const int d = c.d_model, f = c.d_ff, E = c.E, k = c.k, S = c.n_shared, G = L.G;
  const int64_t T = c.T;

  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (T == 0) {
    // No tokens: every gradient is zero.
    struct Z { void* p; size_t bytes; } zs[] = {
        {dW_g, (size_t)d * E * 4}, {db_g, (size_t)E * 4}, {dW1, (size_t)G * d * f * 4}, {db1, (size_t)G * f * 4},
        {dW2, (size_t)G * f * d * 4}, {db2, (size_t)G * d * 4}, {dW3, (size_t)G * d * f * 4}};
    for (const Z& z : zs)
      if (z.p && cudaMemsetAsync(z.p, 0, z.bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  // ---- forward recomputation (padded grouped layout) ----
  RouterArgs ra;
  memset(&ra, 0, sizeof(ra));
  ra.x = x; ra.Wg = W_g; ra.bg = b_g; ra.noise = router_noise; ra.T = T; ra.d = d; ra.E = E; ra.k = k;
  ra.gating = c.gating; ra.dtype = c.dtype; ra.logits_out = (float*)(ws + L.logits);
  ra.topk_idx = (int32_t*)(ws + L.idx); ra.topk_w = (float*)(ws + L.w); ra.lrank = ws + L.lrank;
  ra.hist = (int32_t*)(ws + L.hist); ra.psum = (float*)(ws + L.psum); ra.err = &hdr->err; ra.timeout_ns = timeout;
  ra.nblk = L.nblk;
  ra.bm = router_tile_tokens(c.dtype, c.E);
  if (ec) {
    // the experts choose on the gate probabilities; the gating's backward
    // needs the logits themselves
    ra.scores_em = (float*)(ws + L.ec_scores); ra.logits_out = nullptr; ra.raw_logits = (float*)(ws + L.logits);
    if (cudaMemsetAsync(ws + L.ec_bits, 0, (size_t)T * L.EW * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  // The scan (padded segments) runs in the router's last CTA.
  ScanArgs sa;
  memset(&sa, 0, sizeof(sa));
  sa.T = T; sa.E = E; sa.k = k; sa.S = S; sa.capacity = ec ? -1 : C; sa.alpha = c.alpha; sa.nblk = L.nblk;
  sa.ec_C = ec ? L.ec_C : -1;
  sa.pad_rows = 128; sa.shared_stride = L.Tpad; sa.hist = ra.hist; sa.psum = ra.psum;
  sa.base = (int32_t*)(ws + L.base); sa.n_pre = (int32_t*)(ws + L.npre); sa.counts = (int32_t*)(ws + L.cnt);
  sa.offsets = (int32_t*)(ws + L.offsets); sa.f = (float*)(ws + L.f); sa.P = (float*)(ws + L.P);
  sa.L_aux = (float*)(ws + L.L); sa.route_stats = nullptr; sa.seg = seg; sa.rows_tk = L.rows_routed;
  sa.err = &hdr->err;
  ra.fused_scan = true;
  ra.scan = sa;
  ra.done = &hdr->router_done;
  if (launch_router(ra, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (ec) {
    EcSelectArgs ea;
    ea.scores_em = (const float*)(ws + L.ec_scores); ea.T = T; ea.C = L.ec_C; ea.Cs = L.ec_Cs; ea.E = E;
    ea.EW = L.EW; ea.perm = (int32_t*)(ws + L.ec_perm); ea.w_row = (float*)(ws + L.ec_wrow);
    ea.tok_row = (int32_t*)(ws + L.ec_tokrow); ea.bits = (uint32_t*)(ws + L.ec_bits); ea.err = &hdr->err;
    if (launch_ec_select(ea, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  GatherArgs ga;
  memset(&ga, 0, sizeof(ga));
  ga.x = x; ga.T = T; ga.d = d; ga.E = E; ga.k = k; ga.dtype = c.dtype; ga.capacity = C;
  ga.topk_idx = ra.topk_idx; ga.lrank = ra.lrank; ga.base = sa.base; ga.nblk = L.nblk; ga.bm = ra.bm;
  ga.offsets = sa.offsets;
  ga.slot = (int32_t*)(ws + L.slot); ga.dropped = ws + L.drop; ga.perm_token = nullptr; ga.xperm = ws + L.xperm;
  ga.err = &hdr->err;
  if (ec) {
    EcGatherArgs eg;
    eg.x = x; eg.perm = (const int32_t*)(ws + L.ec_perm); eg.rows = L.rows_routed; eg.C = L.ec_C; eg.Cs = L.ec_Cs;
    eg.d = d; eg.esz = 2; eg.xperm = ws + L.xperm; eg.err = &hdr->err; eg.xs_tok = nullptr; eg.xs_perm = nullptr;
    if (launch_ec_gather(eg, s) != cudaSuccess) return MOE_ERR_CUDA;
  } else if (launch_gather(ga, s) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  PadZeroArgs pz;
  pz.buf = ws + L.xperm; pz.row_bytes = (int64_t)d * 2; pz.G = E; pz.E = E; pz.T = T; pz.counts = sa.counts;
  pz.seg = seg;
  if (launch_pad_zero(pz, s) != cudaSuccess) return MOE_ERR_CUDA;
  const int64_t max_mtiles = L.rows_all / kGemmBM + G;
  GemmArgs g1;
  memset(&g1, 0, sizeof(g1));
  g1.dtype = c.dtype; g1.act = c.act; g1.G = G; g1.K = d; g1.N = f; g1.a_from_out_rows = false; g1.seg = seg;
  g1.A0 = ws + L.xperm; g1.rows_A0 = L.rows_routed; g1.A1 = S > 0 ? x : nullptr; g1.rows_A1 = T;
  g1.B = W1; g1.B3 = W3; g1.Gw = G; g1.bias = b1; g1.C = ws + L.h; g1.max_mtiles = T > 0 ? max_mtiles : 0;
  g1.err = &hdr->err; g1.timeout_ns = timeout; g1.pre_a = ws + L.pre_a; g1.pre_u = swiglu ? ws + L.pre_u : nullptr;
  g1.rows_C = L.rows_all;
  if (launch_grouped_gemm(g1, s) != cudaSuccess) return MOE_ERR_CUDA;
  GemmArgs g2 = g1;
  g2.act = MOE_ACT_NONE; g2.K = f; g2.N = d; g2.a_from_out_rows = true; g2.A0 = ws + L.h; g2.rows_A0 = L.rows_all;
  g2.A1 = nullptr; g2.rows_A1 = 0; g2.B = W2; g2.B3 = nullptr; g2.bias = b2; g2.C = ws + L.o; g2.out_f32 = true;
  g2.pre_a = nullptr; g2.pre_u = nullptr; g2.rows_C = L.rows_all;
  if (launch_grouped_gemm(g2, s) != cudaSuccess) return MOE_ERR_CUDA;

  // ---- backward ----
  CombineBwdArgs cb;
  cb.dy = dy; cb.o = (const float*)(ws + L.o); cb.slot = ga.slot; cb.topk_w = ra.topk_w; cb.T = T; cb.d = d;
  cb.k = k; cb.S = S; cb.rows_routed = L.rows_routed; cb.shared_stride = L.Tpad; cb.dO = ws + L.dO;
  cb.dw = (float*)(ws + L.dw); cb.err = &hdr->err;
  if (ec) {
    EcCombineBwdArgs ecb;
    ecb.dy = dy; ecb.o = (const float*)(ws + L.o); ecb.perm = (const int32_t*)(ws + L.ec_perm);
    ecb.w_row = (const float*)(ws + L.ec_wrow); ecb.rows = L.rows_routed; ecb.C = L.ec_C; ecb.Cs = L.ec_Cs;
    ecb.d = d; ecb.dO = ws + L.dO; ecb.dw_row = (float*)(ws + L.ec_dw); ecb.err = &hdr->err;
    if (launch_ec_combine_bwd(ecb, s) != cudaSuccess) return MOE_ERR_CUDA;
    cb.k = 0; cb.slot = nullptr; cb.topk_w = nullptr;   // the shared rows only
  }
  if ((!ec || S > 0) && launch_combine_bwd(cb, s) != cudaSuccess) return MOE_ERR_CUDA;
  pz.buf = ws + L.dO; pz.G = G;
  if (launch_pad_zero(pz, s) != cudaSuccess) return MOE_ERR_CUDA;
  RouterBwdArgs rb;
  rb.logits = (const float*)(ws + L.logits); rb.topk_idx = ra.topk_idx; rb.topk_w = ra.topk_w;
  rb.dw = cb.dw; rb.n_pre = sa.n_pre; rb.T = T; rb.E = E; rb.k = k; rb.gating = c.gating; rb.alpha = c.alpha;
  rb.dL_aux = dL_aux; rb.dl = (float*)(ws + L.dl); rb.err = &hdr->err;
  if (ec) {
    EcRouterBwdArgs erb;
    erb.logits = (const float*)(ws + L.logits); erb.bits = (const uint32_t*)(ws + L.ec_bits);
    erb.tok_row = (const int32_t*)(ws + L.ec_tokrow); erb.dw_row = (const float*)(ws + L.ec_dw); erb.T = T;
    erb.E = E; erb.EW = L.EW; erb.gating = c.gating; erb.alpha = c.alpha; erb.dL_aux = dL_aux; erb.dl = rb.dl;
    erb.err = &hdr->err;
    if (launch_ec_router_bwd(erb, s) != cudaSuccess) return MOE_ERR_CUDA;
  } else if (launch_router_bwd(rb, s) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  // dH = dO W2^T, activation backward -> dA (, dU)
  BwdGemmArgs bg;
  memset(&bg, 0, sizeof(bg));
  bg.G = G; bg.Gw = G; bg.seg = seg; bg.act = c.act; bg.err = &hdr->err; bg.timeout_ns = timeout;
  const int64_t dgrad_tiles = T > 0 ? (L.rows_all / 256 + G) * ((int64_t)(f + 255) / 256) : 0;
  bg.K = d; bg.N = f; bg.A = ws + L.dO; bg.rows_A = L.rows_all; bg.B = W2; bg.C = ws + L.dA;
  bg.C2 = swiglu ? ws + L.dU : nullptr; bg.pre_a = ws + L.pre_a; bg.pre_u = swiglu ? ws + L.pre_u : nullptr;
  bg.act_bwd = true; bg.max_tiles = dgrad_tiles;
  if (launch_gemm_dgrad(bg, s) != cudaSuccess) return MOE_ERR_CUDA;
  // dX of the grouped rows = dA W1^T (+ dU W3^T)
  BwdGemmArgs bx = bg;
  bx.K = f; bx.N = d; bx.A = ws + L.dA; bx.A2 = swiglu ? ws + L.dU : nullptr; bx.B = W1; bx.B2 = swiglu ? W3 : nullptr;
  bx.C = ws + L.dxp; bx.C2 = nullptr; bx.pre_a = nullptr; bx.pre_u = nullptr; bx.act_bwd = false;
  bx.max_tiles = T > 0 ? (L.rows_all / 256 + G) * ((int64_t)(d + 255) / 256) : 0;
  if (launch_gemm_dgrad(bx, s) != cudaSuccess) return MOE_ERR_CUDA;
  // weight gradients: dW2 = H^T dO, dW1 = X^T dA, dW3 = X^T dU
  BwdGemmArgs bw;
  memset(&bw, 0, sizeof(bw));
  bw.G = G; bw.Gw = G; bw.seg = seg; bw.err = &hdr->err; bw.timeout_ns = timeout;
  bw.M = f; bw.N = d; bw.A = ws + L.h; bw.rows_A = L.rows_all; bw.B = ws + L.dO; bw.rows_B = L.rows_all; bw.C = dW2;
  bw.x_from_asrc = false; bw.max_tiles = (int64_t)G * ((f + 255) / 256) * ((d + 255) / 256);
  if (launch_gemm_wgrad(bw, s) != cudaSuccess) return MOE_ERR_CUDA;
  BwdGemmArgs bw1 = bw;
  bw1.M = d; bw1.N = f; bw1.A = ws + L.xperm; bw1.rows_A = L.rows_routed; bw1.A2 = S > 0 ? x : nullptr;
  bw1.rows_A2 = T;
  bw1.x_from_asrc = true; bw1.B = ws + L.dA; bw1.C = dW1;
  bw1.max_tiles = (int64_t)G * ((d + 255) / 256) * ((f + 255) / 256);
  if (launch_gemm_wgrad(bw1, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (swiglu) {
    BwdGemmArgs bw3 = bw1;
    bw3.B = ws + L.dU; bw3.C = dW3;
    if (launch_gemm_wgrad(bw3, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (b1) {
    ColsumArgs cs;
    cs.buf = ws + L.dA; cs.seg = seg; cs.G = G; cs.N = f; cs.out = db1;
    if (launch_colsum(cs, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (b2) {
    ColsumArgs cs;
    cs.buf = ws + L.dO; cs.seg = seg; cs.G = G; cs.N = d; cs.out = db2;
    if (launch_colsum(cs, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  DxArgs dxa;
  dxa.dxp = (const float*)(ws + L.dxp); dxa.slot = ga.slot; dxa.dl = rb.dl; dxa.Wg = W_g; dxa.T = T; dxa.d = d;
  dxa.k = k; dxa.E = E; dxa.S = S; dxa.rows_routed = L.rows_routed; dxa.shared_stride = L.Tpad; dxa.dx = dx;
  dxa.err = &hdr->err; dxa.ec_bits = nullptr; dxa.ec_tok_row = nullptr; dxa.EW = L.EW;
  if (ec) {
    dxa.k = 0; dxa.slot = nullptr;
    dxa.ec_bits = (const uint32_t*)(ws + L.ec_bits); dxa.ec_tok_row = (const int32_t*)(ws + L.ec_tokrow);
  }
  if (launch_dx(dxa, s) != cudaSuccess) return MOE_ERR_CUDA;
  DwgArgs dg;
  dg.x = x; dg.dl = rb.dl; dg.T = T; dg.d = d; dg.E = E; dg.nchunk = L.nchunk; dg.part = (float*)(ws + L.part);
  dg.bpart = (float*)(ws + L.bpart); dg.dWg = dW_g; dg.dbg = db_g;
  if (launch_dwg(dg, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_check_device_errors(const void* workspace, moe_stream stream) {
  if (!workspace) return MOE_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (h.err & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (h.err & kErrDevice) return MOE_ERR_DEVICE;
  return MOE_OK;
}

size_t moe_grouped_gemm_workspace_size(int32_t G) {
  if (G <= 0) return 0;
  return align_up(sizeof(WsHeader), 256) + align_up((size_t)(6 * G + 1) * 4, 256);
}

moe_status moe_grouped_gemm(int32_t dtype, int32_t act, int32_t G, const int32_t* seg_offsets, int64_t M, int32_t K,
                            int32_t N, const void* A, const void* B, const void* B3, const void* bias, void* C,
                            void* workspace, size_t workspace_bytes, moe_stream stream,
                            const moe_launch_opts* opts) {
  const moe_status st = check_grouped_gemm_args(dtype, act, G, seg_offsets, M, K, N, A, B, B3, bias, C);
  if (st != MOE_OK) return st;
  const size_t need = moe_grouped_gemm_workspace_size(G);
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < need) return MOE_ERR_WORKSPACE;
  return launch_grouped_gemm_on_scratch(dtype, act, G, seg_offsets, M, K, N, A, B, B3, bias, C,
                                        (uint8_t*)workspace, stream, opts);
}

}  // extern "C"
