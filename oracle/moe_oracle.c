/*
 * oracle/moe_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, single-threaded fp64 CPU restatement of the forward pass of a
 * token-choice Mixture-of-Experts feed-forward layer, written step by step
 * from the pages' definitions so that each step can be checked against them
 * by eye.  Only the tests, the package's smoke check and the bench's CPU
 * baseline may load it.  It shares no code, header or constant with the CUDA
 * path: it reads the stored input values (fp32, or bf16 bits) and widens them
 * to double, and does every sum and product in double.
 *
 * Sources (page title, section):
 *   [P1] "MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现"
 *        §1.3 (sparse FFN data flow), §2.1 (router: linear + softmax, top-k,
 *        renormalise), §2.3 (Switch load-balance loss), §3.2 (capacity factor),
 *        §4.1 (the TopKRouter / ExpertFFN / MoEFFN modules).
 *   [P2] "MoE架构解析" §2.1 (token choice), §三 关键技术① (expert capacity,
 *        overflow tokens skip the layer), §四 技术飞跃② (shared experts,
 *        always active), 技术飞跃③ (normalised sigmoid gating).
 *   [P3] "手撕一个极简 MoE-FFN" §三 (Router, top_k_routing, worked example),
 *        §四 (Expert FFN), §五/§六 (weighted sum), §七 (load-balancing loss
 *        with f = counts / (T*k)).
 *   [P4] "Mixture of Experts混合专家模型架构原理与路由策略实现",
 *        门控网络的数学原理 (Gate(x) = softmax(W_g x), W_g is [d_model, E]),
 *        从零实现一个简化版MoE层 (GELU expert).
 *   [P5] "术业有专攻：learn-minimind MoE混合专家模型架构入门指南" §二
 *        (experts are SwiGLU FFNs).
 *
 * Readings taken where the pages are silent or disagree (each is stated at
 * the function that uses it): selection on logits with ties to the lower
 * index; capacity C = ceil(T * cf / E) in fp64, slots given in token order;
 * a dropped slot contributes 0 and the kept weights are not renormalised;
 * shared experts are added with weight 1 after the routed sum; f counts
 * selections before the capacity cut; P under sigmoid gating is the mean of
 * sigma_e / sum_e' sigma_e'; GELU is the exact erf form; SwiGLU is
 * W2 (silu(x W1) * (x W3)); weights are stored [in, out].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ODT_F32 = 0, ODT_BF16 = 1 };
enum { OACT_RELU = 0, OACT_GELU = 1, OACT_SWIGLU = 2 };
enum { OGATE_SOFTMAX = 0, OGATE_SIGMOID_NORM = 1 };

/* Step 0: the stored value widened to double (bf16 -> fp32 bits -> double, exact). */
static double ld(const void* p, int dtype, int64_t i) {
  if (dtype == ODT_F32) return (double)((const float*)p)[i];
  uint32_t u = (uint32_t)((const uint16_t*)p)[i] << 16;
  float v;
  memcpy(&v, &u, 4);
  return (double)v;
}

/* Router logits l[t,e] = b_g[e] + sum_i x[t,i] W_g[i,e]   [P1 §2.1; P3 §三; P4 门控网络的数学原理].
 * W_g is stored [d, E] (the gate formula's [d_model, num_experts]); b_g may be NULL. */
void oracle_router_logits(int64_t T, int d, int E, int dtype, const void* x, const void* Wg,
                          const void* bg, double* logits) {
  for (int64_t t = 0; t < T; ++t) {
    double* l = logits + t * E;
    for (int e = 0; e < E; ++e) l[e] = bg ? ld(bg, dtype, e) : 0.0;
    for (int i = 0; i < d; ++i) {
      double xi = ld(x, dtype, t * d + i);
      for (int e = 0; e < E; ++e) l[e] += xi * ld(Wg, dtype, (int64_t)i * E + e);
    }
  }
}

/* Gate probabilities per token over all E experts.
 *  softmax        p_e = exp(l_e - max) / sum_e' exp(l_e' - max)      [P1 §2.1; P3 §三]
 *  normalised sigmoid: s_e = 1 / (1 + exp(-l_e)),  p_e = s_e / sum_e' s_e'
 *                 (sigmoid per expert, then a global normalisation)  [P2 技术飞跃③]
 * These p feed the balance statistic P_i. */
void oracle_gate_probs(int64_t T, int E, int gating, const double* logits, double* probs) {
  for (int64_t t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    double* p = probs + t * E;
    double z = 0.0;
    if (gating == OGATE_SOFTMAX) {
      double m = l[0];
      for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
      for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - m); z += p[e]; }
    } else {
      for (int e = 0; e < E; ++e) { p[e] = 1.0 / (1.0 + exp(-l[e])); z += p[e]; }
    }
    for (int e = 0; e < E; ++e) p[e] /= z;
  }
}

/* Top-k selection on one row of values: the k largest, listed in descending
 * value, equal values ordered by ascending index.  [P1 §2.1; P3 §三 top_k_routing]
 * Reading: torch.topk leaves the order of ties open; the lower index wins.  A
 * stable insertion sort of the indices 0..E-1 by value realises exactly that. */
void oracle_topk_row(int E, int k, const double* v, int32_t* idx) {
  int order[1024];
  for (int e = 0; e < E; ++e) order[e] = e;
  for (int i = 1; i < E; ++i) {
    int key = order[i], j = i - 1;
    while (j >= 0 && v[order[j]] < v[key]) { order[j + 1] = order[j]; --j; }
    order[j + 1] = key;
  }
  for (int j = 0; j < k; ++j) idx[j] = order[j];
}

/* Selection of every token on its logits.  Softmax and the sigmoid are
 * increasing, so choosing on the logits picks the same experts as choosing on
 * the probabilities, without ties created by rounding of exp. */
void oracle_topk(int64_t T, int E, int k, const double* logits, int32_t* idx) {
  for (int64_t t = 0; t < T; ++t) oracle_topk_row(E, k, logits + t * E, idx + t * k);
}

/* Renormalised top-k weights  w_j = g_j / sum_{j' < k} g_j'   [P1 §2.1; P3 §三]
 * with g = softmax probability, or g = sigmoid(l) for normalised-sigmoid
 * gating (the selected sigmoids divided by their sum) [P2 技术飞跃③]. */
void oracle_topk_weights(int64_t T, int E, int k, int gating, const double* logits,
                         const int32_t* idx, double* w) {
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    if (gating == OGATE_SOFTMAX) {
      oracle_gate_probs(1, E, OGATE_SOFTMAX, l, p);
    } else {
      for (int e = 0; e < E; ++e) p[e] = 1.0 / (1.0 + exp(-l[e]));
    }
    double z = 0.0;
    for (int j = 0; j < k; ++j) z += p[idx[t * k + j]];
    for (int j = 0; j < k; ++j) w[t * k + j] = p[idx[t * k + j]] / z;
  }
  free(p);
}

/* Expert capacity  C = ceil((T / E) * capacity_factor), evaluated as
 * ceil(T * cf / E) in double; cf <= 0 means no limit (returns -1).
 * [P2 §三 关键技术①; P1 §3.2] */
int64_t oracle_capacity(int64_t T, int E, double cf) {
  if (cf <= 0.0) return -1;
  return (int64_t)ceil((double)T * cf / (double)E);
}

/* Capacity, drops and the expert-grouped order of the kept assignments.
 * Walk the tokens in order t = 0..T-1, and each token's choices j = 0..k-1;
 * the assignment takes the next free slot of its expert while fewer than C
 * are taken, otherwise it is dropped (it skips the layer: that slot adds
 * nothing to y) [P2 §三 关键技术①].  Outputs:
 *   n_pre[e]    selections of e before the cut (feeds f_i)
 *   counts[e]   kept assignments of e = min(n_pre[e], C)
 *   offsets[e]  exclusive prefix sum of counts (offsets[E] = total kept)
 *   dropped     1 where the assignment (t,j) was cut
 *   slot        offsets[e] + rank of (t,j) among e's kept assignments, or -1
 *   perm[slot]  the token at each row of the grouped order: experts
 *               ascending, tokens ascending within an expert [P3 §六]. */
void oracle_dispatch(int64_t T, int E, int k, int64_t C, const int32_t* idx, int32_t* n_pre,
                     int32_t* counts, int32_t* offsets, uint8_t* dropped, int32_t* slot, int32_t* perm) {
  int32_t* rank = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T * k + 1));
  for (int e = 0; e < E; ++e) { n_pre[e] = 0; counts[e] = 0; }
  for (int64_t t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      int e = idx[t * k + j];
      n_pre[e] += 1;
      if (C < 0 || counts[e] < C) {
        rank[t * k + j] = counts[e];
        counts[e] += 1;
        dropped[t * k + j] = 0;
      } else {
        rank[t * k + j] = -1;
        dropped[t * k + j] = 1;
      }
    }
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  for (int64_t t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      int64_t a = t * k + j;
      if (dropped[a]) { slot[a] = -1; continue; }
      slot[a] = offsets[idx[a]] + rank[a];
      perm[slot[a]] = (int32_t)t;
    }
  }
  free(rank);
}

/* Activations.  ReLU [P3 §四]; GELU in its exact erf form, the default of
 * F.gelu in the pages' experts [P1 §4.1; P4 简化版MoE层]; SiLU z * sigmoid(z)
 * for the SwiGLU gate [P5 §二]. */
double oracle_act(int act, double z) {
  if (act == OACT_RELU) return z > 0.0 ? z : 0.0;
  if (act == OACT_GELU) return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
  return z / (1.0 + exp(-z));
}

/* One expert on one input row.  Expert g's weights are the g-th slabs of the
 * stacked tensors W1/W3 [G, d, f], W2 [G, f, d], b1 [G, f], b2 [G, d].
 *   ReLU / GELU:  o = W2^T act(W1^T x + b1) + b2         [P3 §四; P1 §4.1; P4]
 *   SwiGLU:       o = W2^T (silu(W1^T x) * (W3^T x))     [P5 §二], no biases.
 * Dropout in the pages' experts is the identity at inference. */
void oracle_expert_ffn(int d, int f, int act, int dtype, int g, const double* xrow, const void* W1,
                       const void* b1, const void* W2, const void* b2, const void* W3, double* out) {
  double* h = (double*)calloc((size_t)f, sizeof(double));
  double* u = (act == OACT_SWIGLU) ? (double*)calloc((size_t)f, sizeof(double)) : NULL;
  const int64_t w1o = (int64_t)g * d * f, w2o = (int64_t)g * f * d;
  if (b1 && act != OACT_SWIGLU)
    for (int j = 0; j < f; ++j) h[j] = ld(b1, dtype, (int64_t)g * f + j);
  for (int i = 0; i < d; ++i) {
    double xi = xrow[i];
    for (int j = 0; j < f; ++j) h[j] += xi * ld(W1, dtype, w1o + (int64_t)i * f + j);
    if (u)
      for (int j = 0; j < f; ++j) u[j] += xi * ld(W3, dtype, w1o + (int64_t)i * f + j);
  }
  for (int j = 0; j < f; ++j)
    h[j] = (act == OACT_SWIGLU) ? oracle_act(OACT_SWIGLU, h[j]) * u[j] : oracle_act(act, h[j]);
  for (int c = 0; c < d; ++c) out[c] = (b2 && act != OACT_SWIGLU) ? ld(b2, dtype, (int64_t)g * d + c) : 0.0;
  for (int j = 0; j < f; ++j) {
    double hj = h[j];
    for (int c = 0; c < d; ++c) out[c] += hj * ld(W2, dtype, w2o + (int64_t)j * d + c);
  }
  free(h);
  free(u);
}

/* Layer output for the listed token rows:
 *   y[t] = sum_{j<k, kept} w_j * E_{idx_j}(x_t)  +  sum_{s<S} E_{E+s}(x_t)
 * summed in that order [P1 §1.3; P3 §五; P2 §四 技术飞跃② for the always-on
 * shared experts, added with weight 1].  A dropped assignment contributes 0 and
 * the kept weights are left as they are [P2 §三 关键技术①]. */
void oracle_layer_rows(int d, int f, int E, int k, int S, int act, int dtype, const int64_t* rows,
                       int64_t nrows, const void* x, const void* W1, const void* b1, const void* W2,
                       const void* b2, const void* W3, const int32_t* idx, const double* w,
                       const uint8_t* dropped, double* y) {
  double* xr = (double*)malloc(sizeof(double) * (size_t)d);
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t t = rows[r];
    double* yr = y + r * d;
    for (int i = 0; i < d; ++i) { xr[i] = ld(x, dtype, t * d + i); yr[i] = 0.0; }
    for (int j = 0; j < k; ++j) {
      if (dropped[t * k + j]) continue;
      oracle_expert_ffn(d, f, act, dtype, idx[t * k + j], xr, W1, b1, W2, b2, W3, o);
      for (int i = 0; i < d; ++i) yr[i] += w[t * k + j] * o[i];
    }
    for (int s = 0; s < S; ++s) {
      oracle_expert_ffn(d, f, act, dtype, E + s, xr, W1, b1, W2, b2, W3, o);
      for (int i = 0; i < d; ++i) yr[i] += o[i];
    }
  }
  free(xr);
  free(o);
}

/* Switch-style balance statistics   [P1 §2.3; P3 §七]
 *   f_i = (selections of i before the capacity cut) / (T * k)
 *   P_i = (1/T) sum_t p[t,i]
 *   L_aux = alpha * E * sum_i f_i * P_i
 * Reading: f divides by T*k as in [P3] §七, so sum_i f_i = 1 and
 * L_aux = alpha exactly when routing is uniform.  T = 0 gives zeros. */
void oracle_balance(int64_t T, int E, int k, double alpha, const int32_t* n_pre, const double* probs,
                    double* f, double* P, double* L_aux) {
  double L = 0.0;
  for (int e = 0; e < E; ++e) {
    double s = 0.0;
    for (int64_t t = 0; t < T; ++t) s += probs[t * E + e];
    f[e] = T > 0 ? (double)n_pre[e] / ((double)T * (double)k) : 0.0;
    P[e] = T > 0 ? s / (double)T : 0.0;
    L += f[e] * P[e];
  }
  *L_aux = alpha * (double)E * L;
}

/* Router noise: the scores get Gaussian noise added before top-k, to
 * encourage exploration of other experts ["Mixture of Experts混合专家模型架构原理
 * 与路由策略实现", 门控网络的数学原理].  The pages give no formula beyond that.
 * Reading: the caller's noise values (already scaled) are added to the logits,
 * and everything after (gating, top-k, weights, P) uses the noisy logits.
 * noise is fp32 [T, E]. */
void oracle_add_noise(int64_t T, int E, double* logits, const float* noise) {
  for (int64_t i = 0; i < T * E; ++i) logits[i] += (double)noise[i];
}

/* Routing-health statistics ["MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch
 * 实现" §3.3: per-expert token counts, the entropy of the routing distribution
 * against ln N, and the variance of expert utilisation / its coefficient of
 * variation].  Reading: the distribution is the pre-capacity selection share
 * f_e = n_e / (T k), so that uniform routing gives entropy ln E:
 *   out[0] = H   = -sum_e f_e ln f_e   (terms with f_e = 0 add 0)
 *   out[1] = Var = (1/E) sum_e (f_e - 1/E)^2
 *   out[2] = CV  = std_e(n_e) / mean_e(n_e) = E sqrt(Var)
 * T = 0 gives zeros. */
void oracle_route_health(int64_t T, int E, int k, const int32_t* n_pre, double* out) {
  out[0] = out[1] = out[2] = 0.0;
  if (T <= 0) return;
  const double tk = (double)T * (double)k;
  double H = 0.0, var = 0.0;
  for (int e = 0; e < E; ++e) {
    const double f = (double)n_pre[e] / tk;
    if (f > 0.0) H -= f * log(f);
    var += (f - 1.0 / E) * (f - 1.0 / E);
  }
  var /= (double)E;
  out[0] = H;
  out[1] = var;
  out[2] = (double)E * sqrt(var);
}

/* ---- expert-choice routing ---------------------------------------------------
 * Each expert chooses the tokens it scores highest, instead of each token
 * choosing experts ["MoE架构解析" §2.2: every expert gets the same load; a
 * token may be chosen by several experts or by none].  Readings: the scores
 * are the gate probabilities s[t,e] (softmax or normalised sigmoid over the
 * experts, as for token choice); expert e takes the C tokens with the largest
 * s[t,e], equal scores going to the lower token index, C = min(T, ceil(T cf /
 * E)) with a capacity factor cf > 0, else min(T, ceil(T k / E)) (the compute
 * of top-k token choice); a token's output is the sum over the experts that
 * chose it, in ascending expert order, of s[t,e] times the expert's output
 * (no renormalisation), plus the shared experts. */

int64_t oracle_ec_capacity(int64_t T, int E, int k, double cf) {
  double c = cf > 0.0 ? ceil((double)T * cf / (double)E) : ceil((double)T * (double)k / (double)E);
  return (int64_t)c < T ? (int64_t)c : T;
}

/* perm[e*C + i]: the i-th chosen token of expert e, tokens ascending.
 * Selection by a stable insertion sort of the token indices by score
 * (descending, equal scores keep ascending token order), then the C chosen
 * tokens listed in token order. */
void oracle_ec_select(int64_t T, int E, int64_t C, const double* scores, int32_t* perm) {
  int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
  uint8_t* chosen = (uint8_t*)malloc((size_t)(T > 0 ? T : 1));
  for (int e = 0; e < E; ++e) {
    for (int64_t t = 0; t < T; ++t) order[t] = (int32_t)t;
    for (int64_t i = 1; i < T; ++i) {
      int32_t key = order[i];
      int64_t j = i - 1;
      while (j >= 0 && scores[(int64_t)order[j] * E + e] < scores[(int64_t)key * E + e]) {
        order[j + 1] = order[j];
        --j;
      }
      order[j + 1] = key;
    }
    for (int64_t t = 0; t < T; ++t) chosen[t] = 0;
    for (int64_t i = 0; i < C; ++i) chosen[order[i]] = 1;
    int64_t n = 0;
    for (int64_t t = 0; t < T; ++t)
      if (chosen[t]) perm[(int64_t)e * C + n++] = (int32_t)t;
  }
  free(order);
  free(chosen);
}

/* Layer output of expert-choice routing for the listed token rows. */
void oracle_ec_layer_rows(int d, int f, int E, int S, int act, int dtype, int64_t T, int64_t C,
                          const int64_t* rows, int64_t nrows, const void* x, const void* W1, const void* b1,
                          const void* W2, const void* b2, const void* W3, const int32_t* perm,
                          const double* scores, double* y) {
  double* xr = (double*)malloc(sizeof(double) * (size_t)d);
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t t = rows[r];
    double* yr = y + r * d;
    for (int i = 0; i < d; ++i) { xr[i] = ld(x, dtype, t * d + i); yr[i] = 0.0; }
    for (int e = 0; e < E; ++e) {
      int hit = 0;
      for (int64_t i = 0; i < C; ++i)
        if (perm[(int64_t)e * C + i] == t) { hit = 1; break; }
      if (!hit) continue;
      oracle_expert_ffn(d, f, act, dtype, e, xr, W1, b1, W2, b2, W3, o);
      const double w = scores[t * E + e];
      for (int i = 0; i < d; ++i) yr[i] += w * o[i];
    }
    for (int s = 0; s < S; ++s) {
      oracle_expert_ffn(d, f, act, dtype, E + s, xr, W1, b1, W2, b2, W3, o);
      for (int i = 0; i < d; ++i) yr[i] += o[i];
    }
  }
  free(xr);
  free(o);
}

/* ---- backward pass ---------------------------------------------------------------
 * Gradients of the scalar  L = sum_t <dy_t, y_t> + dL_aux * L_aux  with respect
 * to x, W_g, b_g, W1, b1, W2, b2, W3 (token-choice routing), for training the
 * layer with the load-balance term added to the main loss ["MoE混合专家模型：
 * Transformer稀疏前馈网络原理与PyTorch实现" §4.3: the aux loss joins the main loss
 * before one backward; "手撕一个极简 MoE-FFN" §七].  Written out from the forward
 * by the chain rule:
 *  - selection, the capacity cut and f are piecewise constant: no gradient;
 *  - y_t = sum_{kept j} w_j o_j + sum_s o_s:  dw_j = <dy_t, o_j>,  do_j = w_j dy_t;
 *  - o = W2^T h + b2:  dh = W2 do,  dW2 += h do^T,  db2 += do;
 *  - h = act(a), a = W1^T x + b1:  da = act'(a) dh;  SwiGLU h = silu(a) u with
 *    u = W3^T x:  da = dh u silu'(a),  du = dh silu(a);
 *  - dx += W1 da (+ W3 du),  dW1 += x da^T,  dW3 += x du^T,  db1 += da;
 *  - renormalised weights w_j = g_j / sum_sel g:  dg_i = (dw_i - sum_j w_j dw_j) /
 *    sum_sel g on the selected experts; softmax g = p: dl = p (dg - <p, dg>);
 *    normalised sigmoid: the selected sigmoids, dl_i = dg_i s_i (1 - s_i);
 *  - L_aux = alpha E sum_e f_e P_e with P_e = mean_t p_te: dp_te = dL_aux alpha E
 *    f_e / T, through softmax as above, or through p = s / sum s for sigmoid;
 *  - l = x W_g + b_g (+ noise): dW_g += x dl^T, db_g += dl, dx += W_g dl.
 * All outputs are fp64 and are overwritten.  dy is fp64 [T, d]. */
static double gelu_grad(double z) {
  /* d/dz [z Phi(z)] = Phi(z) + z phi(z), phi the standard normal density */
  return 0.5 * (1.0 + erf(z / sqrt(2.0))) + z * exp(-0.5 * z * z) / sqrt(2.0 * acos(-1.0));
}
static double sig(double z) { return 1.0 / (1.0 + exp(-z)); }

void oracle_backward(int64_t T, int d, int f, int E, int k, int S, int act, int gating, int dtype, double alpha,
                     double dL_aux, const void* x, const void* W_g, const double* logits, const void* W1,
                     const void* b1, const void* W2, const void* b2, const void* W3, const int32_t* idx,
                     const double* w, const uint8_t* dropped, const int32_t* n_pre, const double* dy, double* dx,
                     double* dWg, double* dbg, double* dW1, double* db1, double* dW2, double* db2, double* dW3) {
  const int G = E + S;
  memset(dx, 0, sizeof(double) * (size_t)(T * d));
  memset(dWg, 0, sizeof(double) * (size_t)d * E);
  memset(dbg, 0, sizeof(double) * (size_t)E);
  memset(dW1, 0, sizeof(double) * (size_t)G * d * f);
  memset(db1, 0, sizeof(double) * (size_t)G * f);
  memset(dW2, 0, sizeof(double) * (size_t)G * f * d);
  memset(db2, 0, sizeof(double) * (size_t)G * d);
  if (dW3) memset(dW3, 0, sizeof(double) * (size_t)G * d * f);
  double* xr = (double*)malloc(sizeof(double) * (size_t)d);
  double* a = (double*)malloc(sizeof(double) * (size_t)f);
  double* u = (double*)malloc(sizeof(double) * (size_t)f);
  double* h = (double*)malloc(sizeof(double) * (size_t)f);
  double* dh = (double*)malloc(sizeof(double) * (size_t)f);
  double* da = (double*)malloc(sizeof(double) * (size_t)f);
  double* du = (double*)malloc(sizeof(double) * (size_t)f);
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  double* dl = (double*)malloc(sizeof(double) * (size_t)E);
  double* dp = (double*)malloc(sizeof(double) * (size_t)E);
  double* dw = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
  const int swiglu = act == OACT_SWIGLU;
  for (int64_t t = 0; t < T; ++t) {
    const double* dyt = dy + t * d;
    for (int i = 0; i < d; ++i) xr[i] = ld(x, dtype, t * d + i);
    /* experts: routed (kept) and shared */
    for (int j = 0; j < k + S; ++j) {
      int g;
      double wj;
      if (j < k) {
        dw[j] = 0.0;
        if (dropped[t * k + j]) continue;
        g = idx[t * k + j];
        wj = w[t * k + j];
      } else {
        g = E + (j - k);
        wj = 1.0;
      }
      const int64_t w1o = (int64_t)g * d * f, w2o = (int64_t)g * f * d;
      for (int c = 0; c < f; ++c) { a[c] = (b1 && !swiglu) ? ld(b1, dtype, (int64_t)g * f + c) : 0.0; u[c] = 0.0; }
      for (int i = 0; i < d; ++i) {
        for (int c = 0; c < f; ++c) a[c] += xr[i] * ld(W1, dtype, w1o + (int64_t)i * f + c);
        if (swiglu)
          for (int c = 0; c < f; ++c) u[c] += xr[i] * ld(W3, dtype, w1o + (int64_t)i * f + c);
      }
      for (int c = 0; c < f; ++c) h[c] = swiglu ? oracle_act(OACT_SWIGLU, a[c]) * u[c] : oracle_act(act, a[c]);
      /* o and dw_j = <dy, o> */
      if (j < k) {
        for (int c = 0; c < d; ++c) o[c] = (b2 && !swiglu) ? ld(b2, dtype, (int64_t)g * d + c) : 0.0;
        for (int r = 0; r < f; ++r)
          for (int c = 0; c < d; ++c) o[c] += h[r] * ld(W2, dtype, w2o + (int64_t)r * d + c);
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += dyt[c] * o[c];
        dw[j] = s;
      }
      /* do = wj dy; dh = W2 do; dW2 += h do^T; db2 += do */
      for (int r = 0; r < f; ++r) {
        double s = 0.0;
        for (int c = 0; c < d; ++c) {
          const double doc = wj * dyt[c];
          s += ld(W2, dtype, w2o + (int64_t)r * d + c) * doc;
          dW2[w2o + (int64_t)r * d + c] += h[r] * doc;
        }
        dh[r] = s;
      }
      if (b2 && !swiglu)
        for (int c = 0; c < d; ++c) db2[(int64_t)g * d + c] += wj * dyt[c];
      /* activation */
      for (int r = 0; r < f; ++r) {
        if (swiglu) {
          const double sa = sig(a[r]);
          da[r] = dh[r] * u[r] * (sa + a[r] * sa * (1.0 - sa));
          du[r] = dh[r] * a[r] * sa;
        } else if (act == OACT_RELU) {
          da[r] = a[r] > 0.0 ? dh[r] : 0.0;
        } else {
          da[r] = dh[r] * gelu_grad(a[r]);
        }
      }
      /* dx, dW1, dW3, db1 */
      for (int i = 0; i < d; ++i) {
        double s = 0.0;
        for (int r = 0; r < f; ++r) {
          s += ld(W1, dtype, w1o + (int64_t)i * f + r) * da[r];
          dW1[w1o + (int64_t)i * f + r] += xr[i] * da[r];
          if (swiglu) {
            s += ld(W3, dtype, w1o + (int64_t)i * f + r) * du[r];
            dW3[w1o + (int64_t)i * f + r] += xr[i] * du[r];
          }
        }
        dx[t * d + i] += s;
      }
      if (b1 && !swiglu)
        for (int r = 0; r < f; ++r) db1[(int64_t)g * f + r] += da[r];
    }
    /* router: through the renormalised weights, then the aux term */
    const double* l = logits + t * E;
    oracle_gate_probs(1, E, gating, l, p);
    for (int e = 0; e < E; ++e) dl[e] = 0.0;
    double zsel = 0.0, wdw = 0.0;
    for (int j = 0; j < k; ++j) {
      const int e = idx[t * k + j];
      zsel += gating == OGATE_SOFTMAX ? p[e] : sig(l[e]);
      wdw += w[t * k + j] * dw[j];
    }
    for (int j = 0; j < k; ++j) {
      const int e = idx[t * k + j];
      if (gating == OGATE_SOFTMAX) {
        /* w = softmax of the selected logits: dl_i = w_i (dw_i - sum w dw) */
        dl[e] += w[t * k + j] * (dw[j] - wdw);
      } else {
        const double se = sig(l[e]);
        dl[e] += (dw[j] - wdw) / zsel * se * (1.0 - se);
      }
    }
    if (dL_aux != 0.0) {
      for (int e = 0; e < E; ++e) dp[e] = dL_aux * alpha * E * ((double)n_pre[e] / ((double)T * k)) / (double)T;
      double s = 0.0;
      for (int e = 0; e < E; ++e) s += p[e] * dp[e];
      if (gating == OGATE_SOFTMAX) {
        for (int e = 0; e < E; ++e) dl[e] += p[e] * (dp[e] - s);
      } else {
        /* p = sig / sum sig:  dsig_e = (dp_e - sum_e' p_e' dp_e') / sum sig;  dl = dsig s (1 - s) */
        double zs = 0.0;
        for (int e = 0; e < E; ++e) zs += sig(l[e]);
        for (int e = 0; e < E; ++e) {
          const double se = sig(l[e]);
          dl[e] += (dp[e] - s) / zs * se * (1.0 - se);
        }
      }
    }
    for (int e = 0; e < E; ++e) {
      dbg[e] += dl[e];
      for (int i = 0; i < d; ++i) dWg[(int64_t)i * E + e] += xr[i] * dl[e];
    }
    for (int i = 0; i < d; ++i) {
      double s = 0.0;
      for (int e = 0; e < E; ++e) s += ld(W_g, dtype, (int64_t)i * E + e) * dl[e];
      dx[t * d + i] += s;
    }
  }
  free(xr); free(a); free(u); free(h); free(dh); free(da); free(du); free(o); free(p); free(dl); free(dp); free(dw);
}

/* ---- backward pass with expert-choice routing --------------------------------------
 * Gradients of the same scalar L = sum_t <dy_t, y_t> + dL_aux * L_aux when each
 * expert chooses its C tokens ["MoE架构解析" §2.2]:
 *   y_t = sum over the experts e that chose t of p_te o_e(x_t) + sum_s o_s(x_t),
 * p the gate probabilities over all E (softmax, or normalised sigmoid), the
 * weights of the sum as they are (no renormalisation).  The choice itself is
 * piecewise constant: no gradient.  By the chain rule:
 *  - dp_te = <dy_t, o_e(x_t)> where e chose t; do_e = p_te dy_t;
 *  - the expert FFN as in the token-choice backward above;
 *  - L_aux = alpha E sum_e f_e P_e with f_e = 1/E (every expert holds C of the
 *    E C selections): dp_te += dL_aux alpha E f_e / T;
 *  - through the gating over all E: softmax dl = p (dp - <p, dp>); normalised
 *    sigmoid p = s / sum s: dl_e = (dp_e - <p, dp>) / sum s * s_e (1 - s_e);
 *  - l = x W_g + b_g (+ noise): dW_g += x dl^T, db_g += dl, dx += W_g dl.
 * perm [E*C]: the chosen tokens of each expert; logits [T, E] (noisy) logits.
 * All outputs fp64, overwritten. */

/* One expert g on one token row xr with output weight wj: adds the expert's
 * parameter gradients (unless dW1 is NULL) and its part of dx_t (dxr), and
 * returns <dy_t, o_g(x_t)>. */
static double expert_row_bwd(int d, int f, int act, int dtype, int g, double wj, const double* xr,
                             const double* dyt, const void* W1, const void* b1, const void* W2, const void* b2,
                             const void* W3, double* dxr, double* dW1, double* db1, double* dW2, double* db2,
                             double* dW3) {
  const int swiglu = act == OACT_SWIGLU;
  const int64_t w1o = (int64_t)g * d * f, w2o = (int64_t)g * f * d;
  double* a = (double*)malloc(sizeof(double) * (size_t)f);
  double* u = (double*)malloc(sizeof(double) * (size_t)f);
  double* h = (double*)malloc(sizeof(double) * (size_t)f);
  double* dh = (double*)malloc(sizeof(double) * (size_t)f);
  double* da = (double*)malloc(sizeof(double) * (size_t)f);
  double* du = (double*)malloc(sizeof(double) * (size_t)f);
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  /* forward of the expert: a = W1^T x + b1 (u = W3^T x), h = act(a) (silu(a) u) */
  for (int c = 0; c < f; ++c) { a[c] = (b1 && !swiglu) ? ld(b1, dtype, (int64_t)g * f + c) : 0.0; u[c] = 0.0; }
  for (int i = 0; i < d; ++i) {
    for (int c = 0; c < f; ++c) a[c] += xr[i] * ld(W1, dtype, w1o + (int64_t)i * f + c);
    if (swiglu)
      for (int c = 0; c < f; ++c) u[c] += xr[i] * ld(W3, dtype, w1o + (int64_t)i * f + c);
  }
  for (int c = 0; c < f; ++c) h[c] = swiglu ? oracle_act(OACT_SWIGLU, a[c]) * u[c] : oracle_act(act, a[c]);
  /* o = W2^T h + b2 and <dy, o> */
  for (int c = 0; c < d; ++c) o[c] = (b2 && !swiglu) ? ld(b2, dtype, (int64_t)g * d + c) : 0.0;
  for (int r = 0; r < f; ++r)
    for (int c = 0; c < d; ++c) o[c] += h[r] * ld(W2, dtype, w2o + (int64_t)r * d + c);
  double dot = 0.0;
  for (int c = 0; c < d; ++c) dot += dyt[c] * o[c];
  /* do = wj dy: dh = W2 do, dW2 += h do^T, db2 += do */
  for (int r = 0; r < f; ++r) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) {
      const double doc = wj * dyt[c];
      acc += ld(W2, dtype, w2o + (int64_t)r * d + c) * doc;
      if (dW1) dW2[w2o + (int64_t)r * d + c] += h[r] * doc;
    }
    dh[r] = acc;
  }
  if (dW1 && b2 && !swiglu)
    for (int c = 0; c < d; ++c) db2[(int64_t)g * d + c] += wj * dyt[c];
  /* activation: da (, du) */
  for (int r = 0; r < f; ++r) {
    if (swiglu) {
      const double sa = sig(a[r]);
      da[r] = dh[r] * u[r] * (sa + a[r] * sa * (1.0 - sa));
      du[r] = dh[r] * a[r] * sa;
    } else if (act == OACT_RELU) {
      da[r] = a[r] > 0.0 ? dh[r] : 0.0;
    } else {
      da[r] = dh[r] * gelu_grad(a[r]);
    }
  }
  /* dx += W1 da (+ W3 du), dW1 += x da^T, dW3 += x du^T, db1 += da */
  for (int i = 0; i < d; ++i) {
    double acc = 0.0;
    for (int r = 0; r < f; ++r) {
      acc += ld(W1, dtype, w1o + (int64_t)i * f + r) * da[r];
      if (dW1) dW1[w1o + (int64_t)i * f + r] += xr[i] * da[r];
      if (swiglu) {
        acc += ld(W3, dtype, w1o + (int64_t)i * f + r) * du[r];
        if (dW1) dW3[w1o + (int64_t)i * f + r] += xr[i] * du[r];
      }
    }
    dxr[i] += acc;
  }
  if (dW1 && b1 && !swiglu)
    for (int r = 0; r < f; ++r) db1[(int64_t)g * f + r] += da[r];
  free(a); free(u); free(h); free(dh); free(da); free(du); free(o);
  return dot;
}

void oracle_ec_backward(int64_t T, int d, int f, int E, int S, int act, int gating, int dtype, double alpha,
                        double dL_aux, int64_t C, const int32_t* perm, const void* x, const void* W_g,
                        const double* logits, const void* W1, const void* b1, const void* W2, const void* b2,
                        const void* W3, const double* dy, double* dx, double* dWg, double* dbg, double* dW1,
                        double* db1, double* dW2, double* db2, double* dW3) {
  const int G = E + S;
  memset(dx, 0, sizeof(double) * (size_t)(T * d));
  memset(dWg, 0, sizeof(double) * (size_t)d * E);
  memset(dbg, 0, sizeof(double) * (size_t)E);
  memset(dW1, 0, sizeof(double) * (size_t)G * d * f);
  memset(db1, 0, sizeof(double) * (size_t)G * f);
  memset(dW2, 0, sizeof(double) * (size_t)G * f * d);
  memset(db2, 0, sizeof(double) * (size_t)G * d);
  if (dW3) memset(dW3, 0, sizeof(double) * (size_t)G * d * f);
  double* xr = (double*)malloc(sizeof(double) * (size_t)d);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  double* dp = (double*)malloc(sizeof(double) * (size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    const double* dyt = dy + t * d;
    double* dxt = dx + t * d;
    for (int i = 0; i < d; ++i) xr[i] = ld(x, dtype, t * d + i);
    const double* l = logits + t * E;
    oracle_gate_probs(1, E, gating, l, p);
    for (int e = 0; e < E; ++e) dp[e] = dL_aux * alpha * E * (1.0 / E) / (double)T;
    /* the experts that chose t, ascending */
    for (int e = 0; e < E; ++e) {
      int chose = 0;
      for (int64_t i = 0; i < C; ++i)
        if (perm[(int64_t)e * C + i] == t) { chose = 1; break; }
      if (chose)
        dp[e] += expert_row_bwd(d, f, act, dtype, e, p[e], xr, dyt, W1, b1, W2, b2, W3, dxt, dW1, db1, dW2, db2,
                                dW3);
    }
    for (int s = 0; s < S; ++s)
      expert_row_bwd(d, f, act, dtype, E + s, 1.0, xr, dyt, W1, b1, W2, b2, W3, dxt, dW1, db1, dW2, db2, dW3);
    /* through the gating over all E */
    double pdp = 0.0;
    for (int e = 0; e < E; ++e) pdp += p[e] * dp[e];
    double zs = 0.0;
    if (gating != OGATE_SOFTMAX)
      for (int e = 0; e < E; ++e) zs += sig(l[e]);
    for (int e = 0; e < E; ++e) {
      double dl;
      if (gating == OGATE_SOFTMAX) {
        dl = p[e] * (dp[e] - pdp);
      } else {
        const double se = sig(l[e]);
        dl = (dp[e] - pdp) / zs * se * (1.0 - se);
      }
      dbg[e] += dl;
      for (int i = 0; i < d; ++i) {
        dWg[(int64_t)i * E + e] += xr[i] * dl;
        dxt[i] += ld(W_g, dtype, (int64_t)i * E + e) * dl;
      }
    }
  }
  free(xr); free(p); free(dp);
}

/* ---- dx of single tokens, for sampled checks at full size ----------------------------
 * With dL_aux = 0 the gradient of x_t depends on token t alone (its routing row,
 * its logits, dy_t): the aux term is what couples the tokens, through n_e and
 * T.  These two functions give dx for the listed token rows only, without the
 * parameter gradients, by the same chain rule as the backward passes above
 * with dL_aux = 0.  Inputs are the rows themselves: x [n, d] (stored dtype),
 * logits [n, E], dy [n, d]; token choice: idx, w, dropped [n, k]; expert choice:
 * chose [n, E] (1 where expert e chose the token). */
void oracle_dx_rows(int64_t n, int d, int f, int E, int k, int S, int act, int gating, int dtype, const void* x,
                    const void* W_g, const double* logits, const void* W1, const void* b1, const void* W2,
                    const void* b2, const void* W3, const int32_t* idx, const double* w, const uint8_t* dropped,
                    const double* dy, double* dx) {
  double* xr = (double*)malloc(sizeof(double) * (size_t)d);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  double* dw = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
  for (int64_t t = 0; t < n; ++t) {
    const double* dyt = dy + t * d;
    double* dxt = dx + t * d;
    for (int i = 0; i < d; ++i) { xr[i] = ld(x, dtype, t * d + i); dxt[i] = 0.0; }
    for (int j = 0; j < k; ++j) {
      dw[j] = 0.0;
      if (dropped[t * k + j]) continue;
      dw[j] = expert_row_bwd(d, f, act, dtype, idx[t * k + j], w[t * k + j], xr, dyt, W1, b1, W2, b2, W3, dxt,
                             NULL, NULL, NULL, NULL, NULL);
    }
    for (int s = 0; s < S; ++s)
      expert_row_bwd(d, f, act, dtype, E + s, 1.0, xr, dyt, W1, b1, W2, b2, W3, dxt, NULL, NULL, NULL, NULL, NULL);
    /* the renormalised weights' gradient on the selected logits */
    const double* l = logits + t * E;
    oracle_gate_probs(1, E, gating, l, p);
    double zsel = 0.0, wdw = 0.0;
    for (int j = 0; j < k; ++j) {
      const int e = idx[t * k + j];
      zsel += gating == OGATE_SOFTMAX ? p[e] : sig(l[e]);
      wdw += w[t * k + j] * dw[j];
    }
    for (int j = 0; j < k; ++j) {
      const int e = idx[t * k + j];
      double dl;
      if (gating == OGATE_SOFTMAX) {
        dl = w[t * k + j] * (dw[j] - wdw);
      } else {
        const double se = sig(l[e]);
        dl = (dw[j] - wdw) / zsel * se * (1.0 - se);
      }
      for (int i = 0; i < d; ++i) dxt[i] += ld(W_g, dtype, (int64_t)i * E + e) * dl;
    }
  }
  free(xr); free(p); free(dw);
}

void oracle_ec_dx_rows(int64_t n, int d, int f, int E, int S, int act, int gating, int dtype, const void* x,
                       const void* W_g, const double* logits, const void* W1, const void* b1, const void* W2,
                       const void* b2, const void* W3, const uint8_t* chose, const double* dy, double* dx) {
  double* xr = (double*)malloc(sizeof(double) * (size_t)d);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  double* dp = (double*)malloc(sizeof(double) * (size_t)E);
  for (int64_t t = 0; t < n; ++t) {
    const double* dyt = dy + t * d;
    double* dxt = dx + t * d;
    for (int i = 0; i < d; ++i) { xr[i] = ld(x, dtype, t * d + i); dxt[i] = 0.0; }
    const double* l = logits + t * E;
    oracle_gate_probs(1, E, gating, l, p);
    for (int e = 0; e < E; ++e) {
      dp[e] = 0.0;
      if (chose[t * E + e])
        dp[e] = expert_row_bwd(d, f, act, dtype, e, p[e], xr, dyt, W1, b1, W2, b2, W3, dxt, NULL, NULL, NULL, NULL,
                               NULL);
    }
    for (int s = 0; s < S; ++s)
      expert_row_bwd(d, f, act, dtype, E + s, 1.0, xr, dyt, W1, b1, W2, b2, W3, dxt, NULL, NULL, NULL, NULL, NULL);
    double pdp = 0.0, zs = 0.0;
    for (int e = 0; e < E; ++e) pdp += p[e] * dp[e];
    if (gating != OGATE_SOFTMAX)
      for (int e = 0; e < E; ++e) zs += sig(l[e]);
    for (int e = 0; e < E; ++e) {
      double dl;
      if (gating == OGATE_SOFTMAX) {
        dl = p[e] * (dp[e] - pdp);
      } else {
        const double se = sig(l[e]);
        dl = (dp[e] - pdp) / zs * se * (1.0 - se);
      }
      for (int i = 0; i < d; ++i) dxt[i] += ld(W_g, dtype, (int64_t)i * E + e) * dl;
    }
  }
  free(xr); free(p); free(dp);
}

/* ---- FP8 (E4M3) experts ---------------------------------------------------------
 * ["MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现" §5.2: the expert
 * parameters are quantised from 16-bit to 8-bit floats, which halves their memory
 * at a usually acceptable loss of quality.]  The pages name the format only.
 * Readings:
 *  - the 8-bit format is E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 *    bits, subnormals, no infinities, largest finite value 448, S.1111.111 NaN);
 *  - encoding rounds to the nearest value, ties to the even mantissa, and
 *    saturates at +-448;
 *  - a vector v has one scale pair: a = max(max_i |v_i|, 2^-60), the encoding
 *    factor r = fl32(448 / a) and the decoding scale s = fl32(a / 448);
 *    q_i = e4m3(fl32(v_i * r)), decoded value s * value(q_i);
 *  - weights: one vector per (expert, output unit), i.e. per column of the
 *    [in, out] slab, stored transposed as [out, in]; activations: one vector per
 *    row of x and per row of the hidden activations h;
 *  - the products of the expert GEMMs are exact and summed in fp64 here; the
 *    scales multiply the sum; h is rounded to bf16 (nearest, ties to even)
 *    before its quantisation, as it is held in bf16 between the two GEMMs. */
static double round_bits(double v, int sig_bits, int min_exp) {
  /* nearest value with sig_bits significant bits (ties to even); quantum never
   * below 2^min_exp */
  if (v == 0.0 || isnan(v)) return v;
  int e;
  frexp(v, &e);                       /* |v| in [2^(e-1), 2^e) */
  int qe = e - sig_bits;
  if (qe < min_exp) qe = min_exp;
  return ldexp(rint(ldexp(v, -qe)), qe);   /* rint: ties to even in the default mode */
}

double oracle_bf16_round(double v) { return round_bits(v, 8, -133); }

double oracle_e4m3_value(uint8_t c) {
  const int E = (c >> 3) & 15, m = c & 7;
  if (E == 15 && m == 7) return NAN;
  const double v = E == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), E - 10);
  return (c & 0x80) ? -v : v;
}

uint8_t oracle_e4m3_encode1(float x) {
  const double v = x;
  if (isnan(v)) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs(v);
  if (a >= 448.0) return sign | 0x7E;                 /* saturate */
  a = round_bits(a, 4, -9);                            /* 4 significant bits; subnormal quantum 2^-9 */
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  if (a < ldexp(1.0, -6)) return sign | (uint8_t)ldexp(a, 9);        /* subnormal: m * 2^-9 */
  int e;
  const double fr = frexp(a, &e);                      /* a = (2 fr) 2^(e-1), 2 fr in [1, 2) */
  const int E = e - 1 + 7, m = (int)((2.0 * fr - 1.0) * 8.0);
  return sign | (uint8_t)(E << 3) | (uint8_t)m;
}

/* value(code) for all 256 codes, filled from oracle_e4m3_value on first use. */
static const double* e4m3_table(void) {
  static double tab[256];
  static int ready = 0;
  if (!ready) {
    for (int c = 0; c < 256; ++c) tab[c] = oracle_e4m3_value((uint8_t)c);
    ready = 1;
  }
  return tab;
}

void oracle_e4m3_encode(int64_t n, const float* x, uint8_t* q) {
  for (int64_t i = 0; i < n; ++i) q[i] = oracle_e4m3_encode1(x[i]);
}

void oracle_quantize_rows(int64_t rows, int64_t cols, const float* v, uint8_t* q, float* s) {
  const float floor_a = (float)ldexp(1.0, -60);
  for (int64_t r = 0; r < rows; ++r) {
    const float* vr = v + r * cols;
    float a = 0.0f;
    for (int64_t i = 0; i < cols; ++i) {
      const float m = fabsf(vr[i]);
      if (m > a) a = m;
    }
    if (a < floor_a) a = floor_a;
    const float rr = 448.0f / a;
    const float ss = a / 448.0f;
    for (int64_t i = 0; i < cols; ++i) {
      const float p = vr[i] * rr;
      q[r * cols + i] = oracle_e4m3_encode1(p);
    }
    s[r] = ss;
  }
}

/* First half of FP8 expert g on one quantised row xq (scale xs): the hidden
 * activations h [f] in fp64, before their bf16 rounding.
 * Weights: Wq [G, out, in] E4M3 codes with scales [G, out]; b1 fp32 or NULL. */
void oracle_fp8_hidden(int d, int f, int act, int g, const uint8_t* xq, float xs, const uint8_t* W1q,
                       const float* s1, const uint8_t* W3q, const float* s3, const float* b1, double* h) {
  const double* V = e4m3_table();
  double* xv = (double*)malloc(sizeof(double) * (size_t)d);
  for (int i = 0; i < d; ++i) xv[i] = V[xq[i]];
  for (int j = 0; j < f; ++j) {
    const uint8_t* w1 = W1q + ((int64_t)g * f + j) * d;
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += xv[i] * V[w1[i]];
    double a = (double)xs * (double)s1[(int64_t)g * f + j] * acc;
    if (act == OACT_SWIGLU) {
      const uint8_t* w3 = W3q + ((int64_t)g * f + j) * d;
      double acc3 = 0.0;
      for (int i = 0; i < d; ++i) acc3 += xv[i] * V[w3[i]];
      const double u = (double)xs * (double)s3[(int64_t)g * f + j] * acc3;
      h[j] = oracle_act(OACT_SWIGLU, a) * u;
    } else {
      if (b1) a += (double)b1[(int64_t)g * f + j];
      h[j] = oracle_act(act, a);
    }
  }
  free(xv);
}

/* Second half: expert output o [d] from the quantised hidden row hq (scale hs). */
void oracle_fp8_out(int d, int f, int act, int g, const uint8_t* hq, float hs, const uint8_t* W2q,
                    const float* s2, const float* b2, double* out) {
  const double* V = e4m3_table();
  double* hv = (double*)malloc(sizeof(double) * (size_t)f);
  for (int j = 0; j < f; ++j) hv[j] = V[hq[j]];
  for (int c = 0; c < d; ++c) {
    const uint8_t* w2 = W2q + ((int64_t)g * d + c) * f;
    double acc = 0.0;
    for (int j = 0; j < f; ++j) acc += hv[j] * V[w2[j]];
    out[c] = (double)hs * (double)s2[(int64_t)g * d + c] * acc;
    if (b2 && act != OACT_SWIGLU) out[c] += (double)b2[(int64_t)g * d + c];
  }
  free(hv);
}

/* FP8 expert g on one quantised row: hidden, bf16 rounding, per-row
 * quantisation of h, output. */
void oracle_fp8_expert_ffn(int d, int f, int act, int g, const uint8_t* xq, float xs, const uint8_t* W1q,
                           const float* s1, const uint8_t* W3q, const float* s3, const float* b1,
                           const uint8_t* W2q, const float* s2, const float* b2, double* out) {
  double* h = (double*)malloc(sizeof(double) * (size_t)f);
  float* hb = (float*)malloc(sizeof(float) * (size_t)f);
  uint8_t* hq = (uint8_t*)malloc((size_t)f);
  oracle_fp8_hidden(d, f, act, g, xq, xs, W1q, s1, W3q, s3, b1, h);
  for (int j = 0; j < f; ++j) hb[j] = (float)oracle_bf16_round(h[j]);    /* exact in fp32 */
  float hs;
  oracle_quantize_rows(1, f, hb, hq, &hs);
  oracle_fp8_out(d, f, act, g, hq, hs, W2q, s2, b2, out);
  free(h);
  free(hb);
  free(hq);
}

/* The layer output of the listed token rows with FP8 experts: x quantised per
 * token row (xq [T, d], xs [T]), then as oracle_layer_rows. */
void oracle_fp8_layer_rows(int d, int f, int E, int k, int S, int act, const int64_t* rows, int64_t nrows,
                           const uint8_t* xq, const float* xs, const uint8_t* W1q, const float* s1,
                           const uint8_t* W3q, const float* s3, const float* b1, const uint8_t* W2q,
                           const float* s2, const float* b2, const int32_t* idx, const double* w,
                           const uint8_t* dropped, double* y) {
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t t = rows[r];
    double* yr = y + r * d;
    for (int i = 0; i < d; ++i) yr[i] = 0.0;
    for (int j = 0; j < k; ++j) {
      if (dropped[t * k + j]) continue;
      oracle_fp8_expert_ffn(d, f, act, idx[t * k + j], xq + t * d, xs[t], W1q, s1, W3q, s3, b1, W2q, s2, b2, o);
      for (int i = 0; i < d; ++i) yr[i] += w[t * k + j] * o[i];
    }
    for (int s = 0; s < S; ++s) {
      oracle_fp8_expert_ffn(d, f, act, E + s, xq + t * d, xs[t], W1q, s1, W3q, s3, b1, W2q, s2, b2, o);
      for (int i = 0; i < d; ++i) yr[i] += o[i];
    }
  }
  free(o);
}

/* Expert-choice layer output with FP8 experts: as oracle_ec_layer_rows, each
 * choosing expert's output from the token's quantised row (xq [T, d], xs [T])
 * through oracle_fp8_expert_ffn. */
void oracle_fp8_ec_layer_rows(int d, int f, int E, int S, int act, int64_t T, int64_t C, const int64_t* rows,
                              int64_t nrows, const uint8_t* xq, const float* xs, const uint8_t* W1q,
                              const float* s1, const uint8_t* W3q, const float* s3, const float* b1,
                              const uint8_t* W2q, const float* s2, const float* b2, const int32_t* perm,
                              const double* scores, double* y) {
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t t = rows[r];
    double* yr = y + r * d;
    for (int i = 0; i < d; ++i) yr[i] = 0.0;
    for (int e = 0; e < E; ++e) {
      int hit = 0;
      for (int64_t i = 0; i < C; ++i)
        if (perm[(int64_t)e * C + i] == t) { hit = 1; break; }
      if (!hit) continue;
      oracle_fp8_expert_ffn(d, f, act, e, xq + t * d, xs[t], W1q, s1, W3q, s3, b1, W2q, s2, b2, o);
      const double w = scores[t * E + e];
      for (int i = 0; i < d; ++i) yr[i] += w * o[i];
    }
    for (int s = 0; s < S; ++s) {
      oracle_fp8_expert_ffn(d, f, act, E + s, xq + t * d, xs[t], W1q, s1, W3q, s3, b1, W2q, s2, b2, o);
      for (int i = 0; i < d; ++i) yr[i] += o[i];
    }
  }
  free(o);
}
