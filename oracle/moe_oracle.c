/*
 * moe_oracle.c -- plain, slow, obviously correct CPU oracle for the
 * Mixture-of-Experts layer forward (route -> routing metadata -> per-expert
 * SwiGLU / SwiGLU-OAI FFN -> gate-weighted combine).
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. It shares no source, header,
 * helper or constant with the CUDA path.
 *
 * Arithmetic: float64 everywhere, rounded to bf16 (round to nearest even)
 * only where the method stores bf16: the gate weights, the expert
 * intermediate h (between the two expert matmuls) and the layer output.
 * No -ffast-math; build with -ffp-contract=off so that x86 and Arm hosts
 * give identical bits. OpenMP splits the FFN over tokens only; each token's
 * arithmetic is sequential, so results do not depend on the thread count.
 *
 * Sources (page title, section):
 *  [R1] "Reuse topk SparseMatrix routing metadata in GPT-OSS MoE forward"
 *       (vLLM PR #45457 report), sections 实现拆解 and 关键源码片段:
 *       topk with apply_softmax=True; mask_metadata {col_sum,
 *       row_sorted_indx, col_sorted_indx}; gate_scal = vals.flatten()[combine_indx];
 *       GatherIndx(combine, dispatch), ScatterIndx(dispatch, combine);
 *       ragged metadata from col_sum.
 *  [R2] "MoE feed-forward performs ~3xnum_experts device->host syncs per
 *       layer, per forward" (MiniMind issue #835), sections Summary and
 *       "It is removable in plain PyTorch": masked per-expert loop
 *       y.index_add_(0, token_idx, expert(x[token_idx]) * weight); stable
 *       sort of the flattened expert ids; tok = order // k.
 *  [R3] "CuteDSL NVFP4 MoE adds SwiGLU-OAI and ReLU2" (vLLM PR #47106
 *       report), sections 关键源码片段 and 评论区精华: interleaved w13
 *       [gate0, up0, gate1, ...] vs packed [gate; up]; SwiGLU-OAI parameters
 *       alpha / beta / limit with defaults 1.702 / 1.0 / 7.0.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - top-k order: descending logit, ties to the lower expert id, compared as
 *    fp32 values (-0.0 ties +0.0); logits must be finite.
 *  - SwiGLU-OAI: gate = min(gate, limit), up = clamp(up, -limit, limit),
 *    h = (gate * sigmoid(alpha * gate)) * (up + beta).
 *  - SwiGLU: h = (gate * sigmoid(gate)) * up; with a clamp limit ("SILU +
 *    clamp") gate and up are clamped as for SwiGLU-OAI first.
 *  - ReLU2 (non-gated, "RELU2_NO_MUL"): h = max(a, 0)^2 of the single w1 row.
 *  - the router weight multiplies the expert output (after w2).
 *  - combine sums a token's k weighted expert outputs in ascending expert
 *    id, the order of the masked per-expert loop.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_NONFINITE 2

#define ORC_GATING_SOFTMAX_TOPK 0
#define ORC_GATING_SOFTMAX_ALL 1
#define ORC_ACT_SWIGLU 0
#define ORC_ACT_SWIGLU_OAI 1
#define ORC_ACT_RELU2 2 /* non-gated: w13 holds I rows (w1 only) */
#define ORC_LAYOUT_PACKED 0
#define ORC_LAYOUT_INTERLEAVED 1

/* ---------------------------------------------------------------- bf16 -- */

/* bf16 bits -> float64 (exact). */
double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* float64 -> bf16 bits, one rounding, to nearest even. bf16 keeps 8
 * significant bits and fp32's exponent range; below 2^-126 it is subnormal
 * with quantum 2^-133. Rounding goes straight from float64 (no fp32 step,
 * which could round twice). */
uint16_t orc_f64_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  uint32_t sign = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (a == 0.0) return (uint16_t)sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
  int ex;
  frexp(a, &ex);                      /* a = m * 2^ex, 0.5 <= m < 1 */
  int q_exp = ex - 8;                 /* quantum of an 8-bit significand */
  if (q_exp < -133) q_exp = -133;     /* subnormal quantum */
  double r = rint(ldexp(a, -q_exp));  /* nearest integer, ties to even */
  r = ldexp(r, q_exp);
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);  /* overflow */
  float f = (float)r;                 /* exact: r has <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

/* ------------------------------------------------------------ routing -- */

/* [R1] 关键源码片段 (topk_fn(logits, k, apply_softmax=True)) and [R2]
 * Summary (top-k weight of the MiniMind gate).
 *
 * Per token: order the experts by (logit descending, expert id ascending)
 * with a stable insertion sort over experts taken in ascending id, keep the
 * first k. Gate weights in float64, rounded once to bf16:
 *   gating 0 (softmax over the k selected): w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0)
 *   gating 1 (softmax over all E):          w_j = p(e_j), p = softmax(all logits)
 * topk_indx [n, k] int32, topk_vals [n, k] bf16 bits. */
int orc_route(const float *logits, int64_t n, int E, int k, int gating,
              int32_t *topk_indx, uint16_t *topk_vals) {
  if (n < 0 || E < 1 || k < 1 || k > E || k > 256) return ORC_BAD_ARG;
  if (gating != ORC_GATING_SOFTMAX_TOPK && gating != ORC_GATING_SOFTMAX_ALL) return ORC_BAD_ARG;
  for (int64_t i = 0; i < n * (int64_t)E; ++i)
    if (!isfinite(logits[i])) return ORC_NONFINITE;
  int *order = (int *)malloc(sizeof(int) * (size_t)E);
  if (!order) return ORC_BAD_ARG;
  for (int64_t t = 0; t < n; ++t) {
    const float *l = logits + t * E;
    /* stable insertion sort: an element moves left only past strictly smaller logits */
    for (int e = 0; e < E; ++e) {
      int pos = e;
      while (pos > 0 && l[order[pos - 1]] < l[e]) {
        order[pos] = order[pos - 1];
        --pos;
      }
      order[pos] = e;
    }
    double w[256];
    if (gating == ORC_GATING_SOFTMAX_TOPK) {
      double l0 = (double)l[order[0]], s = 0.0;
      for (int j = 0; j < k; ++j) s += exp((double)l[order[j]] - l0);
      for (int j = 0; j < k; ++j) w[j] = exp((double)l[order[j]] - l0) / s;
    } else {
      double lmax = (double)l[order[0]], s = 0.0;
      for (int e = 0; e < E; ++e) s += exp((double)l[e] - lmax);
      for (int j = 0; j < k; ++j) w[j] = exp((double)l[order[j]] - lmax) / s;
    }
    for (int j = 0; j < k; ++j) {
      topk_indx[t * k + j] = order[j];
      topk_vals[t * k + j] = orc_f64_to_bf16(w[j]);
    }
  }
  free(order);
  return ORC_OK;
}

/* Expert map (expert parallelism; [R1] 功能与动机 and 风险与影响: the
 * routing of a rank that holds a subset of the experts, where a slot whose
 * expert lives elsewhere is marked -1): expert_map[e] is the local id in
 * [0, E_loc) of global expert e, or -1. A slot f keeps local expert
 * map[indx[f]]; a -1 slot is dropped (it is listed nowhere and contributes
 * nothing to this rank's output). expert_map = NULL: the identity, E_loc = E.
 * Returns the local id of slot f, -1 if dropped, -2 for an invalid map entry. */
static int orc_local(const int32_t *expert_map, int E_loc, int32_t e) {
  if (!expert_map) return e;
  int32_t v = expert_map[e];
  return (v >= -1 && v < E_loc) ? v : -2;
}

/* [R1] 关键源码片段 (routing_data_from_sparse_topk): with f = t*k + j the
 * flat slot index and e(f) its (local) expert,
 *   col_sum[e]        = #{ f : indx[f] = e }                   (histogram)
 *   offs[0] = 0, offs[e+1] = offs[e] + col_sum[e]               (ragged offsets)
 *   col_sorted[p]     = slots listed expert by expert, ascending f within
 *                       an expert (the stable sort of [R2]
 *                       "It is removable in plain PyTorch")     (combine_indx)
 *   row_sorted[f]     = p such that col_sorted[p] = f           (dispatch_indx)
 *   gate_scal[p]      = vals_flat[col_sorted[p]]
 * Gather = (src col_sorted, dst row_sorted); scatter = (src row_sorted,
 * dst col_sorted): the same two arrays. With an expert map the histogram
 * and offsets run over the E_loc local experts, col_sorted / gate_scal list
 * the offs[E_loc] kept slots, and row_sorted[f] = -1 for a dropped slot. */
int orc_metadata(const int32_t *topk_indx, const uint16_t *topk_vals, int64_t n, int E, int k,
                 const int32_t *expert_map, int E_loc, int32_t *col_sum, int32_t *offs,
                 int32_t *col_sorted, int32_t *row_sorted, uint16_t *gate_scal) {
  if (n < 0 || E < 1 || k < 1) return ORC_BAD_ARG;
  if (!expert_map) E_loc = E;
  if (E_loc < 1 || E_loc > E) return ORC_BAD_ARG;
  for (int e = 0; expert_map && e < E; ++e)
    if (orc_local(expert_map, E_loc, e) < -1) return ORC_BAD_ARG;
  int64_t N = n * (int64_t)k;
  for (int64_t f = 0; f < N; ++f)
    if (topk_indx[f] < 0 || topk_indx[f] >= E) return ORC_BAD_ARG;
  for (int e = 0; e < E_loc; ++e) {
    int32_t c = 0;
    for (int64_t f = 0; f < N; ++f) c += (orc_local(expert_map, E_loc, topk_indx[f]) == e);
    col_sum[e] = c;
  }
  offs[0] = 0;
  for (int e = 0; e < E_loc; ++e) offs[e + 1] = offs[e] + col_sum[e];
  int64_t p = 0;
  for (int e = 0; e < E_loc; ++e)
    for (int64_t f = 0; f < N; ++f)
      if (orc_local(expert_map, E_loc, topk_indx[f]) == e) col_sorted[p++] = (int32_t)f;
  for (int64_t f = 0; f < N; ++f) row_sorted[f] = -1;
  for (int64_t q = 0; q < p; ++q) row_sorted[col_sorted[q]] = (int32_t)q;
  for (int64_t q = 0; q < p; ++q) gate_scal[q] = topk_vals[col_sorted[q]];
  return ORC_OK;
}

/* ------------------------------------------------------------- router -- */

/* [R1] 功能与动机 (the router / gate matmul that issue #28986 asks to fuse
 * with expert selection): logits[t, e] = sum_h x[t, h] * w_gate[e, h], in
 * float64, h ascending; the caller rounds to fp32 where the method stores
 * fp32 logits. x [n, H], w_gate [E, H] bf16 bits; out [n, E] float64. */
int orc_router_logits(const uint16_t *x, const uint16_t *w_gate, int64_t n, int E, int H,
                      double *out) {
  if (n < 0 || E < 1 || H < 1) return ORC_BAD_ARG;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t) {
    const uint16_t *xt = x + t * H;
    for (int e = 0; e < E; ++e) {
      const uint16_t *we = w_gate + (int64_t)e * H;
      double s = 0.0;
      for (int h = 0; h < H; ++h) s += orc_bf16_to_f64(xt[h]) * orc_bf16_to_f64(we[h]);
      out[t * E + e] = s;
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------- expert -- */

typedef struct {
  int act;      /* ORC_ACT_* */
  int layout;   /* ORC_LAYOUT_* */
  double alpha; /* SwiGLU-OAI sigmoid scale */
  double beta;  /* SwiGLU-OAI up offset */
  double limit; /* clamp limit; +inf = no clamp */
} orc_act_params;

static double orc_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Rows of one expert's w13: gate and up (2I) for the gated activations,
 * the single w1 projection (I) for ReLU2. */
static int orc_w13_rows(const orc_act_params *prm, int I) {
  return prm->act == ORC_ACT_RELU2 ? I : 2 * I;
}

/* [R3] 实现拆解 / 关键源码片段 / 评论区精华 and [R2] Summary: one expert on
 * one row.
 *   a[r] = sum_h w13[r, h] * x[h]                 r in [0, rows), h ascending
 *   packed:      gate_i = a[i],    up_i = a[I + i]
 *   interleaved: gate_i = a[2i],   up_i = a[2i + 1]
 *   SwiGLU:      g = min(g, limit), u = clamp(u, -limit, limit) (limit +inf
 *                unless set), h_i = (g * sigmoid(g)) * u
 *   SwiGLU-OAI:  g = min(g, limit), u = clamp(u, -limit, limit),
 *                h_i = (g * sigmoid(alpha * g)) * (u + beta)
 *   ReLU2:       h_i = max(a[i], 0)^2               (non-gated, rows = I)
 *   h_i stored as bf16
 *   y[c] = sum_i w2[c, i] * h_i                   c in [0, H), i ascending
 * a_out (rows doubles), h_out (I bf16) may be NULL. */
static int orc_expert_row_impl(const uint16_t *x, const uint16_t *w13, const uint16_t *w2, int H,
                               int I, const orc_act_params *prm, double *a, uint16_t *hb,
                               double *y) {
  const int rows = orc_w13_rows(prm, I);
  for (int r = 0; r < rows; ++r) {
    const uint16_t *wr = w13 + (int64_t)r * H;
    double s = 0.0;
    for (int h = 0; h < H; ++h) s += orc_bf16_to_f64(wr[h]) * orc_bf16_to_f64(x[h]);
    a[r] = s;
  }
  for (int i = 0; i < I; ++i) {
    if (prm->act == ORC_ACT_RELU2) {
      const double r = a[i] > 0.0 ? a[i] : 0.0;
      hb[i] = orc_f64_to_bf16(r * r);
      continue;
    }
    double g, u;
    if (prm->layout == ORC_LAYOUT_PACKED) {
      g = a[i];
      u = a[I + i];
    } else {
      g = a[2 * i];
      u = a[2 * i + 1];
    }
    if (g > prm->limit) g = prm->limit;
    if (u > prm->limit) u = prm->limit;
    if (u < -prm->limit) u = -prm->limit;
    double hv;
    if (prm->act == ORC_ACT_SWIGLU)
      hv = (g * orc_sigmoid(g)) * u;
    else
      hv = (g * orc_sigmoid(prm->alpha * g)) * (u + prm->beta);
    hb[i] = orc_f64_to_bf16(hv);
  }
  for (int c = 0; c < H; ++c) {
    const uint16_t *wc = w2 + (int64_t)c * I;
    double s = 0.0;
    for (int i = 0; i < I; ++i) s += orc_bf16_to_f64(wc[i]) * orc_bf16_to_f64(hb[i]);
    y[c] = s;
  }
  return ORC_OK;
}

static int orc_check_params(const orc_act_params *p) {
  if (!p) return 0;
  if (p->act != ORC_ACT_SWIGLU && p->act != ORC_ACT_SWIGLU_OAI && p->act != ORC_ACT_RELU2)
    return 0;
  if (isnan(p->limit) || p->limit < 0.0) return 0;
  if (p->layout != ORC_LAYOUT_PACKED && p->layout != ORC_LAYOUT_INTERLEAVED) return 0;
  return 1;
}

/* One expert applied to one row (exported for the oracle's own checks). */
int orc_expert_row(const uint16_t *x, const uint16_t *w13, const uint16_t *w2, int H, int I,
                   const orc_act_params *prm, double *a_out, uint16_t *h_out, double *y_out) {
  if (H < 1 || I < 1 || !orc_check_params(prm)) return ORC_BAD_ARG;
  const int rows = orc_w13_rows(prm, I);
  double *a = (double *)malloc(sizeof(double) * (size_t)rows);
  uint16_t *hb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)I);
  if (!a || !hb) { free(a); free(hb); return ORC_BAD_ARG; }
  orc_expert_row_impl(x, w13, w2, H, I, prm, a, hb, y_out);
  if (a_out) memcpy(a_out, a, sizeof(double) * (size_t)rows);
  if (h_out) memcpy(h_out, hb, sizeof(uint16_t) * (size_t)I);
  free(a);
  free(hb);
  return ORC_OK;
}

/* ---------------------------------------------------------------- FFN -- */

/* [R2] Summary (masked loop: y.index_add_(0, token_idx, expert(x) * weight))
 * written per token: for each requested token t, its k (expert, weight)
 * pairs are taken in ascending expert id; each expert output y_e(x_t) is
 * multiplied by the bf16 gate weight and summed in float64; the sum is
 * rounded once to bf16. With an expert map, w13 / w2 hold the E_loc local
 * experts, slot j uses local expert map[e_j], and dropped slots add nothing
 * (their y_slot / h_slot entries are zero).
 *
 * tokens: list of n_sel token ids to compute (NULL = all n, in order).
 * out [n_sel, H] bf16 bits, row s for token tokens[s].
 * y_slot (optional, [n_sel, k, H] float64): gate-weighted expert output of
 *   slot j of the token, in slot order j (not sorted).
 * h_slot (optional, [n_sel, k, I] bf16): the intermediate of slot j. */
int orc_ffn(const uint16_t *x, const int32_t *topk_indx, const uint16_t *topk_vals,
            const uint16_t *w13, const uint16_t *w2, int64_t n, int E, int k, int H, int I,
            const int32_t *expert_map, int E_loc, const orc_act_params *prm,
            const int64_t *tokens, int64_t n_sel, uint16_t *out, double *y_slot,
            uint16_t *h_slot) {
  if (n < 0 || E < 1 || k < 1 || k > E || k > 64 || H < 1 || I < 1 || !orc_check_params(prm))
    return ORC_BAD_ARG;
  if (!expert_map) E_loc = E;
  if (E_loc < 1 || E_loc > E) return ORC_BAD_ARG;
  for (int e = 0; expert_map && e < E; ++e)
    if (orc_local(expert_map, E_loc, e) < -1) return ORC_BAD_ARG;
  if (!tokens) n_sel = n;
  for (int64_t s = 0; s < n_sel; ++s) {
    int64_t t = tokens ? tokens[s] : s;
    if (t < 0 || t >= n) return ORC_BAD_ARG;
    for (int j = 0; j < k; ++j)
      if (topk_indx[t * k + j] < 0 || topk_indx[t * k + j] >= E) return ORC_BAD_ARG;
  }
  int bad = 0;
#pragma omp parallel
  {
    double *a = (double *)malloc(sizeof(double) * 2 * (size_t)I);
    uint16_t *hb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)I);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *acc = (double *)malloc(sizeof(double) * (size_t)H);
    if (!a || !hb || !y || !acc) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t s = 0; s < n_sel; ++s) {
        int64_t t = tokens ? tokens[s] : s;
        const uint16_t *xt = x + t * H;
        for (int c = 0; c < H; ++c) acc[c] = 0.0;
        /* the token's slots in ascending expert id (experts of one token are distinct) */
        int slot_order[64];
        for (int j = 0; j < k; ++j) {
          int pos = j;
          while (pos > 0 && topk_indx[t * k + slot_order[pos - 1]] > topk_indx[t * k + j]) {
            slot_order[pos] = slot_order[pos - 1];
            --pos;
          }
          slot_order[pos] = j;
        }
        for (int jj = 0; jj < k; ++jj) {
          int j = slot_order[jj];
          int e = orc_local(expert_map, E_loc, topk_indx[t * k + j]);
          if (e < 0) { /* dropped: another rank's expert */
            if (y_slot)
              for (int c = 0; c < H; ++c) y_slot[(s * k + j) * H + c] = 0.0;
            if (h_slot) memset(h_slot + (s * k + j) * I, 0, sizeof(uint16_t) * (size_t)I);
            continue;
          }
          double wgt = orc_bf16_to_f64(topk_vals[t * k + j]);
          orc_expert_row_impl(xt, w13 + (int64_t)e * orc_w13_rows(prm, I) * H,
                              w2 + (int64_t)e * H * I, H, I, prm, a, hb, y);
          for (int c = 0; c < H; ++c) acc[c] += y[c] * wgt;
          if (y_slot)
            for (int c = 0; c < H; ++c) y_slot[(s * k + j) * H + c] = y[c] * wgt;
          if (h_slot) memcpy(h_slot + (s * k + j) * I, hb, sizeof(uint16_t) * (size_t)I);
        }
        for (int c = 0; c < H; ++c) out[s * H + c] = orc_f64_to_bf16(acc[c]);
      }
    }
    free(a);
    free(hb);
    free(y);
    free(acc);
  }
  return bad ? ORC_BAD_ARG : ORC_OK;
}

/* Vectorised helper for the checks: float64 array -> bf16 bits. */
void orc_f64_to_bf16_array(const double *v, int64_t m, uint16_t *out) {
  for (int64_t i = 0; i < m; ++i) out[i] = orc_f64_to_bf16(v[i]);
}

/* The number of OpenMP threads the FFN's parallel region runs with (the
 * benchmark states it beside the oracle's timing). */
int orc_num_threads(void) { return omp_get_max_threads(); }
