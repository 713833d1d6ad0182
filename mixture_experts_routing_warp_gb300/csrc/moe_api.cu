// moe_api.cu -- the extern "C" entry points declared in include/moe.h:
// argument validation, workspace carving, and the launch sequence of each
// stage on the caller's stream. No allocation, no synchronisation, no
// device-to-host copy (moe_read_status excepted, documented as debug-only).
#include <math.h>
#include <string.h>

#include "moe_internal.cuh"

using namespace moe;

namespace {

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

moe_status check_sizes(int64_t n, int E, int k, int H, int I, bool need_hi) {
  if (n < 0 || E < 1 || E > kMaxExperts || k < 1 || k > kMaxTopk || k > E)
    return MOE_ERR_INVALID_ARG;
  if (n * (int64_t)k >= (int64_t)INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (need_hi) {
    if (H < 64 || I < 64 || H % 64 != 0 || I % 64 != 0) return MOE_ERR_INVALID_ARG;
    if ((int64_t)2 * I > (int64_t)INT32_MAX / 2 || H > 65536) return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

moe_status resolve_params(const moe_params *p, ActParams &out, int *gating) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (p->gating != MOE_GATING_SOFTMAX_TOPK && p->gating != MOE_GATING_SOFTMAX_ALL)
    return MOE_ERR_INVALID_ARG;
  if (p->activation != MOE_ACT_SWIGLU && p->activation != MOE_ACT_SWIGLU_OAI &&
      p->activation != MOE_ACT_RELU2)
    return MOE_ERR_INVALID_ARG;
  if (p->w13_layout != MOE_W13_PACKED && p->w13_layout != MOE_W13_INTERLEAVED)
    return MOE_ERR_INVALID_ARG;
  if (p->set & ~(MOE_SET_ALPHA | MOE_SET_BETA | MOE_SET_LIMIT)) return MOE_ERR_INVALID_ARG;
  if (p->ffn_kernel != MOE_FFN_AUTO && p->ffn_kernel != MOE_FFN_TILED &&
      p->ffn_kernel != MOE_FFN_SWAP)
    return MOE_ERR_INVALID_ARG;
  out.act = p->activation;
  out.layout = p->w13_layout;
  out.ffn_kernel = p->ffn_kernel;
  if (p->activation == MOE_ACT_SWIGLU_OAI) {
    // Only the parameters the caller set replace the SwiGLU-OAI defaults.
    out.alpha = (p->set & MOE_SET_ALPHA) ? p->alpha : 1.702f;
    out.beta = (p->set & MOE_SET_BETA) ? p->beta : 1.0f;
    out.limit = (p->set & MOE_SET_LIMIT) ? p->limit : 7.0f;
    if (!isfinite(out.alpha) || !isfinite(out.beta) || isnan(out.limit) || out.limit < 0.f)
      return MOE_ERR_INVALID_ARG;
  } else if (p->activation == MOE_ACT_SWIGLU) {
    // SwiGLU takes no alpha / beta; a limit clamps gate and up ("SILU + clamp").
    out.alpha = 1.f;
    out.beta = 0.f;
    out.limit = (p->set & MOE_SET_LIMIT) ? p->limit : INFINITY;
    if (isnan(out.limit) || out.limit < 0.f) return MOE_ERR_INVALID_ARG;
  } else {
    // ReLU2 takes no parameters; a clamp limit is not part of it.
    if (p->set & MOE_SET_LIMIT) return MOE_ERR_UNSUPPORTED;
    out.alpha = 1.f;
    out.beta = 0.f;
    out.limit = INFINITY;
  }
  if (gating) *gating = p->gating;
  return MOE_OK;
}

// True when moe_forward's w13 contraction gathers its own token rows (no
// gather kernel): the swap-operand kernel with at most 2 slots per expert on
// average, where a tile's rows take one tile::gather4 per K step. Measured on
// GPT-OSS decode (32 experts, top-4): 1 token 53.7 -> 52.1 us, 8 tokens equal,
// 64 tokens (~8 rows per expert) 254 -> 256 us.
static bool fused_gather_rows(int64_t n, int32_t E, int32_t k, int ffn_kernel) {
  return ffn_kernel != MOE_FFN_TILED && n * k <= 2 * (int64_t)E;
}

// The per-slot arrays may be NULL when there are no slots (n = 0).
moe_status check_meta(const moe_routing_meta *m, int64_t n) {
  if (!m || !m->col_sum || !m->offs) return MOE_ERR_INVALID_ARG;
  if (n > 0 && (!m->col_sorted || !m->row_sorted || !m->gate_scal)) return MOE_ERR_INVALID_ARG;
  if (!aligned(m->col_sum, 4) || !aligned(m->offs, 4) || !aligned(m->col_sorted, 4) ||
      !aligned(m->row_sorted, 4) || !aligned(m->gate_scal, 2))
    return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

inline moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename T>
T *ws_at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

FfnScratch ffn_scratch(void *ws, const WorkspaceLayout &L) {
  return {ws_at<uint32_t>(ws, L.ctrl), ws_at<uint32_t>(ws, L.sync),
          L.x_sorted > L.sk_part ? ws_at<float>(ws, L.sk_part) : nullptr};
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: not implemented for these arguments";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL: workspace too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device-side wait gave up";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED: pointer breaks the alignment rule";
  }
  return "unknown moe_status";
}

size_t moe_workspace_size(int64_t n, int32_t E, int32_t k, int32_t H, int32_t I) {
  if (check_sizes(n, E, k, H, I, true) != MOE_OK) return 0;
  return workspace_layout(n, E, k, H, I).total;
}

moe_status moe_workspace_regions(int64_t n, int32_t E, int32_t k, int32_t H, int32_t I,
                                 size_t *offset, size_t *bytes) {
  if (!offset || !bytes || check_sizes(n, E, k, H, I, true) != MOE_OK)
    return MOE_ERR_INVALID_ARG;
  const WorkspaceLayout L = workspace_layout(n, E, k, H, I);
  const size_t at[MOE_WS_REGIONS] = {L.ctrl,       L.frows,     L.hist,    L.topk_indx,
                                     L.topk_vals,  L.col_sum,   L.offs,    L.col_sorted,
                                     L.row_sorted, L.gate_scal, L.sync,    L.sk_part,
                                     L.x_sorted,   L.h,         L.y_flat};
  for (int r = 0; r < MOE_WS_REGIONS; ++r) {
    offset[r] = at[r];
    bytes[r] = L.bytes[r];
  }
  return MOE_OK;
}

moe_status moe_workspace_init(void *workspace, size_t workspace_bytes, moe_stream stream) {
  if (!workspace || workspace_bytes < kCtrlBytes) return MOE_ERR_INVALID_ARG;
  if (!aligned(workspace, kAlign)) return MOE_ERR_MISALIGNED;
  return from_cuda(cudaMemsetAsync(workspace, 0, kCtrlBytes, (cudaStream_t)stream));
}

moe_status moe_route(const float *logits, int64_t n, int32_t E, int32_t k, int32_t gating,
                     int32_t *topk_indx, uint16_t *topk_vals, moe_stream stream) {
  moe_status st = check_sizes(n, E, k, 64, 64, false);
  if (st != MOE_OK) return st;
  if (gating != MOE_GATING_SOFTMAX_TOPK && gating != MOE_GATING_SOFTMAX_ALL)
    return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!logits || !topk_indx || !topk_vals) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(topk_indx, 4) || !aligned(topk_vals, 2))
    return MOE_ERR_MISALIGNED;
  return from_cuda(launch_route(logits, n, E, k, gating, topk_indx, topk_vals, nullptr,
                                (cudaStream_t)stream));
}

moe_status moe_build_metadata(const int32_t *topk_indx, const uint16_t *topk_vals, int64_t n,
                              int32_t E, int32_t k, const moe_routing_meta *meta,
                              void *workspace, size_t workspace_bytes, moe_stream stream) {
  moe_status st = check_sizes(n, E, k, 64, 64, false);
  if (st != MOE_OK) return st;
  if ((st = check_meta(meta, n)) != MOE_OK) return st;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(workspace, kAlign)) return MOE_ERR_MISALIGNED;
  const WorkspaceLayout L = workspace_layout(n, E, k, 64, 64);
  if (workspace_bytes < L.topk_indx) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (n > 0 && (!topk_indx || !topk_vals)) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_indx, 4) || !aligned(topk_vals, 2)) return MOE_ERR_MISALIGNED;
  return from_cuda(launch_metadata(topk_indx, topk_vals, n, E, k, *meta,
                                   ws_at<int32_t>(workspace, L.hist),
                                   ws_at<uint32_t>(workspace, L.ctrl), (cudaStream_t)stream));
}

moe_status moe_route_metadata(const float *logits, int64_t n, int32_t E, int32_t k,
                              int32_t gating, int32_t *topk_indx, uint16_t *topk_vals,
                              const moe_routing_meta *meta, void *workspace,
                              size_t workspace_bytes, moe_stream stream) {
  moe_status st = check_sizes(n, E, k, 64, 64, false);
  if (st != MOE_OK) return st;
  if (gating != MOE_GATING_SOFTMAX_TOPK && gating != MOE_GATING_SOFTMAX_ALL)
    return MOE_ERR_INVALID_ARG;
  if ((st = check_meta(meta, n)) != MOE_OK) return st;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(workspace, kAlign)) return MOE_ERR_MISALIGNED;
  const WorkspaceLayout L = workspace_layout(n, E, k, 64, 64);
  if (workspace_bytes < L.topk_indx) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (n > 0 && (!logits || !topk_indx || !topk_vals)) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(topk_indx, 4) || !aligned(topk_vals, 2))
    return MOE_ERR_MISALIGNED;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t *hist = ws_at<int32_t>(workspace, L.hist);
  uint32_t *ctrl = ws_at<uint32_t>(workspace, L.ctrl);
  if (n > 0 && route_metadata_fits(n, k))
    return from_cuda(launch_route_metadata(logits, n, E, k, gating, topk_indx, topk_vals, *meta,
                                           ctrl, s));
  if (launch_route(logits, n, E, k, gating, topk_indx, topk_vals, ctrl, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return from_cuda(launch_metadata(topk_indx, topk_vals, n, E, k, *meta, hist, ctrl, s));
}

moe_status moe_grouped_ffn(const uint16_t *x, const moe_routing_meta *meta, const uint16_t *w13,
                           const uint16_t *w2, int64_t n, int32_t E, int32_t k, int32_t H,
                           int32_t I, const moe_params *params, uint16_t *y_flat,
                           void *workspace, size_t workspace_bytes, moe_stream stream) {
  moe_status st = check_sizes(n, E, k, H, I, true);
  if (st != MOE_OK) return st;
  ActParams act;
  if ((st = resolve_params(params, act, nullptr)) != MOE_OK) return st;
  if ((st = check_meta(meta, n)) != MOE_OK) return st;
  if (n == 0) return MOE_OK;
  if (!x || !w13 || !w2 || !y_flat || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(y_flat, 16) ||
      !aligned(workspace, kAlign))
    return MOE_ERR_MISALIGNED;
  const WorkspaceLayout L = workspace_layout(n, E, k, H, I);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t N = n * k;
  uint16_t *x_sorted = ws_at<uint16_t>(workspace, L.x_sorted);
  const FfnScratch scr = ffn_scratch(workspace, L);
  cudaError_t err = launch_gather_rows(x, meta->row_sorted, n, k, H, x_sorted, scr.sync, s);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  return from_cuda(launch_ffn(x_sorted, meta->offs, meta->col_sorted, meta->gate_scal, w13, w2, N,
                              E, H, I, act, ws_at<uint16_t>(workspace, L.h), y_flat, scr, s));
}

moe_status moe_combine(const uint16_t *y_flat, int64_t n, int32_t k, int32_t H, uint16_t *out,
                       moe_stream stream) {
  if (n < 0 || k < 1 || k > kMaxTopk || H < 64 || H % 64 != 0) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!y_flat || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(y_flat, 16) || !aligned(out, 16)) return MOE_ERR_MISALIGNED;
  return from_cuda(launch_combine(y_flat, n, k, H, out, (cudaStream_t)stream));
}

// Routing comes from `logits`, or, when w_gate is given, from the router
// matmul x . w_gate^T fused with the top-k.
static moe_status forward_impl(const uint16_t *x, const float *logits, const uint16_t *w_gate,
                               const uint16_t *w13,
                               const uint16_t *w2, int64_t n, int32_t E, int32_t k, int32_t H,
                               int32_t I, const moe_params *params, uint16_t *out,
                               int32_t *topk_indx, uint16_t *topk_vals,
                               const moe_routing_meta *meta, void *workspace,
                               size_t workspace_bytes, cudaStream_t s, cudaEvent_t *ev) {
  moe_status st = check_sizes(n, E, k, H, I, true);
  if (st != MOE_OK) return st;
  ActParams act;
  int gating = 0;
  if ((st = resolve_params(params, act, &gating)) != MOE_OK) return st;
  if (meta && (st = check_meta(meta, n)) != MOE_OK) return st;
  if ((topk_indx == nullptr) != (topk_vals == nullptr)) return MOE_ERR_INVALID_ARG;
  // expert parallelism: routing over the E global experts, the metadata and
  // the contractions over the E_loc local ones
  const int32_t *emap = params->expert_map;
  const int32_t E_loc = emap ? params->n_local_experts : E;
  if (E_loc < 1 || E_loc > E) return MOE_ERR_INVALID_ARG;
  if (!aligned(emap, 4)) return MOE_ERR_MISALIGNED;
  if (n == 0) return MOE_OK;
  if (!x || (!logits && !w_gate) || !w13 || !w2 || !out || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16) ||
      !aligned(logits, 4) || !aligned(w_gate, 16) || !aligned(workspace, kAlign) ||
      !aligned(topk_indx, 4) || !aligned(topk_vals, 2))
    return MOE_ERR_MISALIGNED;
  const WorkspaceLayout L = workspace_layout(n, E, k, H, I);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;

  int32_t *indx = topk_indx ? topk_indx : ws_at<int32_t>(workspace, L.topk_indx);
  uint16_t *vals = topk_vals ? topk_vals : ws_at<uint16_t>(workspace, L.topk_vals);
  moe_routing_meta m;
  if (meta) {
    m = *meta;
  } else {
    m.col_sum = ws_at<int32_t>(workspace, L.col_sum);
    m.offs = ws_at<int32_t>(workspace, L.offs);
    m.col_sorted = ws_at<int32_t>(workspace, L.col_sorted);
    m.row_sorted = ws_at<int32_t>(workspace, L.row_sorted);
    m.gate_scal = ws_at<uint16_t>(workspace, L.gate_scal);
  }
  uint32_t *ctrl = ws_at<uint32_t>(workspace, L.ctrl);
  const int64_t N = n * k;
  // k = 1: slot f is token t, so the w2 epilogue writes the output directly
  // (not with an expert map: a token without a local slot needs a zero row,
  // which the combine writes).
  const bool direct = k == 1 && !emap;
  uint16_t *y_flat = direct ? out : ws_at<uint16_t>(workspace, L.y_flat);
  uint16_t *x_sorted = ws_at<uint16_t>(workspace, L.x_sorted);
  uint16_t *h = ws_at<uint16_t>(workspace, L.h);
  const FfnScratch scr = ffn_scratch(workspace, L);
  // Inside a stream capture the records become event-record nodes, so stage
  // timing works for graph replays too.
  auto mark = [&](int i) { return ev ? record_stage_event(ev[i], s) : cudaSuccess; };

  int32_t *hist = ws_at<int32_t>(workspace, L.hist);
  // Where the dispatch rows come from: the w13 contraction gathers them with
  // a row or two per expert; else the cooperative route + metadata kernel
  // copies them after its scatter; else (router matmul path, very large or
  // decode-size batches) the gather kernel.
  const bool fused_gather = fused_gather_rows(n, E_loc, k, act.ffn_kernel);
  const bool rows_in_routing =
      !fused_gather && !w_gate && route_metadata_moves_rows(n, E, k);
  if (w_gate) {
    // router matmul + top-k in one kernel, then the metadata kernel
    if (mark(MOE_STAGE_ROUTE) != cudaSuccess ||
        launch_route_gemm(x, w_gate, n, E, H, k, gating, indx, vals, nullptr, ctrl, s) !=
            cudaSuccess ||
        mark(MOE_STAGE_METADATA) != cudaSuccess ||
        launch_metadata(indx, vals, n, E, k, m, hist, ctrl, s, scr.sync, emap, E_loc) !=
            cudaSuccess)
      return MOE_ERR_CUDA;
  } else if (route_metadata_fits(n, k)) {
    // one cooperative kernel for both stages (and the dispatch rows, unless
    // the w13 contraction gathers them itself); the metadata stage time is 0
    if (mark(MOE_STAGE_ROUTE) != cudaSuccess ||
        launch_route_metadata(logits, n, E, k, gating, indx, vals, m, ctrl, s, scr.sync,
                              emap, E_loc, rows_in_routing ? x : nullptr, H,
                              x_sorted) != cudaSuccess ||
        mark(MOE_STAGE_METADATA) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else {
    if (mark(MOE_STAGE_ROUTE) != cudaSuccess ||
        launch_route(logits, n, E, k, gating, indx, vals, ctrl, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (mark(MOE_STAGE_METADATA) != cudaSuccess ||
        launch_metadata(indx, vals, n, E, k, m, hist, ctrl, s, scr.sync, emap, E_loc) !=
            cudaSuccess)
      return MOE_ERR_CUDA;
  }
  // A row or two per expert: the swap-operand kernel gathers its token rows
  // from x itself (tile::gather4, one instruction per 4 rows). Otherwise they
  // come from X_sorted: a gather4 costs about as much TMA time as a whole 2-D
  // box, so 128 rows per K step as 32 gathers ran w13 3.4x slower at prefill.
  const GatherSrc src{x, n, k};
  if (mark(MOE_STAGE_GATHER) != cudaSuccess ||
      (!fused_gather && !rows_in_routing &&
       launch_gather_rows(x, m.row_sorted, n, k, H, x_sorted, scr.sync, s) != cudaSuccess))
    return MOE_ERR_CUDA;
  if (launch_ffn(x_sorted, m.offs, m.col_sorted, m.gate_scal, w13, w2, N, E_loc, H, I, act, h,
                 y_flat, scr, s, ev ? ev + MOE_STAGE_FFN1 : nullptr,
                 fused_gather ? &src : nullptr) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (mark(MOE_STAGE_COMBINE) != cudaSuccess) return MOE_ERR_CUDA;
  if (!direct &&
      launch_combine(y_flat, n, k, H, out, s, emap ? m.row_sorted : nullptr) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (mark(MOE_STAGE_COUNT) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_ffn_plan(int64_t n, int32_t E, int32_t k, int32_t H, int32_t I,
                        const moe_params *params, int32_t *plan) {
  moe_status st = check_sizes(n, E, k, H, I, true);
  if (st != MOE_OK) return st;
  ActParams act;
  if ((st = resolve_params(params, act, nullptr)) != MOE_OK) return st;
  if (!plan) return MOE_ERR_INVALID_ARG;
  if (act.ffn_kernel == MOE_FFN_TILED) {
    plan[0] = plan[1] = 128;  // BM: token rows per tile of the tokens-on-M kernel
    plan[2] = plan[3] = plan[4] = plan[5] = 0;
    return MOE_OK;
  }
  const SwapPlan p = plan_ffn_swap(n * k, E, H, I, act);
  plan[0] = p.nt1;
  plan[1] = p.nt2;
  plan[2] = p.pair1;
  plan[3] = p.pair2;
  plan[4] = p.decode;
  plan[5] = p.fused;
  return MOE_OK;
}

int32_t moe_forward_launch_count(int64_t n, int32_t E, int32_t k, int32_t H, int32_t I) {
  if (check_sizes(n, E, k, H, I, true) != MOE_OK) return -1;
  if (n == 0) return 0;
  // the same choices forward_impl makes (default kernel: the swap-operand
  // one), then the gather unless w13 or the cooperative routing kernel moves
  // the rows, ffn1 and ffn2 (one launch at decode sizes and on CTA pairs;
  // counted for a gated w13), combine
  const bool gather_kernel =
      !fused_gather_rows(n, E, k, MOE_FFN_AUTO) && !route_metadata_moves_rows(n, E, k);
  ActParams act{};
  act.act = MOE_ACT_SWIGLU;
  act.ffn_kernel = MOE_FFN_AUTO;
  const bool one_ffn_launch = plan_ffn_swap(n * k, E, H, I, act).fused;
  return (route_metadata_fits(n, k) ? 1 : 2) + (gather_kernel ? 1 : 0) +
         (one_ffn_launch ? 1 : 2) + (k > 1 ? 1 : 0);
}

moe_status moe_forward(const uint16_t *x, const float *logits, const uint16_t *w13,
                       const uint16_t *w2, int64_t n, int32_t E, int32_t k, int32_t H, int32_t I,
                       const moe_params *params, uint16_t *out, int32_t *topk_indx,
                       uint16_t *topk_vals, const moe_routing_meta *meta, void *workspace,
                       size_t workspace_bytes, moe_stream stream) {
  return forward_impl(x, logits, nullptr, w13, w2, n, E, k, H, I, params, out, topk_indx,
                      topk_vals, meta, workspace, workspace_bytes, (cudaStream_t)stream, nullptr);
}

moe_status moe_forward_timed(const uint16_t *x, const float *logits, const uint16_t *w13,
                             const uint16_t *w2, int64_t n, int32_t E, int32_t k, int32_t H,
                             int32_t I, const moe_params *params, uint16_t *out,
                             int32_t *topk_indx, uint16_t *topk_vals,
                             const moe_routing_meta *meta, void *workspace,
                             size_t workspace_bytes, void *const *events, int32_t n_events,
                             moe_stream stream) {
  if (!events || n_events != MOE_STAGE_COUNT + 1) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i <= MOE_STAGE_COUNT; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  cudaEvent_t ev[MOE_STAGE_COUNT + 1];
  for (int i = 0; i <= MOE_STAGE_COUNT; ++i) ev[i] = (cudaEvent_t)events[i];
  return forward_impl(x, logits, nullptr, w13, w2, n, E, k, H, I, params, out, topk_indx,
                      topk_vals, meta, workspace, workspace_bytes, (cudaStream_t)stream, ev);
}

moe_status moe_forward_gate(const uint16_t *x, const uint16_t *w_gate, const uint16_t *w13,
                            const uint16_t *w2, int64_t n, int32_t E, int32_t k, int32_t H,
                            int32_t I, const moe_params *params, uint16_t *out,
                            int32_t *topk_indx, uint16_t *topk_vals,
                            const moe_routing_meta *meta, void *workspace,
                            size_t workspace_bytes, moe_stream stream) {
  if (n > 0 && !w_gate) return MOE_ERR_INVALID_ARG;
  return forward_impl(x, nullptr, w_gate, w13, w2, n, E, k, H, I, params, out, topk_indx,
                      topk_vals, meta, workspace, workspace_bytes, (cudaStream_t)stream, nullptr);
}

moe_status moe_route_gemm(const uint16_t *x, const uint16_t *w_gate, int64_t n, int32_t E,
                          int32_t H, int32_t k, int32_t gating, int32_t *topk_indx,
                          uint16_t *topk_vals, float *logits, void *workspace,
                          size_t workspace_bytes, moe_stream stream) {
  moe_status st = check_sizes(n, E, k, H, 64, true);
  if (st != MOE_OK) return st;
  if (gating != MOE_GATING_SOFTMAX_TOPK && gating != MOE_GATING_SOFTMAX_ALL)
    return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!x || !w_gate || !topk_indx || !topk_vals || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_gate, 16) || !aligned(topk_indx, 4) ||
      !aligned(topk_vals, 2) || !aligned(logits, 4) || !aligned(workspace, kAlign))
    return MOE_ERR_MISALIGNED;
  if (workspace_bytes < kCtrlBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(launch_route_gemm(x, w_gate, n, E, H, k, gating, topk_indx, topk_vals, logits,
                                     ws_at<uint32_t>(workspace, 0), (cudaStream_t)stream));
}

moe_status moe_read_status(void *workspace, size_t workspace_bytes, int32_t reset,
                           moe_stream stream) {
  if (!workspace || workspace_bytes < kCtrlBytes) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t word = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (reset) {  // status word and grid-barrier counter back to zero
    if (cudaMemsetAsync(workspace, 0, kCtrlBytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return (moe_status)word;
}

moe_status moe_selftest_wait_timeout(void *workspace, size_t workspace_bytes,
                                     uint64_t timeout_ns, moe_stream stream) {
  if (!workspace || workspace_bytes < kCtrlBytes) return MOE_ERR_INVALID_ARG;
  if (timeout_ns == 0 || timeout_ns > kWaitTimeoutNs) return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_wait_selftest(ws_at<uint32_t>(workspace, 0), timeout_ns,
                                        (cudaStream_t)stream));
}

}  // extern "C"
