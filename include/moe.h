/*
 * moe.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts layer forward.
 *
 * One MoE layer forward in four stages, every stage a CUDA kernel of this
 * library, all enqueued on the caller's stream with no device-to-host
 * readback and no host synchronisation:
 *
 *   1. moe_route           router top-k and gate weights
 *   2. moe_build_metadata  per-expert histogram, ragged offsets, stable
 *                          expert-sorted dispatch / combine indices, gate_scal
 *   3. moe_grouped_ffn     per-expert SwiGLU / SwiGLU-OAI FFN over each
 *                          expert's contiguous slice (grouped GEMM), gate
 *                          scale and scatter back to token-slot order
 *   4. moe_combine         sum of a token's k weighted expert outputs
 *   moe_forward            1 -> 4 in one call
 * and around them: moe_route_metadata (1 + 2 in one kernel),
 * moe_build_metadata_noalloc (2 without a workspace), moe_route_gemm (the
 * router matmul fused with 1), moe_forward_gate (the layer from x and the
 * gate weights), moe_forward_timed (stage events), moe_forward_launch_count,
 * moe_ffn_plan,
 * the workspace calls (moe_workspace_size, moe_workspace_init,
 * moe_workspace_regions), moe_read_status and moe_selftest_wait_timeout.
 *
 * Sources (page title, section):
 *  [R1] "Reuse topk SparseMatrix routing metadata in GPT-OSS MoE forward"
 *       (vLLM PR #45457 report), 实现拆解 and 关键源码片段
 *       (routing_data_from_sparse_topk, topk_fn(logits, k, apply_softmax=True)).
 *  [R2] "MoE feed-forward performs ~3xnum_experts device->host syncs per
 *       layer, per forward" (MiniMind issue #835), Summary and "It is
 *       removable in plain PyTorch".
 *  [R3] "CuteDSL NVFP4 MoE adds SwiGLU-OAI and ReLU2" (vLLM PR #47106
 *       report), 关键源码片段 (apply, reorder_w13_to_w31_for_flashinfer_cutedsl)
 *       and 评论区精华 (parameter defaults).
 *
 * Notation: n tokens, E experts, k experts per token (n_expts_act), H hidden
 * size, I expert intermediate size; f = t*k + j is the flat slot index of
 * token t's j-th choice; p is a position in the expert-sorted order.
 * bf16 values travel as uint16_t bit patterns.
 *
 * Conventions for every call:
 *  - Pointers named d_* / device buffers are CUDA device pointers on the
 *    current device. The caller allocates and owns every buffer, including
 *    the workspace; the library never allocates, frees, synchronises or
 *    copies device-to-host (moe_read_status is the one documented
 *    exception and is for debugging only).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). All
 *    work is enqueued on it; outputs are valid in stream order.
 *  - Arguments are validated on the host before any launch; a rejected call
 *    launches nothing and returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_MISALIGNED / MOE_ERR_WORKSPACE_TOO_SMALL. A failed launch
 *    returns MOE_ERR_CUDA (cudaGetLastError, which does not synchronise).
 *  - n = 0 is a valid no-op.
 *  - Limits: 1 <= E <= 256, 1 <= k <= min(E, 8), n*k < 2^31; H and I
 *    multiples of 64; bf16 tensors 16-byte aligned.
 *  - Device-side waits are bounded. A wait that gives up records
 *    MOE_ERR_TIMEOUT in the workspace's status word and the kernel returns;
 *    read it with moe_read_status.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 4

typedef void *moe_stream;  /* a cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* null pointer, size out of range, bad enum */
  MOE_ERR_UNSUPPORTED = 2,         /* valid request this library does not implement */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < moe_workspace_size(...) */
  MOE_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5,             /* a bounded device-side wait gave up */
  MOE_ERR_MISALIGNED = 6           /* a pointer breaks the 16-byte alignment rule */
} moe_status;

/* Gate weights [R1] 关键源码片段 (apply_softmax=True) and [R2] Summary. */
typedef enum {
  MOE_GATING_SOFTMAX_TOPK = 0, /* softmax over the k selected logits */
  MOE_GATING_SOFTMAX_ALL = 1   /* softmax over all E logits; keep the k selected, no renormalising */
} moe_gating;

/* Expert activation [R3] 实现拆解 (the five activation cases: SILU, SILU +
 * clamp, RELU2_NO_MUL, SWIGLUOAI, SWIGLUOAI_UNINTERLEAVE) and 关键源码片段
 * (apply: SiLU forwards only the clamp limit, SwiGLU-OAI alpha / beta /
 * limit). The two SwiGLU-OAI cases are MOE_ACT_SWIGLU_OAI with the
 * interleaved or the packed w13 layout. */
typedef enum {
  MOE_ACT_SWIGLU = 0,     /* h = silu(g) * u; with MOE_SET_LIMIT ("SILU + clamp")
                             g = min(gate, limit), u = clamp(up, -limit, limit)
                             first, else g = gate, u = up */
  MOE_ACT_SWIGLU_OAI = 1, /* g = min(gate, limit), u = clamp(up, -limit, limit),
                             h = g * sigmoid(alpha * g) * (u + beta) */
  MOE_ACT_RELU2 = 2       /* non-gated: w13 holds one projection of I rows per
                             expert ([E, I, H]), h = max(w1 . x, 0)^2;
                             w13_layout is ignored */
} moe_activation;

/* Row order of the gated w13 [E, 2I, H] [R3] 关键源码片段 (reorder_w13_to_w31_for_flashinfer_cutedsl). */
typedef enum {
  MOE_W13_PACKED = 0,     /* rows [gate_0 .. gate_{I-1}, up_0 .. up_{I-1}] */
  MOE_W13_INTERLEAVED = 1 /* rows [gate_0, up_0, gate_1, up_1, ...] (gpt-oss checkpoints) */
} moe_w13_layout;

/* Flags of moe_params.set: a value whose flag is clear is NOT used; the
 * activation keeps its own default ([R3] 关键源码片段 / 评论区精华: unset
 * parameters must not override the kernel defaults). SwiGLU-OAI defaults:
 * alpha 1.702, beta 1.0, limit 7.0. SwiGLU takes only a limit (no clamp
 * when unset; alpha / beta are ignored). ReLU2 takes none (alpha / beta are
 * ignored, a limit is MOE_ERR_UNSUPPORTED). A limit must be >= 0. */
#define MOE_SET_ALPHA 1u
#define MOE_SET_BETA 2u
#define MOE_SET_LIMIT 4u

/* Which grouped-GEMM kernel runs the two expert contractions of stage 3.
 * Both compute the result moe_grouped_ffn documents (fp32 accumulation, h
 * rounded to bf16); they tile the work differently, so the last bits of an
 * output may differ between them. No counterpart on the pages: a choice of
 * this implementation.
 *   AUTO   = SWAP.
 *   SWAP   128 weight rows x up to 256 sorted rows per tile (the weights on
 *          the MMA's M side; 32-row token tiles when n*k <= 32*E, i.e.
 *          decode). An expert's ragged last token tile runs with the MMA's
 *          N rounded up to 32, so at most 31 idle columns.
 *   TILED  128 sorted rows x 256 weight rows per tile (the tokens on the
 *          MMA's M side); ragged tails cost up to 127 idle MMA rows. */
typedef enum {
  MOE_FFN_AUTO = 0,
  MOE_FFN_TILED = 1,
  MOE_FFN_SWAP = 2
} moe_ffn_kernel;

typedef struct {
  int32_t gating;     /* moe_gating */
  int32_t activation; /* moe_activation */
  int32_t w13_layout; /* moe_w13_layout */
  uint32_t set;       /* MOE_SET_* bits */
  float alpha, beta, limit;
  int32_t ffn_kernel; /* moe_ffn_kernel; 0 = AUTO */
  /* Expert parallelism [R1] 功能与动机 (expert-parallel routing) and 风险与影响
   * (its -1 slots): this rank holds n_local_experts of the E experts.
   * expert_map: device int32 [E], 4-byte aligned, the local id in
   * [0, n_local_experts) of each global expert or -1 for an expert on another
   * rank; NULL = every expert local (n_local_experts is then ignored).
   * Used by moe_forward, moe_forward_gate and moe_forward_timed: top-k runs
   * over the E global logits (topk_indx holds global ids); the metadata
   * covers the local experts (col_sum [n_local_experts], offs
   * [n_local_experts + 1]; the offs[n_local_experts] kept slots are listed in
   * col_sorted / gate_scal; row_sorted is -1 at a dropped slot); w13 / w2
   * hold the n_local_experts local experts; out[t] sums only the token's
   * slots on local experts (a zero row when it has none): this rank's share
   * of the layer output. Entries outside [-1, n_local_experts) count as -1
   * and record MOE_ERR_INVALID_ARG in the status word. The stage entry
   * points ignore the map: moe_grouped_ffn takes E = n_local_experts and the
   * metadata of moe_forward's meta output; moe_combine adds every slot. */
  const int32_t *expert_map;
  int32_t n_local_experts;
} moe_params;

/* Routing metadata [R1] 关键源码片段 (routing_data_from_sparse_topk),
 * all device pointers, caller-owned:
 *   col_sum[E]      per-expert count of routed slots (the histogram; also
 *                   the ragged batch block sizes)
 *   offs[E+1]       exclusive scan of col_sum: expert e owns sorted
 *                   positions [offs[e], offs[e+1])
 *   col_sorted[n*k] combine_indx: p -> f. Slots listed expert by expert,
 *                   ascending f (token order) within an expert: the stable
 *                   sort of [R2] "It is removable in plain PyTorch"
 *   row_sorted[n*k] dispatch_indx: f -> p, the inverse permutation
 *   gate_scal[n*k]  bf16 gate weight in sorted order, topk_vals_flat[col_sorted[p]]
 * GatherIndx = (src col_sorted, dst row_sorted) and ScatterIndx = (src
 * row_sorted, dst col_sorted) are these same two arrays. */
typedef struct {
  int32_t *col_sum;
  int32_t *offs;
  int32_t *col_sorted;
  int32_t *row_sorted;
  uint16_t *gate_scal;
} moe_routing_meta;

/* Version of this ABI (MOE_ABI_VERSION). */
int32_t moe_abi_version(void);

/* Human-readable name of a status code; never NULL. */
const char *moe_status_string(moe_status status);

/* Bytes of workspace that moe_build_metadata, moe_grouped_ffn and
 * moe_forward need for these sizes (a few KB of control and sync data plus,
 * for the FFN, the expert-sorted activations, the intermediate h and the
 * per-slot outputs; for decode sizes, n*k <= 32*E, also 16 MB of
 * fp32 partial sums of the w13 contraction's even split of its work over
 * the SMs). The sync words are rewritten by every FFN call, so one
 * workspace serves one stream at a time. Returns 0 for invalid sizes. */
size_t moe_workspace_size(int64_t n, int32_t E, int32_t k, int32_t H, int32_t I);

/* Where the workspace's regions lie for these sizes (no counterpart on the
 * pages: a debugging aid). Writes MOE_WS_REGIONS byte offsets from the
 * workspace start and the bytes each region uses, in layout order: control
 * block, the fused routing kernel's count rows, metadata histograms, topk_indx, topk_vals, col_sum, offs,
 * col_sorted, row_sorted, gate_scal, contraction sync words, stream-K
 * partial sums, X_sorted [n*k, H], h [n*k, I], y_flat [n*k, H]. Every region
 * starts 256-byte aligned; the bytes between one region's end and the next
 * region's start (and after the last, up to moe_workspace_size) are never
 * written, so a test can fill them with a canary and check them after a
 * forward. offset and bytes are host arrays of MOE_WS_REGIONS entries.
 * Returns MOE_ERR_INVALID_ARG for invalid sizes or null arrays. */
#define MOE_WS_REGIONS 15
moe_status moe_workspace_regions(int64_t n, int32_t E, int32_t k, int32_t H, int32_t I,
                                 size_t *offset, size_t *bytes);

/* Prepare a freshly allocated workspace: zero its control block (the first
 * 4 KB: status word and the grid-barrier counter). Must run once, in stream
 * order, before the workspace's first use; later calls leave the block
 * consistent. */
moe_status moe_workspace_init(void *workspace, size_t workspace_bytes, moe_stream stream);

/* Stage 1 -- router top-k and gate weights. [R1] 关键源码片段
 * (topk_fn(logits, k, apply_softmax=True)), [R2] Summary.
 *   logits     [n, E] fp32, row-major, device. Finite values (NaN sorts last).
 *   topk_indx  [n, k] int32 out: the k experts of largest logit, descending;
 *              equal logits (compared as fp32, -0.0 == +0.0) go to the
 *              lower expert id.
 *   topk_vals  [n, k] bf16 out: gate weights per `gating`, computed in fp32
 *              and rounded to nearest even. */
moe_status moe_route(const float *logits, int64_t n, int32_t E, int32_t k, int32_t gating,
                     int32_t *topk_indx, uint16_t *topk_vals, moe_stream stream);

/* Stage 2 -- routing metadata from a top-k result. [R1] 关键源码片段.
 *   topk_indx [n, k] int32 (each value in [0, E)), topk_vals [n, k] bf16.
 *   meta      the five output arrays described at moe_routing_meta.
 * Bit-reproducible: no atomic decides any position. One cooperative kernel
 * with a bounded grid-wide barrier (MOE_ERR_TIMEOUT in the status word if
 * it gives up). `workspace` as sized by moe_workspace_size and initialised
 * by moe_workspace_init. */
moe_status moe_build_metadata(const int32_t *topk_indx, const uint16_t *topk_vals, int64_t n,
                              int32_t E, int32_t k, const moe_routing_meta *meta,
                              void *workspace, size_t workspace_bytes, moe_stream stream);

/* Stages 1 + 2 in one call -- moe_route followed by moe_build_metadata,
 * same results bit for bit ([R1] 实现拆解 / 关键源码片段: the metadata is
 * built once from the top-k result, with no second pass). Runs as one
 * cooperative kernel (G lanes per token, shared-memory histogram, bounded
 * grid barrier, cross-CTA prefix, stable scatter) when each SM's share of the slots fits in
 * shared memory, else as the two kernels. Workspace as for
 * moe_build_metadata. */
moe_status moe_route_metadata(const float *logits, int64_t n, int32_t E, int32_t k,
                              int32_t gating, int32_t *topk_indx, uint16_t *topk_vals,
                              const moe_routing_meta *meta, void *workspace,
                              size_t workspace_bytes, moe_stream stream);

/* Stage 2 without a workspace -- the paper has no counterpart to this call;
 * it exists for callers that cannot give the library any device memory of
 * their own: a plugin that must enqueue into a framework whose allocator
 * owns all device memory, a latency-critical path where cudaMalloc (which
 * may synchronise the device) is forbidden, or any code that may not
 * allocate where it runs. Same results as moe_build_metadata, bit for bit;
 * it allocates nothing and takes no workspace.
 *   Scratch: a fixed array inside the library (4 KB of control words plus
 *   256 x 256 int32 histogram counters, 266,240 bytes), present on every GPU
 *   that loads the library until the process exits. The grid is capped at
 *   256 CTAs, so every valid size fits; sizes beyond the library's limits
 *   (E > 256, k > 8 or k > E, n*k >= 2^31) return MOE_ERR_INVALID_ARG.
 *   The first call on a device looks up the array's device address (once
 *   per device, with that device current); make that first call before any
 *   stream capture.
 *   Every call shares the one array: calls whose work overlaps on the GPU
 *   (different streams, no ordering between them) race and give wrong
 *   results. Each call clears the control words it needs at zero.
 *   status_out: optional device int32 (NULL = not reported) that receives,
 *   in stream order, the call's device status (MOE_OK, or MOE_ERR_TIMEOUT if
 *   the bounded grid barrier gave up, MOE_ERR_INVALID_ARG if an expert id
 *   was outside [0, E)). */
moe_status moe_build_metadata_noalloc(const int32_t *topk_indx, const uint16_t *topk_vals,
                                      int64_t n, int32_t E, int32_t k,
                                      const moe_routing_meta *meta, int32_t *status_out,
                                      moe_stream stream);

/* Stage 3 -- grouped expert FFN. [R2] Summary and "It is removable in plain
 * PyTorch" (each expert runs on its contiguous slice; the weight multiplies
 * the expert output), [R3] 关键源码片段 (activations, w13 layouts).
 *   x       [n, H] bf16 tokens.
 *   meta    metadata from moe_build_metadata (offs, col_sorted, row_sorted,
 *           gate_scal read).
 *   w13     [E, 2I, H] bf16, row-major (each expert's [2I, H] block in
 *           params->w13_layout order); [E, I, H] for MOE_ACT_RELU2.
 *   w2      [E, H, I] bf16, row-major.
 *   y_flat  [n*k, H] bf16 out, token-slot order: row f = gate_scal[row_sorted[f]]
 *           * (w2_e . h), e = topk_indx_flat[f], h = act(w13_e . x_t) rounded
 *           to bf16; fp32 accumulation in both contractions. */
moe_status moe_grouped_ffn(const uint16_t *x, const moe_routing_meta *meta, const uint16_t *w13,
                           const uint16_t *w2, int64_t n, int32_t E, int32_t k, int32_t H,
                           int32_t I, const moe_params *params, uint16_t *y_flat,
                           void *workspace, size_t workspace_bytes, moe_stream stream);

/* Stage 4 -- combine. [R2] Summary (y.index_add_ of the k weighted expert
 * outputs of each token).
 *   y_flat [n*k, H] bf16, out [n, H] bf16: out[t] = sum_{j<k} y_flat[t*k+j],
 *   summed in fp32 in slot order j, rounded once to bf16. Deterministic. */
moe_status moe_combine(const uint16_t *y_flat, int64_t n, int32_t k, int32_t H, uint16_t *out,
                       moe_stream stream);

/* Stages 1-4 in one call, zero host synchronisations, CUDA-graph friendly.
 *   x [n, H] bf16, logits [n, E] fp32, w13 [E, 2I, H] bf16 ([E, I, H] for
 *   MOE_ACT_RELU2), w2 [E, H, I] bf16, out [n, H] bf16.
 *   The dispatch gather ("It is removable in plain PyTorch": x[tok], tok =
 *   order // k) runs where it costs least: with n*k <= 2E slots and the
 *   swap-operand kernel, the w13 contraction fetches its token rows from x
 *   itself; else, when the cooperative route + metadata kernel runs on at
 *   least half the SMs, it copies the rows into expert-sorted order after
 *   its scatter; else a gather kernel does.
 *   The two expert contractions run as one persistent launch at decode sizes
 *   (n*k <= 32E) and where both use CTA pairs (moe_ffn_plan "fused"): its
 *   CTAs take w2 tiles once other CTAs of the same grid have stored the
 *   expert's h rows, so the grid is sized to what can be resident at once.
 *   Work on other streams that holds SMs for long delays it; a wait past
 *   one second records MOE_ERR_TIMEOUT in the workspace status word (no
 *   hang; moe_read_status).
 *   topk_indx / topk_vals ([n, k]) and meta: optional outputs (NULL = keep
 *   them inside the workspace). When given, all five meta arrays must be
 *   non-NULL. */
moe_status moe_forward(const uint16_t *x, const float *logits, const uint16_t *w13,
                       const uint16_t *w2, int64_t n, int32_t E, int32_t k, int32_t H, int32_t I,
                       const moe_params *params, uint16_t *out, int32_t *topk_indx,
                       uint16_t *topk_vals, const moe_routing_meta *meta, void *workspace,
                       size_t workspace_bytes, moe_stream stream);

/* Stage 1 with the router matmul fused in. [R1] 功能与动机 (issue #28986
 * asks for a fused GPT-OSS router kernel; expert selection is about 3.5 % of
 * a layer; the PR itself leaves the gate matmul untouched).
 *   logits[t, e] = sum_h x[t, h] * w_gate[e, h]   (fp32 accumulation of the
 *   bf16 products), then, in the same kernel, top-k and gate weights
 *   exactly as moe_route computes them from those logits (ties to the lower
 *   expert id; softmax over the k selected or over all E).
 *   x       [n, H] bf16, 16-byte aligned; H a multiple of 64.
 *   w_gate  [E, H] bf16, 16-byte aligned (E <= 256).
 *   topk_indx [n, k] int32, topk_vals [n, k] bf16: outputs.
 *   logits  [n, E] fp32 output, or NULL (then the logits never reach memory).
 *   workspace: at least the 4 KB control block (status of the bounded
 *   waits; moe_workspace_init'ed). */
moe_status moe_route_gemm(const uint16_t *x, const uint16_t *w_gate, int64_t n, int32_t E,
                          int32_t H, int32_t k, int32_t gating, int32_t *topk_indx,
                          uint16_t *topk_vals, float *logits, void *workspace,
                          size_t workspace_bytes, moe_stream stream);

/* moe_forward with the routing computed from x and the gate weights
 * w_gate [E, H] bf16 (moe_route_gemm's kernel, then the metadata kernel)
 * instead of from logits; every other argument as moe_forward. Launches one
 * kernel more than moe_forward when that one fuses route and metadata. */
moe_status moe_forward_gate(const uint16_t *x, const uint16_t *w_gate, const uint16_t *w13,
                            const uint16_t *w2, int64_t n, int32_t E, int32_t k, int32_t H,
                            int32_t I, const moe_params *params, uint16_t *out,
                            int32_t *topk_indx, uint16_t *topk_vals,
                            const moe_routing_meta *meta, void *workspace,
                            size_t workspace_bytes, moe_stream stream);

/* Stage kernels of moe_forward, in launch order (indices of the events of
 * moe_forward_timed). */
#define MOE_STAGE_ROUTE 0    /* top-k + gate weights                       */
#define MOE_STAGE_METADATA 1 /* histogram, offsets, sorted indices         */
#define MOE_STAGE_GATHER 2   /* expert-sorted copy of the token rows       */
#define MOE_STAGE_FFN1 3     /* w13 contraction + activation -> h          */
#define MOE_STAGE_FFN2 4     /* w2 contraction + gate scale + scatter      */
#define MOE_STAGE_COMBINE 5  /* sum over the k slots (no kernel when k = 1) */
#define MOE_STAGE_COUNT 6

/* moe_forward plus timing: `events` holds MOE_STAGE_COUNT + 1 cudaEvent_t
 * handles (created by the caller); events[i] is recorded on `stream` just
 * before stage i's kernel and events[MOE_STAGE_COUNT] after the last one,
 * so cudaEventElapsedTime(events[i], events[i+1]) is stage i's device time.
 * While `stream` is capturing, the records are external
 * (cudaEventRecordExternal), i.e. event-record nodes of the graph.
 * n_events must be MOE_STAGE_COUNT + 1. Same results as moe_forward. */
moe_status moe_forward_timed(const uint16_t *x, const float *logits, const uint16_t *w13,
                             const uint16_t *w2, int64_t n, int32_t E, int32_t k, int32_t H,
                             int32_t I, const moe_params *params, uint16_t *out,
                             int32_t *topk_indx, uint16_t *topk_vals,
                             const moe_routing_meta *meta, void *workspace,
                             size_t workspace_bytes, void *const *events, int32_t n_events,
                             moe_stream stream);

/* Number of kernels moe_forward (and moe_forward_timed) enqueues for these
 * sizes on the current device with the default grouped-GEMM kernel
 * (MOE_FFN_AUTO) and no expert map: route and metadata (one fused kernel
 * when a CTA's slots fit its shared memory, else two), the gather (none when
 * n*k <= 2E, where the w13 contraction gathers, nor when the cooperative
 * routing kernel copies the rows, on at least half the SMs), the two expert
 * contractions (one launch when n*k <= 32E, or when both run 256-row token
 * tiles on CTA pairs; counted for a gated w13) and, when k > 1, the combine;
 * 0 for n = 0; -1 for sizes
 * moe_forward rejects. Host-only: launches nothing. No counterpart on the
 * pages: lets a caller size a CUDA graph or count its launches. */
int32_t moe_forward_launch_count(int64_t n, int32_t E, int32_t k, int32_t H, int32_t I);

/* How moe_grouped_ffn / moe_forward tile the two expert contractions for these
 * sizes and params (no launch; the current device's SM count enters the
 * choice). Writes plan[0..5]: token rows per tile of the w13 and of the w2
 * contraction; 1 if the w13 / the w2 contraction runs on CTA pairs (one
 * M = 256 MMA over two SMs), else 0; 1 for the decode tiling (32-row tiles,
 * the w13 units split evenly over the SMs when they make under two waves);
 * 1 when both contractions run in one launch, whose CTAs take w2 tiles after
 * their w13 work (the decode tiling, and where both run on CTA pairs).
 * With params->ffn_kernel = MOE_FFN_TILED: 128, 128, 0, 0, 0, 0. Returns the
 * validation status of moe_forward for the same arguments (MOE_ERR_INVALID_ARG
 * for a null plan). No counterpart on the pages: introspection for callers
 * and tests. */
moe_status moe_ffn_plan(int64_t n, int32_t E, int32_t k, int32_t H, int32_t I,
                        const moe_params *params, int32_t *plan);

/* DEBUG ONLY -- synchronises `stream`, returns the status word recorded by
 * device-side bounded waits since the last reset (MOE_OK if none). With
 * `reset` non-zero it also zeroes the control block (status word and the
 * grid-barrier counter), which a workspace needs after a MOE_ERR_TIMEOUT
 * before it can be used again. */
moe_status moe_read_status(void *workspace, size_t workspace_bytes, int32_t reset,
                           moe_stream stream);

/* DIAGNOSTIC -- launches one thread that waits, through the library's
 * bounded device-side wait, on a control word that nothing ever sets. After
 * `timeout_ns` (1 .. 1e9) the wait gives up, records MOE_ERR_TIMEOUT in the
 * status word and the kernel returns: the error path of every bounded wait
 * (the metadata kernels' grid barrier is bounded the same way), exercised without
 * a fault or a hang. Read the result with moe_read_status. */
moe_status moe_selftest_wait_timeout(void *workspace, size_t workspace_bytes, uint64_t timeout_ns,
                                     moe_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
