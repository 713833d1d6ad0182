// routing_fused.cu -- router top-k and routing metadata in one cooperative
// kernel (one CTA per SM; a single CTA with no exchange when the batch fits
// one pass), and the entry that picks it or the decode-size kernel.
//
// Sources (page title, section): as routing.cu.
#include "routing_common.cuh"

namespace moe {

// ================================================= fused route + metadata ==
//
// moe_route_metadata / moe_forward's first two stages in one cooperative
// kernel, one CTA per SM: CTA b routes tokens [b*T, b*T + T) (G lanes per
// token as above), keeping its slots and histogram in shared memory, then
// exchanges its counts through 16-bit rows and a grid barrier, and scatters
// its slots from shared memory. With an expert map the metadata
// covers the E_loc local experts and drops the slots of other ranks'
// experts. With x given, the CTA then copies its tokens' rows to their
// sorted positions in X_sorted (the dispatch gather, token-major). Dynamic
// shared memory: the top-k's logit stash ([NQ][1024] float4), then the
// slots' experts (u8) and weights (bf16).
template <int K, int G, int NQ>
__global__ void __launch_bounds__(kFusedThreads, 1) route_metadata_kernel(
    const float *__restrict__ logits, int64_t n, int E, int gating, int T, int vec4,
    int32_t *__restrict__ topk_indx, uint16_t *__restrict__ topk_vals,
    int32_t *__restrict__ col_sum, int32_t *__restrict__ offs, int32_t *__restrict__ col_sorted,
    int32_t *__restrict__ row_sorted, uint16_t *__restrict__ gate_scal,
    uint16_t *__restrict__ rows, uint32_t *ctrl,
    unsigned long long timeout_ns, uint32_t *sync, const int32_t *__restrict__ expert_map,
    int E_loc, const uint4 *__restrict__ x, int vpr, uint4 *__restrict__ x_sorted) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ MetaShared<kFusedThreads> sh;
  __shared__ int s_map_buf[kMaxExperts];
  float4 *stash = reinterpret_cast<float4 *>(smem_raw);
  uint8_t *s_slot_e = smem_raw + (size_t)NQ * kFusedThreads * sizeof(float4);
  uint16_t *s_slot_v = reinterpret_cast<uint16_t *>(s_slot_e + (((size_t)T * K + 15) & ~15ull));

  const int tid = threadIdx.x;
  pdl_launch_dependents();  // the next kernel may be scheduled (it waits for this grid)
  zero_sync_words(sync);
  const int *s_map = load_expert_map(expert_map, E, E_loc, s_map_buf, ctrl);
  for (int e = tid; e < E_loc; e += kFusedThreads) sh.base[e] = 0;
  __syncthreads();

  const int64_t t0 = min(n, (int64_t)blockIdx.x * T);
  const int64_t t1 = min(n, t0 + T);
  constexpr int per_pass = kFusedThreads / G;
  for (int64_t tb = t0; tb < t1; tb += per_pass) {  // uniform over the block
    const int64_t t = tb + tid / G;
    const bool valid = t < t1;
    TopK<K> tk;
    float w[K];
    topk_group<K, G, NQ>(logits + (valid ? t : 0) * E, valid, E, gating, vec4 != 0, tk, w,
                         stash);
    if (valid)
      write_token<K, G, true>(t, t0, tk, w, topk_indx, topk_vals, s_slot_e, s_slot_v, sh.base,
                              s_map);
  }
  __syncthreads();
  // the CTA's top-k outputs leave shared memory while the other CTAs arrive
  const int nslots = (int)(t1 - t0) * K;
  auto write_topk = [&] {
    for (int i = tid; i < nslots; i += kFusedThreads) {
      topk_indx[t0 * K + i] = s_slot_e[i];
      topk_vals[t0 * K + i] = s_slot_v[i];
    }
  };
  if (!meta_exchange_rows(rows, stash, E_loc, sh, col_sum, offs, ctrl, timeout_ns, write_topk))
    return;
  meta_scatter(
      t0 * K, (int)(t1 - t0) * K, E_loc, sh,
      [&](int i, int &e, uint16_t &w) {
        e = s_map ? s_map[s_slot_e[i]] : s_slot_e[i];
        w = s_slot_v[i];
      },
      col_sorted, row_sorted, gate_scal);
  if (x) {
    __syncthreads();  // this CTA's row_sorted entries are written
    copy_token_rows(x, row_sorted, t0, t1, K, vpr, n * K, x_sorted, tid >> 5,
                    kFusedThreads / 32);
  }
}

// Tokens per CTA of the fused kernel: spread over the SMs, a multiple of 4;
// a batch that one pass of one CTA covers (1024 / G tokens) gets one CTA,
// which skips the cross-CTA exchange. With one lane per token (E <= 16) a CTA
// takes at least 32 tokens: the rows are short, and fewer CTAs make the
// exchange cheaper, while at 32 a 4096-token batch still spans 128 CTAs --
// enough for the kernel to copy the dispatch rows itself (MiniMind, E = 4 /
// 8 / 16: 38.6 / 41.2 / 45.7 -> 37.9 / 40.5 / 45.0 us per layer against 128
// tokens per CTA and a gather kernel; the routing call alone 5.83 -> 5.93 us).
int64_t fused_tokens_per_cta(int64_t n, int per_pass) {
  if (n <= per_pass) return (n + 3) / 4 * 4;
  const int sms = device_sm_count();
  int64_t T = (n + sms - 1) / sms;
  if (per_pass >= kFusedThreads && T < 32) T = 32;
  if (T < 4) T = 4;
  return (T + 3) / 4 * 4;
}

// Dynamic shared memory of route_metadata_kernel<K, G, NQ> for T tokens per CTA.
inline size_t fused_smem_bytes(int64_t T, int K, int NQ) {
  const size_t slots = (size_t)T * K;
  return (size_t)NQ * kFusedThreads * sizeof(float4) + ((slots + 15) & ~(size_t)15) + slots * 2;
}

struct RouteMetaLaunch {
  const float *logits;
  int64_t n;
  int E, gating;
  int32_t *indx;
  uint16_t *vals;
  const moe_routing_meta *meta;
  uint32_t *ctrl;
  uint32_t *sync;
  const int32_t *expert_map;
  int E_loc;
  const uint16_t *x;
  int H;
  uint16_t *x_sorted;
  cudaStream_t s;
  template <int K, int G, int NQ>
  cudaError_t go() {
    auto kern = route_metadata_kernel<K, G, NQ>;
    const size_t max_smem = fused_smem_bytes(kSlotCap / K, K, NQ);
    static PerDeviceOnce configured;
    cudaError_t err = configured.run([kern, max_smem] {
      cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
      return e != cudaSuccess ? e : uniform_carveout(kern);
    });
    if (err != cudaSuccess) return err;
    const int64_t T = fused_tokens_per_cta(n, kFusedThreads / G);
    const int64_t B = (n + T - 1) / T;
    int Ti = (int)T;
    int64_t nn = n;
    int E_ = E, g_ = gating;
    int vec4 = (E % 4) == 0 && ((uintptr_t)logits % 16) == 0;
    unsigned long long timeout = kWaitTimeoutNs;
    const uint4 *xv = reinterpret_cast<const uint4 *>(x);
    uint4 *xs = reinterpret_cast<uint4 *>(x_sorted);
    int vpr = H / 8;
    // the count rows follow the control block
    uint16_t *rows = reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(ctrl) + kCtrlBytes);
    void *args[] = {(void *)&logits, (void *)&nn, (void *)&E_, (void *)&g_, (void *)&Ti,
                    (void *)&vec4, (void *)&indx, (void *)&vals, (void *)&meta->col_sum,
                    (void *)&meta->offs, (void *)&meta->col_sorted, (void *)&meta->row_sorted,
                    (void *)&meta->gate_scal, (void *)&rows, (void *)&ctrl, (void *)&timeout, (void *)&sync, (void *)&expert_map,
                    (void *)&E_loc, (void *)&xv, (void *)&vpr, (void *)&xs};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = fused_smem_bytes(T, K, NQ);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = B > 1 ? 1 : 0;  // one CTA needs no co-residency guarantee
    err = cudaLaunchKernelExC(&cfg, (const void *)kern, args);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
  }
};

// True when the fused kernel can take (n, k): each CTA's slots fit in
// shared memory. Otherwise the two kernels run.
bool route_metadata_fits(int64_t n, int k) {
  // the larger of the two T; one CTA per SM, each with a row of counts
  return fused_tokens_per_cta(n, 0) * k <= kSlotCap && device_sm_count() <= kFusedMaxRows;
}

// True when launch_route_metadata, given x, also moves the dispatch rows for
// (n, E, k): the cooperative kernel runs (not the decode-size one) on at
// least half the SMs. Each CTA copies its own tokens' rows, so a narrow grid
// would copy at the pace of a few SMs (GPT-OSS, 64 tokens on one CTA: +25 us;
// MiniMind, 4096 tokens on 32 CTAs: +2 us); at prefill widths the copy
// replaces the gather kernel (GPT-OSS n=8192: 1.153 -> 1.142 ms per layer).
bool route_metadata_moves_rows(int64_t n, int E, int k) {
  if (!route_metadata_fits(n, k) || n * k <= kSmallSlots) return false;
  const int G = E <= 16 ? 1 : E <= 32 ? 2 : E <= 64 ? 4 : 8;  // as dispatch_kg
  const int64_t T = fused_tokens_per_cta(n, kFusedThreads / G);
  return 2 * ((n + T - 1) / T) >= device_sm_count();
}

cudaError_t launch_route_metadata(const float *logits, int64_t n, int E, int k, int gating,
                                  int32_t *topk_indx, uint16_t *topk_vals,
                                  const moe_routing_meta &meta,
                                  uint32_t *ctrl, cudaStream_t s, uint32_t *sync,
                                  const int32_t *expert_map, int E_loc, const uint16_t *x,
                                  int H, uint16_t *x_sorted) {
  if (!expert_map) E_loc = E;
  // every G (<= 8) lanes take a token: n <= 32 tokens fit one 256-thread CTA
  if (n * k <= kSmallSlots)
    return launch_route_metadata_small(logits, (int)n, E, k, gating, topk_indx, topk_vals, meta,
                                       sync, expert_map, E_loc, ctrl, s);
  return dispatch_kg(k, E, RouteMetaLaunch{logits, n, E, gating, topk_indx, topk_vals, &meta,
                                           ctrl, sync, expert_map, E_loc, x, H,
                                           x_sorted, s});
}

}  // namespace moe
