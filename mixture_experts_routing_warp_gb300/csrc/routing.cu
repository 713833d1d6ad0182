// routing.cu -- router top-k, routing metadata, dispatch gather, combine.
//
// Sources (page title, section):
//  "Reuse topk SparseMatrix routing metadata in GPT-OSS MoE forward"
//    (vLLM PR #45457 report), 关键源码片段: topk_fn(logits, k,
//    apply_softmax=True); mask_metadata {col_sum, row_sorted_indx,
//    col_sorted_indx}; gate_scal = vals.flatten()[combine_indx].
//  "MoE feed-forward performs ~3xnum_experts device->host syncs per layer,
//    per forward" (MiniMind issue #835), "It is removable in plain PyTorch":
//    stable sort by expert, tok = order // k, index_select; Summary:
//    y.index_add_ of the weighted expert outputs.
#include <mutex>

#include "routing_common.cuh"

namespace moe {

int device_sm_count() {
  static std::atomic<int> cached[PerDeviceOnce::kMaxDevices] = {};  // per device ordinal
  int dev = 0;
  cudaGetDevice(&dev);
  const bool slot = dev >= 0 && dev < PerDeviceOnce::kMaxDevices;
  if (slot) {
    const int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms < 1) sms = 1;
  if (slot) cached[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

template <int K, int G, int NQ>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(
    const float *__restrict__ logits, int64_t n, int E, int gating, int vec4,
    int32_t *__restrict__ topk_indx, uint16_t *__restrict__ topk_vals) {
  __shared__ float4 stash[NQ * kRouteThreads];  // the top-k's logit stash
  const int64_t groups = (int64_t)gridDim.x * (kRouteThreads / G);
  for (int64_t t0 = (int64_t)blockIdx.x * (kRouteThreads / G); t0 < n; t0 += groups) {
    const int64_t t = t0 + threadIdx.x / G;  // the loop bound is uniform over the block
    const bool valid = t < n;
    TopK<K> tk;
    float w[K];
    topk_group<K, G, NQ>(logits + (valid ? t : 0) * E, valid, E, gating, vec4 != 0, tk, w,
                         stash);
    if (valid) write_token<K, G, false>(t, 0, tk, w, topk_indx, topk_vals, nullptr, nullptr,
                                        nullptr);
  }
}

struct RouteLaunch {
  const float *logits;
  int64_t n;
  int E, gating;
  int32_t *indx;
  uint16_t *vals;
  cudaStream_t s;
  template <int K, int G, int NQ>
  cudaError_t go() {
    const int per_cta = kRouteThreads / G;
    int64_t blocks = (n + per_cta - 1) / per_cta;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    const int vec4 = (E % 4) == 0 && ((uintptr_t)logits % 16) == 0;
    static PerDeviceOnce configured;
    cudaError_t err = configured.run([] { return uniform_carveout(route_kernel<K, G, NQ>); });
    if (err != cudaSuccess) return err;
    route_kernel<K, G, NQ><<<(unsigned)blocks, kRouteThreads, 0, s>>>(logits, n, E, gating, vec4,
                                                                   indx, vals);
    return cudaGetLastError();
  }
};

cudaError_t launch_route(const float *logits, int64_t n, int E, int k, int gating,
                         int32_t *topk_indx, uint16_t *topk_vals, uint32_t *ctrl,
                         cudaStream_t s) {
  (void)ctrl;
  if (n == 0) return cudaSuccess;
  return dispatch_kg(k, E, RouteLaunch{logits, n, E, gating, topk_indx, topk_vals, s});
}

// Metadata from a top-k result in global memory (moe_build_metadata). With
// an expert map, over the E_loc local experts; other ranks' slots dropped.
__global__ void __launch_bounds__(kMetaThreads) metadata_kernel(
    const int32_t *__restrict__ topk_indx, const uint16_t *__restrict__ topk_vals, int N, int E,
    int chunk, int32_t *__restrict__ col_sum, int32_t *__restrict__ offs,
    int32_t *__restrict__ col_sorted, int32_t *__restrict__ row_sorted,
    uint16_t *__restrict__ gate_scal, int32_t *__restrict__ ws_hist, uint32_t *ctrl,
    unsigned long long timeout_ns, uint32_t *sync, const int32_t *__restrict__ expert_map,
    int E_loc) {
  __shared__ MetaShared<kMetaThreads> sh;
  __shared__ int s_map_buf[kMaxExperts];
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  pdl_launch_dependents();  // the next kernel may be scheduled (it waits for this grid)
  zero_sync_words(sync);
  const int *s_map = load_expert_map(expert_map, E, E_loc, s_map_buf, ctrl);
  const int lo = (int)min((int64_t)N, (int64_t)b * chunk);
  const int hi = (int)min((int64_t)N, (int64_t)lo + chunk);
  // local expert of a slot: -1 when dropped (another rank's) or invalid
  auto local = [&](int e) { return (unsigned)e < (unsigned)E ? (s_map ? s_map[e] : e) : -1; };

  for (int e = tid; e < E_loc; e += kMetaThreads) sh.base[e] = 0;
  if (tid == 0) sh.bad = 0;
  __syncthreads();
  for (int f = lo + tid; f < hi; f += kMetaThreads) {
    const int e = __ldg(topk_indx + f);
    if ((unsigned)e >= (unsigned)E) sh.bad = 1;
    const int le = local(e);
    if (le >= 0) atomicAdd(&sh.base[le], 1);
  }
  __syncthreads();
  if (sh.bad && tid == 0) record_status(ctrl, MOE_ERR_INVALID_ARG);

  if (!meta_barrier_prefix(ws_hist, E_loc, sh, col_sum, offs, ctrl, timeout_ns, [] {})) return;
  meta_scatter(
      lo, hi - lo, E_loc, sh,
      [&](int i, int &e, uint16_t &w) {
        e = local(__ldg(topk_indx + lo + i));
        w = __ldg(topk_vals + lo + i);
      },
      col_sorted, row_sorted, gate_scal);
}

int metadata_ctas_per_sm() {
  // CTAs per SM of metadata_kernel, per device ordinal
  static std::atomic<int> cached[PerDeviceOnce::kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool slot = dev >= 0 && dev < PerDeviceOnce::kMaxDevices;
  if (slot) {
    const int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int v = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, metadata_kernel, kMetaThreads, 0) !=
      cudaSuccess)
    return 1;
  v = v > 0 ? v : 1;
  if (slot) cached[dev].store(v, std::memory_order_relaxed);
  return v;
}

cudaError_t launch_metadata_kernel(const int32_t *topk_indx, const uint16_t *topk_vals, int N,
                                   int E, const moe_routing_meta &meta, int32_t *ws_hist,
                                   uint32_t *ctrl, int max_ctas, cudaStream_t s,
                                   uint32_t *sync = nullptr, const int32_t *expert_map = nullptr,
                                   int E_loc = 0) {
  if (!expert_map) E_loc = E;
  static PerDeviceOnce configured;
  {
    cudaError_t err = configured.run([] { return uniform_carveout(metadata_kernel); });
    if (err != cudaSuccess) return err;
  }
  const int64_t slots_per_cta = 1024;
  int64_t B = (N + slots_per_cta - 1) / slots_per_cta;
  const int64_t cap = (int64_t)device_sm_count() * metadata_ctas_per_sm();
  if (B > cap) B = cap;
  if (B > max_ctas) B = max_ctas;
  if (B < 1) B = 1;
  int chunk = (int)((N + B - 1) / B);
  unsigned long long timeout = kWaitTimeoutNs;
  void *args[] = {(void *)&topk_indx, (void *)&topk_vals, (void *)&N, (void *)&E,
                  (void *)&chunk, (void *)&meta.col_sum, (void *)&meta.offs,
                  (void *)&meta.col_sorted, (void *)&meta.row_sorted, (void *)&meta.gate_scal,
                  (void *)&ws_hist, (void *)&ctrl, (void *)&timeout, (void *)&sync,
                  (void *)&expert_map, (void *)&E_loc};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(kMetaThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = B > 1 ? 1 : 0;  // one CTA needs no co-residency guarantee
  cudaError_t err = cudaLaunchKernelExC(&cfg, (const void *)metadata_kernel, args);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_metadata(const int32_t *topk_indx, const uint16_t *topk_vals, int64_t n, int E,
                            int k, const moe_routing_meta &meta, int32_t *ws_hist,
                            uint32_t *ctrl, cudaStream_t s, uint32_t *sync,
                            const int32_t *expert_map, int E_loc) {
  return launch_metadata_kernel(topk_indx, topk_vals, (int)(n * k), E, meta, ws_hist, ctrl,
                                kMetaMaxCtas, s, sync, expert_map, E_loc);
}

// ======================================== metadata without a workspace ==
//
// Some callers cannot hand this library any device memory beyond the
// tensors they already own: code that runs while a framework's allocator
// owns every byte (a plugin asked to enqueue work with no workspace of its
// own), code on a latency-critical path where any cudaMalloc is forbidden
// because it can synchronise the device, or code inside a region that must
// not allocate at all. For them moe_build_metadata_noalloc runs the same
// metadata kernel with its scratch (the control block and the per-CTA
// histograms) in the fixed array below instead of a caller workspace.
//
// The array lives in every GPU that loads the library, until the process
// exits: 4 KB of control words plus 256 CTAs x 256 experts of int32
// counters (266,240 bytes). The kernel never needs more: this variant caps
// its grid at 256 CTAs, each CTA looping over as many slots as it must.
constexpr int kNoAllocMaxCtas = 256;
constexpr size_t kNoAllocScratchBytes =
    kCtrlBytes + (size_t)kNoAllocMaxCtas * (size_t)kMaxExperts * sizeof(int32_t);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device. In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
cudaError_t noalloc_scratch(void **out) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}
}  // namespace

// Same kernel and the same results as launch_metadata; scratch in the
// static array. Clears the control words first (the grid-barrier counter
// and the status word must start at zero; the histograms are overwritten by
// every CTA before they are read), then copies the status word to
// status_out.
cudaError_t launch_metadata_noalloc(const int32_t *topk_indx, const uint16_t *topk_vals,
                                    int64_t n, int E, int k, const moe_routing_meta &meta,
                                    int32_t *status_out, cudaStream_t s) {
  void *scratch = nullptr;
  cudaError_t err = noalloc_scratch(&scratch);
  if (err != cudaSuccess) return err;
  uint32_t *ctrl = static_cast<uint32_t *>(scratch);
  int32_t *hist = reinterpret_cast<int32_t *>(static_cast<char *>(scratch) + kCtrlBytes);
  err = cudaMemsetAsync(scratch, 0, kCtrlBytes, s);
  if (err != cudaSuccess) return err;

  err = launch_metadata_kernel(topk_indx, topk_vals, (int)(n * k), E, meta, hist, ctrl,
                               kNoAllocMaxCtas, s);
  if (err != cudaSuccess) return err;
  if (status_out) {
    err = cudaMemcpyAsync(status_out, ctrl + kCtrlStatus, sizeof(int32_t),
                          cudaMemcpyDeviceToDevice, s);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

// ======================================================= gather rows ==
// X_sorted[p] = x[col_sorted[p] / k]: the dispatch index_select of the
// MiniMind issue ("It is removable in plain PyTorch"), done token-major by
// copy_token_rows: x is read from memory once rather than once per slot.
// (moe_forward runs it only where neither the fused route + metadata kernel
// nor the w13 contraction moves the rows.) Block 0 also zeroes the sync
// words of this forward's expert contractions.
constexpr int kCopyThreads = 256;

constexpr int kChunksPerLane = 4;  // 16-byte chunks in flight per thread (copy_token_rows)

__global__ void __launch_bounds__(kCopyThreads) gather_rows_kernel(
    const uint4 *__restrict__ x, const int32_t *__restrict__ row_sorted, int64_t n, int k,
    int vec_per_row, uint4 *__restrict__ x_sorted, uint32_t *sync) {
  pdl_launch_dependents();
  pdl_wait();  // row_sorted comes from the metadata kernel
  if (sync && blockIdx.x == 0)
    for (int i = threadIdx.x; i < kSyncWords; i += kCopyThreads) sync[i] = 0;
  copy_token_rows(x, row_sorted, 0, n, k, vec_per_row, n * k, x_sorted,
                  (int64_t)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5),
                  (int64_t)gridDim.x * (kCopyThreads / 32));
}

cudaError_t launch_gather_rows(const uint16_t *x, const int32_t *row_sorted, int64_t n, int k,
                               int H, uint16_t *x_sorted, uint32_t *sync, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  static PerDeviceOnce configured;
  {
    cudaError_t err = configured.run([] { return uniform_carveout(gather_rows_kernel); });
    if (err != cudaSuccess) return err;
  }
  const int vpr = H / 8, gpr = (vpr + 32 * kChunksPerLane - 1) / (32 * kChunksPerLane);
  int64_t blocks = (n * gpr + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  cudaError_t err = launch_dependent(gather_rows_kernel, dim3((unsigned)blocks), dim3(kCopyThreads),
                                     0, s, reinterpret_cast<const uint4 *>(x), row_sorted, n, k,
                                     vpr, reinterpret_cast<uint4 *>(x_sorted), sync);
  return err != cudaSuccess ? err : cudaGetLastError();
}

// ============================================================= combine ==
// out[t] = sum_{j<k} y_flat[t*k + j] in fp32, j ascending, one bf16 rounding.
// A warp per (token, group of 64 16-byte chunks), 2 chunks x k slots in
// flight per thread. With row_sorted (an expert map in use), slots without a
// sorted position (another rank's expert: row_sorted -1) are left out; their
// y_flat rows were never written.
__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 &v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] += __uint_as_float(w[q] << 16);
    acc[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
  }
}

template <int K>
__global__ void __launch_bounds__(kCopyThreads) combine_kernel(const uint4 *__restrict__ y_flat,
                                                               int64_t n, int vec_per_row,
                                                               int groups_per_row,
                                                               uint4 *__restrict__ out,
                                                               const int32_t *row_sorted) {
  constexpr int CPL = 2;  // chunks per lane: 2*K loads in flight
  pdl_launch_dependents();
  pdl_wait();  // y_flat comes from the w2 contraction
  const int lane = threadIdx.x & 31;
  const int64_t units = n * groups_per_row;  // (token, group of 64 chunks) per warp
  const int64_t warps = (int64_t)gridDim.x * (kCopyThreads / 32);
  for (int64_t u = (int64_t)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5); u < units;
       u += warps) {
    const int64_t t = u / groups_per_row;
    const int c0 = (int)(u - t * groups_per_row) * 32 * CPL + lane;
    const uint4 *src = y_flat + t * K * vec_per_row;
    bool kept[K];
#pragma unroll
    for (int j = 0; j < K; ++j) kept[j] = !row_sorted || __ldg(row_sorted + t * K + j) >= 0;
    uint4 v[CPL][K];
#pragma unroll
    for (int q = 0; q < CPL; ++q)
#pragma unroll
      for (int j = 0; j < K; ++j)
        v[q][j] = c0 + 32 * q < vec_per_row && kept[j]
                      ? __ldcs(src + (int64_t)j * vec_per_row + c0 + 32 * q)
                      : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const int c = c0 + 32 * q;
      if (c >= vec_per_row) continue;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < K; ++j) add_bf16x8(acc, v[q][j]);
      uint32_t o[4];
#pragma unroll
      for (int w = 0; w < 4; ++w)
        o[w] = (uint32_t)float_to_bf16_bits(acc[2 * w]) |
               ((uint32_t)float_to_bf16_bits(acc[2 * w + 1]) << 16);
      out[t * vec_per_row + c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

cudaError_t launch_combine(const uint16_t *y_flat, int64_t n, int k, int H, uint16_t *out,
                           cudaStream_t s, const int32_t *row_sorted) {
  if (n == 0) return cudaSuccess;
  const int vpr = H / 8, gpr = (vpr + 63) / 64;
  int64_t blocks = (n * gpr + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  const uint4 *y = reinterpret_cast<const uint4 *>(y_flat);
  uint4 *o = reinterpret_cast<uint4 *>(out);
  static PerDeviceOnce configured[9];
  switch (k) {
#define MOE_COMBINE_CASE(K_)                                                       \
  case K_:                                                                         \
    {                                                                              \
      cudaError_t err =                                                            \
          configured[K_].run([] { return uniform_carveout(combine_kernel<K_>); }); \
      if (err != cudaSuccess) return err;                                          \
    }                                                                              \
    {                                                                              \
      cudaError_t err = launch_dependent(combine_kernel<K_>, dim3((unsigned)blocks),  \
                                         dim3(kCopyThreads), 0, s, y, n, vpr, gpr, o,  \
                                         row_sorted);                              \
      if (err != cudaSuccess) return err;                                          \
    }                                                                              \
    break;
    MOE_COMBINE_CASE(1) MOE_COMBINE_CASE(2) MOE_COMBINE_CASE(3) MOE_COMBINE_CASE(4)
    MOE_COMBINE_CASE(5) MOE_COMBINE_CASE(6) MOE_COMBINE_CASE(7) MOE_COMBINE_CASE(8)
#undef MOE_COMBINE_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ======================================================= wait selftest ==
// Waits on a flag that nothing sets, with the same bounded wait as the grid
// barrier, so that a test can see the timeout path record MOE_ERR_TIMEOUT
// and return (no trap, no hang).
__global__ void wait_selftest_kernel(uint32_t *ctrl, unsigned long long timeout_ns) {
  if (threadIdx.x != 0) return;
  const uint32_t *never = ctrl + kCtrlNeverSet;
  const long long deadline = wait_deadline(timeout_ns);
  while (ld_acquire_gpu(never) == 0u) {
    if (clock64() > deadline) {
      record_status(ctrl, MOE_ERR_TIMEOUT);
      return;
    }
    __nanosleep(256);
  }
}

cudaError_t launch_wait_selftest(uint32_t *ctrl, unsigned long long timeout_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(ctrl, timeout_ns);
  return cudaGetLastError();
}

}  // namespace moe

// The C entry point of the no-allocation variant (declared in include/moe.h).
extern "C" moe_status moe_build_metadata_noalloc(const int32_t *topk_indx,
                                                 const uint16_t *topk_vals, int64_t n, int32_t E,
                                                 int32_t k, const moe_routing_meta *meta,
                                                 int32_t *status_out, moe_stream stream) {
  using namespace moe;
  // Sizes beyond what this variant (and its fixed scratch) handles.
  if (n < 0 || E < 1 || E > kMaxExperts || k < 1 || k > kMaxTopk || k > E)
    return MOE_ERR_INVALID_ARG;
  if (n * (int64_t)k >= (int64_t)INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (!meta || !meta->col_sum || !meta->offs) return MOE_ERR_INVALID_ARG;
  if (n > 0 && (!meta->col_sorted || !meta->row_sorted || !meta->gate_scal || !topk_indx ||
                !topk_vals))
    return MOE_ERR_INVALID_ARG;
  auto misaligned = [](const void *p, uintptr_t a) { return ((uintptr_t)p % a) != 0; };
  if (misaligned(meta->col_sum, 4) || misaligned(meta->offs, 4) ||
      misaligned(meta->col_sorted, 4) || misaligned(meta->row_sorted, 4) ||
      misaligned(meta->gate_scal, 2) || misaligned(topk_indx, 4) || misaligned(topk_vals, 2) ||
      misaligned(status_out, 4))
    return MOE_ERR_MISALIGNED;
  cudaError_t err = launch_metadata_noalloc(topk_indx, topk_vals, n, E, k, *meta, status_out,
                                            (cudaStream_t)stream);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
