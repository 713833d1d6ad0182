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
#include <cooperative_groups.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {

int device_sm_count() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

// ================================================================ route ==
//
// One warp per token. Each lane holds the logits of experts lane, lane+32,
// ... as 64-bit keys: high word = an order-preserving image of the fp32
// value (-0.0 folded onto +0.0, NaN below every number), low word = ~e, so
// the largest key is the largest logit and, among equal logits, the lowest
// expert id. k rounds of a warp-shuffle max take the top k in order.

__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 0u;               // NaN: below every number
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7fffffffu) == 0u) u = 0u;  // -0.0 ties +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t key) {
  uint32_t u = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
  return __uint_as_float(u);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
    v = o > v ? o : v;
  }
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

template <int EPL>  // experts per lane: ceil(E / 32)
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int64_t n,
                                                    int E, int k, int gating,
                                                    int32_t *__restrict__ topk_indx,
                                                    uint16_t *__restrict__ topk_vals) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n;
       t += warps_total) {
    const float *row = logits + t * E;
    float v[EPL];
    unsigned long long key[EPL];
#pragma unroll
    for (int c = 0; c < EPL; ++c) {
      const int e = lane + 32 * c;
      if (e < E) {
        v[c] = __ldcs(row + e);
        key[c] = ((unsigned long long)order_key(v[c]) << 32) | (uint32_t)(~(uint32_t)e);
      } else {
        v[c] = 0.f;
        key[c] = 0ull;  // absent: below every present expert (low word of a present one is > 0)
      }
    }
    unsigned long long mine = 0ull;  // lane j keeps the j-th selection
    unsigned long long first = 0ull;
    for (int j = 0; j < k; ++j) {
      unsigned long long best = key[0];
#pragma unroll
      for (int c = 1; c < EPL; ++c) best = key[c] > best ? key[c] : best;
      best = warp_max_u64(best);
      const uint32_t e_best = ~(uint32_t)(best & 0xffffffffu);
      if ((int)(e_best & 31u) == lane) {
#pragma unroll
        for (int c = 0; c < EPL; ++c)
          if ((uint32_t)(lane + 32 * c) == e_best) key[c] = 0ull;
      }
      if (lane == j) mine = best;
      if (j == 0) first = best;
    }
    const float l0 = key_to_float((uint32_t)(first >> 32));
    const float lj = key_to_float((uint32_t)(mine >> 32));
    float denom;
    float num = lane < k ? expf(lj - l0) : 0.f;
    if (gating == MOE_GATING_SOFTMAX_TOPK) {
      denom = warp_sum(num);
    } else {
      float s = 0.f;
#pragma unroll
      for (int c = 0; c < EPL; ++c)
        if (lane + 32 * c < E) s += expf(v[c] - l0);
      denom = warp_sum(s);
    }
    if (lane < k) {
      topk_indx[t * k + lane] = (int32_t)(~(uint32_t)(mine & 0xffffffffu));
      topk_vals[t * k + lane] = float_to_bf16_bits(num / denom);
    }
  }
}

cudaError_t launch_route(const float *logits, int64_t n, int E, int k, int gating,
                         int32_t *topk_indx, uint16_t *topk_vals, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int threads = 256, warps = threads / 32;
  int64_t blocks = (n + warps - 1) / warps;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  const int epl = (E + 31) / 32;
#define ROUTE_CASE(N_)                                                                       \
  case N_:                                                                                   \
    route_kernel<N_><<<(unsigned)blocks, threads, 0, s>>>(logits, n, E, k, gating, topk_indx, \
                                                           topk_vals);                       \
    break;
  switch (epl) {
    ROUTE_CASE(1) ROUTE_CASE(2) ROUTE_CASE(3) ROUTE_CASE(4)
    ROUTE_CASE(5) ROUTE_CASE(6) ROUTE_CASE(7) ROUTE_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef ROUTE_CASE
  return cudaGetLastError();
}

// ============================================================= metadata ==
//
// One cooperative kernel; CTA b owns the contiguous slot range
// [b*chunk, min(N, (b+1)*chunk)).
//  phase 1  shared-memory histogram of the CTA's slots -> ws_hist[b][e]
//  barrier  bounded grid-wide barrier
//  phase 2  total[e] = sum_b ws_hist[b][e], before[e] = sum_{b'<b} ws_hist[b'][e];
//           offs = exclusive scan of total (warp scan); CTA 0 writes
//           col_sum and offs; base[e] = offs[e] + before[e]
//  phase 3  rounds of blockDim slots: a slot's rank among equal experts of
//           its warp (match_any + popc), plus the counts of lower warps,
//           plus base[e] gives its sorted position p. Stable in f with no
//           atomic deciding any position.

constexpr int kMetaThreads = 512;
constexpr int kMetaWarps = kMetaThreads / 32;

__global__ void __launch_bounds__(kMetaThreads) metadata_kernel(
    const int32_t *__restrict__ topk_indx, const uint16_t *__restrict__ topk_vals, int N, int E,
    int chunk, int32_t *__restrict__ col_sum, int32_t *__restrict__ offs,
    int32_t *__restrict__ col_sorted, int32_t *__restrict__ row_sorted,
    uint16_t *__restrict__ gate_scal, int32_t *__restrict__ ws_hist, uint32_t *ctrl,
    unsigned long long timeout_ns) {
  __shared__ int s_base[kMaxExperts];
  __shared__ int s_cnt[kMetaWarps][kMaxExperts];
  __shared__ int s_tot_part[kMetaThreads];
  __shared__ int s_pre_part[kMetaThreads];
  __shared__ int s_bad;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x, B = gridDim.x;
  const int lo = (int)min((int64_t)N, (int64_t)b * chunk);
  const int hi = (int)min((int64_t)N, (int64_t)lo + chunk);

  // ---- phase 1: histogram of this CTA's slots
  for (int e = tid; e < E; e += kMetaThreads) s_base[e] = 0;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int f = lo + tid; f < hi; f += kMetaThreads) {
    const int e = __ldg(topk_indx + f);
    if ((unsigned)e < (unsigned)E) atomicAdd(&s_base[e], 1);
    else s_bad = 1;
  }
  __syncthreads();
  if (s_bad) record_status(ctrl, MOE_ERR_INVALID_ARG);
  for (int e = tid; e < E; e += kMetaThreads) ws_hist[(size_t)b * E + e] = s_base[e];

  if (!grid_barrier(ctrl, timeout_ns)) return;

  // ---- phase 2: per-expert totals and the count in lower CTAs
  const int parts = kMetaThreads / E;  // >= 2 since E <= 256
  {
    int tot = 0, pre = 0;
    if (tid < parts * E) {
      const int e = tid % E, part = tid / E;
      const int b0 = (int)((int64_t)B * part / parts), b1 = (int)((int64_t)B * (part + 1) / parts);
      for (int bb = b0; bb < b1; ++bb) {
        const int v = __ldcg(ws_hist + (size_t)bb * E + e);
        tot += v;
        pre += bb < b ? v : 0;
      }
    }
    s_tot_part[tid] = tot;
    s_pre_part[tid] = pre;
  }
  __syncthreads();
  // warp 0: sums the parts and scans the totals 32 experts at a time
  if (warp == 0) {
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int tot = 0, pre = 0;
      if (e < E)
        for (int part = 0; part < parts; ++part) {
          tot += s_tot_part[part * E + e];
          pre += s_pre_part[part * E + e];
        }
      int incl = tot;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const int excl = carry + incl - tot;
      if (e < E) {
        s_base[e] = excl + pre;
        if (b == 0) {
          col_sum[e] = tot;
          offs[e] = excl;
        }
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (b == 0 && lane == 0) offs[E] = carry;
  }
  __syncthreads();

  // ---- phase 3: stable positions, round by round
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r0 = lo; r0 < hi; r0 += kMetaThreads) {
    for (int e = lane; e < E; e += 32) s_cnt[warp][e] = 0;
    __syncwarp();
    const int f = r0 + tid;
    const bool valid = f < hi;
    int e = valid ? __ldg(topk_indx + f) : -1;
    if ((unsigned)e >= (unsigned)E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0 && rank == 0) s_cnt[warp][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int p = s_base[e] + rank;
      for (int w = 0; w < warp; ++w) p += s_cnt[w][e];
      col_sorted[p] = f;
      row_sorted[f] = p;
      gate_scal[p] = __ldg(topk_vals + f);
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += kMetaThreads) {
      int add = 0;
      for (int w = 0; w < kMetaWarps; ++w) add += s_cnt[w][ee];
      s_base[ee] += add;
    }
    __syncthreads();
  }
}

cudaError_t launch_metadata(const int32_t *topk_indx, const uint16_t *topk_vals, int64_t n, int E,
                            int k, const moe_routing_meta &meta, int32_t *ws_hist,
                            uint32_t *ctrl, cudaStream_t s) {
  const int N = (int)(n * k);
  static int max_resident = 0;  // CTAs per SM of metadata_kernel (same on every GB300)
  if (max_resident == 0) {
    int per_sm = 0;
    cudaError_t err =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, metadata_kernel, kMetaThreads, 0);
    if (err != cudaSuccess) return err;
    max_resident = per_sm > 0 ? per_sm : 1;
  }
  const int64_t slots_per_cta = 1024;
  int64_t B = (N + slots_per_cta - 1) / slots_per_cta;
  const int64_t cap = (int64_t)device_sm_count() * max_resident;
  if (B > cap) B = cap;
  if (B > kMetaMaxCtas) B = kMetaMaxCtas;
  if (B < 1) B = 1;
  int chunk = (int)((N + B - 1) / B);
  unsigned long long timeout = kWaitTimeoutNs;

  void *args[] = {(void *)&topk_indx, (void *)&topk_vals, (void *)&N, (void *)&E,
                  (void *)&chunk, (void *)&meta.col_sum, (void *)&meta.offs,
                  (void *)&meta.col_sorted, (void *)&meta.row_sorted, (void *)&meta.gate_scal,
                  (void *)&ws_hist, (void *)&ctrl, (void *)&timeout};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(kMetaThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelExC(&cfg, (const void *)metadata_kernel, args);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
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
// static array. Clears the control words first (barrier counters and the
// status word must start at zero; the histograms are overwritten by every
// CTA before they are read), then copies the status word to status_out.
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

  int N = (int)(n * k);
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, metadata_kernel, kMetaThreads, 0);
  if (err != cudaSuccess) return err;
  int64_t B = (N + 1023) / 1024;
  const int64_t cap = (int64_t)device_sm_count() * (per_sm > 0 ? per_sm : 1);
  if (B > cap) B = cap;
  if (B > kNoAllocMaxCtas) B = kNoAllocMaxCtas;
  if (B < 1) B = 1;
  int chunk = (int)((N + B - 1) / B);
  unsigned long long timeout = kWaitTimeoutNs;
  void *args[] = {(void *)&topk_indx, (void *)&topk_vals, (void *)&N, (void *)&E,
                  (void *)&chunk, (void *)&meta.col_sum, (void *)&meta.offs,
                  (void *)&meta.col_sorted, (void *)&meta.row_sorted, (void *)&meta.gate_scal,
                  (void *)&hist, (void *)&ctrl, (void *)&timeout};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(kMetaThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelExC(&cfg, (const void *)metadata_kernel, args);
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
// MiniMind issue ("It is removable in plain PyTorch"), 16 bytes per thread.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4 *__restrict__ x,
                                                          const int32_t *__restrict__ col_sorted,
                                                          int64_t N, int k, int vec_per_row,
                                                          uint4 *__restrict__ x_sorted) {
  const int64_t total = N * vec_per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = i / vec_per_row;
    const int c = (int)(i - p * vec_per_row);
    const int32_t f = __ldg(col_sorted + p);
    // positions whose slot carried an out-of-range expert id are never
    // written by the metadata kernel (which flags MOE_ERR_INVALID_ARG)
    if ((uint32_t)f >= (uint32_t)N) continue;
    x_sorted[i] = __ldg(x + (int64_t)(f / k) * vec_per_row + c);
  }
}

cudaError_t launch_gather_rows(const uint16_t *x, const int32_t *col_sorted, int64_t N, int k,
                               int H, uint16_t *x_sorted, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  const int vpr = H / 8;
  int64_t blocks = (N * vpr + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  gather_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const uint4 *>(x),
                                                      col_sorted, N, k, vpr,
                                                      reinterpret_cast<uint4 *>(x_sorted));
  return cudaGetLastError();
}

// ============================================================= combine ==
// out[t] = sum_{j<k} y_flat[t*k + j] in fp32, j ascending, one bf16 rounding.
__global__ void __launch_bounds__(256) combine_kernel(const uint4 *__restrict__ y_flat, int64_t n,
                                                      int k, int vec_per_row,
                                                      uint4 *__restrict__ out) {
  const int64_t total = n * vec_per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / vec_per_row;
    const int c = (int)(i - t * vec_per_row);
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int j = 0; j < k; ++j) {
      const uint4 v = __ldcs(y_flat + (t * k + j) * vec_per_row + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += __uint_as_float(w[q] << 16);
        acc[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = (uint32_t)float_to_bf16_bits(acc[2 * q]) |
             ((uint32_t)float_to_bf16_bits(acc[2 * q + 1]) << 16);
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_combine(const uint16_t *y_flat, int64_t n, int k, int H, uint16_t *out,
                           cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int vpr = H / 8;
  int64_t blocks = (n * vpr + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  combine_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const uint4 *>(y_flat), n, k,
                                                  vpr, reinterpret_cast<uint4 *>(out));
  return cudaGetLastError();
}

// ======================================================= wait selftest ==
// Waits on a flag that nothing sets, with the same bounded wait as the grid
// barrier, so that a test can see the timeout path record MOE_ERR_TIMEOUT
// and return (no trap, no hang).
__global__ void wait_selftest_kernel(uint32_t *ctrl, unsigned long long timeout_ns) {
  if (threadIdx.x != 0) return;
  const uint32_t *never = ctrl + kCtrlBarGen + 1;  // a word no kernel writes
  const unsigned long long t0 = global_timer_ns();
  while (ld_acquire_gpu(never) == 0u) {
    if (global_timer_ns() - t0 > timeout_ns) {
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
