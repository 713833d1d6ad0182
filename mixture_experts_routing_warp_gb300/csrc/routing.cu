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

#include "moe_internal.cuh"

namespace moe {

int device_sm_count() {
  static int cached[64] = {};  // per device ordinal
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms < 1) sms = 1;
  if (dev >= 0 && dev < 64) cached[dev] = sms;
  return sms;
}

// ================================================================ route ==
//
// Router top-k. G consecutive lanes share a token (G = 1, 2, 4, 8 for E up
// to 16, 32, 64, 256: at most 16 elements per lane up to E = 128, so that
// enough warps are in flight to hide the compare chains): lane g of the
// group loads the 16-byte
// chunks g, g+G, g+2G, ... of the token's fp32 row (all its loads in flight
// at once; the G lanes of a token read adjacent chunks), and keeps the K
// largest 32-bit order keys (an order-preserving image of the value: -0.0
// folded onto +0.0, NaN = 1 below every number) of its elements in
// registers. Within a lane the elements arrive in ascending expert id and
// a key enters only if strictly larger, so equal logits keep the lower id;
// the lanes of a group then merge their lists in log2(G) shuffle steps,
// ordering by (value descending, expert id ascending). Gate weights:
// softmax in fp32 over the K selected (or over all E), rounded to bf16.

constexpr int kRouteThreads = 256;
constexpr int kFusedThreads = 1024;
constexpr int kSlotCap = 8192;  // slots a fused CTA keeps in shared memory

// Top-K of token row `row` (E fp32) by the G lanes of a group; lane g =
// lane % G. On return every lane of the group holds the merged list and
// the K gate weights. `valid` is uniform within a group.
__device__ __forceinline__ unsigned long long pack_key(uint32_t key, int e) {
  return ((unsigned long long)key << 32) | (uint32_t)~(uint32_t)e;
}

// compare-exchange: a gets the larger, b the smaller
__device__ __forceinline__ void cx(unsigned long long &a, unsigned long long &b) {
  const bool s = b > a;
  const unsigned long long hi = s ? b : a, lo = s ? a : b;
  a = hi;
  b = lo;
}

__device__ __forceinline__ void sort4_desc(unsigned long long (&c)[4]) {
  cx(c[0], c[1]);
  cx(c[2], c[3]);
  cx(c[0], c[2]);
  cx(c[1], c[3]);
  cx(c[1], c[2]);
}

// top <- the 4 largest of top (sorted) and o (sorted), sorted descending:
// elementwise max of top and reversed o is bitonic; two half-cleaner stages.
__device__ __forceinline__ void merge4_desc(unsigned long long (&top)[4],
                                            const unsigned long long (&o)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) top[j] = top[j] > o[3 - j] ? top[j] : o[3 - j];
  cx(top[0], top[2]);
  cx(top[1], top[3]);
  cx(top[0], top[1]);
  cx(top[2], top[3]);
}

// vec4: rows are 16-byte aligned (E % 4 == 0 and a 16-byte aligned base),
// so a chunk is one 128-bit load; otherwise four 32-bit loads.
template <int K, int G, int NQ>  // NQ chunks of 4 elements per lane: NQ*4*G >= E
__device__ __forceinline__ void topk_group(const float *__restrict__ row, bool valid, int E,
                                           int gating, bool vec4, TopK<K> &tk, float (&w)[K]) {
  const int lane = threadIdx.x & 31, g = lane % G;
  tk.init();
  const int nq = (E + 3) >> 2;  // chunks of 4 elements in the row
  float4 x[NQ];
  if (vec4) {
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      const int q = i * G + g;
      x[i] = (valid && q < nq) ? __ldg(reinterpret_cast<const float4 *>(row) + q)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  } else {
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      const int e0 = (i * G + g) * 4;
      const bool ok = valid && e0 < E;
      x[i].x = ok ? __ldg(row + e0) : 0.f;
      x[i].y = ok && e0 + 1 < E ? __ldg(row + e0 + 1) : 0.f;
      x[i].z = ok && e0 + 2 < E ? __ldg(row + e0 + 2) : 0.f;
      x[i].w = ok && e0 + 3 < E ? __ldg(row + e0 + 3) : 0.f;
    }
  }
  if constexpr (K <= 4) {
    // Branch-free: packed keys ((order key << 32) | ~id) are unique and
    // "larger" means (value descending, id ascending). Sort each chunk of 4
    // with a 5-comparator network, then bitonic-merge the sorted 4-lists
    // (inside the lane, then across the G lanes), keeping the top 4.
    unsigned long long top[4];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      const int e0 = (i * G + g) * 4;
      unsigned long long c[4];
      c[0] = e0 < E ? pack_key(order_key(x[i].x), e0) : 0ull;
      c[1] = e0 + 1 < E ? pack_key(order_key(x[i].y), e0 + 1) : 0ull;
      c[2] = e0 + 2 < E ? pack_key(order_key(x[i].z), e0 + 2) : 0ull;
      c[3] = e0 + 3 < E ? pack_key(order_key(x[i].w), e0 + 3) : 0ull;
      sort4_desc(c);
      if (i == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) top[j] = c[j];
      } else {
        merge4_desc(top, c);
      }
    }
#pragma unroll
    for (int off = 1; off < G; off <<= 1) {
      unsigned long long o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] = __shfl_xor_sync(0xffffffffu, top[j], off);
      merge4_desc(top, o);
    }
#pragma unroll
    for (int j = 0; j < K; ++j) {
      tk.key[j] = (uint32_t)(top[j] >> 32);
      tk.e[j] = (int)~(uint32_t)top[j];
    }
  } else {
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      const int e0 = (i * G + g) * 4;
      if (e0 < E) {
        tk.push_ascending(order_key(x[i].x), e0);
        if (e0 + 1 < E) tk.push_ascending(order_key(x[i].y), e0 + 1);
        if (e0 + 2 < E) tk.push_ascending(order_key(x[i].z), e0 + 2);
        if (e0 + 3 < E) tk.push_ascending(order_key(x[i].w), e0 + 3);
      }
    }
#pragma unroll
    for (int off = 1; off < G; off <<= 1) {  // butterfly merge inside the group
      uint32_t pk[K];
      int pe[K];
#pragma unroll
      for (int i = 0; i < K; ++i) {
        pk[i] = __shfl_xor_sync(0xffffffffu, tk.key[i], off);
        pe[i] = __shfl_xor_sync(0xffffffffu, tk.e[i], off);
      }
#pragma unroll
      for (int i = 0; i < K; ++i) tk.push_any(pk[i], pe[i]);
    }
  }
  const float v0 = key_to_float(tk.key[0]);
  float ex[K];
  float denom = 0.f;
#pragma unroll
  for (int i = 0; i < K; ++i) {
    ex[i] = expf(key_to_float(tk.key[i]) - v0);
    denom += ex[i];
  }
  if (gating == MOE_GATING_SOFTMAX_ALL) {
    float s = 0.f;  // this lane's elements, ascending chunks, then a fixed tree
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      const int e0 = (i * G + g) * 4;
      if (e0 < E) s += expf(x[i].x - v0);
      if (e0 + 1 < E) s += expf(x[i].y - v0);
      if (e0 + 2 < E) s += expf(x[i].z - v0);
      if (e0 + 3 < E) s += expf(x[i].w - v0);
    }
#pragma unroll
    for (int off = 1; off < G; off <<= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    denom = s;
  }
#pragma unroll
  for (int i = 0; i < K; ++i) w[i] = ex[i] / denom;
}

// Outputs of one token: lane g of the group writes entries j = g, g+G, ...
template <int K, int G, bool KEEP>
__device__ __forceinline__ void write_token(int64_t t, int64_t t0, const TopK<K> &tk,
                                            const float (&w)[K], int32_t *__restrict__ topk_indx,
                                            uint16_t *__restrict__ topk_vals, uint8_t *s_slot_e,
                                            uint16_t *s_slot_v, int *s_hist) {
  const int g = (threadIdx.x & 31) % G;
#pragma unroll
  for (int j = 0; j < K; ++j) {
    if (j % G != g) continue;
    const uint16_t wb = float_to_bf16_bits(w[j]);
    if (!KEEP) {  // KEEP: the caller writes the outputs from the slots
      topk_indx[t * K + j] = tk.e[j];
      topk_vals[t * K + j] = wb;
    } else {
      const int s = (int)(t - t0) * K + j;
      s_slot_e[s] = (uint8_t)tk.e[j];
      s_slot_v[s] = wb;
      atomicAdd(&s_hist[tk.e[j]], 1);
    }
  }
}

template <int K, int G, int NQ>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(
    const float *__restrict__ logits, int64_t n, int E, int gating, int vec4,
    int32_t *__restrict__ topk_indx, uint16_t *__restrict__ topk_vals) {
  const int64_t groups = (int64_t)gridDim.x * (kRouteThreads / G);
  for (int64_t t0 = (int64_t)blockIdx.x * (kRouteThreads / G); t0 < n; t0 += groups) {
    const int64_t t = t0 + threadIdx.x / G;  // the loop bound is uniform over the block
    const bool valid = t < n;
    TopK<K> tk;
    float w[K];
    topk_group<K, G, NQ>(logits + (valid ? t : 0) * E, valid, E, gating, vec4 != 0, tk, w);
    if (valid) write_token<K, G, false>(t, 0, tk, w, topk_indx, topk_vals, nullptr, nullptr,
                                        nullptr);
  }
}

template <typename F>
cudaError_t dispatch_kg(int k, int E, F &&f) {
  // (G, NQ) by expert count: E <= 16: (1, 4); <= 32: (2, 4); <= 64: (4, 4);
  // <= 128: (8, 4); <= 256: (8, 8)
#define MOE_G_CASES(K_)                                   \
  if (E <= 16) return f.template go<K_, 1, 4>();          \
  if (E <= 32) return f.template go<K_, 2, 4>();          \
  if (E <= 64) return f.template go<K_, 4, 4>();          \
  if (E <= 128) return f.template go<K_, 8, 4>();         \
  return f.template go<K_, 8, 8>();
  switch (k) {
    case 1: MOE_G_CASES(1)
    case 2: MOE_G_CASES(2)
    case 3: MOE_G_CASES(3)
    case 4: MOE_G_CASES(4)
    case 5: MOE_G_CASES(5)
    case 6: MOE_G_CASES(6)
    case 7: MOE_G_CASES(7)
    default: MOE_G_CASES(8)
  }
#undef MOE_G_CASES
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
    static bool configured = false;
    if (!configured) {
      cudaError_t err = uniform_carveout(route_kernel<K, G, NQ>);
      if (err != cudaSuccess) return err;
      configured = true;
    }
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

// ============================================================= metadata ==
//
// Cross-CTA part of the metadata, shared by the kernels below. CTA b of B
// owns a contiguous range of slots and counts them per expert in shared
// memory. Then:
//  barrier  the counts go to row b of ws_hist (stride = E rounded up to 4);
//           bounded grid barrier
//  prefix   (expert group of 4, part of the rows) threads load the rows as
//           int4, all rows of a batch in flight together:
//           total[e] = sum_b counts[b][e], before[e] = sum_{b'<b} counts[b'][e];
//           parts summed per expert, warp 0 scans: offs = exclusive scan of
//           total; CTA 0 writes col_sum and offs; base[e] = offs[e] + before[e]
//  scatter  rounds of blockDim slots: a slot's rank among equal experts of
//           its warp (match_any + popc) plus the slots of that expert in
//           lower warps plus base[e] is its sorted position p. Stable in f;
//           no atomic decides any position.

constexpr int kMetaThreads = 512;   // metadata_kernel
constexpr int kMaxParts = 32;

template <int THREADS>
struct __align__(16) MetaShared {  // tot / pre take int4 stores
  static constexpr int kWarps = THREADS / 32;
  // rows loaded together per thread in the prefix (fewer with more threads:
  // registers per thread halve, rows per thread halve)
  static constexpr int kBatch = THREADS >= 1024 ? 8 : 16;
  static constexpr int kPartInts = 1024;  // parts * stride never exceeds this
  int base[kMaxExperts];
  int cnt[kWarps][kMaxExperts];
  int tot[kPartInts];
  int pre[kPartInts];
  int bad;
};

// Threads of the prefix: `parts` groups of E4 threads, each part summing a
// range of CTA rows into tot/pre[part * stride ..]; parts * stride must fit
// in kPartInts and parts * E4 in the block.
__host__ __device__ __forceinline__ int prefix_parts(int threads, int stride) {
  int parts = threads / (stride / 4);
  if (parts > kMaxParts) parts = kMaxParts;
  if (parts > 1024 / stride) parts = 1024 / stride;
  return parts < 1 ? 1 : parts;
}

__host__ __device__ __forceinline__ int hist_stride(int E) { return (E + 3) & ~3; }

// Warp 0: exclusive scan of the totals sh.tot[0..E) 32 experts at a time;
// sh.base[e] = offs[e] + sh.pre[e]; CTA 0 writes col_sum and offs.
template <int THREADS>
__device__ void meta_scan(int E, MetaShared<THREADS> &sh, int32_t *__restrict__ col_sum,
                          int32_t *__restrict__ offs) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == 0) {
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int tot = e < E ? sh.tot[e] : 0;
      const int pre = e < E ? sh.pre[e] : 0;
      int incl = tot;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const int excl = carry + incl - tot;
      if (e < E) {
        sh.base[e] = excl + pre;
        if (blockIdx.x == 0) {
          col_sum[e] = tot;
          offs[e] = excl;
        }
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (blockIdx.x == 0 && lane == 0) offs[E] = carry;
  }
  __syncthreads();
}

// Publish this CTA's counts (in sh.base[0..E)), pass the grid barrier, read
// every CTA's and build sh.base = offs + before. `between` runs (every
// thread) after this CTA's arrival and before its wait. Returns false after
// a timeout.
template <int THREADS, typename Between>
__device__ bool meta_barrier_prefix(int32_t *__restrict__ ws_hist, int E, MetaShared<THREADS> &sh,
                                    int32_t *__restrict__ col_sum, int32_t *__restrict__ offs,
                                    uint32_t *ctrl, unsigned long long timeout_ns,
                                    Between between) {
  const int tid = threadIdx.x;
  const int b = blockIdx.x, B = gridDim.x;
  const int stride = hist_stride(E), E4 = stride / 4;
  if (B == 1) {  // one CTA holds every slot: no exchange, no barrier
    between();
    for (int e = tid; e < E; e += THREADS) {
      sh.tot[e] = sh.base[e];
      sh.pre[e] = 0;
    }
    __syncthreads();
    meta_scan(E, sh, col_sum, offs);
    return true;
  }
  int32_t *row = ws_hist + (size_t)b * stride;
  for (int e = tid; e < stride; e += THREADS) row[e] = e < E ? sh.base[e] : 0;
  const uint32_t arrived = grid_arrive(ctrl);
  between();
  if (!grid_wait(ctrl, arrived, timeout_ns)) return false;

  const int parts = prefix_parts(THREADS, stride);
  if (tid < parts * E4) {
    const int g = tid % E4, part = tid / E4;
    const int b0 = (int)((int64_t)B * part / parts), b1 = (int)((int64_t)B * (part + 1) / parts);
    int4 tot = make_int4(0, 0, 0, 0), pre = make_int4(0, 0, 0, 0);
    for (int base = b0; base < b1; base += MetaShared<THREADS>::kBatch) {
      int4 v[MetaShared<THREADS>::kBatch];
#pragma unroll
      for (int q = 0; q < MetaShared<THREADS>::kBatch; ++q)
        v[q] = base + q < b1
                   ? __ldcg(reinterpret_cast<const int4 *>(ws_hist + (size_t)(base + q) * stride) +
                            g)
                   : make_int4(0, 0, 0, 0);
#pragma unroll
      for (int q = 0; q < MetaShared<THREADS>::kBatch; ++q) {
        tot.x += v[q].x;
        tot.y += v[q].y;
        tot.z += v[q].z;
        tot.w += v[q].w;
        if (base + q < b) {
          pre.x += v[q].x;
          pre.y += v[q].y;
          pre.z += v[q].z;
          pre.w += v[q].w;
        }
      }
    }
    reinterpret_cast<int4 *>(sh.tot + part * stride)[g] = tot;
    reinterpret_cast<int4 *>(sh.pre + part * stride)[g] = pre;
  }
  __syncthreads();
  for (int e = tid; e < E; e += THREADS) {  // sum the parts, one thread per expert
    int tot = 0, pre = 0;
    for (int part = 0; part < parts; ++part) {
      tot += sh.tot[part * stride + e];
      pre += sh.pre[part * stride + e];
    }
    sh.tot[e] = tot;  // part 0's row now holds the sums
    sh.pre[e] = pre;
  }
  __syncthreads();
  meta_scan(E, sh, col_sum, offs);
  return true;
}

template <int THREADS, typename Get>
__device__ void meta_scatter(int64_t f_lo, int count, int E, MetaShared<THREADS> &sh, Get get,
                             int32_t *__restrict__ col_sorted, int32_t *__restrict__ row_sorted,
                             uint16_t *__restrict__ gate_scal) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r0 = 0; r0 < count; r0 += THREADS) {
    for (int e = lane; e < E; e += 32) sh.cnt[warp][e] = 0;
    __syncwarp();
    const int i = r0 + tid;
    int e = -1;
    uint16_t w = 0;
    if (i < count) get(i, e, w);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0 && rank == 0) sh.cnt[warp][e] = __popc(peers);
    __syncthreads();
    // cnt[w][e] -> base[e] + (slots of expert e in warps < w); base[e] += all
    for (int ee = tid; ee < E; ee += THREADS) {
      int run = sh.base[ee];
#pragma unroll
      for (int ww = 0; ww < MetaShared<THREADS>::kWarps; ++ww) {
        const int c = sh.cnt[ww][ee];
        sh.cnt[ww][ee] = run;
        run += c;
      }
      sh.base[ee] = run;
    }
    __syncthreads();
    if (e >= 0) {
      const int p = sh.cnt[warp][e] + rank;
      const int32_t f = (int32_t)(f_lo + i);
      col_sorted[p] = f;
      row_sorted[f] = p;
      gate_scal[p] = w;
    }
    __syncthreads();
  }
}

// Metadata from a top-k result in global memory (moe_build_metadata).
__global__ void __launch_bounds__(kMetaThreads) metadata_kernel(
    const int32_t *__restrict__ topk_indx, const uint16_t *__restrict__ topk_vals, int N, int E,
    int chunk, int32_t *__restrict__ col_sum, int32_t *__restrict__ offs,
    int32_t *__restrict__ col_sorted, int32_t *__restrict__ row_sorted,
    uint16_t *__restrict__ gate_scal, int32_t *__restrict__ ws_hist, uint32_t *ctrl,
    unsigned long long timeout_ns) {
  __shared__ MetaShared<kMetaThreads> sh;
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  pdl_launch_dependents();  // the gather may be scheduled (it waits for this grid)
  const int lo = (int)min((int64_t)N, (int64_t)b * chunk);
  const int hi = (int)min((int64_t)N, (int64_t)lo + chunk);

  for (int e = tid; e < E; e += kMetaThreads) sh.base[e] = 0;
  if (tid == 0) sh.bad = 0;
  __syncthreads();
  for (int f = lo + tid; f < hi; f += kMetaThreads) {
    const int e = __ldg(topk_indx + f);
    if ((unsigned)e < (unsigned)E) atomicAdd(&sh.base[e], 1);
    else sh.bad = 1;
  }
  __syncthreads();
  if (sh.bad && tid == 0) record_status(ctrl, MOE_ERR_INVALID_ARG);

  if (!meta_barrier_prefix(ws_hist, E, sh, col_sum, offs, ctrl, timeout_ns, [] {})) return;
  meta_scatter(
      lo, hi - lo, E, sh,
      [&](int i, int &e, uint16_t &w) {
        e = __ldg(topk_indx + lo + i);
        if ((unsigned)e >= (unsigned)E) e = -1;
        w = __ldg(topk_vals + lo + i);
      },
      col_sorted, row_sorted, gate_scal);
}

int metadata_ctas_per_sm() {
  static int per_sm = 0;  // CTAs per SM of metadata_kernel (same on every GB300)
  if (per_sm == 0) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, metadata_kernel, kMetaThreads, 0) !=
        cudaSuccess)
      return 1;
    per_sm = v > 0 ? v : 1;
  }
  return per_sm;
}

cudaError_t launch_metadata_kernel(const int32_t *topk_indx, const uint16_t *topk_vals, int N,
                                   int E, const moe_routing_meta &meta, int32_t *ws_hist,
                                   uint32_t *ctrl, int max_ctas, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t err = uniform_carveout(metadata_kernel);
    if (err != cudaSuccess) return err;
    configured = true;
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
                  (void *)&ws_hist, (void *)&ctrl, (void *)&timeout};
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
                            uint32_t *ctrl, cudaStream_t s) {
  return launch_metadata_kernel(topk_indx, topk_vals, (int)(n * k), E, meta, ws_hist, ctrl,
                                kMetaMaxCtas, s);
}

// ================================================= fused route + metadata ==
//
// moe_route_metadata / moe_forward's first two stages in one cooperative
// kernel, one CTA per SM: CTA b routes tokens [b*T, b*T + T) (G lanes per
// token as above), keeping its slots and histogram in shared memory, then
// publishes, gathers and scatters its slots from shared memory.
template <int K, int G, int NQ>
__global__ void __launch_bounds__(kFusedThreads, 1) route_metadata_kernel(
    const float *__restrict__ logits, int64_t n, int E, int gating, int T, int vec4,
    int32_t *__restrict__ topk_indx, uint16_t *__restrict__ topk_vals,
    int32_t *__restrict__ col_sum, int32_t *__restrict__ offs, int32_t *__restrict__ col_sorted,
    int32_t *__restrict__ row_sorted, uint16_t *__restrict__ gate_scal,
    int32_t *__restrict__ ws_hist, uint32_t *ctrl, unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ MetaShared<kFusedThreads> sh;
  uint8_t *s_slot_e = smem_raw;
  uint16_t *s_slot_v = reinterpret_cast<uint16_t *>(smem_raw + (((size_t)T * K + 15) & ~15ull));

  const int tid = threadIdx.x;
  pdl_launch_dependents();  // the gather may be scheduled (it waits for this grid)
  for (int e = tid; e < E; e += kFusedThreads) sh.base[e] = 0;
  __syncthreads();

  const int64_t t0 = min(n, (int64_t)blockIdx.x * T);
  const int64_t t1 = min(n, t0 + T);
  constexpr int per_pass = kFusedThreads / G;
  for (int64_t tb = t0; tb < t1; tb += per_pass) {  // uniform over the block
    const int64_t t = tb + tid / G;
    const bool valid = t < t1;
    TopK<K> tk;
    float w[K];
    topk_group<K, G, NQ>(logits + (valid ? t : 0) * E, valid, E, gating, vec4 != 0, tk, w);
    if (valid)
      write_token<K, G, true>(t, t0, tk, w, topk_indx, topk_vals, s_slot_e, s_slot_v, sh.base);
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
  if (!meta_barrier_prefix(ws_hist, E, sh, col_sum, offs, ctrl, timeout_ns, write_topk)) return;
  meta_scatter(
      t0 * K, (int)(t1 - t0) * K, E, sh,
      [&](int i, int &e, uint16_t &w) {
        e = s_slot_e[i];
        w = s_slot_v[i];
      },
      col_sorted, row_sorted, gate_scal);
}

// Tokens per CTA of the fused kernel: spread over the SMs, a multiple of 4;
// a batch that one pass of one CTA covers (1024 / G tokens) gets one CTA,
// which skips the cross-CTA exchange.
int64_t fused_tokens_per_cta(int64_t n, int per_pass) {
  if (n <= per_pass) return (n + 3) / 4 * 4;
  const int sms = device_sm_count();
  int64_t T = (n + sms - 1) / sms;
  if (T < 4) T = 4;
  return (T + 3) / 4 * 4;
}

struct RouteMetaLaunch {
  const float *logits;
  int64_t n;
  int E, gating;
  int32_t *indx;
  uint16_t *vals;
  const moe_routing_meta *meta;
  int32_t *ws_hist;
  uint32_t *ctrl;
  cudaStream_t s;
  template <int K, int G, int NQ>
  cudaError_t go() {
    const int64_t T = fused_tokens_per_cta(n, kFusedThreads / G);
    const int64_t B = (n + T - 1) / T;
    const size_t slots = (size_t)T * K;
    const size_t smem = ((slots + 15) & ~(size_t)15) + slots * 2;
    auto kern = route_metadata_kernel<K, G, NQ>;
    static bool configured = false;
    if (!configured) {
      const int max_smem = kSlotCap * 3 + 16;
      cudaError_t e1 =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
      if (e1 != cudaSuccess) return e1;
      if ((e1 = uniform_carveout(kern)) != cudaSuccess) return e1;
      configured = true;
    }
    cudaError_t err = cudaSuccess;
    int Ti = (int)T;
    int64_t nn = n;
    int E_ = E, g_ = gating;
    int vec4 = (E % 4) == 0 && ((uintptr_t)logits % 16) == 0;
    unsigned long long timeout = kWaitTimeoutNs;
    void *args[] = {(void *)&logits, (void *)&nn, (void *)&E_, (void *)&g_, (void *)&Ti,
                    (void *)&vec4, (void *)&indx, (void *)&vals, (void *)&meta->col_sum, (void *)&meta->offs,
                    (void *)&meta->col_sorted, (void *)&meta->row_sorted,
                    (void *)&meta->gate_scal, (void *)&ws_hist, (void *)&ctrl,
                    (void *)&timeout};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = smem;
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
  return fused_tokens_per_cta(n, 0) * k <= kSlotCap;  // the larger of the two T
}

// ----------------------------------------- route + metadata, decode sizes --
// n*k <= 32 slots (a decode step): one CTA of kSmallThreads. The top-k as
// above (G lanes per token); then warp 0 alone builds the metadata: the
// histogram from shared-memory counts, the exclusive scan into offs, and
// each slot's position offs[e] + (slots of e with a lower flat index), the
// rank among the lanes that hold the same expert (__match_any_sync). The
// same results as the cooperative kernel, with one CTA and two barriers.
constexpr int kSmallThreads = 256;
constexpr int kSmallSlots = 32;

template <int K, int G, int NQ>
__global__ void __launch_bounds__(kSmallThreads) route_metadata_small_kernel(
    const float *__restrict__ logits, int n, int E, int gating, int vec4,
    int32_t *__restrict__ topk_indx, uint16_t *__restrict__ topk_vals,
    int32_t *__restrict__ col_sum, int32_t *__restrict__ offs, int32_t *__restrict__ col_sorted,
    int32_t *__restrict__ row_sorted, uint16_t *__restrict__ gate_scal) {
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_e[kSmallSlots];
  __shared__ uint16_t s_w[kSmallSlots];
  const int tid = threadIdx.x, lane = tid & 31;
  pdl_launch_dependents();  // the gather may be scheduled (it waits for this grid)
  for (int e = tid; e < E; e += kSmallThreads) s_cnt[e] = 0;
  __syncthreads();
  {
    const int t = tid / G, g = lane % G;
    const bool valid = t < n;
    TopK<K> tk;
    float w[K];
    topk_group<K, G, NQ>(logits + (valid ? t : 0) * (int64_t)E, valid, E, gating, vec4 != 0, tk,
                         w);
    if (valid) {
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (j % G != g) continue;
        const int f = t * K + j;
        const uint16_t wb = float_to_bf16_bits(w[j]);
        topk_indx[f] = tk.e[j];
        topk_vals[f] = wb;
        s_e[f] = tk.e[j];
        s_w[f] = wb;
        atomicAdd(&s_cnt[tk.e[j]], 1);
      }
    }
  }
  __syncthreads();
  if (tid < 32) {
    int carry = 0;  // exclusive scan of the counts, 32 experts at a time
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int cnt = e < E ? s_cnt[e] : 0;
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < E) {
        col_sum[e] = cnt;
        offs[e] = carry + incl - cnt;
        s_cnt[e] = carry + incl - cnt;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) offs[E] = carry;
    __syncwarp();
    const int N = n * K;
    const int e = lane < N ? s_e[lane] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (lane < N) {
      const int p = s_cnt[e] + __popc(peers & ((1u << lane) - 1u));
      col_sorted[p] = lane;
      row_sorted[lane] = p;
      gate_scal[p] = s_w[lane];
    }
  }
}

struct RouteMetaSmallLaunch {
  const float *logits;
  int n, E, gating;
  int32_t *indx;
  uint16_t *vals;
  const moe_routing_meta *meta;
  cudaStream_t s;
  template <int K, int G, int NQ>
  cudaError_t go() {
    auto kern = route_metadata_small_kernel<K, G, NQ>;
    static bool configured = false;
    if (!configured) {
      cudaError_t err = uniform_carveout(kern);
      if (err != cudaSuccess) return err;
      configured = true;
    }
    const int vec4 = (E % 4) == 0 && ((uintptr_t)logits % 16) == 0;
    kern<<<1, kSmallThreads, 0, s>>>(logits, n, E, gating, vec4, indx, vals, meta->col_sum,
                                      meta->offs, meta->col_sorted, meta->row_sorted,
                                      meta->gate_scal);
    return cudaGetLastError();
  }
};

cudaError_t launch_route_metadata(const float *logits, int64_t n, int E, int k, int gating,
                                  int32_t *topk_indx, uint16_t *topk_vals,
                                  const moe_routing_meta &meta, int32_t *ws_hist,
                                  uint32_t *ctrl, cudaStream_t s) {
  // every G (<= 8) lanes take a token: n <= 32 tokens fit one 256-thread CTA
  if (n * k <= kSmallSlots)
    return dispatch_kg(k, E, RouteMetaSmallLaunch{logits, (int)n, E, gating, topk_indx,
                                                  topk_vals, &meta, s});
  return dispatch_kg(k, E, RouteMetaLaunch{logits, n, E, gating, topk_indx, topk_vals, &meta,
                                           ws_hist, ctrl, s});
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
// MiniMind issue ("It is removable in plain PyTorch"), done token-major: a
// warp per (token t, group of 128 16-byte chunks) reads its chunks of x[t]
// once (up to 4 loads in flight per thread) and writes them to the k sorted
// positions row_sorted[t*k + j] of the token's slots, so x is read from
// memory once rather than once per slot.
constexpr int kCopyThreads = 256;

constexpr int kChunksPerLane = 4;  // 16-byte chunks in flight per thread

__global__ void __launch_bounds__(kCopyThreads) gather_rows_kernel(
    const uint4 *__restrict__ x, const int32_t *__restrict__ row_sorted, int64_t n, int k,
    int vec_per_row, int groups_per_row, uint4 *__restrict__ x_sorted) {
  pdl_launch_dependents();
  pdl_wait();  // row_sorted comes from the metadata kernel
  const int lane = threadIdx.x & 31;
  const int64_t N = n * k;
  const int64_t units = n * groups_per_row;  // (token, group of 32 * kChunksPerLane chunks)
  const int64_t warps = (int64_t)gridDim.x * (kCopyThreads / 32);
  for (int64_t u = (int64_t)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5); u < units;
       u += warps) {
    const int64_t t = u / groups_per_row;
    const int c0 = (int)(u - t * groups_per_row) * 32 * kChunksPerLane + lane;
    const uint4 *src = x + t * vec_per_row;
    uint4 v[kChunksPerLane];
#pragma unroll
    for (int q = 0; q < kChunksPerLane; ++q)
      if (c0 + 32 * q < vec_per_row) v[q] = __ldcs(src + c0 + 32 * q);
    for (int j = 0; j < k; ++j) {
      const int32_t p = __ldg(row_sorted + t * k + j);
      // a slot whose expert id was out of range has no position (the metadata
      // kernel flags MOE_ERR_INVALID_ARG)
      if ((uint32_t)p >= (uint32_t)N) continue;
      uint4 *dst = x_sorted + (int64_t)p * vec_per_row;
#pragma unroll
      for (int q = 0; q < kChunksPerLane; ++q)
        if (c0 + 32 * q < vec_per_row) dst[c0 + 32 * q] = v[q];
    }
  }
}

cudaError_t launch_gather_rows(const uint16_t *x, const int32_t *row_sorted, int64_t n, int k,
                               int H, uint16_t *x_sorted, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    cudaError_t err = uniform_carveout(gather_rows_kernel);
    if (err != cudaSuccess) return err;
    configured = true;
  }
  const int vpr = H / 8, gpr = (vpr + 32 * kChunksPerLane - 1) / (32 * kChunksPerLane);
  int64_t blocks = (n * gpr + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  cudaError_t err = launch_dependent(gather_rows_kernel, dim3((unsigned)blocks), dim3(kCopyThreads),
                                     0, s, reinterpret_cast<const uint4 *>(x), row_sorted, n, k,
                                     vpr, gpr, reinterpret_cast<uint4 *>(x_sorted));
  return err != cudaSuccess ? err : cudaGetLastError();
}

// ============================================================= combine ==
// out[t] = sum_{j<k} y_flat[t*k + j] in fp32, j ascending, one bf16 rounding.
// A warp per (token, group of 64 16-byte chunks), 2 chunks x k slots in
// flight per thread.
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
                                                               uint4 *__restrict__ out) {
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
    uint4 v[CPL][K];
#pragma unroll
    for (int q = 0; q < CPL; ++q)
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (c0 + 32 * q < vec_per_row)
          v[q][j] = __ldcs(src + (int64_t)j * vec_per_row + c0 + 32 * q);
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
                           cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int vpr = H / 8, gpr = (vpr + 63) / 64;
  int64_t blocks = (n * gpr + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  const uint4 *y = reinterpret_cast<const uint4 *>(y_flat);
  uint4 *o = reinterpret_cast<uint4 *>(out);
  static bool configured[9] = {};
  switch (k) {
#define MOE_COMBINE_CASE(K_)                                                       \
  case K_:                                                                         \
    if (!configured[K_]) {                                                         \
      cudaError_t err = uniform_carveout(combine_kernel<K_>);                      \
      if (err != cudaSuccess) return err;                                          \
      configured[K_] = true;                                                       \
    }                                                                              \
    {                                                                              \
      cudaError_t err = launch_dependent(combine_kernel<K_>, dim3((unsigned)blocks),  \
                                         dim3(kCopyThreads), 0, s, y, n, vpr, gpr, o); \
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
