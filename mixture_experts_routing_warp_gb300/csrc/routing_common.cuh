// routing_common.cuh -- device code shared by the routing kernels (router
// top-k, metadata): the G-lane top-k, the per-token output writer, the
// (K, G, NQ) dispatch, and the metadata phases (per-CTA counts, cross-CTA
// prefix, stable scatter). The kernels themselves live in routing.cu,
// routing_fused.cu and routing_small.cu, compiled in parallel.
//
// Sources (page title, section): as routing.cu.
#pragma once

#include "tc_ptx.cuh"

namespace moe {

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

// The kernels that build the routing metadata also zero the per-forward sync
// words of the expert contractions (block 0; `sync` may be null): the w13
// contraction reads them only after these grids have completed
// (griddepcontrol.wait), and the previous forward's contractions have
// completed before these grids start (they are not dependent launches).
__device__ __forceinline__ void zero_sync_words(uint32_t *sync) {
  if (sync && blockIdx.x == 0)
    for (int i = threadIdx.x; i < kSyncWords; i += blockDim.x) sync[i] = 0;
}
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

// 32-bit selection keys. trunc_key replaces the IDB low bits of the order
// key by (2^IDB - 1 - e): keys are unique, and a larger key has a larger
// value in the upper 32 - IDB bits of the order key or, on equal upper bits,
// a lower expert id. Two elements whose upper bits differ are ordered as their
// exact (value, id) keys are; only elements that share the upper bits can be
// ordered differently (their low value bits are ignored).
template <int IDB>
__device__ __forceinline__ uint32_t trunc_key(float v, int e) {
  constexpr uint32_t m = (1u << IDB) - 1u;
  return (order_key(v) & ~m) | (m - (uint32_t)e);
}

__device__ __forceinline__ void cx32(uint32_t &a, uint32_t &b) {
  const uint32_t hi = max(a, b), lo = min(a, b);
  a = hi;
  b = lo;
}

__device__ __forceinline__ void sort4_desc32(uint32_t (&c)[4]) {
  cx32(c[0], c[1]);
  cx32(c[2], c[3]);
  cx32(c[0], c[2]);
  cx32(c[1], c[3]);
  cx32(c[1], c[2]);
}

// top <- the 4 largest of top and o (both sorted descending), sorted; the
// 4 smallest are dropped, and `dropped` keeps the largest key ever dropped.
__device__ __forceinline__ void merge4_desc32(uint32_t (&top)[4], const uint32_t (&o)[4],
                                              uint32_t &dropped) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    dropped = max(dropped, min(top[j], o[3 - j]));
    top[j] = max(top[j], o[3 - j]);
  }
  cx32(top[0], top[2]);
  cx32(top[1], top[3]);
  cx32(top[0], top[1]);
  cx32(top[2], top[3]);
}

constexpr int ilog2_ce(int v) { return v <= 1 ? 0 : 1 + ilog2_ce(v / 2); }

// vec4: rows are 16-byte aligned (E % 4 == 0 and a 16-byte aligned base),
// so a chunk is one 128-bit load; otherwise four 32-bit loads.
//
// K <= 4: the G lanes select on 32-bit trunc_keys (IDB = log2(NQ * 4 * G)
// id bits): each lane sorts its 4-element chunks with a 5-comparator network
// and bitonic-merges the sorted 4-lists (inside the lane, then across the G
// lanes), keeping the top 4. The selection S = s_1..s_K is exact -- the same
// experts in the same order as with full (value, id) keys -- when the upper
// bits h of the selected keys are pairwise distinct and no other element
// shares h(s_K): then every selected element beats every other on its upper
// bits alone. Each lane checks the second condition on its own top 5 (its
// final local top-4 list and the largest key its local merges dropped): an
// unselected element y of the lane with h(y) = h(s_K) either is among those
// five, or lies below five of the lane's elements that beat it, one of which
// is then unselected with h = h(s_K) as well, or is the fifth itself when the
// lane's top 4 are S. A warp with a token that fails the test (equal upper
// bits near the cut: ties, near-ties, NaN) redoes its tokens on 64-bit
// (order key, ~id) keys. The selected logits are read back from `stash`,
// where each lane leaves its chunks ([NQ][blockDim.x] float4, this thread's
// column), so the gate weights see the exact values.
template <int K, int G, int NQ>  // NQ chunks of 4 elements per lane: NQ*4*G >= E
__device__ __forceinline__ void topk_group(const float *__restrict__ row, bool valid, int E,
                                           int gating, bool vec4, TopK<K> &tk, float (&w)[K],
                                           float4 *stash) {
  const int lane = threadIdx.x & 31, g = lane % G;
  tk.init();
  // a warp without a token (the tail of a CTA's range) has nothing to rank;
  // the test is warp-uniform, so the shuffles below stay warp-complete
  if (!__any_sync(0xffffffffu, valid)) {
#pragma unroll
    for (int j = 0; j < K; ++j) w[j] = 0.f;
    return;
  }
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
    constexpr int IDB = ilog2_ce(NQ * 4 * G);
    static_assert((1 << IDB) == NQ * 4 * G, "NQ * 4 * G must be a power of two");
    __syncwarp();  // the group's reads of the previous pass's stash are done
#pragma unroll
    for (int i = 0; i < NQ; ++i) stash[i * blockDim.x + threadIdx.x] = x[i];
    uint32_t top[4], dropped = 0u;
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      if (i > 0 && i * G * 4 >= E) break;  // uniform: no lane's chunk holds an expert
      const int e0 = (i * G + g) * 4;
      uint32_t c[4];
      c[0] = e0 < E ? trunc_key<IDB>(x[i].x, e0) : 0u;
      c[1] = e0 + 1 < E ? trunc_key<IDB>(x[i].y, e0 + 1) : 0u;
      c[2] = e0 + 2 < E ? trunc_key<IDB>(x[i].z, e0 + 2) : 0u;
      c[3] = e0 + 3 < E ? trunc_key<IDB>(x[i].w, e0 + 3) : 0u;
      sort4_desc32(c);
      if (i == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) top[j] = c[j];
      } else {
        merge4_desc32(top, c, dropped);
      }
    }
    const uint32_t local[4] = {top[0], top[1], top[2], top[3]};
#pragma unroll
    for (int off = 1; off < G; off <<= 1) {
      uint32_t o[4], unused = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] = __shfl_xor_sync(0xffffffffu, top[j], off);
      merge4_desc32(top, o, unused);
    }
    // exactness: distinct upper bits among the selected, and s_K's upper
    // bits on no other element of this lane's top 5
    bool exact = true;
#pragma unroll
    for (int j = 1; j < K; ++j) exact = exact && (top[j - 1] >> IDB) != (top[j] >> IDB);
    const uint32_t sk = top[K - 1], hk = sk >> IDB;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      exact = exact && !(local[j] != sk && local[j] != 0u && (local[j] >> IDB) == hk);
    exact = exact && !(dropped != 0u && (dropped >> IDB) == hk);
    if (__all_sync(0xffffffffu, exact || !valid)) {
      __syncwarp();  // the group's stash entries are written
      const float *sf = reinterpret_cast<const float *>(stash);
      const int base = threadIdx.x - g;  // the group's first thread
#pragma unroll
      for (int j = 0; j < K; ++j) {
        const int e = (int)((1u << IDB) - 1u - (top[j] & ((1u << IDB) - 1u)));
        const int q = e >> 2;
        const float v = sf[((q / G) * (int)blockDim.x + base + q % G) * 4 + (e & 3)];
        tk.key[j] = order_key(v);
        tk.e[j] = e;
      }
    } else {
      // Exact selection on packed 64-bit keys ((order key << 32) | ~id):
      // the same networks on unique keys whose order is (value descending,
      // id ascending).
      unsigned long long top64[4];
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        if (i > 0 && i * G * 4 >= E) break;  // uniform: no lane's chunk holds an expert
        const int e0 = (i * G + g) * 4;
        unsigned long long c[4];
        c[0] = e0 < E ? pack_key(order_key(x[i].x), e0) : 0ull;
        c[1] = e0 + 1 < E ? pack_key(order_key(x[i].y), e0 + 1) : 0ull;
        c[2] = e0 + 2 < E ? pack_key(order_key(x[i].z), e0 + 2) : 0ull;
        c[3] = e0 + 3 < E ? pack_key(order_key(x[i].w), e0 + 3) : 0ull;
        sort4_desc(c);
        if (i == 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j) top64[j] = c[j];
        } else {
          merge4_desc(top64, c);
        }
      }
#pragma unroll
      for (int off = 1; off < G; off <<= 1) {
        unsigned long long o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = __shfl_xor_sync(0xffffffffu, top64[j], off);
        merge4_desc(top64, o);
      }
#pragma unroll
      for (int j = 0; j < K; ++j) {
        tk.key[j] = (uint32_t)(top64[j] >> 32);
        tk.e[j] = (int)~(uint32_t)top64[j];
      }
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
// KEEP: the slots stay in shared memory (global expert ids) and are counted
// per local expert (s_map: local id of each global expert or -1, null for
// the identity; a -1 slot is not counted).
template <int K, int G, bool KEEP>
__device__ __forceinline__ void write_token(int64_t t, int64_t t0, const TopK<K> &tk,
                                            const float (&w)[K], int32_t *__restrict__ topk_indx,
                                            uint16_t *__restrict__ topk_vals, uint8_t *s_slot_e,
                                            uint16_t *s_slot_v, int *s_hist,
                                            const int *s_map = nullptr) {
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
      const int le = s_map ? s_map[tk.e[j]] : tk.e[j];
      if (le >= 0) atomicAdd(&s_hist[le], 1);
    }
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

// ------------------------------------------------ 16-bit count rows ----
//
// The cooperative route + metadata kernel's exchange: CTA b writes its counts
// as row b of `rows` ([kFusedMaxRows][S] u16, S = E rounded up to 8: a CTA
// holds at most kSlotCap = 8192 slots), passes the bounded grid barrier, and
// copies all B rows into its shared memory with bulk copies (TMA, whole
// 128-byte lines: when every CTA reads the same few tens of KB at once, one
// request per line keeps the lines' L2 slices far less busy than a 16-byte
// load per row and column). Threads then sum columns of the rows in parts,
// and an exclusive scan over experts, 32 experts per warp in parallel, gives
// offs; base[e] = offs[e] + the counts of expert e in lower CTAs.
constexpr uint32_t kBulkChunk = 32768;  // bytes per bulk copy

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// sh.base[0..E) holds this CTA's counts; on return sh.base = offs + before,
// and CTA 0 has written col_sum and offs. `staging` is shared memory for B
// rows (B * S * 2 bytes, 16-byte aligned), free at this point. `between`
// runs (every thread) after this CTA's arrival and before its wait. Returns
// false after a timeout.
template <int THREADS, typename Between>
__device__ bool meta_exchange_rows(uint16_t *__restrict__ rows, void *staging, int E,
                                   MetaShared<THREADS> &sh, int32_t *__restrict__ col_sum,
                                   int32_t *__restrict__ offs, uint32_t *ctrl,
                                   unsigned long long timeout_ns, Between between) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = gridDim.x, b = blockIdx.x;
  const int S = (E + 7) & ~7, S8 = S / 8;  // u16 counts per row, int4 per row
  __shared__ int s_chunk[kMaxExperts / 32];
  __shared__ __align__(8) uint64_t s_bar;
  int nparts = 1;
  if (B == 1) {  // one CTA holds every slot: no exchange, no barrier
    between();
    for (int e = tid; e < S; e += THREADS) {
      sh.tot[e] = e < E ? sh.base[e] : 0;
      sh.pre[e] = 0;
    }
  } else {
    const uint32_t bar = tc::smem_u32(&s_bar);
    if (tid == 0) {
      tc::mbar_init(bar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < S8; i += THREADS) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = i * 8 + 2 * q;
        const uint32_t lo = e < E ? (uint32_t)sh.base[e] : 0u;
        const uint32_t hi = e + 1 < E ? (uint32_t)sh.base[e + 1] : 0u;
        w[q] = lo | (hi << 16);
      }
      reinterpret_cast<int4 *>(rows + (size_t)b * S)[i] =
          make_int4((int)w[0], (int)w[1], (int)w[2], (int)w[3]);
    }
    const uint32_t arrived = grid_arrive(ctrl);  // (its __syncthreads covers the init)
    between();
    if (!grid_wait(ctrl, arrived, timeout_ns)) return false;
    const uint32_t bytes = (uint32_t)B * (uint32_t)S * 2u;
    if (tid == 0) {
      tc::fence_proxy_async_global();  // the acquired rows, for the bulk copies
      tc::mbar_arrive_expect_tx(bar, bytes);
      for (uint32_t off = 0; off < bytes; off += kBulkChunk)
        bulk_load(tc::smem_u32(staging) + off, reinterpret_cast<const uint8_t *>(rows) + off,
                  min(kBulkChunk, bytes - off), bar);
    }
    bool ok = tc::mbar_try_wait(bar, 0);
    if (!ok) {
      const long long deadline = wait_deadline(timeout_ns);
      while (!(ok = tc::mbar_try_wait(bar, 0)))
        if (clock64() > deadline) break;
    }
    if (__syncthreads_or(!ok)) {
      if (tid == 0) record_status(ctrl, MOE_ERR_TIMEOUT);
      tc::wait_drain(bar, 0, timeout_ns);  // no copy may still write here at exit
      return false;
    }
    // part q of nparts sums rows [B q / nparts, B (q + 1) / nparts) of each column
    nparts = min(32, THREADS / S);
    const int part = tid / S, e = tid % S;
    if (part < nparts) {
      const uint16_t *rs = reinterpret_cast<const uint16_t *>(staging);
      const int r0 = B * part / nparts, r1 = B * (part + 1) / nparts;
      int t = 0, p = 0;
#pragma unroll 4
      for (int r = r0; r < r1; ++r) {
        const int c = rs[r * S + e];
        t += c;
        p += r < b ? c : 0;
      }
      sh.tot[part * S + e] = t;
      sh.pre[part * S + e] = p;
    }
  }
  __syncthreads();
  // sums over the parts, then an exclusive scan over experts: warp c scans
  // experts [32c, 32c + 32), the chunk totals are added afterwards
  int tot = 0, pre = 0, incl = 0;
  if (warp * 32 < E) {  // warp-uniform
    if (tid < E) {
      for (int q = 0; q < nparts; ++q) {
        tot += sh.tot[q * S + tid];
        pre += sh.pre[q * S + tid];
      }
    }
    incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) s_chunk[warp] = incl;
  }
  __syncthreads();
  if (tid < E) {
    int carry = 0;
    for (int c = 0; c < warp; ++c) carry += s_chunk[c];
    const int excl = carry + incl - tot;
    sh.base[tid] = excl + pre;
    if (b == 0) {
      col_sum[tid] = tot;
      offs[tid] = excl;
      if (tid == E - 1) offs[E] = excl + tot;
    }
  }
  __syncthreads();
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
    if (i < count) {
      get(i, e, w);
      // a dropped slot (expert on another rank, or an invalid id) has no
      // sorted position
      if (e < 0) row_sorted[f_lo + i] = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0 && rank == 0) sh.cnt[warp][e] = __popc(peers);
    __syncthreads();
    // cnt[w][e] -> base[e] + (slots of expert e in warps < w); base[e] += all
    for (int ee = tid; ee < E; ee += THREADS) {  // consecutive experts: no bank conflicts
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

// Expert map (expert parallelism): the local id of each of the E global
// experts, or -1 for an expert on another rank, copied to shared memory.
// An entry outside [-1, E_loc) is treated as -1 and flags
// MOE_ERR_INVALID_ARG. Returns the table, or null (identity) without a map.
__device__ __forceinline__ const int *load_expert_map(const int32_t *expert_map, int E, int E_loc,
                                                      int *s_map, uint32_t *ctrl) {
  if (!expert_map) return nullptr;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int v = expert_map[e];
    const bool ok = v >= -1 && v < E_loc;
    if (!ok && ctrl) record_status(ctrl, MOE_ERR_INVALID_ARG);
    s_map[e] = ok ? v : -1;
  }
  return s_map;
}

// Dispatch rows X_sorted[row_sorted[t*k + j]] = x[t] for tokens [t_lo, t_hi)
// ("It is removable in plain PyTorch": x[tok], tok = order // k), token-major:
// a warp per (token, group of 128 16-byte chunks), 4 chunks in flight per
// lane, x[t] read once and written to the token's k sorted positions; a
// position outside [0, N) (a dropped slot) is skipped. row_sorted is read
// through L2 (the calling kernel may have written it). `warp` of `warps`:
// this warp's share of the (token, group) units.
__device__ __forceinline__ void copy_token_rows(const uint4 *__restrict__ x,
                                                const int32_t *row_sorted, int64_t t_lo,
                                                int64_t t_hi, int k, int vpr, int64_t N,
                                                uint4 *__restrict__ x_sorted, int64_t warp,
                                                int64_t warps) {
  constexpr int kChunks = 4;  // 16-byte chunks in flight per lane
  const int lane = threadIdx.x & 31;
  const int gpr = (vpr + 32 * kChunks - 1) / (32 * kChunks);
  const int64_t units = (t_hi - t_lo) * gpr;
  for (int64_t u = warp; u < units; u += warps) {
    const int64_t t = t_lo + u / gpr;
    const int c0 = (int)(u % gpr) * 32 * kChunks + lane;
    const uint4 *src = x + t * vpr;
    uint4 v[kChunks];
#pragma unroll
    for (int q = 0; q < kChunks; ++q)
      if (c0 + 32 * q < vpr) v[q] = __ldcs(src + c0 + 32 * q);
    for (int j = 0; j < k; ++j) {
      const int32_t p = __ldcg(row_sorted + t * k + j);
      if ((uint64_t)(uint32_t)p >= (uint64_t)N) continue;
      uint4 *dst = x_sorted + (int64_t)p * vpr;
#pragma unroll
      for (int q = 0; q < kChunks; ++q)
        if (c0 + 32 * q < vpr) dst[c0 + 32 * q] = v[q];
    }
  }
}

// Decode sizes (n*k <= kSmallSlots): route + metadata in one CTA
// (routing_small.cu).
constexpr int kSmallSlots = 32;
cudaError_t launch_route_metadata_small(const float *logits, int n, int E, int k, int gating,
                                        int32_t *topk_indx, uint16_t *topk_vals,
                                        const moe_routing_meta &meta, uint32_t *sync,
                                        const int32_t *expert_map, int E_loc, uint32_t *ctrl,
                                        cudaStream_t s);

}  // namespace moe
