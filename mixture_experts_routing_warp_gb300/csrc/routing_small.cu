// routing_small.cu -- router top-k and routing metadata for decode sizes
// (n*k <= 32 slots) in one CTA.
//
// Sources (page title, section): as routing.cu.
#include "routing_common.cuh"

namespace moe {

// ----------------------------------------- route + metadata, decode sizes --
// n*k <= 32 slots (a decode step): one CTA of kSmallThreads. The top-k of
// routing_common.cuh (G lanes per token); then warp 0 alone builds the metadata: the
// histogram from shared-memory counts, the exclusive scan into offs, and
// each slot's position offs[e] + (slots of e with a lower flat index), the
// rank among the lanes that hold the same expert (__match_any_sync). The
// same results as the cooperative kernel, with one CTA and two barriers.
// With an expert map the metadata covers the E_loc local experts and a slot
// of another rank's expert gets no position (row_sorted -1).
constexpr int kSmallThreads = 256;

template <int K, int G, int NQ>
__global__ void __launch_bounds__(kSmallThreads) route_metadata_small_kernel(
    const float *__restrict__ logits, int n, int E, int gating, int vec4,
    int32_t *__restrict__ topk_indx, uint16_t *__restrict__ topk_vals,
    int32_t *__restrict__ col_sum, int32_t *__restrict__ offs, int32_t *__restrict__ col_sorted,
    int32_t *__restrict__ row_sorted, uint16_t *__restrict__ gate_scal, uint32_t *sync,
    const int32_t *__restrict__ expert_map, int E_loc, uint32_t *ctrl) {
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_map_buf[kMaxExperts];
  __shared__ int s_e[kSmallSlots];
  __shared__ uint16_t s_w[kSmallSlots];
  __shared__ float4 stash[NQ * kSmallThreads];  // the top-k's logit stash
  const int tid = threadIdx.x, lane = tid & 31;
  pdl_launch_dependents();  // the next kernel may be scheduled (it waits for this grid)
  zero_sync_words(sync);
  const int *s_map = load_expert_map(expert_map, E, E_loc, s_map_buf, ctrl);
  for (int e = tid; e < E_loc; e += kSmallThreads) s_cnt[e] = 0;
  __syncthreads();
  {
    const int t = tid / G, g = lane % G;
    const bool valid = t < n;
    TopK<K> tk;
    float w[K];
    topk_group<K, G, NQ>(logits + (valid ? t : 0) * (int64_t)E, valid, E, gating, vec4 != 0, tk,
                         w, stash);
    if (valid) {
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (j % G != g) continue;
        const int f = t * K + j;
        const uint16_t wb = float_to_bf16_bits(w[j]);
        const int le = s_map ? s_map[tk.e[j]] : tk.e[j];
        topk_indx[f] = tk.e[j];
        topk_vals[f] = wb;
        s_e[f] = le;
        s_w[f] = wb;
        if (le >= 0) atomicAdd(&s_cnt[le], 1);
      }
    }
  }
  __syncthreads();
  if (tid < 32) {
    int carry = 0;  // exclusive scan of the counts, 32 experts at a time
    for (int e0 = 0; e0 < E_loc; e0 += 32) {
      const int e = e0 + lane;
      const int cnt = e < E_loc ? s_cnt[e] : 0;
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < E_loc) {
        col_sum[e] = cnt;
        offs[e] = carry + incl - cnt;
        s_cnt[e] = carry + incl - cnt;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) offs[E_loc] = carry;
    __syncwarp();
    const int N = n * K;
    const int e = lane < N ? s_e[lane] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (lane < N && e < 0) row_sorted[lane] = -1;  // another rank's expert
    if (lane < N && e >= 0) {
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
  uint32_t *sync;
  const int32_t *expert_map;
  int E_loc;
  uint32_t *ctrl;
  cudaStream_t s;
  template <int K, int G, int NQ>
  cudaError_t go() {
    auto kern = route_metadata_small_kernel<K, G, NQ>;
    static PerDeviceOnce configured;
    cudaError_t err = configured.run([kern] { return uniform_carveout(kern); });
    if (err != cudaSuccess) return err;
    const int vec4 = (E % 4) == 0 && ((uintptr_t)logits % 16) == 0;
    kern<<<1, kSmallThreads, 0, s>>>(logits, n, E, gating, vec4, indx, vals, meta->col_sum,
                                      meta->offs, meta->col_sorted, meta->row_sorted,
                                      meta->gate_scal, sync, expert_map, E_loc, ctrl);
    return cudaGetLastError();
  }
};

cudaError_t launch_route_metadata_small(const float *logits, int n, int E, int k, int gating,
                                        int32_t *topk_indx, uint16_t *topk_vals,
                                        const moe_routing_meta &meta, uint32_t *sync,
                                        const int32_t *expert_map, int E_loc, uint32_t *ctrl,
                                        cudaStream_t s) {
  return dispatch_kg(k, E, RouteMetaSmallLaunch{logits, n, E, gating, topk_indx, topk_vals,
                                                &meta, sync, expert_map, E_loc, ctrl, s});
}

}  // namespace moe
