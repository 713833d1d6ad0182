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
// Router top-k, one warp per token. A CTA owns a contiguous block of tokens;
// their logit rows are staged into shared memory with cp.async.bulk in
// chunks of 32 tokens, one mbarrier per chunk, so warps start on the first
// chunk while the others are still in flight. Lane l holds experts
// [l*EPL, l*EPL + EPL) as 32-bit order keys (an order-preserving image of
// the fp32 value: -0.0 folded onto +0.0, NaN = 1 below every number,
// absent experts = 0). Each of the k rounds takes the warp maximum with
// redux.sync; among lanes holding it the lowest lane (lowest expert ids)
// wins, and within that lane the lowest slot, so equal logits go to the
// lower expert id. Gate weights: softmax in fp32 over the k selected
// (or over all E), rounded to bf16.

constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kChunkTok = 32;                 // tokens per staged chunk (one mbarrier)
constexpr int kMaxChunks = 32;                // chunks per staging round
constexpr int kStageBytes = 96 * 1024;        // staging buffer per CTA
constexpr int kStagePad = 1024;               // vector over-read slack after the last row
constexpr int kSlotCap = 8192;                // slots a fused CTA keeps in shared memory

__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 1u;                       // NaN: below every number, above "absent"
  const uint32_t u = __float_as_uint(v + 0.0f);  // -0.0 + 0.0 = +0.0: the two zeros tie
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Tokens [r0, r0 + ntok) of one staging round: rows in smem (row j at
// stage + j*E). Returns in lanes r < k the r-th expert and its weight.
template <int EPL, bool VEC>
__device__ __forceinline__ void topk_row(const float *row, int E, int k, int gating, int lane,
                                         int &sel_e, float &sel_w) {
  float v[EPL];
  if (VEC && EPL >= 4) {
#pragma unroll
    for (int q = 0; q < EPL / 4; ++q) {
      const float4 x = reinterpret_cast<const float4 *>(row + lane * EPL)[q];
      v[4 * q] = x.x;
      v[4 * q + 1] = x.y;
      v[4 * q + 2] = x.z;
      v[4 * q + 3] = x.w;
    }
  } else if (VEC && EPL == 2) {
    const float2 x = reinterpret_cast<const float2 *>(row + lane * 2)[0];
    v[0] = x.x;
    v[1] = x.y;
  } else {
#pragma unroll
    for (int c = 0; c < EPL; ++c) v[c] = row[min(lane * EPL + c, E - 1)];
  }
  uint32_t key[EPL];
  uint32_t lmax = 0u;
#pragma unroll
  for (int c = 0; c < EPL; ++c) {
    key[c] = (lane * EPL + c < E) ? order_key(v[c]) : 0u;
    lmax = max(lmax, key[c]);
  }
  uint32_t m0 = 0u, my_key = 0u;
  int my_e = 0;
  for (int r = 0; r < k; ++r) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, lmax);
    const unsigned holders = __ballot_sync(0xffffffffu, lmax == m);
    const int wl = __ffs(holders) - 1;
    int e_sel = 0;
    if (lane == wl) {
      int cw = EPL - 1;
#pragma unroll
      for (int c = EPL - 1; c >= 0; --c)
        if (key[c] == m) cw = c;
      e_sel = lane * EPL + cw;
      lmax = 0u;
#pragma unroll
      for (int c = 0; c < EPL; ++c) {
        if (c == cw) key[c] = 0u;
        lmax = max(lmax, key[c]);
      }
    }
    e_sel = __shfl_sync(0xffffffffu, e_sel, wl);
    if (lane == r) {
      my_e = e_sel;
      my_key = m;
    }
    if (r == 0) m0 = m;
  }
  const float v0 = key_to_float(m0);
  const float num = lane < k ? expf(key_to_float(my_key) - v0) : 0.f;
  float denom;
  if (gating == MOE_GATING_SOFTMAX_TOPK) {
    denom = num;  // lanes >= k hold 0; k <= 8
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
  } else {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < EPL; ++c)
      if (lane * EPL + c < E) s += expf(v[c] - v0);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    denom = s;
  }
  sel_e = my_e;
  sel_w = num / denom;
}

// Staged routing of tokens [t0, t1) by one CTA. Chunk barriers `bars`
// (kMaxChunks of them, initialised with count 1) keep their phases in
// `phase_bits` across rounds. With KEEP, the CTA's slots (expert, bf16
// weight) also go to s_slot_e / s_slot_v (index (t - t0)*k + j) and to the
// shared histogram s_hist.
template <int EPL, bool VEC, bool KEEP>
__device__ void route_block(const float *__restrict__ logits, int64_t t0, int64_t t1, int E, int k,
                            int gating, int TR, bool bulk_ok, int32_t *__restrict__ topk_indx,
                            uint16_t *__restrict__ topk_vals, float *stage, uint64_t *bars,
                            uint32_t &phase_bits, unsigned *s_plain, uint8_t *s_slot_e,
                            uint16_t *s_slot_v, int *s_hist, uint32_t *ctrl,
                            unsigned long long timeout_ns) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int64_t r0 = t0; r0 < t1; r0 += TR) {
    const int ntok = (int)min((int64_t)TR, t1 - r0);
    const int nch = (ntok + kChunkTok - 1) / kChunkTok;
    __syncthreads();  // the previous round's rows are no longer read
    if (tid == 0) {
      unsigned plain = 0;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      for (int c = 0; c < nch; ++c) {
        const int rows = min(kChunkTok, ntok - c * kChunkTok);
        const uint32_t bytes = (uint32_t)rows * (uint32_t)E * 4u;
        if (bulk_ok && (bytes & 15u) == 0) {
          const uint32_t bar = (uint32_t)__cvta_generic_to_shared(bars + c);
          const uint32_t dst =
              (uint32_t)__cvta_generic_to_shared(stage + (size_t)c * kChunkTok * E);
          const float *src = logits + (r0 + (int64_t)c * kChunkTok) * E;
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                       "r"(bytes)
                       : "memory");
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
              "[%3];" ::"r"(dst),
              "l"(src), "r"(bytes), "r"(bar)
              : "memory");
        } else {
          plain |= 1u << c;
        }
      }
      *s_plain = plain;
    }
    __syncthreads();
    const unsigned plain = *s_plain;
    if (plain) {  // chunks that cannot go through the bulk copy (size or alignment)
      for (int c = 0; c < nch; ++c) {
        if (!(plain >> c & 1u)) continue;
        const int rows = min(kChunkTok, ntok - c * kChunkTok);
        const float *src = logits + (r0 + (int64_t)c * kChunkTok) * E;
        float *dst = stage + (size_t)c * kChunkTok * E;
        for (int i = tid; i < rows * E; i += kRouteThreads) dst[i] = src[i];
      }
      __syncthreads();
    }
    const uint32_t used = (nch >= 32 ? 0xffffffffu : ((1u << nch) - 1u)) & ~plain;
    for (int j = warp; j < ntok; j += kRouteWarps) {
      const int c = j / kChunkTok;
      if (!(plain >> c & 1u)) {
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(bars + c);
        const uint32_t parity = (phase_bits >> c) & 1u;
        bool ok = false;
        const unsigned long long t_start = global_timer_ns();
        while (true) {
          uint32_t done;
          asm volatile(
              "{\n\t.reg .pred p;\n\t"
              "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
              "selp.u32 %0, 1, 0, p;\n\t}"
              : "=r"(done)
              : "r"(bar), "r"(parity)
              : "memory");
          if (done) {
            ok = true;
            break;
          }
          if (global_timer_ns() - t_start > timeout_ns) break;
        }
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) record_status(ctrl, MOE_ERR_TIMEOUT);
          continue;
        }
      }
      int e_sel;
      float w;
      topk_row<EPL, VEC>(stage + (size_t)j * E, E, k, gating, lane, e_sel, w);
      if (lane < k) {
        const int64_t t = r0 + j;
        const uint16_t wb = float_to_bf16_bits(w);
        topk_indx[t * k + lane] = e_sel;
        topk_vals[t * k + lane] = wb;
        if (KEEP) {
          const int i = (int)(t - t0) * k + lane;
          s_slot_e[i] = (uint8_t)e_sel;
          s_slot_v[i] = wb;
          atomicAdd(&s_hist[e_sel], 1);
        }
      }
    }
    phase_bits ^= used;
  }
}

__device__ __forceinline__ float *aligned_stage(uint8_t *raw) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(raw);
  return reinterpret_cast<float *>(raw + ((128u - (a & 127u)) & 127u));
}

__device__ __forceinline__ void init_chunk_bars(uint64_t *bars) {
  if (threadIdx.x == 0) {
    for (int c = 0; c < kMaxChunks; ++c)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
                       (uint32_t)__cvta_generic_to_shared(bars + c))
                   : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
}

template <int EPL, bool VEC>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(
    const float *__restrict__ logits, int64_t n, int E, int k, int gating, int T, int TR,
    int bulk_ok, int32_t *__restrict__ topk_indx, uint16_t *__restrict__ topk_vals,
    uint32_t *ctrl, unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kMaxChunks];
  __shared__ unsigned s_plain;
  float *stage = aligned_stage(smem_raw);
  init_chunk_bars(bars);
  uint32_t phase_bits = 0;
  const int64_t t0 = (int64_t)blockIdx.x * T;
  const int64_t t1 = min(n, t0 + T);
  route_block<EPL, VEC, false>(logits, t0, t1, E, k, gating, TR, bulk_ok != 0, topk_indx,
                               topk_vals, stage, bars, phase_bits, &s_plain, nullptr, nullptr,
                               nullptr, ctrl, timeout_ns);
}

// Tokens per staging round for E experts: whole chunks, at most kMaxChunks,
// within kStageBytes.
int staging_round_tokens(int E) {
  int chunks = kStageBytes / (kChunkTok * E * 4);
  if (chunks > kMaxChunks) chunks = kMaxChunks;
  if (chunks < 1) chunks = 1;
  return chunks * kChunkTok;
}

int epl_for(int E) { return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : 8; }

template <typename F>
cudaError_t dispatch_epl(int E, F &&f) {
  const bool vec = (E % 4) == 0;
  switch (epl_for(E)) {
    case 1: return vec ? f.template go<1, true>() : f.template go<1, false>();
    case 2: return vec ? f.template go<2, true>() : f.template go<2, false>();
    case 4: return vec ? f.template go<4, true>() : f.template go<4, false>();
    default: return vec ? f.template go<8, true>() : f.template go<8, false>();
  }
}

struct RouteLaunch {
  const float *logits;
  int64_t n;
  int E, k, gating;
  int32_t *indx;
  uint16_t *vals;
  uint32_t *ctrl;
  cudaStream_t s;
  template <int EPL, bool VEC>
  cudaError_t go() {
    const int sms = device_sm_count();
    int64_t T = (n + 2 * sms - 1) / (2 * sms);  // about two CTAs per SM
    T = (T + 3) / 4 * 4;
    if (T < 4) T = 4;
    const int TR = (int)min((int64_t)staging_round_tokens(E), (T + kChunkTok - 1) / kChunkTok *
                                                                 kChunkTok);
    const int smem = TR * E * 4 + kStagePad + 128;
    auto kern = route_kernel<EPL, VEC>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kStageBytes + kStagePad + 128);
    if (err != cudaSuccess) return err;
    const int bulk_ok = ((uintptr_t)logits % 16) == 0;
    const int64_t blocks = (n + T - 1) / T;
    kern<<<(unsigned)blocks, kRouteThreads, smem, s>>>(logits, n, E, k, gating, (int)T, TR,
                                                       bulk_ok, indx, vals, ctrl,
                                                       kWaitTimeoutNs);
    return cudaGetLastError();
  }
};

cudaError_t launch_route(const float *logits, int64_t n, int E, int k, int gating,
                         int32_t *topk_indx, uint16_t *topk_vals, uint32_t *ctrl,
                         cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  return dispatch_epl(E, RouteLaunch{logits, n, E, k, gating, topk_indx, topk_vals, ctrl, s});
}

// ============================================================= metadata ==
//
// Cross-CTA part of the metadata, shared by the kernels below. CTA b of B
// owns a contiguous range of slots. After its shared-memory histogram is
// published to ws_hist[b][0..E) (row stride `stride` = E rounded up to 4)
// and the bounded grid barrier:
//  prefix  total[e] = sum_b ws_hist[b][e] and before[e] = sum_{b'<b}
//          ws_hist[b'][e], read as int4 by (expert group, part of the CTA
//          rows) threads, parts summed and scanned by warp 0:
//          offs = exclusive scan of total; CTA 0 writes col_sum and offs;
//          base[e] = offs[e] + before[e]
//  scatter rounds of blockDim slots: a slot's rank among equal experts of
//          its warp (match_any + popc) plus the counts of lower warps plus
//          base[e] is its sorted position p. Stable in f; no atomic decides
//          any position.

constexpr int kMetaThreads = 512;
constexpr int kMetaWarps = kMetaThreads / 32;
constexpr int kMaxParts = 32;

struct MetaShared {
  int base[kMaxExperts];
  int cnt[kMetaWarps][kMaxExperts];
  int tot[2048];
  int pre[2048];
  int bad;
};

__device__ __forceinline__ int hist_stride(int E) { return (E + 3) & ~3; }

__device__ void meta_prefix(const int32_t *__restrict__ ws_hist, int E, MetaShared &sh,
                            int32_t *__restrict__ col_sum, int32_t *__restrict__ offs) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x, B = gridDim.x;
  const int stride = hist_stride(E), E4 = stride / 4;
  int parts = kMetaThreads / E4;
  if (parts > kMaxParts) parts = kMaxParts;
  if (tid < parts * E4) {
    const int g = tid % E4, part = tid / E4;
    const int b0 = (int)((int64_t)B * part / parts), b1 = (int)((int64_t)B * (part + 1) / parts);
    int4 tot = make_int4(0, 0, 0, 0), pre = make_int4(0, 0, 0, 0);
#pragma unroll 4
    for (int bb = b0; bb < b1; ++bb) {
      const int4 v = __ldcg(reinterpret_cast<const int4 *>(ws_hist + (size_t)bb * stride) + g);
      tot.x += v.x;
      tot.y += v.y;
      tot.z += v.z;
      tot.w += v.w;
      if (bb < b) {
        pre.x += v.x;
        pre.y += v.y;
        pre.z += v.z;
        pre.w += v.w;
      }
    }
    reinterpret_cast<int4 *>(sh.tot + part * stride)[g] = tot;
    reinterpret_cast<int4 *>(sh.pre + part * stride)[g] = pre;
  }
  __syncthreads();
  if (warp == 0) {  // sum the parts, scan the totals 32 experts at a time
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int tot = 0, pre = 0;
      if (e < E)
        for (int part = 0; part < parts; ++part) {
          tot += sh.tot[part * stride + e];
          pre += sh.pre[part * stride + e];
        }
      int incl = tot;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const int excl = carry + incl - tot;
      if (e < E) {
        sh.base[e] = excl + pre;
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
}

// Positions of slots [f_lo, f_lo + count); slot i's expert and weight come
// from get(i) -> (e, w) (e = -1 for an invalid id).
template <typename Get>
__device__ void meta_scatter(int64_t f_lo, int count, int E, MetaShared &sh, Get get,
                             int32_t *__restrict__ col_sorted, int32_t *__restrict__ row_sorted,
                             uint16_t *__restrict__ gate_scal) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r0 = 0; r0 < count; r0 += kMetaThreads) {
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
    if (e >= 0) {
      int p = sh.base[e] + rank;
      for (int ww = 0; ww < warp; ++ww) p += sh.cnt[ww][e];
      const int32_t f = (int32_t)(f_lo + i);
      col_sorted[p] = f;
      row_sorted[f] = p;
      gate_scal[p] = w;
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += kMetaThreads) {
      int add = 0;
      for (int ww = 0; ww < kMetaWarps; ++ww) add += sh.cnt[ww][ee];
      sh.base[ee] += add;
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
  __shared__ MetaShared sh;
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  const int lo = (int)min((int64_t)N, (int64_t)b * chunk);
  const int hi = (int)min((int64_t)N, (int64_t)lo + chunk);
  const int stride = hist_stride(E);

  for (int e = tid; e < stride; e += kMetaThreads) sh.base[e] = 0;
  if (tid == 0) sh.bad = 0;
  __syncthreads();
  for (int f = lo + tid; f < hi; f += kMetaThreads) {
    const int e = __ldg(topk_indx + f);
    if ((unsigned)e < (unsigned)E) atomicAdd(&sh.base[e], 1);
    else sh.bad = 1;
  }
  __syncthreads();
  if (sh.bad) record_status(ctrl, MOE_ERR_INVALID_ARG);
  for (int e = tid; e < stride; e += kMetaThreads) ws_hist[(size_t)b * stride + e] = sh.base[e];

  if (!grid_barrier(ctrl, timeout_ns)) return;
  meta_prefix(ws_hist, E, sh, col_sum, offs);
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
  cfg.numAttrs = 1;
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
// moe_forward's first two stages in one cooperative kernel, one CTA per SM:
// CTA b routes tokens [b*T, b*T + T) (staged as above) keeping its slots
// and histogram in shared memory, publishes the histogram, passes the
// bounded grid barrier, and scatters its slots from shared memory.
template <int EPL, bool VEC>
__global__ void __launch_bounds__(kRouteThreads, 1) route_metadata_kernel(
    const float *__restrict__ logits, int64_t n, int E, int k, int gating, int T, int TR,
    int bulk_ok, int32_t *__restrict__ topk_indx, uint16_t *__restrict__ topk_vals,
    int32_t *__restrict__ col_sum, int32_t *__restrict__ offs, int32_t *__restrict__ col_sorted,
    int32_t *__restrict__ row_sorted, uint16_t *__restrict__ gate_scal,
    int32_t *__restrict__ ws_hist, uint32_t *ctrl, unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ MetaShared sh;
  __shared__ __align__(8) uint64_t bars[kMaxChunks];
  __shared__ unsigned s_plain;
  float *stage = aligned_stage(smem_raw);
  uint8_t *s_slot_e = reinterpret_cast<uint8_t *>(stage) + (size_t)TR * E * 4 + kStagePad;
  uint16_t *s_slot_v = reinterpret_cast<uint16_t *>(s_slot_e + (((size_t)T * k + 15) & ~15ull));

  const int tid = threadIdx.x;
  const int stride = hist_stride(E);
  for (int e = tid; e < stride; e += kRouteThreads) sh.base[e] = 0;
  init_chunk_bars(bars);
  __syncthreads();

  const int64_t t0 = min(n, (int64_t)blockIdx.x * T);
  const int64_t t1 = min(n, t0 + T);
  uint32_t phase_bits = 0;
  route_block<EPL, VEC, true>(logits, t0, t1, E, k, gating, TR, bulk_ok != 0, topk_indx,
                              topk_vals, stage, bars, phase_bits, &s_plain, s_slot_e, s_slot_v,
                              sh.base, ctrl, timeout_ns);
  __syncthreads();
  for (int e = tid; e < stride; e += kRouteThreads)
    ws_hist[(size_t)blockIdx.x * stride + e] = sh.base[e];

  if (!grid_barrier(ctrl, timeout_ns)) return;
  meta_prefix(ws_hist, E, sh, col_sum, offs);
  meta_scatter(
      t0 * k, (int)(t1 - t0) * k, E, sh,
      [&](int i, int &e, uint16_t &w) {
        e = s_slot_e[i];
        w = s_slot_v[i];
      },
      col_sorted, row_sorted, gate_scal);
}

struct RouteMetaLaunch {
  const float *logits;
  int64_t n;
  int E, k, gating;
  int32_t *indx;
  uint16_t *vals;
  const moe_routing_meta *meta;
  int32_t *ws_hist;
  uint32_t *ctrl;
  cudaStream_t s;
  template <int EPL, bool VEC>
  cudaError_t go() {
    const int sms = device_sm_count();
    int64_t B = (n + 3) / 4;
    if (B > sms) B = sms;
    if (B < 1) B = 1;
    int64_t T = (n + B - 1) / B;
    T = (T + 3) / 4 * 4;
    B = (n + T - 1) / T;
    if (B < 1) B = 1;
    const int TR = (int)min((int64_t)staging_round_tokens(E),
                            (T + kChunkTok - 1) / kChunkTok * kChunkTok);
    const size_t slots = (size_t)T * k;
    const size_t smem = 128 + (size_t)TR * E * 4 + kStagePad + ((slots + 15) & ~(size_t)15) +
                        slots * 2;
    auto kern = route_metadata_kernel<EPL, VEC>;
    const int max_smem = 128 + kStageBytes + kStagePad + kSlotCap * 3 + 16;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (err != cudaSuccess) return err;
    int bulk_ok = ((uintptr_t)logits % 16) == 0;
    int Ti = (int)T;
    int64_t nn = n;
    int E_ = E, k_ = k, g_ = gating;
    unsigned long long timeout = kWaitTimeoutNs;
    void *args[] = {(void *)&logits, (void *)&nn, (void *)&E_, (void *)&k_, (void *)&g_,
                    (void *)&Ti, (void *)&TR, (void *)&bulk_ok, (void *)&indx, (void *)&vals,
                    (void *)&meta->col_sum, (void *)&meta->offs, (void *)&meta->col_sorted,
                    (void *)&meta->row_sorted, (void *)&meta->gate_scal, (void *)&ws_hist,
                    (void *)&ctrl, (void *)&timeout};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelExC(&cfg, (const void *)kern, args);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
  }
};

// True when the fused kernel can take (n, k): each CTA's slots fit in
// shared memory. Otherwise moe_forward runs route_kernel + metadata_kernel.
bool route_metadata_fits(int64_t n, int k) {
  const int sms = device_sm_count();
  int64_t T = (n + sms - 1) / sms;
  T = (T + 3) / 4 * 4;
  return T * k <= kSlotCap;
}

cudaError_t launch_route_metadata(const float *logits, int64_t n, int E, int k, int gating,
                                  int32_t *topk_indx, uint16_t *topk_vals,
                                  const moe_routing_meta &meta, int32_t *ws_hist,
                                  uint32_t *ctrl, cudaStream_t s) {
  return dispatch_epl(E, RouteMetaLaunch{logits, n, E, k, gating, topk_indx, topk_vals, &meta,
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
