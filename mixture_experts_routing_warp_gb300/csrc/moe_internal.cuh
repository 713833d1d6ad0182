// moe_internal.cuh -- shared pieces of the CUDA path: workspace layout,
// bounded device-side waits, bf16 helpers, kernel launcher declarations.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------- limits --
constexpr int kMaxExperts = 256;
constexpr int kMaxTopk = 8;
constexpr int kMetaMaxCtas = 1024;       // cap on the metadata kernel's grid
constexpr size_t kCtrlBytes = 4096;      // control block at the start of the workspace
constexpr size_t kAlign = 256;

// Control block words (uint32 index into the control block).
constexpr int kCtrlStatus = 0;           // sticky moe_status from device-side waits
constexpr int kCtrlBarArrive = 32;       // grid barrier counter (top bit flips per barrier)
constexpr int kCtrlNeverSet = 96;        // a word no kernel writes (bounded-wait self-test)

// Per-forward synchronisation words of the expert contractions, zeroed by the
// routing kernels (or the dispatch gather) of each forward:
//   [kSyncReady, +kMaxExperts): per-expert completion counts of the w13
//     contraction; the w2 contraction starts an expert's tiles once complete;
//   [kSyncSk, +4 * kSkMaxCtas): arrival counters (per first CTA of a split
//     tile and TMEM lane quarter) of the w13 contraction's decode stream-K
//     partition;
//   [kSyncSk2, +4 * kSkMaxCtas): the same for the w2 tiles of a decode
//     launch that runs both contractions.
constexpr int kSkMaxCtas = 256;
constexpr int kSyncReady = 0;
constexpr int kSyncSk = kMaxExperts;
constexpr int kSyncSk2 = kSyncSk + 4 * kSkMaxCtas;
constexpr int kSyncWords = kMaxExperts + 2 * 4 * kSkMaxCtas;
// Decode tiling (32-row token tiles, stream-K) applies when n*k <= 32 * E.
constexpr int kDecodeRowsPerExpert = 32;
// fp32 partial sums per stream-K CTA: 2 slots (the CTA's first and last
// piece) x 2 contractions (w13, then w2 in a launch that runs both) x 128
// weight rows x 32 token columns.
constexpr size_t kSkPartFloats = 2 * 2 * 128 * 32;

// Default limit of a device-side wait (ns). Legitimate waits last microseconds.
constexpr unsigned long long kWaitTimeoutNs = 1000000000ull;

// Count rows of the cooperative route + metadata kernel (routing_common.cuh):
// kFusedMaxRows rows (one per CTA, one CTA per SM) of up to kMaxExperts
// 16-bit counts, right after the control block.
constexpr int kFusedMaxRows = 256;
constexpr size_t kFusedRowsBytes = (size_t)kFusedMaxRows * kMaxExperts * 2;

// ------------------------------------------------------ workspace layout --
struct WorkspaceLayout {
  size_t ctrl, frows, hist, topk_indx, topk_vals, col_sum, offs, col_sorted, row_sorted, gate_scal;
  size_t sync, sk_part, x_sorted, h, y_flat, total;
  size_t bytes[MOE_WS_REGIONS];  // bytes each region uses, in layout order
  int regions;
};

// What the expert contractions use besides their operands: the control
// block (status word), the per-forward sync words, the stream-K partials
// (null when the workspace has none: n*k > 32 * E).
struct FfnScratch {
  uint32_t *ctrl;
  uint32_t *sync;
  float *sk_part;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Regions: control block; the route + metadata kernel's count rows;
// per-CTA histograms of the metadata kernel; the
// routing result and metadata used when moe_forward's caller keeps them
// internal; the sync words of the expert contractions; the decode stream-K
// partial sums (n*k <= 32 * E only); the expert-sorted activations X_sorted
// [N, H]; the intermediate h [N, I]; the per-slot outputs y_flat [N, H]
// (at k = 1 used only with an expert map, where the combine writes the zero
// rows of tokens without a local slot). N = n * k.
inline WorkspaceLayout workspace_layout(int64_t n, int E, int k, int H, int I) {
  WorkspaceLayout L{};
  const size_t N = (size_t)n * (size_t)k;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, kAlign);
    L.bytes[L.regions++] = bytes;
    return at;
  };
  L.ctrl = take(kCtrlBytes);
  L.frows = take(kFusedRowsBytes);  // at kCtrlBytes: right after the control block
  L.hist = take((size_t)kMetaMaxCtas * (size_t)((E + 3) & ~3) * 4);  // rows padded to 4
  L.topk_indx = take(N * 4);
  L.topk_vals = take(N * 2);
  L.col_sum = take((size_t)E * 4);
  L.offs = take((size_t)(E + 1) * 4);
  L.col_sorted = take(N * 4);
  L.row_sorted = take(N * 4);
  L.gate_scal = take(N * 2);
  L.sync = take((size_t)kSyncWords * 4);
  L.sk_part = take(N <= (size_t)kDecodeRowsPerExpert * (size_t)E
                       ? (size_t)kSkMaxCtas * kSkPartFloats * 4
                       : 0);
  L.x_sorted = take(N * (size_t)H * 2);
  L.h = take(N * (size_t)I * 2);
  L.y_flat = take(N * (size_t)H * 2);
  L.total = o;
  return L;
}

// ------------------------------------------------------- device helpers --
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// ------------------------------------------------------------- clusters --
// Rank of this CTA in its cluster, the cluster's CTA count and its index in
// the grid (x); a launch without cluster dimensions is a cluster of one.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_ctas() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster; orders shared-memory writes (and
// mbarrier initialisation) before the other CTAs' accesses that follow.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ int ld_shared_cluster(uint32_t cluster_addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// Sticky first error in the control block (no-op without one, as for
// moe_route, which takes no workspace).
__device__ __forceinline__ void record_status(uint32_t *ctrl, moe_status s) {
  if (ctrl) atomicCAS(ctrl + kCtrlStatus, (uint32_t)MOE_OK, (uint32_t)s);
}

// Deadline of a bounded wait in SM clock cycles: timeout_ns at 3 cycles/ns,
// so the real limit is at least timeout_ns (clocks <= 2.1 GHz) and at most
// 3x it at low clocks. clock64 is a cheap per-SM counter; reading it costs
// nothing like %globaltimer, so it is only sampled after a poll misses.
__device__ __forceinline__ long long wait_deadline(unsigned long long timeout_ns) {
  return clock64() + (long long)(timeout_ns * 3ull);
}

// Grid-wide barrier for a cooperative launch, bounded by `timeout_ns`.
// Thread 0 of each CTA adds to one counter with release semantics: CTA 0
// adds 2^31 - (gridDim.x - 1), the others 1, so when every CTA has arrived
// the counter's top bit has flipped and its low bits are back where they
// started (no reset step, and any grid size may use the same counter next
// time). Each thread 0 then polls with acquire loads until the top bit
// differs from the value its own add returned. Returns false (and records
// MOE_ERR_TIMEOUT) when the wait gives up; the caller must then return
// without touching shared outputs. After a timeout the counter is off and
// later barriers on this workspace time out too, until the control block is
// cleared (moe_read_status with reset).
// The barrier in two halves, so that a CTA can do work that the other CTAs
// do not wait for between its arrival and its wait: grid_arrive (every
// thread; returns thread 0's old counter value) and grid_wait (every thread,
// with that value).
__device__ __forceinline__ uint32_t grid_arrive(uint32_t *ctrl) {
  __syncthreads();
  uint32_t old = 0;
  if (threadIdx.x == 0) {
    const uint32_t inc = blockIdx.x == 0 ? (0x80000000u - (gridDim.x - 1u)) : 1u;
    old = atom_add_release_gpu(ctrl + kCtrlBarArrive, inc);
  }
  return old;
}

__device__ __forceinline__ bool grid_wait(uint32_t *ctrl, uint32_t old,
                                          unsigned long long timeout_ns) {
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    uint32_t *ctr = ctrl + kCtrlBarArrive;
    int ok = 1;
    if (((ld_acquire_gpu(ctr) ^ old) & 0x80000000u) == 0u) {
      const long long deadline = wait_deadline(timeout_ns);
      while (((ld_acquire_gpu(ctr) ^ old) & 0x80000000u) == 0u) {
        if (clock64() > deadline) {
          ok = 0;
          record_status(ctrl, MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

__device__ __forceinline__ bool grid_barrier(uint32_t *ctrl, unsigned long long timeout_ns) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t *ctr = ctrl + kCtrlBarArrive;
    const uint32_t inc = blockIdx.x == 0 ? (0x80000000u - (gridDim.x - 1u)) : 1u;
    const uint32_t old = atom_add_release_gpu(ctr, inc);
    int ok = 1;
    if (((ld_acquire_gpu(ctr) ^ old) & 0x80000000u) == 0u) {
      const long long deadline = wait_deadline(timeout_ns);
      while (((ld_acquire_gpu(ctr) ^ old) & 0x80000000u) == 0u) {
        if (clock64() > deadline) {
          ok = 0;
          record_status(ctrl, MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&h);
}

// Router top-k keys: an order-preserving 32-bit image of an fp32 logit
// (-0.0 folded onto +0.0, NaN = 1 below every number, 0 below everything),
// and a K-entry list kept in (key descending, expert id ascending) order.
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 1u;                         // NaN: below every number
  const uint32_t u = __float_as_uint(v + 0.0f);  // -0.0 + 0.0 = +0.0: the two zeros tie
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

template <int K>
struct TopK {
  uint32_t key[K];
  int e[K];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int i = 0; i < K; ++i) {
      key[i] = 0u;  // below every present element
      e[i] = 0x7fffffff;
    }
  }
  // Elements arriving in ascending id: enter only if strictly larger.
  __device__ __forceinline__ void push_ascending(uint32_t kv, int ev) {
    if (kv > key[K - 1]) {
#pragma unroll
      for (int i = K - 1; i > 0; --i) {
        const bool above = kv > key[i - 1];
        const bool here = kv > key[i];
        key[i] = above ? key[i - 1] : (here ? kv : key[i]);
        e[i] = above ? e[i - 1] : (here ? ev : e[i]);
      }
      if (kv > key[0]) {
        key[0] = kv;
        e[0] = ev;
      }
    }
  }
  // Any order: (key descending, id ascending).
  __device__ __forceinline__ static bool before(uint32_t ka, int ea, uint32_t kb, int eb) {
    return ka > kb || (ka == kb && ea < eb);
  }
  __device__ __forceinline__ void push_any(uint32_t kv, int ev) {
    if (before(kv, ev, key[K - 1], e[K - 1])) {
#pragma unroll
      for (int i = K - 1; i > 0; --i) {
        const bool above = before(kv, ev, key[i - 1], e[i - 1]);
        const bool here = before(kv, ev, key[i], e[i]);
        key[i] = above ? key[i - 1] : (here ? kv : key[i]);
        e[i] = above ? e[i - 1] : (here ? ev : e[i]);
      }
      if (before(kv, ev, key[0], e[0])) {
        key[0] = kv;
        e[0] = ev;
      }
    }
  }
};

// Resolved activation parameters handed to the FFN kernels.
struct ActParams {
  int act;         // moe_activation
  int layout;      // moe_w13_layout
  float alpha, beta, limit;
  int ffn_kernel;  // moe_ffn_kernel (host-side choice of the GEMM kernel)
};

// Logistic sigmoid 1 / (1 + e^-x) = 1 / (1 + 2^(-x log2 e)) on the special
// function unit: one ex2.approx and one rcp.approx (each within a few fp32
// ulp; subnormals flushed), far below the bf16 rounding of h that follows.
// The short-K epilogues are instruction-bound, and this is a fraction of the
// instructions of expf and an IEEE division. x -> -inf: 2^(+inf) = +inf and
// its reciprocal 0; x -> +inf: 2^(-inf) = 0 and the result 1.
__device__ __forceinline__ float sigmoid_fast(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return r;
}

// Gated activations of (gate, up). SwiGLU: (g * sigmoid(g)) * u, with
// g = min(g, limit), u = clamp(u, -limit, limit) first when a limit is set.
// SwiGLU-OAI: the same clamps, then (g * sigmoid(alpha g)) * (u + beta).
__device__ __forceinline__ float activate(float g, float u, const ActParams &p) {
  if (p.act == MOE_ACT_SWIGLU_OAI) {
    g = fminf(g, p.limit);
    u = fminf(fmaxf(u, -p.limit), p.limit);
    return (g * sigmoid_fast(p.alpha * g)) * (u + p.beta);
  }
  if (p.limit < INFINITY) {
    g = fminf(g, p.limit);
    u = fminf(fmaxf(u, -p.limit), p.limit);
  }
  return (g * sigmoid_fast(g)) * u;
}

// The non-gated ReLU2: max(a, 0)^2.
__device__ __forceinline__ float relu2(float a) {
  const float r = fmaxf(a, 0.0f);
  return r * r;
}

// Rows of one expert's w13: 2I (gate and up) or I (ReLU2).
inline int w13_rows(const ActParams &p, int I) { return p.act == MOE_ACT_RELU2 ? I : 2 * I; }

// Stage-timing event record: a plain record on an eager stream, an external
// record (an event-record node of the graph) while the stream is capturing.
inline cudaError_t record_stage_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  cudaError_t err = cudaStreamIsCapturing(s, &st);
  if (err != cudaSuccess) return err;
  return st == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
             : cudaEventRecord(ev, s);
}

// Programmatic dependent launch. The kernels after the first of a forward
// (gather, the two expert contractions, combine) are launched with
// launch_dependent(): they may be scheduled while the previous kernel of the
// stream still runs, do their set-up (barriers, TMEM, tensor-map prefetch),
// and call pdl_wait() -- a hardware wait for the previous grid to complete
// and its writes to be visible -- before reading anything it (or an earlier
// kernel) wrote. Every kernel calls pdl_launch_dependents() early so that
// the next one can be scheduled; all of its own CTAs are resident by then.
// One exception: the swap-operand w13 kernel triggers after its pdl_wait, and
// the w2 kernel that follows does not pdl_wait; it waits per expert on the
// w13 kernel's completion counters instead (everything older than the w13
// kernel is complete once the w13 kernel has passed its own pdl_wait).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Every kernel of the library asks for the same L1 / shared-memory split
// (all shared: the grouped GEMM needs ~200 KB), so that consecutive kernels
// never wait for an SM to drain and reconfigure. Call once per kernel and
// device before its first launch there (through PerDeviceOnce).
template <typename Kern>
inline cudaError_t uniform_carveout(Kern kern) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

// A kernel's function attributes (cudaFuncSetAttribute) belong to the
// context of the device that is current when they are set, so each device
// ordinal is configured on its own. run(fn) calls fn once per device, the
// first time any thread calls it with that device current; concurrent first
// calls serialise on a mutex, later calls cost one atomic load. A failed fn
// is retried on the next call.
class PerDeviceOnce {
 public:
  static constexpr int kMaxDevices = 64;
  template <typename F>
  cudaError_t run(F &&fn) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    err = fn();
    if (err == cudaSuccess) done_[dev].store(true, std::memory_order_release);
    return err;
  }

 private:
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices] = {};
};

// ----------------------------------------------------- kernel launchers --
// launch_ffn records ev_ffn[0] before the w13 kernel and ev_ffn[1] before the
// w2 kernel when ev_ffn is given (stage timing of moe_forward_timed).
// All return the launch's cudaError_t (cudaGetLastError after the launch).
int device_sm_count();

cudaError_t launch_route(const float *logits, int64_t n, int E, int k, int gating,
                         int32_t *topk_indx, uint16_t *topk_vals, uint32_t *ctrl,
                         cudaStream_t s);

// Fused route + metadata (one cooperative kernel) for moe_forward, when
// route_metadata_fits(n, k).
bool route_metadata_fits(int64_t n, int k);
cudaError_t launch_route_metadata(const float *logits, int64_t n, int E, int k, int gating,
                                  int32_t *topk_indx, uint16_t *topk_vals,
                                  const moe_routing_meta &meta, uint32_t *ctrl, cudaStream_t s, uint32_t *sync = nullptr,
                                  const int32_t *expert_map = nullptr, int E_loc = 0,
                                  const uint16_t *x = nullptr, int H = 0,
                                  uint16_t *x_sorted = nullptr);
// launch_route_metadata with x given copies the dispatch rows into x_sorted;
// moe_forward gives it x exactly when this holds for (n, E, k) (the
// cooperative kernel runs on at least half the SMs).
bool route_metadata_moves_rows(int64_t n, int E, int k);

// sync (may be null): the kSyncWords per-forward sync words of the expert
// contractions, zeroed by these kernels (and by the gather)
cudaError_t launch_metadata(const int32_t *topk_indx, const uint16_t *topk_vals, int64_t n, int E,
                            int k, const moe_routing_meta &meta, int32_t *ws_hist,
                            uint32_t *ctrl, cudaStream_t s, uint32_t *sync = nullptr,
                            const int32_t *expert_map = nullptr, int E_loc = 0);

// X_sorted[row_sorted[t*k + j]] = x[t] for the n tokens' k slots.
// sync (may be null): the kSyncWords sync words the gather zeroes
cudaError_t launch_gather_rows(const uint16_t *x, const int32_t *row_sorted, int64_t n, int k,
                               int H, uint16_t *x_sorted, uint32_t *sync, cudaStream_t s);

// row_sorted (may be null): leave out the slots whose row_sorted is -1
cudaError_t launch_combine(const uint16_t *y_flat, int64_t n, int k, int H, uint16_t *out,
                           cudaStream_t s, const int32_t *row_sorted = nullptr);

// The unsorted tokens x [n, H] and k, for the w13 contraction's fused
// dispatch gather: sorted row p is x[col_sorted[p] / k].
struct GatherSrc {
  const uint16_t *x;
  int64_t n;
  int k;
};

// The two expert contractions. The w13 one reads its token rows from
// x_sorted, or, with `gather` (swap-operand kernel only), straight from the
// unsorted tokens.
cudaError_t launch_ffn(const uint16_t *x_sorted, const int32_t *offs, const int32_t *col_sorted,
                       const uint16_t *gate_scal, const uint16_t *w13, const uint16_t *w2,
                       int64_t N, int E, int H, int I, const ActParams &act, uint16_t *h_buf,
                       uint16_t *y_flat, const FfnScratch &scr, cudaStream_t s,
                       cudaEvent_t *ev_ffn = nullptr, const GatherSrc *gather = nullptr);

// Tiling of the swap-operand contractions for N rows (host only): token-tile
// rows of each, weight tiles per expert of the w13 one, CTA pairs, decode
// tiling (32-row tiles; the w13 work may then split its units evenly over
// the grid), both contractions in one launch.
struct SwapPlan {
  int nt1, nt2, f_tiles1;
  bool decode, pair1, pair2, fused;
};
SwapPlan plan_ffn_swap(int64_t N, int E, int H, int I, const ActParams &act);

// The swap-operand grouped GEMM (weights on the MMA's M side, token tiles
// of 32 or 256 rows); launch_ffn hands over to it unless act.ffn_kernel is
// MOE_FFN_TILED.
cudaError_t launch_ffn_swap(const uint16_t *x_sorted, const int32_t *offs,
                            const int32_t *col_sorted, const uint16_t *gate_scal,
                            const uint16_t *w13, const uint16_t *w2, int64_t N, int E, int H,
                            int I, const ActParams &act, uint16_t *h_buf, uint16_t *y_flat,
                            const FfnScratch &scr, cudaStream_t s, cudaEvent_t *ev_ffn,
                            const GatherSrc *gather);

// Router matmul fused with the top-k (the tokens-on-M GEMM, EPI_ROUTE).
cudaError_t launch_route_gemm(const uint16_t *x, const uint16_t *w_gate, int64_t n, int E, int H,
                              int k, int gating, int32_t *topk_indx, uint16_t *topk_vals,
                              float *logits, uint32_t *ctrl, cudaStream_t s);

cudaError_t launch_wait_selftest(uint32_t *ctrl, unsigned long long timeout_ns, cudaStream_t s);

}  // namespace moe
