// grouped_gemm.cu -- the two expert contractions of the MoE layer as one
// persistent, warp-specialised tcgen05 grouped GEMM for sm_103a.
//
// Sources (page title, section):
//  "MoE feed-forward performs ~3xnum_experts device->host syncs per layer,
//    per forward" (MiniMind issue #835), "It is removable in plain PyTorch":
//    each expert runs on its contiguous slice of the expert-sorted rows;
//    Summary: the router weight multiplies the expert output.
//  "CuteDSL NVFP4 MoE adds SwiGLU-OAI and ReLU2" (vLLM PR #47106 report),
//    关键源码片段: SwiGLU / SwiGLU-OAI, interleaved [gate0, up0, ...] and
//    packed [gate; up] w13 rows.
//  "Reuse topk SparseMatrix routing metadata in GPT-OSS MoE forward" (vLLM
//    PR #45457 report), 关键源码片段: gate_scal in sorted order and the
//    scatter (row_sorted, col_sorted) back to token-slot order.
//
// ffn1:  h[p, :]            = act(w13_e . X_sorted[p])         (EPI_ACT)
// ffn2:  y_flat[col_sorted[p], :] = gate_scal[p] * (w2_e . h[p]) (EPI_SCATTER)
// for p in expert e's slice [offs[e], offs[e+1]).
//
// Per CTA (one per SM, persistent over tiles t = blockIdx.x + i*gridDim.x):
//   warp 0      TMA producer: A tile [128 x 64] of the sorted rows and B tile
//               [256 x 64] of the expert's weight rows, 128B-swizzled, into a
//               4-stage shared-memory ring (full/empty mbarriers)
//   warp 1      allocates 512 TMEM columns; one thread issues
//               tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, M=128, N=256,
//               K=16) into one of two 256-column accumulators, commits
//               stage releases and "accumulator full"
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows (warp w reads
//               TMEM lanes 32*(w%4)..), activation or gate scale, bf16
//               stores; "accumulator empty" lets the next tile's MMAs reuse it
// Ragged per-expert tiles come from offs on the device: m-tile counts per
// expert, a prefix over experts in shared memory, and a binary search per
// tile. Rows of a tile past the expert's slice are computed and dropped.
// Every mbarrier wait is bounded: on timeout the kernel records
// MOE_ERR_TIMEOUT, the other roles see the abort flag and leave, in-flight
// copies and MMAs are drained (bounded), TMEM is freed, and the kernel returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                 // rows per tile (UMMA M)
constexpr int BN = 256;                 // accumulator columns per tile (UMMA N)
constexpr int BK = 64;                  // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int UK = 16;                  // K per tcgen05.mma (kind::f16)
constexpr int STAGES = 4;
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB
constexpr int B_BYTES = BN * BK * 2;    // 32 KB
constexpr int kTmemCols = 2 * BN;       // two fp32 accumulators
constexpr int kNumBars = 2 * STAGES + 2 + 2 + 1;
constexpr int kSmemBytes = 1024 /*alignment slack*/ + STAGES * (A_BYTES + B_BYTES) +
                           kNumBars * 8 + 16 + 2 * (kMaxExperts + 1) * 4 + 16;

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 =
// 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

enum { EPI_ACT = 0, EPI_SCATTER = 1 };

struct GemmArgs {
  const int32_t *offs;
  int E;
  int num_kb;      // K / BK
  int n_tiles;     // tiles along N
  int I, H;
  ActParams act;
  uint16_t *h_out;               // ffn1: h [N, I]
  const int32_t *col_sorted;     // ffn2
  const uint16_t *gate_scal;     // ffn2
  uint16_t *y_out;               // ffn2: y_flat [N or n, H]
  uint32_t *ctrl;
  unsigned long long timeout_ns;
};

// ------------------------------------------------------------ PTX wrappers --
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows
// of 128 bytes, 8-row groups 1024 bytes apart (SBO); LBO unused for this
// layout; bits 46-47 = 1 (descriptor version); bits 61-63 = 2 (SWIZZLE_128B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

#define TMEM_LD32(taddr, r)                                                                      \
  asm volatile(                                                                                  \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "   \
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "    \
      "%28, %29, %30, %31}, [%32];"                                                              \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),           \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),           \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])            \
      : "r"(taddr))

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bounded mbarrier wait. Returns false when this wait gave up (records
// MOE_ERR_TIMEOUT and raises the CTA's abort flag) or another role already
// aborted.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int *abort_flag, const GemmArgs &a) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long deadline = wait_deadline(a.timeout_ns);
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 15u) == 0) {
      if (*abort_flag) return false;
      if (clock64() > deadline) {
        *abort_flag = 1;
        record_status(a.ctrl, MOE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait used while draining, independent of the abort flag.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity,
                                           unsigned long long timeout_ns) {
  const long long deadline = wait_deadline(timeout_ns);
  while (!mbar_try_wait(bar, parity))
    if (clock64() > deadline) return;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)float_to_bf16_bits(lo) | ((uint32_t)float_to_bf16_bits(hi) << 16);
}

struct Tile {
  int e, m0, m_end, nt;
};

__device__ __forceinline__ Tile decode_tile(int t, int n_tiles, const int *s_tstart,
                                            const int *s_offs, int E) {
  Tile d;
  const int mt = t / n_tiles;
  d.nt = t - mt * n_tiles;
  int lo = 0, hi = E - 1;  // last expert whose first m-tile is <= mt owns it
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tstart[mid] <= mt) lo = mid;
    else hi = mid - 1;
  }
  d.e = lo;
  d.m0 = s_offs[lo] + (mt - s_tstart[lo]) * BM;
  d.m_end = min(d.m0 + BM, s_offs[lo + 1]);
  return d;
}

// ------------------------------------------------------------------ kernel --
template <int EPI, bool PACKED>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
  volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_offs = reinterpret_cast<int *>(tmem_slot + 4);
  int *s_tstart = s_offs + (kMaxExperts + 1);

  const uint32_t sA_addr = smem_u32(sA), sB_addr = smem_u32(sB);
  const uint32_t full0 = smem_u32(bars);
  auto full_bar = [&](int s) { return full0 + 8u * s; };
  auto empty_bar = [&](int s) { return full0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return full0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return full0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = full0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (int i = threadIdx.x; i <= E; i += kThreads) s_offs[i] = args.offs[i];
  __syncthreads();
  if (warp == 0) {  // exclusive prefix of m-tiles over experts
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int cnt = e < E ? (s_offs[e + 1] - s_offs[e] + BM - 1) / BM : 0;
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < E) s_tstart[e] = carry + incl - cnt;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_tstart[E] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_tstart[E] * args.n_tiles;
  const int num_kb = args.num_kb;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // stages filled whose consumption we have not seen
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        const Tile d = decode_tile(t, args.n_tiles, s_tstart, s_offs, E);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, args)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), A_BYTES + B_BYTES);
          tma_load_2d(sA_addr + stage * A_BYTES, &tmap_a, full_bar(stage), kb * BK, d.m0);
          if (PACKED) {
            tma_load_3d(sB_addr + stage * B_BYTES, &tmap_b, full_bar(stage), kb * BK,
                        d.nt * (BN / 2), d.e);
            tma_load_3d(sB_addr + stage * B_BYTES + B_BYTES / 2, &tmap_b, full_bar(stage),
                        kb * BK, args.I + d.nt * (BN / 2), d.e);
          } else {
            tma_load_3d(sB_addr + stage * B_BYTES, &tmap_b, full_bar(stage), kb * BK, d.nt * BN,
                        d.e);
          }
          issued = issued < STAGES ? issued + 1 : STAGES;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // wait (bounded) for the copies already issued into the ring to land
        for (uint32_t i = 0; i < issued; ++i) {
          int s = stage - 1 - (int)i;
          uint32_t ph = phase;
          if (s < 0) {
            s += STAGES;
            ph ^= 1u;
          }
          wait_drain(full_bar(s), ph, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, s_abort, args)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, s_abort, args)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sw128_desc(sA_addr + stage * A_BYTES);
          const uint64_t bdesc = sw128_desc(sB_addr + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk)  // +32 bytes along K per step = +2 in the descriptor
            umma_bf16(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, (kb | kk) != 0 ? 1u : 0u);
          umma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(tfull_bar(acc));
      }
      // every MMA issued so far completes before the drain barrier fires
      umma_commit(drain_bar);
      wait_drain(drain_bar, 0, 100000000ull);
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int row = q * 32 + lane;
    int local = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++local) {
      const Tile d = decode_tile(t, args.n_tiles, s_tstart, s_offs, E);
      const int acc = local & 1;
      const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
      if (!wait_bounded(tfull_bar(acc), acc_phase, s_abort, args)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      const int p = d.m0 + row;
      const bool valid = p < d.m_end;
      if (EPI == EPI_ACT) {
        uint16_t *hrow = args.h_out + (size_t)p * args.I;
        if (PACKED) {
          // columns [0,128) gate_j, [128,256) up_j -> h columns nt*128 + j
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t g[32], u[32];
            TMEM_LD32(tbase + c * 32, g);
            TMEM_LD32(tbase + 128 + c * 32, u);
            tmem_wait_ld();
            const int col = d.nt * 128 + c * 32;
            if (valid && col < args.I) {
              uint32_t o[16];
#pragma unroll
              for (int j = 0; j < 16; ++j)
                o[j] = pack_bf16x2(
                    activate(__uint_as_float(g[2 * j]), __uint_as_float(u[2 * j]), args.act),
                    activate(__uint_as_float(g[2 * j + 1]), __uint_as_float(u[2 * j + 1]),
                             args.act));
              uint4 *dst = reinterpret_cast<uint4 *>(hrow + col);
#pragma unroll
              for (int v = 0; v < 4; ++v)
                dst[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
            }
          }
        } else {
          // columns (2j, 2j+1) = (gate_j, up_j) -> h columns nt*128 + j
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t r[32];
            TMEM_LD32(tbase + c * 32, r);
            tmem_wait_ld();
            const int col = d.nt * 128 + c * 16;
            if (valid && col < args.I) {
              uint32_t o[8];
#pragma unroll
              for (int j = 0; j < 8; ++j)
                o[j] = pack_bf16x2(
                    activate(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]), args.act),
                    activate(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]),
                             args.act));
              uint4 *dst = reinterpret_cast<uint4 *>(hrow + col);
              dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
              dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            }
          }
        }
      } else {
        float g = 0.f;
        uint16_t *yrow = nullptr;
        if (valid) {
          g = bf16_bits_to_float(args.gate_scal[p]);
          yrow = args.y_out + (size_t)args.col_sorted[p] * args.H;
        }
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
          TMEM_LD32(tbase + c * 32, r);
          tmem_wait_ld();
          const int col = d.nt * BN + c * 32;
          if (valid && col < args.H) {
            uint32_t o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              o[j] = pack_bf16x2(__uint_as_float(r[2 * j]) * g, __uint_as_float(r[2 * j + 1]) * g);
            uint4 *dst = reinterpret_cast<uint4 *>(yrow + col);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// -------------------------------------------------------------- host side --
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 [rows, cols] row-major, boxes of 64 columns x box_rows rows, 128B swizzle.
bool map_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [E, rows, cols] row-major, boxes of 64 columns x box_rows rows x 1 expert.
bool map_3d(CUtensorMap *m, const void *base, uint64_t E, uint64_t rows, uint64_t cols,
            uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, rows, E};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {BK, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, bool PACKED>
cudaError_t launch_gemm(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a,
                        cudaStream_t s) {
  auto kern = grouped_gemm_kernel<EPI, PACKED>;
  static bool attr_set = false;  // one value for every device of the process
  if (!attr_set) {
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    if ((err = uniform_carveout(kern)) != cudaSuccess) return err;
    attr_set = true;
  }
  kern<<<device_sm_count(), kThreads, kSmemBytes, s>>>(ta, tb, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn(const uint16_t *x_sorted, const int32_t *offs, const int32_t *col_sorted,
                       const uint16_t *gate_scal, const uint16_t *w13, const uint16_t *w2,
                       int64_t N, int E, int H, int I, const ActParams &act, uint16_t *h_buf,
                       uint16_t *y_flat, uint32_t *ctrl, cudaStream_t s, cudaEvent_t *ev_ffn) {
  if (N == 0) return cudaSuccess;
  const bool packed = act.layout == MOE_W13_PACKED;
  CUtensorMap ta1, tb1, ta2, tb2;
  if (!map_2d(&ta1, x_sorted, (uint64_t)N, (uint64_t)H, BM) ||
      !map_3d(&tb1, w13, (uint64_t)E, 2ull * I, (uint64_t)H, packed ? BN / 2 : BN) ||
      !map_2d(&ta2, h_buf, (uint64_t)N, (uint64_t)I, BM) ||
      !map_3d(&tb2, w2, (uint64_t)E, (uint64_t)H, (uint64_t)I, BN))
    return cudaErrorInvalidValue;

  GemmArgs a{};
  a.offs = offs;
  a.E = E;
  a.I = I;
  a.H = H;
  a.act = act;
  a.h_out = h_buf;
  a.col_sorted = col_sorted;
  a.gate_scal = gate_scal;
  a.y_out = y_flat;
  a.ctrl = ctrl;
  a.timeout_ns = kWaitTimeoutNs;

  if (ev_ffn && record_stage_event(ev_ffn[0], s) != cudaSuccess) return cudaErrorUnknown;
  a.num_kb = H / BK;
  a.n_tiles = (I + BN / 2 - 1) / (BN / 2);  // each tile yields 128 h columns
  cudaError_t err = packed ? launch_gemm<EPI_ACT, true>(ta1, tb1, a, s)
                           : launch_gemm<EPI_ACT, false>(ta1, tb1, a, s);
  if (err != cudaSuccess) return err;

  if (ev_ffn && record_stage_event(ev_ffn[1], s) != cudaSuccess) return cudaErrorUnknown;
  a.num_kb = I / BK;
  a.n_tiles = (H + BN - 1) / BN;
  return launch_gemm<EPI_SCATTER, false>(ta2, tb2, a, s);
}

}  // namespace moe
