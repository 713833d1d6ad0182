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
// ffn1:  h[p, :]            = act(w13_e . X_sorted[p])         (EPI_ACT,
//        gated; EPI_RELU2: h = max(w1_e . X_sorted[p], 0)^2, non-gated)
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
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;                 // rows per tile (UMMA M)
constexpr int BN = 256;                 // accumulator columns per tile (UMMA N)
constexpr int BK = 64;                  // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int UK = 16;                  // K per tcgen05.mma (kind::f16)
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB

// Ring configuration by the B rows a stage holds (RB): 256 weight rows for
// the expert contractions (4 stages of 48 KB); the router's few gate rows
// leave room for a deeper ring (RB = 32: 9 stages of 20 KB), which is what
// keeps enough bytes in flight per SM when only n / 128 SMs have a tile.
template <int RB>
struct TCfg {
  static constexpr int kBBytes = RB * BK * 2;
  static constexpr int kStages =
      196608 / (A_BYTES + kBBytes) < 12 ? 196608 / (A_BYTES + kBBytes) : 12;
  static constexpr int kTmemCols = 2 * RB;  // two fp32 accumulators of RB columns
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 1;
  static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kStages * (A_BYTES + kBBytes) +
                                    kNumBars * 8 + 16 + 2 * (kMaxExperts + 1) * 4 + 16;
  static_assert(RB == 32 || RB == 64 || RB == 128 || RB == 256, "B rows per stage");
};

constexpr uint32_t kIdesc = make_idesc_bf16(BM, BN);

enum { EPI_ACT = 0, EPI_SCATTER = 1, EPI_RELU2 = 2, EPI_ROUTE = 3 };

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
  // router (EPI_ROUTE): one dense group of dense_rows tokens (offs == NULL),
  // B = the gate weights [n_experts, H]; per token the top-k of its logits
  int64_t dense_rows;
  int b_rows;  // weight rows of a stage's B box and the MMA's N (BN; the router: E to 16)
  int n_experts, topk, gating;
  int32_t *topk_indx;
  uint16_t *topk_vals;
  float *logits_out;             // [n, n_experts] fp32, or NULL
  uint32_t *ctrl;
  unsigned long long timeout_ns;
};

// ------------------------------------------------------------------ kernel --
template <int EPI, bool PACKED, int RB>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b, const GemmArgs args) {
  using C = TCfg<RB>;
  constexpr int STAGES = C::kStages;
  constexpr int B_BYTES = C::kBBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
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
  pdl_launch_dependents();

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
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  pdl_wait();  // offs and the operands come from earlier kernels of the stream
  if (args.offs) {
    for (int i = threadIdx.x; i <= E; i += kThreads) s_offs[i] = args.offs[i];
  } else if (threadIdx.x == 0) {  // one dense group (the router)
    s_offs[0] = 0;
    s_offs[1] = (int)args.dense_rows;
  }
  __syncthreads();
  if (warp == 0) row_tile_prefix(s_offs, E, BM, s_tstart);
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
        const Tile d = decode_tile(t, args.n_tiles, s_tstart, s_offs, E, BM);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, args.ctrl, args.timeout_ns)) {
            ok = false;
            break;
          }
          // B rows past b_rows keep stale data: the MMA's N stops at b_rows
          mbar_arrive_expect_tx(full_bar(stage), (uint32_t)(A_BYTES + args.b_rows * BK * 2));
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
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, s_abort, args.ctrl, args.timeout_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * RB);
        const uint32_t idesc = args.b_rows == BN ? kIdesc : make_idesc_bf16(BM, args.b_rows);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, s_abort, args.ctrl, args.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sw128_desc(sA_addr + stage * A_BYTES);
          const uint64_t bdesc = sw128_desc(sB_addr + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk)  // +32 bytes along K per step = +2 in the descriptor
            umma_bf16(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
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
      const Tile d = decode_tile(t, args.n_tiles, s_tstart, s_offs, E, BM);
      const int acc = local & 1;
      const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
      if (!wait_bounded(tfull_bar(acc), acc_phase, s_abort, args.ctrl, args.timeout_ns)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * RB);
      const int p = d.m0 + row;
      const bool valid = p < d.m_end;
      if (EPI == EPI_ROUTE) {
        // this thread's row holds token p's logits in columns [0, n_experts):
        // keep the top 8 by (value descending, expert id ascending), columns
        // arriving in ascending expert id
        const int En = args.n_experts;
        const int nchunk = (En + 31) / 32;
        float *lrow = (valid && args.logits_out) ? args.logits_out + (size_t)p * En : nullptr;
        TopK<8> tk;
        tk.init();
#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
          uint32_t r[32];
          TMEM_LD32(tbase + c * 32, r);
          tmem_wait_ld(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int e = c * 32 + i;
            if (e < En) {
              const float v = __uint_as_float(r[i]);
              if (lrow) lrow[e] = v;
              tk.push_ascending(order_key(v), e);
            }
          }
        }
        const int K = args.topk;
        const float v0 = key_to_float(tk.key[0]);
        float ex[8], denom = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          ex[j] = j < K ? expf(key_to_float(tk.key[j]) - v0) : 0.f;
          denom += ex[j];
        }
        if (args.gating == MOE_GATING_SOFTMAX_ALL) {  // uniform: every lane reads TMEM
          float sum = 0.f;
#pragma unroll 1
          for (int c = 0; c < nchunk; ++c) {
            uint32_t r[32];
            TMEM_LD32(tbase + c * 32, r);
            tmem_wait_ld(r);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i < En) sum += expf(__uint_as_float(r[i]) - v0);
          }
          denom = sum;
        }
        if (valid) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < K) {
              args.topk_indx[(size_t)p * K + j] = tk.e[j];
              args.topk_vals[(size_t)p * K + j] = float_to_bf16_bits(ex[j] / denom);
            }
        }
      } else if (EPI == EPI_RELU2) {
        // column j of the tile is h column nt*256 + j
        uint16_t *hrow = args.h_out + (size_t)p * args.I;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
          TMEM_LD32(tbase + c * 32, r);
          tmem_wait_ld(r);
          const int col = d.nt * BN + c * 32;
          if (valid && col < args.I) {
            uint32_t o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              o[j] = pack_bf16x2(relu2(__uint_as_float(r[2 * j])),
                                 relu2(__uint_as_float(r[2 * j + 1])));
            uint4 *dst = reinterpret_cast<uint4 *>(hrow + col);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
          }
        }
      } else if (EPI == EPI_ACT) {
        uint16_t *hrow = args.h_out + (size_t)p * args.I;
        if (PACKED) {
          // columns [0,128) gate_j, [128,256) up_j -> h columns nt*128 + j
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t g[32], u[32];
            TMEM_LD32(tbase + c * 32, g);
            TMEM_LD32(tbase + 128 + c * 32, u);
            tmem_wait_ld(g, u);
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
            tmem_wait_ld(r);
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
          tmem_wait_ld(r);
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
                 "r"(C::kTmemCols)
                 : "memory");
  }
}

template <int EPI, bool PACKED, int RB = BN>
cudaError_t launch_gemm(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a,
                        cudaStream_t s) {
  using C = TCfg<RB>;
  auto kern = grouped_gemm_kernel<EPI, PACKED, RB>;
  static PerDeviceOnce attr_set;
  {
    cudaError_t err = attr_set.run([kern] {
      cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
      return e != cudaSuccess ? e : uniform_carveout(kern);
    });
    if (err != cudaSuccess) return err;
  }
  const cudaError_t err = launch_dependent(kern, dim3(device_sm_count()), dim3(kThreads),
                                           C::kSmemBytes, s, ta, tb, a);
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace

// Router matmul with the top-k in its epilogue: logits = x . w_gate^T
// (tokens on the MMA's M side, the E <= 256 gate rows on N), then per token
// the k largest logits (ties to the lower expert id) and their gate weights.
cudaError_t launch_route_gemm(const uint16_t *x, const uint16_t *w_gate, int64_t n, int E, int H,
                              int k, int gating, int32_t *topk_indx, uint16_t *topk_vals,
                              float *logits, uint32_t *ctrl, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  CUtensorMap ta, tb;
  const int b_rows = (E + 15) / 16 * 16;  // the MMA's N: a multiple of 16
  if (!map_2d(&ta, x, (uint64_t)n, (uint64_t)H, BM) ||
      !map_3d(&tb, w_gate, 1ull, (uint64_t)E, (uint64_t)H, (uint32_t)b_rows))
    return cudaErrorInvalidValue;
  GemmArgs a{};
  a.b_rows = b_rows;
  a.offs = nullptr;
  a.dense_rows = n;
  a.E = 1;
  a.num_kb = H / BK;
  a.n_tiles = 1;  // E <= 256 columns
  a.n_experts = E;
  a.topk = k;
  a.gating = gating;
  a.topk_indx = topk_indx;
  a.topk_vals = topk_vals;
  a.logits_out = logits;
  a.ctrl = ctrl;
  a.timeout_ns = kWaitTimeoutNs;
  if (b_rows <= 32) return launch_gemm<EPI_ROUTE, false, 32>(ta, tb, a, s);
  if (b_rows <= 64) return launch_gemm<EPI_ROUTE, false, 64>(ta, tb, a, s);
  if (b_rows <= 128) return launch_gemm<EPI_ROUTE, false, 128>(ta, tb, a, s);
  return launch_gemm<EPI_ROUTE, false, 256>(ta, tb, a, s);
}

cudaError_t launch_ffn(const uint16_t *x_sorted, const int32_t *offs, const int32_t *col_sorted,
                       const uint16_t *gate_scal, const uint16_t *w13, const uint16_t *w2,
                       int64_t N, int E, int H, int I, const ActParams &act, uint16_t *h_buf,
                       uint16_t *y_flat, const FfnScratch &scr, cudaStream_t s,
                       cudaEvent_t *ev_ffn, const GatherSrc *gather) {
  if (N == 0) return cudaSuccess;
  if (act.ffn_kernel != MOE_FFN_TILED)  // AUTO: the swap-operand kernel at every size
    return launch_ffn_swap(x_sorted, offs, col_sorted, gate_scal, w13, w2, N, E, H, I, act, h_buf,
                           y_flat, scr, s, ev_ffn, gather);
  if (gather) return cudaErrorInvalidValue;  // the tokens-on-M kernel reads x_sorted
  uint32_t *ctrl = scr.ctrl;
  const bool relu2_act = act.act == MOE_ACT_RELU2;
  const bool packed = !relu2_act && act.layout == MOE_W13_PACKED;
  CUtensorMap ta1, tb1, ta2, tb2;
  if (!map_2d(&ta1, x_sorted, (uint64_t)N, (uint64_t)H, BM) ||
      !map_3d(&tb1, w13, (uint64_t)E, (uint64_t)w13_rows(act, I), (uint64_t)H,
              packed ? BN / 2 : BN) ||
      !map_2d(&ta2, h_buf, (uint64_t)N, (uint64_t)I, BM) ||
      !map_3d(&tb2, w2, (uint64_t)E, (uint64_t)H, (uint64_t)I, BN))
    return cudaErrorInvalidValue;

  GemmArgs a{};
  a.b_rows = BN;
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
  cudaError_t err;
  if (relu2_act) {
    a.n_tiles = (I + BN - 1) / BN;  // each tile yields 256 h columns
    err = launch_gemm<EPI_RELU2, false>(ta1, tb1, a, s);
  } else {
    a.n_tiles = (I + BN / 2 - 1) / (BN / 2);  // each tile yields 128 h columns
    err = packed ? launch_gemm<EPI_ACT, true>(ta1, tb1, a, s)
                 : launch_gemm<EPI_ACT, false>(ta1, tb1, a, s);
  }
  if (err != cudaSuccess) return err;

  if (ev_ffn && record_stage_event(ev_ffn[1], s) != cudaSuccess) return cudaErrorUnknown;
  a.num_kb = I / BK;
  a.n_tiles = (H + BN - 1) / BN;
  return launch_gemm<EPI_SCATTER, false>(ta2, tb2, a, s);
}

}  // namespace moe
