// grouped_gemm_swap.cu -- the expert contractions for small per-expert
// batches (decode): the same persistent, warp-specialised tcgen05 design as
// grouped_gemm.cu with the operands swapped, so that the weights fill the
// MMA's M side and the few token rows its N side.
//
// Sources (page title, section): as grouped_gemm.cu -- "MoE feed-forward
// performs ~3xnum_experts device->host syncs per layer, per forward"
// (contiguous per-expert slices, weight on the output), "CuteDSL NVFP4 MoE
// adds SwiGLU-OAI and ReLU2" (activations, w13 layouts), "Reuse topk
// SparseMatrix routing metadata in GPT-OSS MoE forward" (gate_scal, scatter).
//
// A tile is (expert e, 32 sorted rows of e's slice, 128 weight rows):
//   D[w, j] = sum_k W_e[f0 + w, k] * A[m0 + j, k]      (w < 128, j < 32)
// with tcgen05.mma M=128 (weight rows), N=32 (tokens), fp32 in TMEM. A tile
// reads its 128 x K weight slice once and the 32 x K token rows, so a decode
// step streams each touched expert's weights through all SMs.
//   ffn1, interleaved w13: weight rows 2i / 2i+1 are gate_i / up_i, in
//     adjacent TMEM lanes: one shuffle pairs them.
//   ffn1, packed w13: the gate rows and the up rows of the same h columns go
//     to two accumulators, so each thread holds its pair.
//   ffn1, ReLU2 (non-gated): weight row f0 + w is h column f0 + w.
//   ffn2: y_flat[col_sorted[m0 + j], f0 + w] = gate_scal[m0 + j] * D[w, j].
//
// Warps: 0 TMA producer, 1 TMEM allocation + MMA issue, 2-5 epilogue (warp
// q reads TMEM lanes 32*(q%4)..). Every mbarrier wait is bounded.
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int SW_M = 128;  // weight rows per tile (UMMA M)
constexpr int SW_N = 32;   // token rows per tile (UMMA N)
constexpr int SW_BK = 64;
constexpr int SW_UK = 16;
constexpr int SW_EPI_WARPS = 4;
constexpr int SW_THREADS = (2 + SW_EPI_WARPS) * 32;
constexpr int SW_A_BYTES = SW_M * SW_BK * 2;  // 16 KB of weights
constexpr int SW_B_BYTES = SW_N * SW_BK * 2;  // 4 KB of token rows
constexpr uint32_t kSwIdesc = make_idesc_bf16(SW_M, SW_N);

enum { SW_ACT = 0, SW_SCATTER = 1, SW_RELU2 = 2 };

template <bool DUAL>  // DUAL: gate and up weight tiles in each stage
struct SwCfg {
  static constexpr int kA = DUAL ? 2 : 1;
  static constexpr int kStages = DUAL ? 5 : 8;
  static constexpr int kStageBytes = kA * SW_A_BYTES + SW_B_BYTES;  // a multiple of 1 KB
  static constexpr int kAccCols = kA * SW_N;                        // one accumulator buffer
  static constexpr int kTmemCols = 2 * kAccCols;                    // 64 or 128 (power of 2)
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 1;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kNumBars * 8 + 16 +
                                    2 * (kMaxExperts + 1) * 4 + 16;
};

struct SwArgs {
  const int32_t *offs;
  int E;
  int num_kb;   // K / 64
  int f_tiles;  // weight-row tiles per expert
  int I, H;
  ActParams act;
  uint16_t *h_out;
  const int32_t *col_sorted;
  const uint16_t *gate_scal;
  uint16_t *y_out;
  uint32_t *ctrl;
  unsigned long long timeout_ns;
};

template <int EPI, bool PACKED>
__global__ void __launch_bounds__(SW_THREADS, 1)
    grouped_gemm_swap_kernel(const __grid_constant__ CUtensorMap tmap_w,
                             const __grid_constant__ CUtensorMap tmap_x, const SwArgs args) {
  constexpr bool DUAL = EPI == SW_ACT && PACKED;
  using C = SwCfg<DUAL>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kStageBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
  volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_offs = reinterpret_cast<int *>(tmem_slot + 4);
  int *s_tstart = s_offs + (kMaxExperts + 1);

  const uint32_t stage0 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars);
  auto full_bar = [&](int s) { return full0 + 8u * s; };
  auto empty_bar = [&](int s) { return full0 + 8u * (C::kStages + s); };
  auto tfull_bar = [&](int b) { return full0 + 8u * (2 * C::kStages + b); };
  auto tempty_bar = [&](int b) { return full0 + 8u * (2 * C::kStages + 2 + b); };
  const uint32_t drain_bar = full0 + 8u * (2 * C::kStages + 4);
  auto a_addr = [&](int s, int which) { return stage0 + s * C::kStageBytes + which * SW_A_BYTES; };
  auto b_addr = [&](int s) { return stage0 + s * C::kStageBytes + C::kA * SW_A_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), SW_EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (int i = threadIdx.x; i <= E; i += SW_THREADS) s_offs[i] = args.offs[i];
  __syncthreads();
  if (warp == 0) row_tile_prefix(s_offs, E, SW_N, s_tstart);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_tstart[E] * args.f_tiles;
  const int num_kb = args.num_kb;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        const Tile d = decode_tile(t, args.f_tiles, s_tstart, s_offs, E, SW_N);
        const int f0 = d.nt * SW_M;  // first weight row of the tile
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, args.ctrl, args.timeout_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), C::kStageBytes);
          tma_load_3d(a_addr(stage, 0), &tmap_w, full_bar(stage), kb * SW_BK, f0, d.e);
          if (DUAL)
            tma_load_3d(a_addr(stage, 1), &tmap_w, full_bar(stage), kb * SW_BK, args.I + f0, d.e);
          tma_load_2d(b_addr(stage), &tmap_x, full_bar(stage), kb * SW_BK, d.m0);
          issued = issued < (uint32_t)C::kStages ? issued + 1 : (uint32_t)C::kStages;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (uint32_t i = 0; i < issued; ++i) {
          int s = stage - 1 - (int)i;
          uint32_t ph = phase;
          if (s < 0) {
            s += C::kStages;
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
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, s_abort, args.ctrl, args.timeout_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kAccCols);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, s_abort, args.ctrl, args.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc0 = sw128_desc(a_addr(stage, 0));
          const uint64_t bdesc = sw128_desc(b_addr(stage));
          const bool first = kb == 0;
#pragma unroll
          for (int kk = 0; kk < SW_BK / SW_UK; ++kk)
            umma_bf16(d_tmem, adesc0 + 2u * kk, bdesc + 2u * kk, kSwIdesc,
                      (first && kk == 0) ? 0u : 1u);
          if (DUAL) {
            const uint64_t adesc1 = sw128_desc(a_addr(stage, 1));
#pragma unroll
            for (int kk = 0; kk < SW_BK / SW_UK; ++kk)
              umma_bf16(d_tmem + SW_N, adesc1 + 2u * kk, bdesc + 2u * kk, kSwIdesc,
                        (first && kk == 0) ? 0u : 1u);
          }
          umma_commit(empty_bar(stage));
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(tfull_bar(acc));
      }
      umma_commit(drain_bar);
      wait_drain(drain_bar, 0, 100000000ull);
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    // TMEM is read in 8-column chunks (tokens) up to the tile's valid rows:
    // decode tiles hold a few tokens, so the work and the code stay small.
    const int q = warp & 3;       // TMEM lane quarter this warp may read
    const int w = q * 32 + lane;  // weight row within the tile
    int local = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++local) {
      const Tile d = decode_tile(t, args.f_tiles, s_tstart, s_offs, E, SW_N);
      const int acc = local & 1;
      const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
      if (!wait_bounded(tfull_bar(acc), acc_phase, s_abort, args.ctrl, args.timeout_ns)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols);
      const int rows = d.m_end - d.m0;   // valid token columns of the tile
      const int frow = d.nt * SW_M + w;  // weight row of this thread
      int dst_mine = 0;
      float g_mine = 0.f;
      if (EPI == SW_SCATTER && lane < rows) {  // lane j: token j's destination and weight
        dst_mine = args.col_sorted[d.m0 + lane];
        g_mine = bf16_bits_to_float(args.gate_scal[d.m0 + lane]);
      }
      for (int c0 = 0; c0 < rows; c0 += 8) {
        uint32_t r0[8], r1[8];
        TMEM_LD8(taddr + c0, r0);
        if (DUAL) TMEM_LD8(taddr + SW_N + c0, r1);
        tmem_wait_ld();
        if (EPI == SW_SCATTER) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int j = c0 + i;
            const int dst = __shfl_sync(0xffffffffu, dst_mine, j & 31);
            const float g = __shfl_sync(0xffffffffu, g_mine, j & 31);
            if (j < rows && frow < args.H)
              args.y_out[(size_t)dst * args.H + frow] =
                  float_to_bf16_bits(__uint_as_float(r0[i]) * g);
          }
        } else if (EPI == SW_RELU2) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (c0 + i < rows && frow < args.I)
              args.h_out[(size_t)(d.m0 + c0 + i) * args.I + frow] =
                  float_to_bf16_bits(relu2(__uint_as_float(r0[i])));
        } else if (DUAL) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (c0 + i < rows && frow < args.I)
              args.h_out[(size_t)(d.m0 + c0 + i) * args.I + frow] = float_to_bf16_bits(
                  activate(__uint_as_float(r0[i]), __uint_as_float(r1[i]), args.act));
        } else {
          // weight rows 2i (gate) and 2i+1 (up) sit in lanes 2i, 2i+1
          const int c = frow >> 1;  // h column of this pair
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float mine = __uint_as_float(r0[i]);
            const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
            if ((lane & 1) == 0 && c0 + i < rows && c < args.I)
              args.h_out[(size_t)(d.m0 + c0 + i) * args.I + c] =
                  float_to_bf16_bits(activate(mine, other, args.act));
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

template <int EPI, bool PACKED>
cudaError_t launch_swap(const CUtensorMap &tw, const CUtensorMap &tx, const SwArgs &a,
                        cudaStream_t s) {
  constexpr bool DUAL = EPI == SW_ACT && PACKED;
  auto kern = grouped_gemm_swap_kernel<EPI, PACKED>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           SwCfg<DUAL>::kSmemBytes);
    if (err != cudaSuccess) return err;
    if ((err = uniform_carveout(kern)) != cudaSuccess) return err;
    attr_set = true;
  }
  kern<<<device_sm_count(), SW_THREADS, SwCfg<DUAL>::kSmemBytes, s>>>(tw, tx, a);
  return cudaGetLastError();
}

}  // namespace

bool use_swap_ffn(int64_t N, int E) { return N <= (int64_t)SW_N * E; }

cudaError_t launch_ffn_swap(const uint16_t *x_sorted, const int32_t *offs,
                            const int32_t *col_sorted, const uint16_t *gate_scal,
                            const uint16_t *w13, const uint16_t *w2, int64_t N, int E, int H,
                            int I, const ActParams &act, uint16_t *h_buf, uint16_t *y_flat,
                            uint32_t *ctrl, cudaStream_t s, cudaEvent_t *ev_ffn) {
  if (N == 0) return cudaSuccess;
  const bool relu2_act = act.act == MOE_ACT_RELU2;
  const bool packed = !relu2_act && act.layout == MOE_W13_PACKED;
  CUtensorMap tw1, tx1, tw2, tx2;
  if (!map_3d(&tw1, w13, (uint64_t)E, (uint64_t)w13_rows(act, I), (uint64_t)H, SW_M) ||
      !map_2d(&tx1, x_sorted, (uint64_t)N, (uint64_t)H, SW_N) ||
      !map_3d(&tw2, w2, (uint64_t)E, (uint64_t)H, (uint64_t)I, SW_M) ||
      !map_2d(&tx2, h_buf, (uint64_t)N, (uint64_t)I, SW_N))
    return cudaErrorInvalidValue;
  SwArgs a{};
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
  a.num_kb = H / SW_BK;
  a.f_tiles = (w13_rows(act, I) / (packed ? 2 : 1) + SW_M - 1) / SW_M;
  cudaError_t err = relu2_act ? launch_swap<SW_RELU2, false>(tw1, tx1, a, s)
                    : packed  ? launch_swap<SW_ACT, true>(tw1, tx1, a, s)
                              : launch_swap<SW_ACT, false>(tw1, tx1, a, s);
  if (err != cudaSuccess) return err;

  if (ev_ffn && record_stage_event(ev_ffn[1], s) != cudaSuccess) return cudaErrorUnknown;
  a.num_kb = I / SW_BK;
  a.f_tiles = (H + SW_M - 1) / SW_M;
  return launch_swap<SW_SCATTER, false>(tw2, tx2, a, s);
}

}  // namespace moe
