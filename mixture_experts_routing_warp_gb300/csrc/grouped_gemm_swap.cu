// grouped_gemm_swap.cu -- the expert contractions with the operands swapped:
// the weights fill the MMA's M side (128 weight rows per tile) and the
// expert-sorted token rows its N side. The same persistent, warp-specialised
// tcgen05 design as grouped_gemm.cu.
//
// Sources (page title, section): as grouped_gemm.cu -- "MoE feed-forward
// performs ~3xnum_experts device->host syncs per layer, per forward"
// (contiguous per-expert slices, weight on the output), "CuteDSL NVFP4 MoE
// adds SwiGLU-OAI and ReLU2" (activations, w13 layouts), "Reuse topk
// SparseMatrix routing metadata in GPT-OSS MoE forward" (gate_scal, scatter).
//
// A tile is (expert e, up to NT sorted rows of e's slice, 128 weight rows):
//   D[w, j] = sum_k W_e[f0 + w, k] * A[m0 + j, k]      (w < 128, j < rows)
// with tcgen05.mma M=128 (weight rows) and N = rows rounded up to 32 (so an
// expert's last, ragged token tile costs at most 31 idle columns, not up to
// 127 idle MMA rows as with tokens on M), fp32 in TMEM.
//   NT = 32: decode, a handful of tokens per expert; the weights stream
//     through all SMs.
//   NT = 32 .. 256: prefill; per contraction the NT with the least
//     estimated time (waves x per-tile cost; 256: the same MMA shape as
//     tokens-on-M tiles, on a CTA pair).
// Epilogues:
//   ffn1, interleaved w13: weight rows 2i / 2i+1 are gate_i / up_i, in
//     adjacent TMEM lanes: one shuffle pairs them.
//   ffn1, packed w13: loaded through a 4-D tensor map that interleaves the
//     gate and up rows of the same h columns on the way into shared memory,
//     so the tile is the interleaved layout's and so is the epilogue.
//   ffn1, ReLU2 (non-gated): weight row f0 + w is h column f0 + w.
//   ffn2: y_flat[col_sorted[m0 + j], f0 + w] = gate_scal[m0 + j] * D[w, j].
// TMEM is read in chunks of 32 (then 8) token columns up to the tile's rows.
//
// Token rows come from X_sorted (the expert-sorted copy that the gather
// kernel or the routing kernel writes) as 2-D boxes, or, with at most 2 slots
// per expert, straight from the unsorted
// x: the producer warp reads the tile's rows col_sorted[p] / k and each lane
// fetches 4 of them per K step with tile::gather4 (one-row boxes). A gather4
// costs about as much TMA time as a whole box, so wide tiles keep X_sorted.
//
// Between the contractions: the w13 kernel counts, per expert, the tiles
// whose h rows are stored; the w2 kernel waits for those counts instead of
// for the whole w13 grid, so its tiles of finished experts run on the SMs
// that w13 CTAs leave in their last wave. One SM streams a weight tile at
// roughly 70 GB/s at most, so a decode w13 contraction with fewer than two
// waves of tiles splits its (tile, K step) units evenly over the grid
// (stream-K) instead of leaving most SMs idle behind a few whole tiles.
// At decode sizes, and where both contractions run 256-row tiles on CTA
// pairs, one launch runs both: each CTA takes its w2 tiles (in reverse CTA
// order, or at decode split the same way under one wave) after its w13 work;
// at decode it fetches a w2 tile's weights into free stages before the
// tile's h rows are complete.
//
// Warps: 0 TMA producer, 1 TMEM allocation + MMA issue, then the epilogue
// warps (4; 8 for tiles wider than 32 rows, two per TMEM lane quarter): warp
// q reads TMEM lanes 32*(q%4).. . Every mbarrier and counter wait is bounded.
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int SW_M = 128;  // weight rows per tile (UMMA M)
constexpr int SW_BK = 64;
constexpr int SW_UK = 16;
constexpr int SW_A_BYTES = SW_M * SW_BK * 2;  // 16 KB of weights
constexpr int SW_NGRAN = 32;                  // token-column granularity of a tile's MMA N
constexpr int SW_SMEM_RING = 192 * 1024;      // bytes of stage ring at most

enum { SW_ACT = 0, SW_SCATTER = 1, SW_RELU2 = 2 };

// epilogue warps: one per TMEM lane quarter for decode tiles, two (taking
// alternate token chunks) for wider tiles
constexpr int sw_epi_warps(int nt) { return nt > SW_NGRAN ? 8 : 4; }

// PAIR: a CTA pair runs one MMA of M = 256 (cta_group::2); each CTA's stage
// holds its 128 weight rows and half of the tile's token rows.
template <int NT, bool PAIR = false>
struct SwCfg {
  static constexpr int kBBytes = (PAIR ? NT / 2 : NT) * SW_BK * 2;  // token rows of one stage
  static constexpr int kStageBytes = SW_A_BYTES + kBBytes;  // a multiple of 1 KB
  // pairs: 7 stages of 32 KB, which fit only without the 1 KB alignment slack
  static constexpr int kRing = PAIR ? 7 * 32 * 1024 : SW_SMEM_RING;
  static constexpr int kStages = kRing / kStageBytes < 8 ? kRing / kStageBytes : 8;
  static constexpr int kSlack = PAIR ? 0 : 1024;  // PAIR: the base must be 1024-aligned
  static constexpr int kEpiWarps = sw_epi_warps(NT);
  static constexpr int kThreads = (2 + kEpiWarps) * 32;
  static constexpr int kAccCols = NT;              // one accumulator buffer
  static constexpr int kTmemCols = 2 * kAccCols;   // a power of 2 in [64, 512]
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 1;
  static constexpr int kSmemBytes = kSlack + kStages * kStageBytes + kNumBars * 8 + 16 +
                                    2 * (kMaxExperts + 1) * 4 + 16;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns");
  static_assert(NT % SW_NGRAN == 0 && NT <= 256, "token tile");
  static_assert(kStages >= 4, "pipeline depth");
  static_assert(!PAIR || NT > SW_NGRAN, "CTA pairs: wide token tiles");
  static_assert((PAIR ? NT / 2 : NT) <= 4 * 32, "a gathering lane fetches 4 token rows");
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
  // Expert handoff between the two contractions. The w13 kernel adds one to
  // ready_out[e] per epilogue warp and tile of expert e once the tile's h
  // rows are stored; the w2 kernel loads expert e's h rows once ready_in[e]
  // reaches ceil(rows_e / ready_nt) * ready_per_tile, and meanwhile streams
  // the tile's weight rows (w, w_rows per expert) into L2.
  uint32_t *ready_out;
  const uint32_t *ready_in;
  int ready_nt, ready_per_tile;
  const uint16_t *w;
  int w_rows;
  // Dispatch gather fused into the token-operand loads (w13 contraction):
  // with gather_rows set, sorted row p is token gather_rows[p] / gather_k of
  // the unsorted tokens that tmap_x maps with one-row boxes, and the producer
  // warp fetches each tile's rows with tile::gather4 (one lane per 4 rows).
  const int32_t *gather_rows;
  int gather_k;
  // Decode stream-K (NT = 32, the w13 contraction when it has fewer than two
  // waves of tiles): CTA c owns the (tile, K step) units
  // [c * U / G, (c + 1) * U / G) of U = tiles * num_kb. A tile cut by a CTA
  // boundary is computed in pieces; each piece stores its fp32 partial sums
  // in its CTA's slot of sk_part, and the last piece to arrive on the tile's
  // counters (sk_cnt, per first CTA and TMEM lane quarter) adds them up in
  // piece order and applies the epilogue: no CTA waits for another.
  int stream_k;
  uint32_t *sk_cnt;
  float *sk_part;
  // Both contractions in one launch (decode tiling): once a CTA has done its
  // w13 work it runs w2 tiles (num_kb2 K steps, f_tiles2 weight tiles per
  // expert, through the second pair of tensor maps), each after its expert's
  // h rows are complete (ready_in, the counts ready_out collects). With
  // stream_k and less than one wave of w2 tiles, the w2 units are split
  // evenly over the grid as well (counters sk_cnt + 4 * kSkMaxCtas, the
  // second half of each partial slot).
  int num_kb2, f_tiles2;
};

// ------------------------------------------------------------- stream-K --
__device__ __forceinline__ int64_t sk_lo(int64_t c, int64_t U, int G) { return c * U / G; }
// CTA owning unit u: the largest c with sk_lo(c) <= u
__device__ __forceinline__ int sk_cta(int64_t u, int64_t U, int G) {
  return (int)(((u + 1) * G + U - 1) / U - 1);
}
// Pieces of the tile whose units start at u0: the CTAs c_first..c_last that
// own at least one of its units (with fewer units than CTAs, some CTAs in
// between own none).
__device__ __forceinline__ int sk_pieces(int c_first, int c_last, int64_t U, int G) {
  int pieces = 0;
  for (int c = c_first; c <= c_last; ++c) pieces += sk_lo(c, U, G) < sk_lo(c + 1, U, G);
  return pieces;
}

// One unit of a CTA's work: K steps [k_lo, k_hi) of tile t of contraction
// ph (0: the kernel's own; 1: the w2 tiles of a launch that runs both).
struct Work {
  int t, k_lo, k_hi, ph;
};

// The CTA's work items in order: whole tiles t = first + i * step, or
// (stream-K) the pieces of its unit range; then, in a launch that runs both
// contractions, whole w2 tiles t = (step - 1 - first) + i * step of total2
// (in reverse CTA order, so the CTAs left with one w13 tile fewer -- the last
// total % step -- take one w2 tile more), or with stream_k2 the pieces of its
// range of the w2 units. Every role walks the same list.
struct WorkIter {
  int64_t u, hi, u2, hi2;
  int t, total, kb;
  bool sk, sk2;
  int step;
  int t2, total2, kb2;
  // first, step: this CTA's (or CTA pair's) index and the number of them;
  // stream_k / stream_k2: split the first / second contraction's units
  __device__ WorkIter(bool stream_k, int total_tiles, int num_kb, int first, int step_,
                      int total2_ = 0, int num_kb2 = 0, bool stream_k2 = false)
      : u(0), hi(0), u2(0), hi2(0), t(first), total(total_tiles), kb(num_kb), sk(stream_k),
        sk2(stream_k2), step(step_), t2(step_ - 1 - first), total2(total2_), kb2(num_kb2) {
    if (sk) {
      const int64_t U = (int64_t)total * kb;
      u = sk_lo(first, U, step);
      hi = sk_lo(first + 1, U, step);
    }
    if (sk2) {
      const int64_t U2 = (int64_t)total2 * kb2;
      u2 = sk_lo(first, U2, step);
      hi2 = sk_lo(first + 1, U2, step);
    }
  }
  // the next piece of [u, hi) in tiles of k units
  __device__ static bool piece(int64_t &u, int64_t hi, int k, Work &w) {
    if (u >= hi) return false;
    w.t = (int)(u / k);
    const int64_t base = (int64_t)w.t * k, end = base + k < hi ? base + k : hi;
    w.k_lo = (int)(u - base);
    w.k_hi = (int)(end - base);
    u = end;
    return true;
  }
  __device__ bool next(Work &w) {
    w.ph = 0;
    if (sk) {
      if (piece(u, hi, kb, w)) return true;
    } else if (t < total) {
      w.t = t;
      w.k_lo = 0;
      w.k_hi = kb;
      t += step;
      return true;
    }
    w.ph = 1;
    if (sk2) return piece(u2, hi2, kb2, w);
    if (t2 >= total2) return false;
    w.t = t2;
    w.k_lo = 0;
    w.k_hi = kb2;
    t2 += step;
    return true;
  }
};

// Producer side of the handoff for tile (e, weight rows f0..), K steps
// [k_lo, k_hi) of num_kb: true once expert e's h rows are complete and
// visible to this thread's TMA loads. Meanwhile the weights of those K
// steps are fetched into L2.
__device__ __forceinline__ bool wait_expert_ready(const SwArgs &args, int e, int f0, int num_kb,
                                                  int k_lo, int k_hi, const int *s_offs,
                                                  volatile int *abort_flag) {
  const int rows = s_offs[e + 1] - s_offs[e];
  const uint32_t need =
      (uint32_t)((rows + args.ready_nt - 1) / args.ready_nt) * (uint32_t)args.ready_per_tile;
  const uint32_t *p = args.ready_in + e;
  if (ld_acquire_gpu(p) < need) {
    // the tile's weight rows are contiguous: W[e, f0 .. f0 + wr, 0 .. K)
    const int K = num_kb * SW_BK;
    const int wr = args.w_rows - f0 < SW_M ? args.w_rows - f0 : SW_M;
    const char *base = reinterpret_cast<const char *>(args.w + ((size_t)e * args.w_rows + f0) * K);
    // kept in L2 (evict_last) against the w13 contraction's streaming loads
    const uint64_t keep = l2_policy_evict_last();
    if (k_lo == 0 && k_hi == num_kb) {
      const uint32_t bytes = (uint32_t)wr * (uint32_t)K * 2u;
      for (uint32_t o = 0; o < bytes; o += 65536u)
        prefetch_l2_hint(base + o, bytes - o < 65536u ? bytes - o : 65536u, keep);
    } else {  // a piece of the tile: its K range of every row
      const uint32_t seg = (uint32_t)(k_hi - k_lo) * SW_BK * 2u;
      for (int r = 0; r < wr; ++r)
        prefetch_l2_hint(base + ((size_t)r * K + (size_t)k_lo * SW_BK) * 2, seg, keep);
    }
    const long long deadline = wait_deadline(args.timeout_ns);
    uint32_t spins = 0;
    while (ld_acquire_gpu(p) < need) {
      __nanosleep(64);
      if ((++spins & 15u) == 0) {
        if (*abort_flag) return false;
        if (clock64() > deadline) {
          *abort_flag = 1;
          record_status(args.ctrl, MOE_ERR_TIMEOUT);
          return false;
        }
      }
    }
  }
  fence_proxy_async_global();
  return true;
}

template <int W>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[W]) {
  static_assert(W == 8 || W == 32, "chunk width");
  if constexpr (W == 32) {
    TMEM_LD32(taddr, r);
  } else {
    TMEM_LD8(taddr, r);
  }
}

// Per-warp epilogue state of one tile.
struct EpiTile {
  uint32_t taddr;  // this warp's lanes, the tile's accumulator buffer
  int m0, rows;    // first sorted row, valid token columns
  int frow;        // weight row of this thread
  int lane;
  int dst_base;    // 32-token group whose scatter targets the lanes hold
  int dst_mine;    // lane l: destination row of token dst_base + l
  float g_mine;    // lane l: gate weight of token dst_base + l
};

// Token columns [c0, c0 + W) of the tile, accumulators r0 as fp32 bits:
// apply the epilogue. FULL: every column of the chunk is a valid token row
// (no per-column bounds test). Stores walk a row pointer instead of
// recomputing 64-bit offsets.
template <int EPI, int W, bool FULL = false>
__device__ __forceinline__ void epi_apply(EpiTile &t, int c0, const uint32_t (&r0)[W],
                                          const SwArgs &args) {
  const int nvalid = t.rows - c0;  // columns of this chunk holding tokens
  if constexpr (EPI == SW_SCATTER) {
    const int base = c0 & ~31;
    if (base != t.dst_base) {  // warp-uniform: next 32-token group
      t.dst_base = base;
      const int j = base + t.lane;
      t.dst_mine = j < t.rows ? args.col_sorted[t.m0 + j] : 0;
      t.g_mine = j < t.rows ? bf16_bits_to_float(args.gate_scal[t.m0 + j]) : 0.f;
    }
    if (t.frow < args.H) {
      uint16_t *col = args.y_out + t.frow;
#pragma unroll
      for (int i = 0; i < W; ++i) {
        const int j = c0 + i;
        const int dst = __shfl_sync(0xffffffffu, t.dst_mine, j & 31);
        const float g = __shfl_sync(0xffffffffu, t.g_mine, j & 31);
        if (FULL || i < nvalid)
          col[(size_t)dst * args.H] = float_to_bf16_bits(__uint_as_float(r0[i]) * g);
      }
    }
  } else if constexpr (EPI == SW_RELU2) {
    if (t.frow < args.I) {
      uint16_t *dst = args.h_out + (size_t)(t.m0 + c0) * args.I + t.frow;
#pragma unroll
      for (int i = 0; i < W; ++i, dst += args.I)
        if (FULL || i < nvalid) *dst = float_to_bf16_bits(relu2(__uint_as_float(r0[i])));
    }
  } else {
    // Weight rows 2i (gate) and 2i+1 (up) sit in lanes 2i, 2i+1 (either
    // layout: the packed one is interleaved by its tensor map). For each
    // pair of tokens (j, j+1) the even lane computes token j and the odd
    // lane token j+1: one shuffle hands over the missing operand.
    const int c = t.frow >> 1;  // h column of this lane pair
    const int odd = t.lane & 1;
    const bool col_ok = c < args.I;
    uint16_t *dst = args.h_out + (size_t)(t.m0 + c0 + odd) * args.I + c;
    const size_t step = 2 * (size_t)args.I;
#pragma unroll
    for (int i = 0; i < W; i += 2, dst += step) {
      const float a = __uint_as_float(r0[i]), b = __uint_as_float(r0[i + 1]);
      const float recv = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
      const float g = odd ? recv : a;  // even: gate_j (own), up_j (recv)
      const float u = odd ? b : recv;  // odd: gate_j+1 (recv), up_j+1 (own)
      if (col_ok && (FULL || i + odd < nvalid)) *dst = float_to_bf16_bits(activate(g, u, args.act));
    }
  }
}

// Token columns [c0, c0 + W) of the tile: read TMEM, apply the epilogue.
template <int EPI, int W, bool FULL = false>
__device__ __forceinline__ void epi_chunk(EpiTile &t, int c0, const SwArgs &args) {
  uint32_t r0[W];
  tmem_ld<W>(t.taddr + c0, r0);
  tmem_wait_ld(r0);
  epi_apply<EPI, W, FULL>(t, c0, r0, args);
}

// A whole tile's token columns for one epilogue warp: chunks of 32 columns
// (every column valid), then of 8; a lane quarter's kPer warps take
// alternate chunks (`half`: this warp's turn).
template <int EPI, int NT, int kPer>
__device__ __forceinline__ void epi_tile(EpiTile &et, int half, const SwArgs &args) {
  int c0 = 0;
  if constexpr (NT > SW_NGRAN) {
    const int full = et.rows & ~31;
    for (int c = 32 * half; c < full; c += 32 * kPer) epi_chunk<EPI, 32, true>(et, c, args);
    c0 = full;
  }
  for (int c = c0 + 8 * half; c < et.rows; c += 8 * kPer) epi_chunk<EPI, 8>(et, c, args);
}

// The w13 epilogue's handoff: this warp's h rows of a tile of expert e are
// stored; count them for the w2 kernel (the warp barrier orders every lane's
// stores before lane 0's release).
__device__ __forceinline__ void publish_ready(const SwArgs &args, int e, int lane) {
  fence_proxy_async_global();  // h rows -> the w2 kernel's TMA loads
  __syncwarp();
  if (lane == 0) atom_add_release_gpu(args.ready_out + e, 1u);
}

// A piece of a split tile (decode stream-K). The warp stores its partial
// sums (32 weight rows x the tile's token columns) in this
// CTA's slot -- slot 0 for the piece that starts the CTA's unit range, 1 for
// the one that ends it --, releases the accumulator buffer and counts the
// piece. The warp that counts the tile's last piece of its lane quarter adds
// the pieces' partials in piece order (a fixed order: the result does not
// depend on which piece finishes last) and applies the epilogue.
// ph: the contraction (0: w13; 1: the w2 tiles of a launch that runs both,
// with their own counters and the second half of each slot).
template <int EPI, int NT>
__device__ __forceinline__ void sk_piece(EpiTile &et, const SwArgs &args, int ph, int64_t u0,
                                         int c_first, int c_last, int pieces, int k_lo,
                                         int64_t U, int G, int q, int e, uint32_t tempty) {
  constexpr size_t kSlot = kSkPartFloats / 2;
  static_assert(2 * SW_M * NT <= (int)kSlot, "partial slot");
  const int w_row = q * 32 + et.lane;
  const int my_slot = u0 + k_lo == sk_lo(blockIdx.x, U, G) ? 0 : 1;
  float *const part0 = args.sk_part + (size_t)ph * SW_M * NT;
  uint32_t *const cnt = args.sk_cnt + (size_t)ph * 4 * kSkMaxCtas;
  float *mine = part0 + ((size_t)blockIdx.x * 2 + my_slot) * kSlot;
  for (int c = 0; c < et.rows; c += 8) {
    uint32_t r0[8];
    tmem_ld<8>(et.taddr + c, r0);
    tmem_wait_ld(r0);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c + i < et.rows) mine[(size_t)(c + i) * SW_M + w_row] = __uint_as_float(r0[i]);
  }
  tc_fence_before();
  __syncwarp();
  // the warp barrier orders every lane's partial stores before lane 0's
  // release; lane 0's acquire and the next warp barrier order the last
  // piece's reads of the other partials after their stores
  uint32_t old = 0;
  if (et.lane == 0) {
    mbar_arrive(tempty);
    old = atom_add_acq_rel_gpu(cnt + (size_t)c_first * 4 + q, 1u);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != (uint32_t)pieces - 1) return;
  __syncwarp();
  for (int c = 0; c < et.rows; c += 8) {
    float s0[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s0[i] = 0.f;
    for (int cta = c_first; cta <= c_last; ++cta) {
      const int64_t lo = sk_lo(cta, U, G);
      if (lo == sk_lo(cta + 1, U, G)) continue;  // owns no unit
      const int slot = (u0 > lo ? u0 : lo) == lo ? 0 : 1;
      const float *part = part0 + ((size_t)cta * 2 + slot) * kSlot;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (c + i < et.rows) s0[i] += __ldcg(part + (size_t)(c + i) * SW_M + w_row);
    }
    uint32_t r0[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) r0[i] = __float_as_uint(s0[i]);
    epi_apply<EPI, 8>(et, c, r0, args);
  }
  if (args.ready_out && ph == 0) publish_ready(args, e, et.lane);
}

// PACKED: the weights are a packed gated w13, read through the 4-D map that
// interleaves gate and up rows (box coordinates: column, 0, pair, expert).
// FUSE: the w13 contraction (EPI) and then the w2 one (gate scale + scatter,
// weights tmap_w2, h rows tmap_h) in one launch; its CTAs wait only for h
// rows that other CTAs of the same grid, all resident, compute first.
template <int EPI, bool PACKED, int NT, bool PAIR, bool FUSE>
__global__ void __launch_bounds__(SwCfg<NT, PAIR>::kThreads, 1)
    grouped_gemm_swap_kernel(const __grid_constant__ CUtensorMap tmap_w,
                             const __grid_constant__ CUtensorMap tmap_x,
                             const __grid_constant__ CUtensorMap tmap_w2,
                             const __grid_constant__ CUtensorMap tmap_h, const SwArgs args) {
  static_assert(!PACKED || EPI == SW_ACT, "the packed layout is a gated w13");
  static_assert(!FUSE || EPI != SW_SCATTER, "a fused launch starts with the w13 contraction");
  using C = SwCfg<NT, PAIR>;
  // PAIR: tiles of 256 weight rows; this CTA's half starts at row `rank` * 128
  constexpr int kTileRows = PAIR ? 2 * SW_M : SW_M;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  if (C::kSlack == 0 && (raw_addr & 1023u) != 0) {
    // no room to align the stages (128-byte swizzle needs 1024): refuse, in
    // every CTA alike (the same address in both CTAs of a pair)
    if (threadIdx.x == 0) record_status(args.ctrl, MOE_ERR_UNSUPPORTED);
    return;
  }
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
  auto a_addr = [&](int s) { return stage0 + s * C::kStageBytes; };
  auto b_addr = [&](int s) { return stage0 + s * C::kStageBytes + SW_A_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  const int first = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int step = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  if (!args.ready_out) pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), C::kEpiWarps * (PAIR ? 2 : 1));  // the leader's counts both CTAs
    }
    mbar_init(drain_bar, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
    if constexpr (FUSE) {
      prefetch_tmap(&tmap_w2);
      prefetch_tmap(&tmap_h);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {  // one warp of each CTA of the pair, collectively
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(C::kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(C::kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  // offs and the operands come from earlier kernels of the stream. The w2
  // kernel of a handoff skips the grid-wide wait: the w13 kernel triggered it
  // only after its own pdl_wait, so everything but h is complete, and h is
  // waited for per expert.
  if (FUSE || !args.ready_in) pdl_wait();
  if (args.ready_out) pdl_launch_dependents();
  for (int i = threadIdx.x; i <= E; i += C::kThreads) s_offs[i] = args.offs[i];
  __syncthreads();
  if (warp == 0) row_tile_prefix(s_offs, E, NT, s_tstart);
  tc_fence_before();
  if constexpr (PAIR) {
    cluster_sync();  // both CTAs' barriers and TMEM exist before any cross-CTA use
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_tstart[E] * args.f_tiles;
  const int num_kb = args.num_kb;
  const int total2 = FUSE ? s_tstart[E] * args.f_tiles2 : 0;  // w2 tiles after the w13 work
  const int num_kb2 = FUSE ? args.num_kb2 : 0;
  // stream-K pays only where whole tiles leave a large last wave idle; with
  // two or more waves, CTAs that finish early start the next contraction
  const bool sk = NT == SW_NGRAN && args.stream_k && total < 2 * (int)gridDim.x;
  // the w2 tiles of a fused launch: split only under one wave (GPT-OSS n = 1:
  // 92 tiles, 52.1 -> 50.8 us; at n = 4, ~2 waves, the split lost 3 us)
  const bool sk2 = FUSE && NT == SW_NGRAN && args.stream_k && total2 < (int)gridDim.x;
  // K steps of a fused launch's w2 tile whose weights may be fetched before
  // the expert's h rows are complete: the whole ring
  constexpr int kPreload = C::kStages;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    // Lane 0 waits for free stages and issues the weight (and plain token)
    // copies; with the fused gather every lane then fetches four token rows.
    const bool gather_rows = args.gather_rows != nullptr;
    const uint64_t read_once = l2_policy_evict_first();
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok = true;
    int ready_e = -1;  // expert whose h rows this warp has seen complete
    WorkIter it(sk, total, num_kb, first, step, total2, num_kb2, sk2);
    Work w;
    while (ok && it.next(w)) {
      const bool p1 = FUSE && w.ph == 1;  // a w2 tile of a fused launch
      const Tile d = decode_tile(w.t, p1 ? args.f_tiles2 : args.f_tiles, s_tstart, s_offs, E, NT);
      const int f0 = d.nt * kTileRows + (int)rank * SW_M;  // first weight row of this CTA
      const bool gather = gather_rows && !p1;
      const CUtensorMap *mw = p1 ? &tmap_w2 : &tmap_w;
      const CUtensorMap *mx = p1 ? &tmap_h : &tmap_x;
      // PAIR: the MMA reads its first n_mma / 2 token rows from the leader
      // and the rest from the peer
      const int rows = d.m_end - d.m0;
      const int n_mma = (rows + SW_NGRAN - 1) / SW_NGRAN * SW_NGRAN;
      const int m_b = d.m0 + (int)rank * (n_mma / 2);
      // Token rows a CTA gathers: only the tile's own, in groups of 4 (a
      // group's padding reads row 0). The MMA's padding rows up to n_mma keep
      // stale data: they feed only columns the epilogue discards.
      const int half = n_mma / 2;
      const int n_lead = PAIR ? (rows < half ? rows : half) : rows;
      const int n_peer = PAIR && rows > half ? rows - half : 0;
      const int n_cta = rank ? n_peer : n_lead;
      int g0 = 0, g1 = 0, g2 = 0, g3 = 0;  // this lane's 4 token rows
      if (gather && 4 * lane < n_cta) {
        const int p = m_b + 4 * lane;
        g0 = p < d.m_end ? args.gather_rows[p] / args.gather_k : 0;
        g1 = p + 1 < d.m_end ? args.gather_rows[p + 1] / args.gather_k : 0;
        g2 = p + 2 < d.m_end ? args.gather_rows[p + 2] / args.gather_k : 0;
        g3 = p + 3 < d.m_end ? args.gather_rows[p + 3] / args.gather_k : 0;
      }
      // stage bytes: weights, then the token rows (the gathered groups of
      // both CTAs of a pair; a plain box always its full height)
      const uint32_t b_bytes = gather ? 512u * (uint32_t)((n_lead + 3) / 4 + (n_peer + 3) / 4)
                                      : (uint32_t)(PAIR ? 2 : 1) * C::kBBytes;
      const uint32_t tx_bytes = (uint32_t)(PAIR ? 2 : 1) * SW_A_BYTES + b_bytes;
      int pre = 0;  // K steps whose weights went out before the expert's h was ready
      if ((FUSE ? p1 : args.ready_in != nullptr) && d.e != ready_e) {
        const int kbt = p1 ? num_kb2 : num_kb;
        if constexpr (FUSE && !PAIR) {
          // A w2 tile of a fused launch: its weights need no h, so the
          // weights of up to kPreload K steps go into free stages first and
          // their h boxes follow once the expert's h rows are complete.
          if (lane == 0) {
            const int s0 = stage;
            while (ok && pre < w.k_hi - w.k_lo && pre < kPreload) {
              ok = wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, args.ctrl, args.timeout_ns);
              if (!ok) break;
              mbar_arrive_expect_tx(full_bar(stage), tx_bytes);
              tma_load_3d_hint(a_addr(stage), mw, full_bar(stage), (w.k_lo + pre) * SW_BK, f0,
                               d.e, read_once);
              ++pre;
              issued = issued < (uint32_t)C::kStages ? issued + 1 : (uint32_t)C::kStages;
              if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (ok) ok = wait_expert_ready(args, d.e, f0, kbt, w.k_lo, w.k_hi, s_offs, s_abort);
            // the h boxes of those stages, after a failed wait too, so that
            // every posted stage completes (in-bounds reads) and the drain ends
            for (int i = 0; i < pre; ++i) {
              const int si = (s0 + i) % C::kStages;
              tma_load_2d(b_addr(si), mx, full_bar(si), (w.k_lo + i) * SW_BK, d.m0);
            }
          }
          pre = __shfl_sync(0xffffffffu, pre, 0);
          stage = __shfl_sync(0xffffffffu, stage, 0);
          phase = __shfl_sync(0xffffffffu, phase, 0);
          issued = __shfl_sync(0xffffffffu, issued, 0);
        } else {
          if (lane == 0)
            ok = wait_expert_ready(args, d.e, f0, kbt, w.k_lo, w.k_hi, s_offs, s_abort);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        ready_e = d.e;
      }
      for (int kb = w.k_lo + pre; kb < w.k_hi; ++kb) {
        if (lane == 0)
          ok = wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, args.ctrl, args.timeout_ns);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        if constexpr (PAIR) {
          // both CTAs' copies complete on the leader's full barrier
          const uint32_t fb = map_to_rank(full_bar(stage), 0);
          if (lane == 0) {
            if (leader) mbar_arrive_expect_tx(full_bar(stage), tx_bytes);
            if (PACKED && !p1)
              tma_load_4d_pair(a_addr(stage), mw, fb, kb * SW_BK, 0, f0 / 2, d.e);
            else
              tma_load_3d_pair(a_addr(stage), mw, fb, kb * SW_BK, f0, d.e);
            if (!gather) tma_load_2d_pair(b_addr(stage), mx, fb, kb * SW_BK, m_b);
          }
          __syncwarp();
          if (gather && 4 * lane < n_cta)
            tma_gather4_pair(b_addr(stage) + 512u * lane, &tmap_x, fb, kb * SW_BK, g0, g1, g2, g3);
        } else {
          if (lane == 0) {
            mbar_arrive_expect_tx(full_bar(stage), tx_bytes);
            if constexpr (NT == SW_NGRAN) {
              // decode: every weight line is read once (evict_first), leaving
              // L2 to the w2 tiles fetched ahead while their expert's h is
              // still being computed (GPT-OSS n = 4 / 8 / 64: 109.6 / 162.6 /
              // 255.7 -> 108.5 / 160.9 / 253.2 us per layer)
              if (PACKED && !p1)
                tma_load_4d_hint(a_addr(stage), mw, full_bar(stage), kb * SW_BK, 0, f0 / 2, d.e,
                                 read_once);
              else
                tma_load_3d_hint(a_addr(stage), mw, full_bar(stage), kb * SW_BK, f0, d.e,
                                 read_once);
            } else if (PACKED && !p1) {
              tma_load_4d(a_addr(stage), mw, full_bar(stage), kb * SW_BK, 0, f0 / 2, d.e);
            } else {
              tma_load_3d(a_addr(stage), mw, full_bar(stage), kb * SW_BK, f0, d.e);
            }
            if (!gather) tma_load_2d(b_addr(stage), mx, full_bar(stage), kb * SW_BK, d.m0);
          }
          __syncwarp();  // the expected bytes are posted before any gathered row lands
          if (gather && 4 * lane < n_cta)
            tma_gather4(b_addr(stage) + 512u * lane, &tmap_x, full_bar(stage), kb * SW_BK, g0, g1,
                        g2, g3);
        }
        issued = issued < (uint32_t)C::kStages ? issued + 1 : (uint32_t)C::kStages;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // a pair's copies complete on the leader's barriers: the leader drains
    // (the peer stays resident until the final cluster barrier)
    if (!ok && leader && lane == 0) {
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
  } else if (warp == 1) {
    // ------------------------------------- MMA issuer (a pair's leader) --
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      WorkIter it(sk, total, num_kb, first, step, total2, num_kb2, sk2);
      Work w;
      for (; ok && it.next(w); ++local) {
        const Tile d = decode_tile(w.t, FUSE && w.ph == 1 ? args.f_tiles2 : args.f_tiles,
                                   s_tstart, s_offs, E, NT);
        const int rows = d.m_end - d.m0;
        // MMA N: the tile's rows rounded up to 32 (a multiple of 16, <= 256)
        const int n_mma = (rows + SW_NGRAN - 1) / SW_NGRAN * SW_NGRAN;
        const uint32_t idesc = make_idesc_bf16(kTileRows, n_mma);
        const int acc = local & 1;
        const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, s_abort, args.ctrl, args.timeout_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kAccCols);
        for (int kb = w.k_lo; kb < w.k_hi; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, s_abort, args.ctrl, args.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t acc_k0 = kb != w.k_lo ? 1u : 0u;  // first K step: overwrite
          tc_fence_after();
          const uint64_t adesc0 = sw128_desc(a_addr(stage));
          const uint64_t bdesc = sw128_desc(b_addr(stage));
#pragma unroll
          for (int kk = 0; kk < SW_BK / SW_UK; ++kk) {
            if constexpr (PAIR)
              umma_bf16_pair(d_tmem, adesc0 + 2u * kk, bdesc + 2u * kk, idesc, acc_k0 | (kk != 0));
            else
              umma_bf16(d_tmem, adesc0 + 2u * kk, bdesc + 2u * kk, idesc, acc_k0 | (kk != 0));
          }
          if constexpr (PAIR)
            umma_commit_pair(empty_bar(stage), 0x3);
          else
            umma_commit(empty_bar(stage));
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) {
          if constexpr (PAIR)
            umma_commit_pair(tfull_bar(acc), 0x3);
          else
            umma_commit(tfull_bar(acc));
        }
      }
      if constexpr (PAIR)
        umma_commit_pair(drain_bar, 0x1);
      else
        umma_commit(drain_bar);
      wait_drain(drain_bar, 0, 100000000ull);
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    const int q = warp & 3;             // TMEM lane quarter this warp may read
    const int half = (warp - 2) >> 2;   // which of the quarter's warps: chunk parity
    constexpr int kPer = C::kEpiWarps / 4;  // warps per lane quarter
    int local = 0;
    WorkIter it(sk, total, num_kb, first, step, total2, num_kb2, sk2);
    Work w;
    const int G = (int)gridDim.x;
    for (; it.next(w); ++local) {
      const bool p1 = FUSE && w.ph == 1;  // a w2 tile of a fused launch
      const Tile d = decode_tile(w.t, p1 ? args.f_tiles2 : args.f_tiles, s_tstart, s_offs, E, NT);
      const int acc = local & 1;
      const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
      if (!wait_bounded(tfull_bar(acc), acc_phase, s_abort, args.ctrl, args.timeout_ns)) break;
      tc_fence_after();
      EpiTile et;
      et.taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols);
      et.m0 = d.m0;
      et.rows = d.m_end - d.m0;
      et.frow = d.nt * kTileRows + (int)rank * SW_M + q * 32 + lane;
      et.lane = lane;
      et.dst_base = -1;
      et.dst_mine = 0;
      et.g_mine = 0.f;
      if constexpr (NT == SW_NGRAN) {
        if (p1 ? sk2 : sk) {
          const int kbt = p1 ? num_kb2 : num_kb;  // K steps of this contraction's tiles
          const int64_t U = (int64_t)(p1 ? total2 : total) * kbt;
          const int64_t u0 = (int64_t)w.t * kbt;
          const int c_first = sk_cta(u0, U, G), c_last = sk_cta(u0 + kbt - 1, U, G);
          if (c_last > c_first) {
            const int pieces = sk_pieces(c_first, c_last, U, G);
            if (p1)
              sk_piece<SW_SCATTER, NT>(et, args, 1, u0, c_first, c_last, pieces, w.k_lo, U, G,
                                       q, d.e, tempty_bar(acc));
            else
              sk_piece<EPI, NT>(et, args, 0, u0, c_first, c_last, pieces, w.k_lo, U, G, q, d.e,
                                tempty_bar(acc));
            continue;  // the piece released its accumulator buffer
          }
        }
      }
      if (p1)
        epi_tile<SW_SCATTER, NT, kPer>(et, half, args);
      else
        epi_tile<EPI, NT, kPer>(et, half, args);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && !leader)
          mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
        else
          mbar_arrive(tempty_bar(acc));
      }
      if (args.ready_out && !p1) publish_ready(args, d.e, lane);
    }
  }

  tc_fence_before();
  if constexpr (PAIR) {
    cluster_sync();  // the leader's MMAs into the peer's TMEM are complete
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(C::kTmemCols)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(C::kTmemCols)
                   : "memory");
  }
}

// tw2 / th: the w2 weights and h rows of a fused launch (FUSE), else unused.
template <int EPI, bool PACKED, int NT, bool PAIR = false, bool FUSE = false>
cudaError_t launch_swap(const CUtensorMap &tw, const CUtensorMap &tx, const CUtensorMap &tw2,
                        const CUtensorMap &th, const SwArgs &a, cudaStream_t s) {
  using C = SwCfg<NT, PAIR>;
  auto kern = grouped_gemm_swap_kernel<EPI, PACKED, NT, PAIR, FUSE>;
  static PerDeviceOnce attr_set;
  {
    cudaError_t err = attr_set.run([kern] {
      cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
      return e != cudaSuccess ? e : uniform_carveout(kern);
    });
    if (err != cudaSuccess) return err;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(PAIR ? device_sm_count() & ~1 : device_sm_count());
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;  // PAIR: two CTAs per cluster
  attr[1].val.clusterDim.x = PAIR ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  if constexpr (FUSE) {
    // CTAs of a fused launch wait for h rows that other CTAs compute: the
    // grid is only as large as can be resident at once (queried once per
    // device; the kernel takes any grid size)
    static std::atomic<int> resident[PerDeviceOnce::kMaxDevices] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const bool slot = dev >= 0 && dev < PerDeviceOnce::kMaxDevices;
    int fit = slot ? resident[dev].load(std::memory_order_relaxed) : 0;
    if (fit <= 0) {
      int n = 0;
      cudaError_t e;
      if constexpr (PAIR) {
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        n *= 2;
      } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::kThreads, C::kSmemBytes);
        n *= device_sm_count();
      }
      if (e != cudaSuccess) return e;
      if (n < (PAIR ? 2 : 1)) return cudaErrorInvalidConfiguration;
      fit = n;
      if (slot) resident[dev].store(fit, std::memory_order_relaxed);
    }
    if ((int)cfg.gridDim.x > fit) cfg.gridDim.x = (unsigned)(PAIR ? fit & ~1 : fit);
  }
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kern, tw, tx, tw2, th, a);
  return err != cudaSuccess ? err : cudaGetLastError();
}

// CTA pairs (M = 256 per MMA) for 256-row token tiles: each SM then reads
// 32 KB per K step instead of 48 KB, so the same shared memory keeps 7 K
// steps in flight instead of 4.
constexpr bool use_pair(int nt) { return nt == 256; }

// The w13 contraction at token-tile width NT. A packed gated w13 goes
// through the interleaving 4-D map: the kernel sees the interleaved layout.
// With `gather` the token rows come from the unsorted x (one-row boxes).
template <int NT>
cudaError_t swap_ffn1(const uint16_t *x_sorted, const uint16_t *w13, int64_t N, int E, int H,
                      int I, const ActParams &act, SwArgs a, cudaStream_t s,
                      const GatherSrc *gather) {
  const bool relu2_act = act.act == MOE_ACT_RELU2;
  const bool packed = !relu2_act && act.layout == MOE_W13_PACKED;
  constexpr bool PAIR = use_pair(NT);
  constexpr int tile_rows = PAIR ? 2 * SW_M : SW_M;
  CUtensorMap tw, tx;
  const bool w_ok =
      packed ? map_w13_packed_interleaved(&tw, w13, (uint64_t)E, (uint64_t)I, (uint64_t)H, SW_M / 2)
             : map_3d(&tw, w13, (uint64_t)E, (uint64_t)w13_rows(act, I), (uint64_t)H, SW_M);
  const bool x_ok = gather ? map_2d_rows(&tx, gather->x, (uint64_t)gather->n, (uint64_t)H)
                           : map_2d(&tx, x_sorted, (uint64_t)N, (uint64_t)H, PAIR ? NT / 2 : NT);
  if (!w_ok || !x_ok) return cudaErrorInvalidValue;
  if (gather) {
    a.gather_rows = a.col_sorted;
    a.gather_k = gather->k;
  }
  a.num_kb = H / SW_BK;
  a.f_tiles = (w13_rows(act, I) + tile_rows - 1) / tile_rows;
  return relu2_act ? launch_swap<SW_RELU2, false, NT, PAIR>(tw, tx, tw, tx, a, s)
         : packed  ? launch_swap<SW_ACT, true, NT, PAIR>(tw, tx, tw, tx, a, s)
                   : launch_swap<SW_ACT, false, NT, PAIR>(tw, tx, tw, tx, a, s);
}

// The w2 contraction (gate scale + scatter) at token-tile width NT.
template <int NT>
cudaError_t swap_ffn2(const uint16_t *h_buf, const uint16_t *w2, int64_t N, int E, int H, int I,
                      SwArgs a, cudaStream_t s) {
  constexpr bool PAIR = use_pair(NT);
  const int tile_rows = PAIR ? 2 * SW_M : SW_M;
  CUtensorMap tw, tx;
  if (!map_3d(&tw, w2, (uint64_t)E, (uint64_t)H, (uint64_t)I, SW_M) ||
      !map_2d(&tx, h_buf, (uint64_t)N, (uint64_t)I, PAIR ? NT / 2 : NT))
    return cudaErrorInvalidValue;
  a.num_kb = I / SW_BK;
  a.f_tiles = (H + tile_rows - 1) / tile_rows;
  return launch_swap<SW_SCATTER, false, NT, PAIR>(tw, tx, tw, tx, a, s);
}

// Both contractions of the decode tiling (32-row token tiles, one CTA per
// SM) in one launch: the w13 work (stream-K when short), then whole w2
// tiles, each waiting for its expert's h rows. It saves the second launch,
// its set-up, and the gap between a w13 CTA leaving an SM and a w2 CTA
// arriving there.
template <int NT>
cudaError_t swap_ffn_fused(const uint16_t *x_sorted, const uint16_t *w13, const uint16_t *h_buf,
                           const uint16_t *w2, int64_t N, int E, int H, int I,
                           const ActParams &act, SwArgs a, cudaStream_t s,
                           const GatherSrc *gather) {
  constexpr bool PAIR = use_pair(NT);
  constexpr int tile_rows = PAIR ? 2 * SW_M : SW_M;
  const bool relu2_act = act.act == MOE_ACT_RELU2;
  const bool packed = !relu2_act && act.layout == MOE_W13_PACKED;
  CUtensorMap tw, tx, tw2, th;
  const bool w_ok =
      packed ? map_w13_packed_interleaved(&tw, w13, (uint64_t)E, (uint64_t)I, (uint64_t)H, SW_M / 2)
             : map_3d(&tw, w13, (uint64_t)E, (uint64_t)w13_rows(act, I), (uint64_t)H, SW_M);
  const bool x_ok = gather ? map_2d_rows(&tx, gather->x, (uint64_t)gather->n, (uint64_t)H)
                           : map_2d(&tx, x_sorted, (uint64_t)N, (uint64_t)H, PAIR ? NT / 2 : NT);
  if (!w_ok || !x_ok || !map_3d(&tw2, w2, (uint64_t)E, (uint64_t)H, (uint64_t)I, SW_M) ||
      !map_2d(&th, h_buf, (uint64_t)N, (uint64_t)I, PAIR ? NT / 2 : NT))
    return cudaErrorInvalidValue;
  if (gather) {
    a.gather_rows = a.col_sorted;
    a.gather_k = gather->k;
  }
  a.num_kb = H / SW_BK;
  a.f_tiles = (w13_rows(act, I) + tile_rows - 1) / tile_rows;
  a.num_kb2 = I / SW_BK;
  a.f_tiles2 = (H + tile_rows - 1) / tile_rows;
  // arrivals per token tile: every epilogue warp of every w13 weight tile
  // (a pair tile counts both CTAs' warps)
  a.ready_nt = NT;
  a.ready_per_tile = a.f_tiles * (PAIR ? 2 : 1) * sw_epi_warps(NT);
  return relu2_act ? launch_swap<SW_RELU2, false, NT, PAIR, true>(tw, tx, tw2, th, a, s)
         : packed  ? launch_swap<SW_ACT, true, NT, PAIR, true>(tw, tx, tw2, th, a, s)
                   : launch_swap<SW_ACT, false, NT, PAIR, true>(tw, tx, tw2, th, a, s);
}

// Token-tile width of a contraction with f_tiles weight tiles per expert and
// num_kb K steps: the NT that minimises waves * (per-tile cost + num_kb *
// cost of one K step). A K step reads a 16 KB weight tile and NT token rows
// (128 B each; half of them per CTA of a pair) from shared memory at ~128 B
// per cycle, and issues MMAs worth ~1.45 cycles per token column: narrow
// tiles are bound by the shared-memory reads. A tile also costs a fixed
// ~1450 of these units (start-up and hand-over between tiles, measured at
// K = 512: 8 K steps took the time of ~12), so short contractions favour
// fewer, wider tiles. Tiles are estimated as (ceil(N / NT) + min(E, N)) *
// f_tiles (each expert's ragged last tile).
int pick_token_tile(int64_t N, int E, int f_tiles, int num_kb) {
  constexpr double kTileCost = 1450.0;
  const int64_t sms = device_sm_count();
  int best = 32;
  double best_t = 1e300;
  for (int nt = 256; nt >= 32; nt /= 2) {
    const int64_t tiles = ((N + nt - 1) / nt + (N < E ? N : E)) * (int64_t)f_tiles;
    const double smem = 128.0 + (use_pair(nt) ? nt / 2 : nt), mma = 1.45 * nt;
    const double t = (double)((tiles + sms - 1) / sms) *
                     (kTileCost + (double)num_kb * (smem > mma ? smem : mma));
    if (t < best_t) {
      best_t = t;
      best = nt;
    }
  }
  return best;
}

}  // namespace

// Both contractions in one launch where both run on CTA pairs (256-row token
// tiles): same-box A/B, GPT-OSS prefill n = 8192 1.17 -> 1.14 ms, the skewed
// 128-expert n = 16384 layer 2.182 -> 2.145 ms. Where w2 would pick narrower
// tiles (MiniMind: 128 rows on single CTAs), forcing pairs on it lost 1.3 us.
constexpr bool kFusePairs = true;

SwapPlan plan_ffn_swap(int64_t N, int E, int H, int I, const ActParams &act) {
  SwapPlan p{};
  p.f_tiles1 = (w13_rows(act, I) + SW_M - 1) / SW_M;
  // a handful of rows per expert (decode): 32-row token tiles for both, the
  // w13 (tile, K step) units split evenly over the grid when short
  p.nt1 = p.nt2 = SW_NGRAN;
  p.decode = N <= (int64_t)kDecodeRowsPerExpert * E;
  if (!p.decode) {
    p.nt1 = pick_token_tile(N, E, p.f_tiles1, H / SW_BK);
    p.nt2 = pick_token_tile(N, E, (H + SW_M - 1) / SW_M, I / SW_BK);
  }
  p.pair1 = use_pair(p.nt1);
  p.pair2 = use_pair(p.nt2);
  // both contractions in one launch (it needs every CTA of the grid
  // resident at once): the decode tiling, and 256-row tiles on CTA pairs for
  // both
  p.fused = p.decode || (kFusePairs && p.pair1 && p.pair2);
  return p;
}

cudaError_t launch_ffn_swap(const uint16_t *x_sorted, const int32_t *offs,
                            const int32_t *col_sorted, const uint16_t *gate_scal,
                            const uint16_t *w13, const uint16_t *w2, int64_t N, int E, int H,
                            int I, const ActParams &act, uint16_t *h_buf, uint16_t *y_flat,
                            const FfnScratch &scr, cudaStream_t s, cudaEvent_t *ev_ffn,
                            const GatherSrc *gather) {
  if (N == 0) return cudaSuccess;
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
  a.ctrl = scr.ctrl;
  a.timeout_ns = kWaitTimeoutNs;
  const SwapPlan plan = plan_ffn_swap(N, E, H, I, act);
  const int f_tiles1 = plan.f_tiles1, nt1 = plan.nt1, nt2 = plan.nt2;
  a.stream_k = plan.decode && scr.sync && scr.sk_part && device_sm_count() <= kSkMaxCtas;
  if (ev_ffn && record_stage_event(ev_ffn[0], s) != cudaSuccess) return cudaErrorUnknown;
  // the w13 kernel publishes per-expert completion; the w2 kernel waits on it
  uint32_t *ready = scr.sync ? scr.sync + kSyncReady : nullptr;
  a.ready_out = ready;
  if (a.stream_k) {
    a.sk_cnt = scr.sync + kSyncSk;
    a.sk_part = scr.sk_part;
  }
  if (plan.fused) {
    // one launch; the w2 weights are fetched into L2 while a tile waits
    a.ready_in = ready;
    a.w = w2;
    a.w_rows = H;
    const cudaError_t err =
        plan.decode ? swap_ffn_fused<SW_NGRAN>(x_sorted, w13, h_buf, w2, N, E, H, I, act, a, s,
                                              gather)
                    : swap_ffn_fused<256>(x_sorted, w13, h_buf, w2, N, E, H, I, act, a, s,
                                          gather);
    if (err != cudaSuccess) return err;
    return ev_ffn ? record_stage_event(ev_ffn[1], s) : cudaSuccess;
  }
  cudaError_t err;
  switch (nt1) {
    case 32: err = swap_ffn1<32>(x_sorted, w13, N, E, H, I, act, a, s, gather); break;
    case 64: err = swap_ffn1<64>(x_sorted, w13, N, E, H, I, act, a, s, gather); break;
    case 128: err = swap_ffn1<128>(x_sorted, w13, N, E, H, I, act, a, s, gather); break;
    default: err = swap_ffn1<256>(x_sorted, w13, N, E, H, I, act, a, s, gather); break;
  }
  if (err != cudaSuccess) return err;
  if (ev_ffn && record_stage_event(ev_ffn[1], s) != cudaSuccess) return cudaErrorUnknown;
  a.ready_out = nullptr;
  a.ready_in = ready;
  a.ready_nt = nt1;
  // arrivals per token tile: every epilogue warp of every weight tile (a
  // CTA pair's tile covers 256 weight rows with both CTAs' warps)
  a.ready_per_tile = (plan.pair1 ? (f_tiles1 + 1) / 2 * 2 : f_tiles1) * sw_epi_warps(nt1);
  a.w = w2;
  a.w_rows = H;
  a.stream_k = 0;  // whole w2 tiles: they start as soon as w13 CTAs leave SMs free
  switch (nt2) {
    case 32: return swap_ffn2<32>(h_buf, w2, N, E, H, I, a, s);
    case 64: return swap_ffn2<64>(h_buf, w2, N, E, H, I, a, s);
    case 128: return swap_ffn2<128>(h_buf, w2, N, E, H, I, a, s);
    default: return swap_ffn2<256>(h_buf, w2, N, E, H, I, a, s);
  }
}

}  // namespace moe
