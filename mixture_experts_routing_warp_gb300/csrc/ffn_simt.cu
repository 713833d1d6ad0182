// ffn_simt.cu -- grouped expert FFN on CUDA cores (fp32 FMA).
//
// The per-expert FFN of the MiniMind issue ("It is removable in plain
// PyTorch": each expert runs on its contiguous slice of the sorted rows) with
// the activations and w13 layouts of "CuteDSL NVFP4 MoE adds SwiGLU-OAI and
// ReLU2" (关键源码片段). Ragged per-expert batches are scheduled on the
// device from offs: m-tile index -> (expert, first row), no host readback.
#include "moe_internal.cuh"

namespace moe {

constexpr int SB_M = 64, SB_N = 64, SB_K = 32, SB_THREADS = 256;

// Map this CTA's m-tile index to (expert, row range) from offs (device).
__device__ __forceinline__ bool find_mtile(const int32_t *offs, int E, int mt, int tile_m,
                                           int &e_out, int &row0, int &row1) {
  __shared__ int s_e, s_r0, s_r1;
  if (threadIdx.x == 0) {
    int acc = 0, found = -1, r0 = 0, r1 = 0;
    for (int e = 0; e < E; ++e) {
      const int lo = offs[e], hi = offs[e + 1];
      const int tiles = (hi - lo + tile_m - 1) / tile_m;
      if (mt < acc + tiles) {
        found = e;
        r0 = lo + (mt - acc) * tile_m;
        r1 = min(hi, r0 + tile_m);
        break;
      }
      acc += tiles;
    }
    s_e = found;
    s_r0 = r0;
    s_r1 = r1;
  }
  __syncthreads();
  e_out = s_e;
  row0 = s_r0;
  row1 = s_r1;
  return s_e >= 0;
}

// h[p, c] = act(gate . x_p, up . x_p) for the expert owning row p.
__global__ void __launch_bounds__(SB_THREADS) ffn1_simt_kernel(
    const uint16_t *__restrict__ xs, const int32_t *__restrict__ offs, int E, int H, int I,
    const uint16_t *__restrict__ w13, ActParams act, uint16_t *__restrict__ h_buf) {
  __shared__ float sA[SB_K][SB_M + 4];
  __shared__ float sG[SB_K][SB_N + 4];
  __shared__ float sU[SB_K][SB_N + 4];
  int e, row0, row1;
  if (!find_mtile(offs, E, blockIdx.x, SB_M, e, row0, row1)) return;
  const int rows = row1 - row0;
  const int c0 = blockIdx.y * SB_N;
  const uint16_t *W = w13 + (size_t)e * 2 * I * H;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  float accG[4][4] = {}, accU[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += SB_K) {
    for (int i = tid; i < SB_M * SB_K; i += SB_THREADS) {
      const int r = i / SB_K, kk = i % SB_K;
      sA[kk][r] = r < rows ? bf16_bits_to_float(xs[(size_t)(row0 + r) * H + k0 + kk]) : 0.f;
    }
    for (int i = tid; i < SB_N * SB_K; i += SB_THREADS) {
      const int c = i / SB_K, kk = i % SB_K, col = c0 + c;
      float g = 0.f, u = 0.f;
      if (col < I) {
        const int gr = act.layout == MOE_W13_PACKED ? col : 2 * col;
        const int ur = act.layout == MOE_W13_PACKED ? I + col : 2 * col + 1;
        g = bf16_bits_to_float(W[(size_t)gr * H + k0 + kk]);
        u = bf16_bits_to_float(W[(size_t)ur * H + k0 + kk]);
      }
      sG[kk][c] = g;
      sU[kk][c] = u;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < SB_K; ++kk) {
      float a[4], g[4], u[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[q] = sA[kk][ty * 4 + q];
        g[q] = sG[kk][tx * 4 + q];
        u[q] = sU[kk][tx * 4 + q];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          accG[i][j] = fmaf(a[i], g[j], accG[i][j]);
          accU[i][j] = fmaf(a[i], u[j], accU[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = ty * 4 + i, c = c0 + tx * 4 + j;
      if (r < rows && c < I)
        h_buf[(size_t)(row0 + r) * I + c] = float_to_bf16_bits(activate(accG[i][j], accU[i][j], act));
    }
}

// y_flat[col_sorted[p], c] = gate_scal[p] * (w2_e[c, :] . h_p)
__global__ void __launch_bounds__(SB_THREADS) ffn2_simt_kernel(
    const uint16_t *__restrict__ h_buf, const int32_t *__restrict__ offs,
    const int32_t *__restrict__ col_sorted, const uint16_t *__restrict__ gate_scal, int E, int H,
    int I, const uint16_t *__restrict__ w2, uint16_t *__restrict__ y_flat) {
  __shared__ float sA[SB_K][SB_M + 4];
  __shared__ float sB[SB_K][SB_N + 4];
  int e, row0, row1;
  if (!find_mtile(offs, E, blockIdx.x, SB_M, e, row0, row1)) return;
  const int rows = row1 - row0;
  const int c0 = blockIdx.y * SB_N;
  const uint16_t *W = w2 + (size_t)e * H * I;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < I; k0 += SB_K) {
    for (int i = tid; i < SB_M * SB_K; i += SB_THREADS) {
      const int r = i / SB_K, kk = i % SB_K;
      sA[kk][r] = r < rows ? bf16_bits_to_float(h_buf[(size_t)(row0 + r) * I + k0 + kk]) : 0.f;
    }
    for (int i = tid; i < SB_N * SB_K; i += SB_THREADS) {
      const int c = i / SB_K, kk = i % SB_K, col = c0 + c;
      sB[kk][c] = col < H ? bf16_bits_to_float(W[(size_t)col * I + k0 + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < SB_K; ++kk) {
      float a[4], bb[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[q] = sA[kk][ty * 4 + q];
        bb[q] = sB[kk][tx * 4 + q];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= rows) continue;
    const int p = row0 + r;
    const float g = bf16_bits_to_float(gate_scal[p]);
    const size_t dst = (size_t)col_sorted[p] * H;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + tx * 4 + j;
      if (c < H) y_flat[dst + c] = float_to_bf16_bits(acc[i][j] * g);
    }
  }
}

cudaError_t launch_ffn(const uint16_t *x_sorted, const int32_t *offs, const int32_t *col_sorted,
                       const uint16_t *gate_scal, const uint16_t *w13, const uint16_t *w2,
                       int64_t N, int E, int H, int I, const ActParams &act, uint16_t *h_buf,
                       uint16_t *y_flat, uint32_t *ctrl, cudaStream_t s, cudaEvent_t *ev_ffn) {
  (void)ctrl;
  if (N == 0) return cudaSuccess;
  if (ev_ffn && cudaEventRecord(ev_ffn[0], s) != cudaSuccess) return cudaErrorUnknown;
  const unsigned mtiles = (unsigned)((N + SB_M - 1) / SB_M + E);
  ffn1_simt_kernel<<<dim3(mtiles, (I + SB_N - 1) / SB_N), SB_THREADS, 0, s>>>(x_sorted, offs, E, H,
                                                                             I, w13, act, h_buf);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (ev_ffn && cudaEventRecord(ev_ffn[1], s) != cudaSuccess) return cudaErrorUnknown;
  ffn2_simt_kernel<<<dim3(mtiles, (H + SB_N - 1) / SB_N), SB_THREADS, 0, s>>>(
      h_buf, offs, col_sorted, gate_scal, E, H, I, w2, y_flat);
  return cudaGetLastError();
}

}  // namespace moe
