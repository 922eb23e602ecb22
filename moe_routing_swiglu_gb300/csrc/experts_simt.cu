// K7: FP32 SwiGLU experts on CUDA cores (FP32 FMA only, no TF32: the F32
// contract is a max-abs error of 1e-4, which TF32's 10-bit mantissa misses).
//
// Per dispatched row r of expert e ("tiny-llm deep dive 5: ops.rs", section
// on SiLU; ruDNN user guide, section 5 for the weight shapes):
//   gate/up pass:  h[r, i] = SiLU(sum_c gate[e, i, c] x[r, c]) * sum_c up[e, i, c] x[r, c]
//   down pass:     y[r, n] = sum_i down[e, n, i] h[r, i]
// Both are grouped GEMMs over the experts' row ranges; tiles are 64 rows x
// 64 columns, 256 threads, each thread a 4 x 4 block of outputs.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int SB_M = 64, SB_N = 64, SB_K = 16, SB_THREADS = 256;

// Gather mode (gate/up only, row_src != nullptr): row r of the A operand is
// a[(row_src[r] / top_k) * K ...], the token's row of x.
template <bool GATE_UP>
__global__ void __launch_bounds__(SB_THREADS) experts_simt_kernel(
    const float* __restrict__ a, const uint32_t* __restrict__ row_src, int top_k, int64_t a_rows,
    const uint32_t* __restrict__ offsets, int E, const float* __restrict__ w0, const float* __restrict__ w1,
    int64_t K, int64_t N, int64_t rows_total, float* __restrict__ out, float* __restrict__ out_g,
    float* __restrict__ out_u) {
  __shared__ uint32_t tile_start[ROUTE_MAX_E + 1];
  __shared__ float As[SB_K][SB_M + 4];
  __shared__ float B0s[SB_K][SB_N + 4];
  __shared__ float B1s[GATE_UP ? SB_K : 1][SB_N + 4];
  grid_dependency_wait();
  launch_dependents();
  const int n_tiles = static_cast<int>((N + SB_N - 1) / SB_N);
  if (threadIdx.x < 32) build_tile_prefix(offsets, E, SB_M, n_tiles, tile_start);
  __syncthreads();
  const uint32_t tile = blockIdx.x;
  if (tile >= tile_start[E]) return;
  TileCoord tc = decode_tile(tile, tile_start, E, offsets, SB_M, n_tiles);
  // Rows past rows_total (only possible with inconsistent offsets) are skipped.
  if (static_cast<int64_t>(tc.row0) >= rows_total) return;
  if (static_cast<int64_t>(tc.row0) + tc.rows > rows_total) tc.rows = static_cast<int>(rows_total - tc.row0);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t n0 = static_cast<int64_t>(tc.n) * SB_N;
  const float* wg = w0 + static_cast<int64_t>(tc.e) * N * K;
  const float* wu = GATE_UP ? w1 + static_cast<int64_t>(tc.e) * N * K : nullptr;

  float acc0[4][4], acc1[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { acc0[i][j] = 0.0f; acc1[i][j] = 0.0f; }

  const int lr = threadIdx.x / 4;        // 0..63: row of the A / B tile this thread loads
  const int lk = (threadIdx.x % 4) * 4;  // 0,4,8,12: first k of its 4 loads
  const float* a_row = nullptr;          // this thread's A row, or nullptr for zeros
  if (lr < tc.rows) {
    int64_t src = static_cast<int64_t>(tc.row0) + lr;
    if (row_src != nullptr) src = row_src[src] / static_cast<uint32_t>(top_k);
    if (src < a_rows) a_row = a + src * K;
  }
  for (int64_t k0 = 0; k0 < K; k0 += SB_K) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t kk = k0 + lk + q;
      const bool kin = kk < K;
      As[lk + q][lr] = (kin && a_row != nullptr) ? a_row[kk] : 0.0f;
      const int64_t n = n0 + lr;
      B0s[lk + q][lr] = (kin && n < N) ? wg[n * K + kk] : 0.0f;
      if constexpr (GATE_UP) B1s[lk + q][lr] = (kin && n < N) ? wu[n * K + kk] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SB_K; ++kk) {
      float av[4], b0[4], b1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b0[j] = B0s[kk][tx * 4 + j];
        if constexpr (GATE_UP) b1[j] = B1s[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc0[i][j] = fmaf(av[i], b0[j], acc0[i][j]);
          if constexpr (GATE_UP) acc1[i][j] = fmaf(av[i], b1[j], acc1[i][j]);
        }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= tc.rows) continue;
    float* dst = out + (static_cast<int64_t>(tc.row0) + r) * N;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float v = acc0[i][j];
      if constexpr (GATE_UP) {
        if (out_g != nullptr) {  // training: keep the pre-activations
          out_g[(static_cast<int64_t>(tc.row0) + r) * N + n] = v;
          out_u[(static_cast<int64_t>(tc.row0) + r) * N + n] = acc1[i][j];
        }
        v = v / (1.0f + expf(-v)) * acc1[i][j];
      }
      dst[n] = v;
    }
  }
}

int64_t tile_bound(int64_t rows, int E, int bm, int64_t n_tiles) {
  const int64_t m_tiles = rows / bm + (rows < E ? rows : E);
  return m_tiles * n_tiles;
}

}  // namespace

cudaError_t launch_experts_simt_f32(bool gate_up, const float* a, const TcGather* gather, const TcCache* cache,
                                    const uint32_t* offsets, int E, int64_t rows, const float* w0,
                                    const float* w1, int64_t H, int64_t I, float* out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if ((gather != nullptr || cache != nullptr) && !gate_up) return cudaErrorInvalidValue;
  const float* src = gather != nullptr ? static_cast<const float*>(gather->x) : a;
  const uint32_t* row_src = gather != nullptr ? gather->row_src : nullptr;
  const int top_k = gather != nullptr ? gather->top_k : 1;
  const int64_t a_rows = gather != nullptr ? gather->x_rows : rows;
  if (gate_up) {
    const int64_t g = tile_bound(rows, E, SB_M, (I + SB_N - 1) / SB_N);
    return launch_dependent(experts_simt_kernel<true>, dim3(static_cast<unsigned>(g)), dim3(SB_THREADS), 0, stream,
                            src, row_src, top_k, a_rows, offsets, E, w0, w1, H, I, rows, out,
                            cache != nullptr ? static_cast<float*>(cache->g) : nullptr,
                            cache != nullptr ? static_cast<float*>(cache->u) : nullptr);
  } else {
    const int64_t g = tile_bound(rows, E, SB_M, (H + SB_N - 1) / SB_N);
    return launch_dependent(experts_simt_kernel<false>, dim3(static_cast<unsigned>(g)), dim3(SB_THREADS), 0, stream,
                            a, static_cast<const uint32_t*>(nullptr), 1, rows, offsets, E, w0,
                            static_cast<const float*>(nullptr), I, H, rows, out, static_cast<float*>(nullptr),
                            static_cast<float*>(nullptr));
  }
  return cudaGetLastError();
}

}  // namespace moe
