// Backward of combine and of the SwiGLU experts (ruDNN user guide, section 12:
// combine_backward returns dexpert and FP32 dweights; the forward cache's
// backward returns the dispatched rows' input gradient and FP32 gradients of
// gate, up and down).
//
// Per dispatched row r of expert e, with g = W_gate[e] x_r, u = W_up[e] x_r,
// h = SiLU(g) * u, y = W_down[e] h and dy the row's gradient:
//   dh = W_down[e]^T dy                       (dgrad GEMM, K = H)
//   dg = dh * u * SiLU'(g), du = dh * SiLU(g) (elementwise, FP32)
//   dx = W_gate[e]^T dg + W_up[e]^T du        (dgrad GEMM, K = I, two terms)
//   ddown[e] += dy h^T, dgate[e] += dg x^T, dup[e] += du x^T  (wgrad GEMMs,
//   K = the expert's rows)
// SiLU'(g) = s (1 + g (1 - s)) with s the logistic function of g.
// Here the GEMMs accumulate in FP32 on CUDA cores (64 x 64 output tiles, 4 x 4
// per thread): the F32 experts' path (no TF32, as in the forward); F16/BF16
// run them on the tensor cores (experts_bwd_tc.cu, with the SiLU backward in
// the dgrad epilogue). dh stays FP32, dg and du are rounded to the dtype like
// the forward's activations, the weight gradients are FP32.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int TB_M = 64, TB_N = 64, TB_K = 16, TB_THREADS = 256;

// ------------------------------------------------------------------ combine backward
// dexpert[r] = w[s] * dout[s / k] and dweights[s] = <dout[s / k], y[r]> (FP32:
// each lane's columns in order, then a butterfly over the warp) for every
// dispatched row r, s = row_src[r]. One warp per row, so y is read and
// dexpert written as sequential row streams (in slot order both would be
// scattered 4 KB rows: measured 1.4x slower). A row is real when
// inv[row_src[r]] == r (row_src past the dispatched rows is not consulted
// otherwise); warp r also gives slot r a NaN dweight when inv[r] is out of
// range (such a slot has no row). Lane l owns the NV-element vectors at
// columns (l + 32 i) * NV (16-byte vectors when rows are 16-byte multiples).
template <typename T, int NV>
struct VecIO {
  static __device__ __forceinline__ void load(const T* p, float (&v)[NV]) {
    if constexpr (NV * sizeof(T) == 16) {
      const uint4 raw = *reinterpret_cast<const uint4*>(p);
      const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = to_f32(e[i]);
    } else {
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = to_f32(p[i]);
    }
  }
  static __device__ __forceinline__ void store(T* p, const float (&v)[NV]) {
    if constexpr (NV * sizeof(T) == 16) {
      uint4 raw;
      T* e = reinterpret_cast<T*>(&raw);
#pragma unroll
      for (int i = 0; i < NV; ++i) e[i] = from_f32<T>(v[i]);
      *reinterpret_cast<uint4*>(p) = raw;
    } else {
#pragma unroll
      for (int i = 0; i < NV; ++i) p[i] = from_f32<T>(v[i]);
    }
  }
};

template <typename T, typename TW, int NV>
__global__ void __launch_bounds__(256) combine_backward_kernel(
    const T* __restrict__ y, const uint32_t* __restrict__ inv, const uint32_t* __restrict__ row_src,
    const TW* __restrict__ w, const T* __restrict__ dout, int k, int64_t H, uint32_t nslots,
    T* __restrict__ dexpert, float* __restrict__ dweights) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const float qnan = __int_as_float(0x7FC00000);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < nslots;
       r += warps) {
    if (lane == 0 && inv[r] >= nslots) dweights[r] = qnan;  // slot r has no row
    const uint32_t s = row_src[r];
    if (s >= nslots || inv[s] != static_cast<uint32_t>(r)) continue;
    const int64_t t = s / static_cast<uint32_t>(k);
    const float wq = to_f32(w[s]);
    float part = 0.0f;
    for (int64_t c = static_cast<int64_t>(lane) * NV; c < H; c += 32 * NV) {
      float go[NV], yv[NV], dv[NV];
      VecIO<T, NV>::load(dout + t * H + c, go);
      VecIO<T, NV>::load(y + r * H + c, yv);
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        part = fmaf(go[i], yv[i], part);
        dv[i] = wq * go[i];
      }
      VecIO<T, NV>::store(dexpert + r * H + c, dv);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(FULL_MASK, part, off);
    if (lane == 0) dweights[s] = part;
  }
}

// ------------------------------------------------------------------ SiLU backward
// dg = dh * u * SiLU'(g), du = dh * SiLU(g), rounded to the dtype.
template <typename T>
__global__ void silu_backward_kernel(const float* __restrict__ dh, const T* __restrict__ g,
                                     const T* __restrict__ u, int64_t n, T* __restrict__ dg, T* __restrict__ du) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float dgv, duv;
    silu_mul_backward(dh[i], to_f32(g[i]), to_f32(u[i]), &dgv, &duv);
    dg[i] = from_f32<T>(dgv);
    du[i] = from_f32<T>(duv);
  }
}

// ------------------------------------------------------------------ dgrad GEMM
// out[r, n] = sum_k A1[r, k] W1[e][k][n] (+ sum_k A2[r, k] W2[e][k][n]) for the
// rows r of expert e (rows from the offsets); W is [E, K, N] row-major.
template <typename TA, typename TO, bool DUAL>
__global__ void __launch_bounds__(TB_THREADS) dgrad_kernel(
    const TA* __restrict__ a1, const TA* __restrict__ w1, const TA* __restrict__ a2, const TA* __restrict__ w2,
    const uint32_t* __restrict__ offsets, int E, int64_t K, int64_t N, int64_t rows_total, TO* __restrict__ out) {
  __shared__ uint32_t tile_start[ROUTE_MAX_E + 1];
  __shared__ float As[TB_K][TB_M + 4];
  __shared__ float Ws[TB_K][TB_N + 4];
  const int n_tiles = static_cast<int>((N + TB_N - 1) / TB_N);
  if (threadIdx.x < 32) build_tile_prefix(offsets, E, TB_M, n_tiles, tile_start);
  __syncthreads();
  const uint32_t tile = blockIdx.x;
  if (tile >= tile_start[E]) return;
  TileCoord tc = decode_tile(tile, tile_start, E, offsets, TB_M, n_tiles);
  if (static_cast<int64_t>(tc.row0) >= rows_total) return;
  if (static_cast<int64_t>(tc.row0) + tc.rows > rows_total) tc.rows = static_cast<int>(rows_total - tc.row0);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t n0 = static_cast<int64_t>(tc.n) * TB_N;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  const int lr = threadIdx.x / 4, lk = (threadIdx.x % 4) * 4;   // A tile loads: row lr, k lk..lk+3
  const int wk = threadIdx.x / 16, wn = (threadIdx.x % 16) * 4; // W tile loads: k wk, n wn..wn+3
  for (int pass = 0; pass < (DUAL ? 2 : 1); ++pass) {
    const TA* a = pass == 0 ? a1 : a2;
    const TA* wt = (pass == 0 ? w1 : w2) + static_cast<int64_t>(tc.e) * K * N;
    for (int64_t k0 = 0; k0 < K; k0 += TB_K) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t kk = k0 + lk + q;
        As[lk + q][lr] = (kk < K && lr < tc.rows) ? to_f32(a[(static_cast<int64_t>(tc.row0) + lr) * K + kk]) : 0.0f;
        const int64_t kw = k0 + wk;
        const int64_t n = n0 + wn + q;
        Ws[wk][wn + q] = (kw < K && n < N) ? to_f32(wt[kw * N + n]) : 0.0f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < TB_K; ++kk) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = Ws[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= tc.rows) continue;
    TO* dst = out + (static_cast<int64_t>(tc.row0) + r) * N;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n < N) dst[n] = from_f32<TO>(acc[i][j]);
    }
  }
}

// ------------------------------------------------------------------ wgrad GEMM
// out1[e][m][n] = sum_{r in expert e} A1[r, m] B[r, n] (and out2 with A2):
// grid = E x (M/64) x (N/64) tiles; an expert without rows writes zeros.
template <typename TA, bool DUAL>
__global__ void __launch_bounds__(TB_THREADS) wgrad_kernel(
    const TA* __restrict__ a1, const TA* __restrict__ a2, const TA* __restrict__ b,
    const uint32_t* __restrict__ offsets, int64_t M, int64_t N, int64_t rows_total, float* __restrict__ out1,
    float* __restrict__ out2) {
  __shared__ float A1s[TB_K][TB_M + 4];
  __shared__ float A2s[DUAL ? TB_K : 1][TB_M + 4];
  __shared__ float Bs[TB_K][TB_N + 4];
  const int m_tiles = static_cast<int>((M + TB_M - 1) / TB_M);
  const int n_tiles = static_cast<int>((N + TB_N - 1) / TB_N);
  const int e = blockIdx.x / (m_tiles * n_tiles);
  const int rem = blockIdx.x % (m_tiles * n_tiles);
  const int64_t m0 = static_cast<int64_t>(rem / n_tiles) * TB_M;
  const int64_t n0 = static_cast<int64_t>(rem % n_tiles) * TB_N;
  int64_t r_lo = offsets[e], r_hi = offsets[e + 1];
  if (r_hi > rows_total) r_hi = rows_total;
  if (r_lo > r_hi) r_lo = r_hi;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc1[4][4], acc2[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { acc1[i][j] = 0.0f; acc2[i][j] = 0.0f; }
  const int lk = threadIdx.x / 16, lc = (threadIdx.x % 16) * 4;  // loads: row lk of the chunk, cols lc..lc+3
  for (int64_t r0 = r_lo; r0 < r_hi; r0 += TB_K) {
    const int64_t r = r0 + lk;
    const bool rin = r < r_hi;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t m = m0 + lc + q, n = n0 + lc + q;
      A1s[lk][lc + q] = (rin && m < M) ? to_f32(a1[r * M + m]) : 0.0f;
      if constexpr (DUAL) A2s[lk][lc + q] = (rin && m < M) ? to_f32(a2[r * M + m]) : 0.0f;
      Bs[lk][lc + q] = (rin && n < N) ? to_f32(b[r * N + n]) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TB_K; ++kk) {
      float av[4], a2v[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = A1s[kk][ty * 4 + i];
        if constexpr (DUAL) a2v[i] = A2s[kk][ty * 4 + i];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc1[i][j] = fmaf(av[i], bv[j], acc1[i][j]);
          if constexpr (DUAL) acc2[i][j] = fmaf(a2v[i], bv[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n >= N) continue;
      const int64_t o = (static_cast<int64_t>(e) * M + m) * N + n;
      out1[o] = acc1[i][j];
      if constexpr (DUAL) out2[o] = acc2[i][j];
    }
  }
}

int64_t tile_bound(int64_t rows, int E, int bm, int64_t n_tiles) {
  const int64_t m_tiles = rows / bm + (rows < E ? rows : E);
  return m_tiles * n_tiles;
}

template <typename T>
cudaError_t backward_t(const TrainBuffers& b, const uint32_t* offsets, int E, int64_t rows, int64_t H, int64_t I,
                       cudaStream_t s) {
  const T* dy = static_cast<const T*>(b.dy);
  // dh = dy W_down (W_down [E, H, I]: K = H, N = I), FP32
  {
    const int64_t g = tile_bound(rows, E, TB_M, (I + TB_N - 1) / TB_N);
    dgrad_kernel<T, float, false><<<static_cast<unsigned>(g), TB_THREADS, 0, s>>>(
        dy, static_cast<const T*>(b.down), nullptr, nullptr, offsets, E, H, I, rows, b.dh);
  }
  // dg, du
  {
    const int64_t n = rows * I;
    const int blocks = static_cast<int>(n / 256 + 1 < 152 * 16 ? n / 256 + 1 : 152 * 16);
    silu_backward_kernel<T><<<blocks, 256, 0, s>>>(b.dh, static_cast<const T*>(b.g), static_cast<const T*>(b.u), n,
                                                   static_cast<T*>(b.dg), static_cast<T*>(b.du));
  }
  // dx = dg W_gate + du W_up (W [E, I, H]: K = I, N = H)
  {
    const int64_t g = tile_bound(rows, E, TB_M, (H + TB_N - 1) / TB_N);
    dgrad_kernel<T, T, true><<<static_cast<unsigned>(g), TB_THREADS, 0, s>>>(
        static_cast<const T*>(b.dg), static_cast<const T*>(b.gate), static_cast<const T*>(b.du),
        static_cast<const T*>(b.up), offsets, E, I, H, rows, static_cast<T*>(b.dx));
  }
  // ddown[e] = dy^T h ([H, I]); dgate[e], dup[e] = dg^T x, du^T x ([I, H])
  {
    const int64_t tiles = ((H + TB_M - 1) / TB_M) * ((I + TB_N - 1) / TB_N) * E;
    wgrad_kernel<T, false><<<static_cast<unsigned>(tiles), TB_THREADS, 0, s>>>(
        dy, nullptr, static_cast<const T*>(b.h), offsets, H, I, rows, b.ddown, nullptr);
    const int64_t tiles2 = ((I + TB_M - 1) / TB_M) * ((H + TB_N - 1) / TB_N) * E;
    wgrad_kernel<T, true><<<static_cast<unsigned>(tiles2), TB_THREADS, 0, s>>>(
        static_cast<const T*>(b.dg), static_cast<const T*>(b.du), static_cast<const T*>(b.x), offsets, I, H, rows,
        b.dgate, b.dup);
  }
  return cudaGetLastError();
}

template <typename T, typename TW>
cudaError_t combine_backward_t(const void* y, const uint32_t* inv, const uint32_t* row_src, const void* w,
                               const void* dout, int64_t T_tokens, int k, int64_t H, void* dexpert, float* dweights,
                               cudaStream_t s) {
  const uint32_t nslots = static_cast<uint32_t>(T_tokens * k);
  const int64_t want = (static_cast<int64_t>(nslots) + 7) / 8;  // eight rows (warps) per block
  const int blocks = static_cast<int>(want < 65536 ? want : 65536);
  constexpr int NV = 16 / static_cast<int>(sizeof(T));
  const bool vec = (H * static_cast<int64_t>(sizeof(T))) % 16 == 0 && reinterpret_cast<uintptr_t>(y) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(dout) % 16 == 0 && reinterpret_cast<uintptr_t>(dexpert) % 16 == 0;
  const auto* yp = static_cast<const T*>(y);
  const auto* wp = static_cast<const TW*>(w);
  const auto* dp = static_cast<const T*>(dout);
  auto* ep = static_cast<T*>(dexpert);
  if (vec)
    combine_backward_kernel<T, TW, NV><<<blocks, 256, 0, s>>>(yp, inv, row_src, wp, dp, k, H, nslots, ep, dweights);
  else
    combine_backward_kernel<T, TW, 1><<<blocks, 256, 0, s>>>(yp, inv, row_src, wp, dp, k, H, nslots, ep, dweights);
  return cudaGetLastError();
}

template <typename T>
cudaError_t combine_backward_w(const void* y, const uint32_t* inv, const uint32_t* row_src, const void* w,
                               moe_dtype wdt, const void* dout, int64_t T_tokens, int k, int64_t H, void* dexpert,
                               float* dweights, cudaStream_t s) {
  switch (wdt) {
    case MOE_F32:
      return combine_backward_t<T, float>(y, inv, row_src, w, dout, T_tokens, k, H, dexpert, dweights, s);
    case MOE_F16:
      return combine_backward_t<T, __half>(y, inv, row_src, w, dout, T_tokens, k, H, dexpert, dweights, s);
    default:
      return combine_backward_t<T, __nv_bfloat16>(y, inv, row_src, w, dout, T_tokens, k, H, dexpert, dweights, s);
  }
}

}  // namespace

cudaError_t launch_combine_backward(const void* y_dispatched, moe_dtype dtype, const uint32_t* inv,
                                    const uint32_t* row_src, const void* weights, moe_dtype weights_dtype,
                                    const void* grad_out, int64_t T, int top_k, int64_t H, void* dexpert,
                                    float* dweights, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  switch (dtype) {
    case MOE_F32:
      return combine_backward_w<float>(y_dispatched, inv, row_src, weights, weights_dtype, grad_out, T, top_k, H,
                                       dexpert, dweights, stream);
    case MOE_F16:
      return combine_backward_w<__half>(y_dispatched, inv, row_src, weights, weights_dtype, grad_out, T, top_k, H,
                                        dexpert, dweights, stream);
    default:
      return combine_backward_w<__nv_bfloat16>(y_dispatched, inv, row_src, weights, weights_dtype, grad_out, T,
                                               top_k, H, dexpert, dweights, stream);
  }
}


cudaError_t launch_experts_backward(moe_dtype dtype, const TrainBuffers& b, const uint32_t* offsets, int E,
                                    int64_t rows, int64_t H, int64_t I, cudaStream_t stream) {
  if (rows == 0) {
    // No rows: every weight gradient is zero.
    cudaError_t err = cudaMemsetAsync(b.dgate, 0, sizeof(float) * E * I * H, stream);
    if (err == cudaSuccess) err = cudaMemsetAsync(b.dup, 0, sizeof(float) * E * I * H, stream);
    if (err == cudaSuccess) err = cudaMemsetAsync(b.ddown, 0, sizeof(float) * E * H * I, stream);
    return err;
  }
  switch (dtype) {
    case MOE_F32: return backward_t<float>(b, offsets, E, rows, H, I, stream);
    case MOE_F16: return backward_t<__half>(b, offsets, E, rows, H, I, stream);
    default: return backward_t<__nv_bfloat16>(b, offsets, E, rows, H, I, stream);
  }
}

}  // namespace moe
