// K5: weighted combine back to token order (ruDNN user guide, section 6:
// combine restores token order through the dispatch mapping and merges the
// expert outputs with the routing weights).
//
// out[t, :] = sum_{j=0..k-1} w[t, j] * y[inv[t*k + j], :], accumulated in FP32
// in slot order j = 0, 1, ..., k-1, then rounded to the output dtype. One
// block per token (grid-stride): the token's k row numbers and weights are
// staged in shared memory (the threads that stage them also ask L2 to fetch
// each whole slot row in one bulk prefetch), then each thread owns 16-byte
// vectors of the row and keeps 4 slot-row loads in flight before their
// in-order FMAs. No atomics, so the result does not depend on scheduling. A slot whose inv
// entry is INVALID_ROW (an index >= E at dispatch), or any entry >= T*k,
// makes its token's row NaN instead of reading out of range.
//
// The same kernel without weights is dispatch_backward (ruDNN user guide,
// section 12): dx[t, :] = sum_j dinput[inv[t*k + j], :], the dispatched rows'
// gradients added back onto their token in slot order, with no routing
// weight applied again.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int COMBINE_MAX_K = 1024;  // top_k <= E <= 1024

template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__half> { static constexpr int N = 8; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float (&v)[Vec<T>::N]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
  for (int i = 0; i < Vec<T>::N; ++i) v[i] = to_f32(e[i]);
}

template <typename T>
__device__ __forceinline__ void store_vec(T* p, const float (&v)[Vec<T>::N]) {
  uint4 raw;
  T* e = reinterpret_cast<T*>(&raw);
#pragma unroll
  for (int i = 0; i < Vec<T>::N; ++i) e[i] = from_f32<T>(v[i]);
  *reinterpret_cast<uint4*>(p) = raw;
}

template <typename T, typename TW, bool VEC, bool WEIGHTED>
__global__ void __launch_bounds__(256) combine_kernel(const T* __restrict__ y,
                                                      const uint32_t* __restrict__ inv,
                                                      const TW* __restrict__ w, int64_t T_tokens,
                                                      int k, int64_t H, uint32_t rows,
                                                      T* __restrict__ out) {
  constexpr int NV = VEC ? Vec<T>::N : 1;
  constexpr int G = 4;  // slot rows whose loads are in flight together
  __shared__ uint32_t s_row[COMBINE_MAX_K];
  __shared__ float s_w[COMBINE_MAX_K];
  __shared__ int s_bad;
  grid_dependency_wait();
  launch_dependents();
  const float qnan = __int_as_float(0x7FC00000);
  for (int64_t t = blockIdx.x; t < T_tokens; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
      const uint32_t r = inv[t * k + j];
      s_row[j] = r < rows ? r : 0u;           // an invalid entry reads row 0 ...
      s_w[j] = WEIGHTED ? to_f32(w[t * k + j]) : 1.0f;
      if (r >= rows) s_bad = 1;               // ... and the whole row becomes NaN
      // The whole slot row into L2 in one request, ahead of the loads below.
      else if (VEC) prefetch_l2_bulk(y + static_cast<int64_t>(r) * H, static_cast<uint32_t>(H * sizeof(T)));
    }
    __syncthreads();
    const bool bad = s_bad != 0;
    for (int64_t c = static_cast<int64_t>(threadIdx.x) * NV; c < H; c += static_cast<int64_t>(blockDim.x) * NV) {
      float acc[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) acc[i] = 0.0f;
      int j0 = 0;
      for (; j0 + G <= k; j0 += G) {
        float v[G][NV];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const T* src = y + static_cast<int64_t>(s_row[j0 + g]) * H + c;
          if constexpr (VEC) load_vec<T>(src, v[g]);
          else v[g][0] = to_f32(src[0]);
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int i = 0; i < NV; ++i) acc[i] = fmaf(s_w[j0 + g], v[g][i], acc[i]);
      }
      for (; j0 < k; ++j0) {
        float v[NV];
        const T* src = y + static_cast<int64_t>(s_row[j0]) * H + c;
        if constexpr (VEC) load_vec<T>(src, v);
        else v[0] = to_f32(src[0]);
#pragma unroll
        for (int i = 0; i < NV; ++i) acc[i] = fmaf(s_w[j0], v[i], acc[i]);
      }
      if (bad) {
#pragma unroll
        for (int i = 0; i < NV; ++i) acc[i] = qnan;
      }
      T* dst = out + t * H + c;
      if constexpr (VEC) {
        store_vec<T>(dst, acc);
      } else {
        dst[0] = from_f32<T>(acc[0]);
      }
    }
  }
}

template <typename T, typename TW, bool WEIGHTED = true>
cudaError_t launch_combine_t(const void* y, const uint32_t* inv, const void* w, int64_t T_tokens,
                             int k, int64_t H, void* out, cudaStream_t stream) {
  const int blocks = static_cast<int>(T_tokens < 65536 ? T_tokens : 65536);
  const bool vec = (H * static_cast<int64_t>(sizeof(T))) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(y) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(out) % 16 == 0;
  int threads = 256;
  const int64_t per_thread = vec ? Vec<T>::N : 1;
  while (threads > 32 && static_cast<int64_t>(threads / 2) * per_thread >= H) threads /= 2;
  auto kern = vec ? combine_kernel<T, TW, true, WEIGHTED> : combine_kernel<T, TW, false, WEIGHTED>;
  return launch_dependent(kern, dim3(blocks), dim3(threads), 0, stream, static_cast<const T*>(y), inv,
                          static_cast<const TW*>(w), T_tokens, k, H, static_cast<uint32_t>(T_tokens * k),
                          static_cast<T*>(out));
}

template <typename T>
cudaError_t launch_combine_w(const void* y, const uint32_t* inv, const void* w, moe_dtype wdt,
                             int64_t T_tokens, int k, int64_t H, void* out, cudaStream_t stream) {
  switch (wdt) {
    case MOE_F32: return launch_combine_t<T, float>(y, inv, w, T_tokens, k, H, out, stream);
    case MOE_F16: return launch_combine_t<T, __half>(y, inv, w, T_tokens, k, H, out, stream);
    default: return launch_combine_t<T, __nv_bfloat16>(y, inv, w, T_tokens, k, H, out, stream);
  }
}

}  // namespace

cudaError_t launch_combine(const void* y_dispatched, moe_dtype dtype, const uint32_t* inv,
                           const void* weights, moe_dtype weights_dtype, int64_t T, int top_k,
                           int64_t H, void* out, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  switch (dtype) {
    case MOE_F32:
      return launch_combine_w<float>(y_dispatched, inv, weights, weights_dtype, T, top_k, H, out, stream);
    case MOE_F16:
      return launch_combine_w<__half>(y_dispatched, inv, weights, weights_dtype, T, top_k, H, out, stream);
    default:
      return launch_combine_w<__nv_bfloat16>(y_dispatched, inv, weights, weights_dtype, T, top_k, H, out, stream);
  }
}

cudaError_t launch_dispatch_backward(const void* dinput, moe_dtype dtype, const uint32_t* inv, int64_t T,
                                     int top_k, int64_t H, void* dx, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  switch (dtype) {
    case MOE_F32: return launch_combine_t<float, float, false>(dinput, inv, nullptr, T, top_k, H, dx, stream);
    case MOE_F16: return launch_combine_t<__half, float, false>(dinput, inv, nullptr, T, top_k, H, dx, stream);
    default: return launch_combine_t<__nv_bfloat16, float, false>(dinput, inv, nullptr, T, top_k, H, dx, stream);
  }
}

}  // namespace moe
