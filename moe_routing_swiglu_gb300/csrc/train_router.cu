// Router weights of a fixed selection and their gradient, one warp per token.
//
// ruDNN user guide, section 12 "First-order MoE training":
// selected_router_weights gives FP32 weights of the given indices (softmax over
// all E experts, or the sigmoid of each selected logit), optionally divided by
// their sum over the slots, then multiplied by scale; selected_router_backward
// gives the gradient of those weights with respect to the logits, in the
// logits dtype. Repeated indices gather (each slot is its own term); an index
// outside 0..E-1 makes the whole row NaN, with no out-of-range access.
//
// With c = scale, g the FP32 weight gradient, and (renormalize) w~_j the
// renormalized unscaled weights, G = sum_j g_j w~_j:
//   softmax          dl_m = c (sum_{j: i_j = m} g_j p_j - P_m sum_j g_j p_j)
//   softmax + renorm dl_m = c sum_{j: i_j = m} w~_j (g_j - G)
//                    (p / sum_sel p = exp(l_i) / sum_sel exp(l): the full
//                    softmax denominator cancels)
//   sigmoid          dl_m = c sum_{j: i_j = m} g_j s_j (1 - s_j)
//   sigmoid + renorm dl_m = c sum_{j: i_j = m} s_j (1 - s_j) / S (g_j - G)
// Slot contributions to one logit are added in slot order.
//
// Layout: lane l holds experts l*V .. l*V+V-1 (V = ceil(E/32) rounded to a
// power of two); slot j lives on lane j % 32, word j / 32 (top_k <= 64). The
// softmax numerators are kept in a warp-private shared buffer in id order and
// summed left to right.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int RW_WARPS = 8;

template <typename TI>
__device__ __forceinline__ int64_t load_index(const TI* p) {
  return static_cast<int64_t>(p[0]);
}

template <typename TL, typename TI, int V, bool BACKWARD>
__global__ void __launch_bounds__(RW_WARPS * 32)
    router_kernel(const TL* __restrict__ logits, int64_t T, int E, const TI* __restrict__ indices, int k,
                  RouterParams p, float* __restrict__ weights, const float* __restrict__ grad,
                  TL* __restrict__ dlogits) {
  __shared__ __align__(16) float e_sm[RW_WARPS][32 * V];
  const int lane = threadIdx.x & 31;
  float* my_e = e_sm[threadIdx.x >> 5];
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const float qnan = __int_as_float(0x7FC00000);
  const bool softmax = p.scoring == 0;

  for (int64_t t = warp0; t < T; t += nwarps) {
    const TL* row = logits + t * E;
    // Slots of this token (j = lane, lane + 32).
    int64_t sid[2] = {0, 0};
    bool bad = false;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int j = q * 32 + lane;
      if (j < k) {
        sid[q] = load_index(indices + t * k + j);
        bad |= sid[q] < 0 || sid[q] >= E;
      }
    }
    bad = __any_sync(FULL_MASK, bad);
    if (bad) {
      if (!BACKWARD) {
        for (int j = lane; j < k; j += 32) weights[t * k + j] = qnan;
      } else {
        for (int i = lane; i < E; i += 32) dlogits[t * E + i] = from_f32<TL>(qnan);
      }
      continue;
    }

    // Unscaled, unnormalized selected values v_j and, for softmax, the full
    // probabilities P_i (each lane its V experts).
    float P[V];
    float v[2] = {0.0f, 0.0f};
    if (softmax) {
      float l[V];
      float m = -INFINITY;
#pragma unroll
      for (int q = 0; q < V; ++q) {
        const int id = lane * V + q;
        l[q] = id < E ? to_f32(row[id]) : -INFINITY;
        m = fmaxf(m, l[q]);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, off));
#pragma unroll
      for (int q = 0; q < V; ++q) {
        const int id = lane * V + q;
        if (id < E) my_e[id] = expf(__fsub_rn(l[q], m));
      }
      __syncwarp();
      float s = 0.0f;
      for (int i = 0; i < E; ++i) s = __fadd_rn(s, my_e[i]);
#pragma unroll
      for (int q = 0; q < V; ++q) {
        const int id = lane * V + q;
        P[q] = id < E ? __fdiv_rn(my_e[id], s) : 0.0f;
      }
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (q * 32 + lane < k) v[q] = __fdiv_rn(my_e[sid[q]], s);
      __syncwarp();
    } else {
#pragma unroll
      for (int q = 0; q < V; ++q) P[q] = 0.0f;
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (q * 32 + lane < k) {
          const float x = to_f32(row[sid[q]]);
          v[q] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-x)));
        }
    }

    // Renormalize over the slots, in slot order.
    float z = 1.0f;
    if (p.renormalize) {
      z = 0.0f;
      for (int j = 0; j < k; ++j) z = __fadd_rn(z, __shfl_sync(FULL_MASK, j < 32 ? v[0] : v[1], j & 31));
    }

    if (!BACKWARD) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = q * 32 + lane;
        if (j < k) {
          const float wv = p.renormalize ? __fdiv_rn(v[q], z) : v[q];
          weights[t * k + j] = __fmul_rn(wv, p.scale);
        }
      }
      continue;
    }

    // ---- backward
    float g[2] = {0.0f, 0.0f};
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (q * 32 + lane < k) g[q] = grad[t * k + q * 32 + lane];
    // Per-slot coefficient c_j: the amount slot j adds to dl at its expert;
    // `dense` multiplies P_m at every expert (softmax without renormalize).
    float coef[2] = {0.0f, 0.0f};
    float dense = 0.0f;
    if (p.renormalize) {
      float G = 0.0f;
      for (int j = 0; j < k; ++j) {
        const float vj = __shfl_sync(FULL_MASK, j < 32 ? v[0] : v[1], j & 31);
        const float gj = __shfl_sync(FULL_MASK, j < 32 ? g[0] : g[1], j & 31);
        G = fmaf(gj, __fdiv_rn(vj, z), G);
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float wt = __fdiv_rn(v[q], z);
        const float d = softmax ? wt : __fdiv_rn(v[q] * (1.0f - v[q]), z);
        coef[q] = p.scale * d * (g[q] - G);
      }
    } else {
      float A = 0.0f;
      if (softmax)
        for (int j = 0; j < k; ++j) {
          const float vj = __shfl_sync(FULL_MASK, j < 32 ? v[0] : v[1], j & 31);
          const float gj = __shfl_sync(FULL_MASK, j < 32 ? g[0] : g[1], j & 31);
          A = fmaf(gj, vj, A);
        }
#pragma unroll
      for (int q = 0; q < 2; ++q) coef[q] = p.scale * g[q] * (softmax ? v[q] : v[q] * (1.0f - v[q]));
      dense = softmax ? -p.scale * A : 0.0f;
    }
    float dl[V];
#pragma unroll
    for (int q = 0; q < V; ++q) dl[q] = dense * P[q];
    for (int j = 0; j < k; ++j) {
      const float cj = __shfl_sync(FULL_MASK, j < 32 ? coef[0] : coef[1], j & 31);
      const int64_t ij = __shfl_sync(FULL_MASK, j < 32 ? sid[0] : sid[1], j & 31);
      if (lane == static_cast<int>(ij / V)) {
        const int slot = static_cast<int>(ij % V);
#pragma unroll
        for (int q = 0; q < V; ++q)
          if (q == slot) dl[q] = __fadd_rn(dl[q], cj);
      }
    }
#pragma unroll
    for (int q = 0; q < V; ++q) {
      const int id = lane * V + q;
      if (id < E) dlogits[t * E + id] = from_f32<TL>(dl[q]);
    }
  }
}

template <typename TL, typename TI, bool BACKWARD>
cudaError_t launch_v(const void* logits, int64_t T, int E, const void* idx, int k, const RouterParams& p,
                     float* weights, const float* grad, void* dlogits, cudaStream_t s) {
  const int64_t want = (T + RW_WARPS - 1) / RW_WARPS;
  const int blocks = static_cast<int>(want < 65535 * 8 ? want : 65535 * 8);
  const TL* lg = static_cast<const TL*>(logits);
  const TI* ix = static_cast<const TI*>(idx);
  TL* dl = static_cast<TL*>(dlogits);
  const int th = RW_WARPS * 32;
  if (E <= 32) router_kernel<TL, TI, 1, BACKWARD><<<blocks, th, 0, s>>>(lg, T, E, ix, k, p, weights, grad, dl);
  else if (E <= 64) router_kernel<TL, TI, 2, BACKWARD><<<blocks, th, 0, s>>>(lg, T, E, ix, k, p, weights, grad, dl);
  else if (E <= 128) router_kernel<TL, TI, 4, BACKWARD><<<blocks, th, 0, s>>>(lg, T, E, ix, k, p, weights, grad, dl);
  else if (E <= 256) router_kernel<TL, TI, 8, BACKWARD><<<blocks, th, 0, s>>>(lg, T, E, ix, k, p, weights, grad, dl);
  else if (E <= 512) router_kernel<TL, TI, 16, BACKWARD><<<blocks, th, 0, s>>>(lg, T, E, ix, k, p, weights, grad, dl);
  else router_kernel<TL, TI, 32, BACKWARD><<<blocks, th, 0, s>>>(lg, T, E, ix, k, p, weights, grad, dl);
  return cudaGetLastError();
}

template <typename TL, bool BACKWARD>
cudaError_t launch_i(const void* logits, int64_t T, int E, const void* idx, int itype, int k,
                     const RouterParams& p, float* weights, const float* grad, void* dlogits, cudaStream_t s) {
  switch (itype) {
    case 0: return launch_v<TL, uint32_t, BACKWARD>(logits, T, E, idx, k, p, weights, grad, dlogits, s);
    case 1: return launch_v<TL, int32_t, BACKWARD>(logits, T, E, idx, k, p, weights, grad, dlogits, s);
    default: return launch_v<TL, int64_t, BACKWARD>(logits, T, E, idx, k, p, weights, grad, dlogits, s);
  }
}

template <bool BACKWARD>
cudaError_t launch_router(const void* logits, moe_dtype dtype, int64_t T, int E, const void* idx, int itype,
                          int k, const RouterParams& p, float* weights, const float* grad, void* dlogits,
                          cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  switch (dtype) {
    case MOE_F32: return launch_i<float, BACKWARD>(logits, T, E, idx, itype, k, p, weights, grad, dlogits, s);
    case MOE_F16: return launch_i<__half, BACKWARD>(logits, T, E, idx, itype, k, p, weights, grad, dlogits, s);
    default: return launch_i<__nv_bfloat16, BACKWARD>(logits, T, E, idx, itype, k, p, weights, grad, dlogits, s);
  }
}

}  // namespace

cudaError_t launch_router_weights(const void* logits, moe_dtype dtype, int64_t T, int E, const void* indices,
                                  int index_type, int top_k, const RouterParams& p, float* weights,
                                  cudaStream_t stream) {
  return launch_router<false>(logits, dtype, T, E, indices, index_type, top_k, p, weights, nullptr, nullptr,
                              stream);
}

cudaError_t launch_router_backward(const void* logits, moe_dtype dtype, int64_t T, int E, const void* indices,
                                   int index_type, int top_k, const RouterParams& p, const float* grad_weights,
                                   void* dlogits, cudaStream_t stream) {
  return launch_router<true>(logits, dtype, T, E, indices, index_type, top_k, p, nullptr, grad_weights, dlogits,
                             stream);
}

}  // namespace moe
