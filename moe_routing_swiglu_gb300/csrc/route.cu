// K1: softmax / top-k routing, one warp per token.
//
// ruDNN user guide, section 4 "Routing contract": softmax over all E experts
// in FP32, then top-k with ties to the lower expert id, optional renormalize,
// then a cast to the logits dtype; rows with a NaN, a +inf or only -inf keep
// NaN weights. The max-shifted softmax follows "tiny-llm deep dive 5: ops.rs"
// (section on softmax).
//
// Layout: lane l of the warp holds experts l*V .. l*V+V-1 (V = ceil(E/32)
// rounded up to a power of two), so walking lanes then registers visits the
// experts in id order. That lets every lane form the softmax denominator as a
// left-to-right FP32 sum over experts 0..E-1 (the broadcast order below), the
// same order the oracle uses, so FP32 weights differ only by expf's ulps.
// Selection is k rounds of a warp arg-max on (logit, id) with the order
// "larger logit, then smaller id"; the winner's lane marks it taken.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__device__ __forceinline__ bool better(float va, uint32_t ia, float vb, uint32_t ib) {
  return va > vb || (va == vb && ia < ib);
}

template <typename TL, int V>
__global__ void __launch_bounds__(256) route_kernel(const TL* __restrict__ logits, int64_t T,
                                                    int E, int k, int renormalize,
                                                    uint32_t* __restrict__ indices,
                                                    TL* __restrict__ weights,
                                                    float* __restrict__ weights32) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

  for (int64_t t = warp0; t < T; t += nwarps) {
    const TL* row = logits + t * E;
    float l[V];
    bool nonfinite = false, all_neg_inf = true;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int id = lane * V + v;
      l[v] = id < E ? to_f32(row[id]) : -INFINITY;
      if (id < E) {
        nonfinite |= isnan(l[v]) || l[v] == INFINITY;
        all_neg_inf &= l[v] == -INFINITY;
      }
    }
    nonfinite = __any_sync(FULL_MASK, nonfinite);
    all_neg_inf = __all_sync(FULL_MASK, all_neg_inf);
    uint32_t* idx_row = indices + t * k;
    if (nonfinite || all_neg_inf) {
      // All probabilities of such a row are NaN: NaN weights, and the tie
      // rule over all-equal keys picks ids 0..k-1.
      for (int j = lane; j < k; j += 32) {
        idx_row[j] = static_cast<uint32_t>(j);
        weights[t * k + j] = from_f32<TL>(__int_as_float(0x7FC00000));
        if (weights32 != nullptr) weights32[t * k + j] = __int_as_float(0x7FC00000);
      }
      continue;
    }

    // m = max_i l_i (exact, order-free); absent slots hold -inf.
    float m = -INFINITY;
#pragma unroll
    for (int v = 0; v < V; ++v) m = fmaxf(m, l[v]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, off));

    // e_i = exp(l_i - m) in FP32.
    float e[V];
#pragma unroll
    for (int v = 0; v < V; ++v) e[v] = (lane * V + v) < E ? expf(__fsub_rn(l[v], m)) : 0.0f;

    // s = e_0 + e_1 + ... + e_{E-1}, left to right, identical on every lane.
    float s = 0.0f;
    for (int src = 0; src < 32; ++src) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const float ev = __shfl_sync(FULL_MASK, e[v], src);
        if (src * V + v < E) s = __fadd_rn(s, ev);
      }
    }

    // k rounds of arg-max over untaken experts; slot j keeps round j's winner.
    uint32_t taken = 0;
    float z = 0.0f;        // sum of selected p in slot order (renormalize)
    float p_keep[V];       // slot j's p lives on lane j % 32, register j / 32
    uint32_t id_keep[V];
#pragma unroll
    for (int q = 0; q < V; ++q) { p_keep[q] = 0.0f; id_keep[q] = 0; }
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      uint32_t bi = 0xFFFFFFFFu;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const uint32_t id = static_cast<uint32_t>(lane * V + v);
        if (id < static_cast<uint32_t>(E) && !((taken >> v) & 1u) && better(l[v], id, bv, bi)) {
          bv = l[v];
          bi = id;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(FULL_MASK, bv, off);
        const uint32_t oi = __shfl_xor_sync(FULL_MASK, bi, off);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      const int owner = static_cast<int>(bi / V);
      const int slot = static_cast<int>(bi % V);
      float ew = 0.0f;
#pragma unroll
      for (int v = 0; v < V; ++v) if (v == slot) ew = e[v];
      ew = __shfl_sync(FULL_MASK, ew, owner);
      if (lane == owner) taken |= 1u << slot;
      const float p = __fdiv_rn(ew, s);
      z = __fadd_rn(z, p);
#pragma unroll
      for (int q = 0; q < V; ++q) {
        if (q == (j >> 5) && lane == (j & 31)) { p_keep[q] = p; id_keep[q] = bi; }
      }
    }

#pragma unroll
    for (int q = 0; q < V; ++q) {
      const int j = q * 32 + lane;
      if (j < k) {
        const float w = renormalize ? __fdiv_rn(p_keep[q], z) : p_keep[q];
        idx_row[j] = id_keep[q];
        weights[t * k + j] = from_f32<TL>(w);
        if (weights32 != nullptr) weights32[t * k + j] = w;
      }
    }
  }
}

template <typename TL>
cudaError_t launch_route_t(const void* logits, int64_t T, int E, int k, bool renorm,
                           uint32_t* indices, void* weights, float* w32, cudaStream_t stream) {
  const int threads = 256;
  const int64_t want = (T + 7) / 8;
  const int blocks = static_cast<int>(want < 65535 * 8 ? want : 65535 * 8);
  const TL* lg = static_cast<const TL*>(logits);
  TL* w = static_cast<TL*>(weights);
  const int r = renorm ? 1 : 0;
  if (E <= 32) route_kernel<TL, 1><<<blocks, threads, 0, stream>>>(lg, T, E, k, r, indices, w, w32);
  else if (E <= 64) route_kernel<TL, 2><<<blocks, threads, 0, stream>>>(lg, T, E, k, r, indices, w, w32);
  else if (E <= 128) route_kernel<TL, 4><<<blocks, threads, 0, stream>>>(lg, T, E, k, r, indices, w, w32);
  else if (E <= 256) route_kernel<TL, 8><<<blocks, threads, 0, stream>>>(lg, T, E, k, r, indices, w, w32);
  else if (E <= 512) route_kernel<TL, 16><<<blocks, threads, 0, stream>>>(lg, T, E, k, r, indices, w, w32);
  else route_kernel<TL, 32><<<blocks, threads, 0, stream>>>(lg, T, E, k, r, indices, w, w32);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const void* logits, moe_dtype dtype, int64_t T, int E, int top_k,
                         bool renormalize, uint32_t* indices, void* weights, float* weights_fp32,
                         cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  switch (dtype) {
    case MOE_F32:
      return launch_route_t<float>(logits, T, E, top_k, renormalize, indices, weights, weights_fp32, stream);
    case MOE_F16:
      return launch_route_t<__half>(logits, T, E, top_k, renormalize, indices, weights, weights_fp32, stream);
    default:
      return launch_route_t<__nv_bfloat16>(logits, T, E, top_k, renormalize, indices, weights, weights_fp32, stream);
  }
}

}  // namespace moe
