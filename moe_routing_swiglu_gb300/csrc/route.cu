// K1: softmax / top-k routing, one warp per token (the per-token routing,
// its contract and its layout are in route_softmax.cuh).
#include "moe_common.cuh"
#include "moe_internal.h"
#include "route_softmax.cuh"

namespace moe {
namespace {

constexpr int ROUTE_WARPS = 8;

template <typename TL, int V>
__global__ void __launch_bounds__(ROUTE_WARPS * 32) route_kernel(const TL* __restrict__ logits, int64_t T,
                                                                 int E, int k, int renormalize,
                                                                 uint32_t* __restrict__ indices,
                                                                 TL* __restrict__ weights,
                                                                 float* __restrict__ weights32) {
  __shared__ __align__(16) float e_sm[ROUTE_WARPS][32 * V];
  grid_dependency_wait();
  launch_dependents();
  const int lane = threadIdx.x & 31;
  float* my_e = e_sm[threadIdx.x >> 5];
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = warp0; t < T; t += nwarps) {
    uint32_t slot_id[V];
    route_token<TL, V>(logits, t, E, k, renormalize, lane, my_e, indices, weights, weights32, slot_id);
  }
}

template <typename TL>
cudaError_t launch_route_t(const void* logits, int64_t T, int E, int k, bool renorm,
                           uint32_t* indices, void* weights, float* w32, cudaStream_t stream) {
  const int threads = ROUTE_WARPS * 32;
  const int64_t want = (T + ROUTE_WARPS - 1) / ROUTE_WARPS;
  const int blocks = static_cast<int>(want < 65535 * 8 ? want : 65535 * 8);
  const TL* lg = static_cast<const TL*>(logits);
  TL* w = static_cast<TL*>(weights);
  const int r = renorm ? 1 : 0;
  auto kern = route_kernel<TL, 32>;
  if (E <= 32) kern = route_kernel<TL, 1>;
  else if (E <= 64) kern = route_kernel<TL, 2>;
  else if (E <= 128) kern = route_kernel<TL, 4>;
  else if (E <= 256) kern = route_kernel<TL, 8>;
  else if (E <= 512) kern = route_kernel<TL, 16>;
  return launch_dependent(kern, dim3(blocks), dim3(threads), 0, stream, lg, T, E, k, r, indices, w, w32);
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
