// Grouped, bias-corrected sigmoid routing, one warp per token (the
// per-token routing, its contract, its exactness argument and its layout are
// in route_grouped.cuh).
#include "moe_common.cuh"
#include "moe_internal.h"
#include "route_grouped.cuh"

namespace moe {
namespace {

constexpr int GR_WARPS = 8;

template <typename TL, int V>
__global__ void __launch_bounds__(GR_WARPS * 32)
    route_grouped_kernel(const TL* __restrict__ logits, const float* __restrict__ bias, int64_t T, int E,
                         GroupRouteParams p, uint32_t* __restrict__ indices, TL* __restrict__ weights,
                         float* __restrict__ weights32) {
  __shared__ float bias_sm[ROUTE_MAX_E];
  __shared__ uint8_t grp_sm[ROUTE_MAX_E];
  __shared__ __align__(16) float c_sm[GR_WARPS][32 * V];
  grid_dependency_wait();
  launch_dependents();
  const int lane = threadIdx.x & 31;
  float* my_c = c_sm[threadIdx.x >> 5];

  bool bias_nan = false;
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    const float b = bias != nullptr ? bias[i] : 0.0f;
    bias_sm[i] = b;
    bias_nan |= isnan(b);
    grp_sm[i] = static_cast<uint8_t>(i / p.group_size);
  }
  bias_nan = __syncthreads_or(bias_nan) != 0;

  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = warp0; t < T; t += nwarps) {
    uint32_t keep_id[2];
    route_token_grouped<TL, V>(logits, t, E, p, bias_sm, grp_sm, bias_nan, lane, my_c, indices, weights, weights32,
                               keep_id);
  }
}

template <typename TL>
cudaError_t launch_t(const void* logits, int64_t T, int E, const float* bias, const GroupRouteParams& p,
                     uint32_t* indices, void* weights, float* w32, cudaStream_t stream) {
  const int threads = GR_WARPS * 32;
  const int64_t want = (T + GR_WARPS - 1) / GR_WARPS;
  const int blocks = static_cast<int>(want < 65535 * 8 ? want : 65535 * 8);
  const TL* lg = static_cast<const TL*>(logits);
  TL* w = static_cast<TL*>(weights);
  auto kern = route_grouped_kernel<TL, 32>;
  if (E <= 32) kern = route_grouped_kernel<TL, 1>;
  else if (E <= 64) kern = route_grouped_kernel<TL, 2>;
  else if (E <= 128) kern = route_grouped_kernel<TL, 4>;
  else if (E <= 256) kern = route_grouped_kernel<TL, 8>;
  else if (E <= 512) kern = route_grouped_kernel<TL, 16>;
  return launch_dependent(kern, dim3(blocks), dim3(threads), 0, stream, lg, bias, T, E, p, indices, w, w32);
}

}  // namespace

static_assert(grouped_detail::GR_MAX_GROUPS <= 128, "the selected-group mask holds 128 groups");

cudaError_t launch_route_sigmoid_grouped(const void* logits, moe_dtype dtype, int64_t T, int E,
                                         const float* bias, const GroupRouteParams& p, uint32_t* indices,
                                         void* weights, float* weights_fp32, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  switch (dtype) {
    case MOE_F32:
      return launch_t<float>(logits, T, E, bias, p, indices, weights, weights_fp32, stream);
    case MOE_F16:
      return launch_t<__half>(logits, T, E, bias, p, indices, weights, weights_fp32, stream);
    default:
      return launch_t<__nv_bfloat16>(logits, T, E, bias, p, indices, weights, weights_fp32, stream);
  }
}

}  // namespace moe
