// K2: compact per-expert dispatch (ruDNN user guide, section 5 "Expert
// weights and dispatch": no capacity dropping; a saved mapping restores
// token order). "PyTorch general ops", section 4 (gather/scatter), motivates
// handing the index table to the compute kernels instead of pre-gathering;
// the optional x_dispatched copy below serves the split API.
//
// The flat slots f = t*k + j are cut into chunks of DISPATCH_CHUNK. Three
// passes make the layout stable (row order inside an expert = ascending f)
// without atomics on the output:
//   1. count:   per-chunk expert histogram          -> scratch[c][e]
//   2. scan:    per expert, exclusive prefix over chunks plus the expert's
//               offset                               -> scratch[c][e] = first row
//               and counts / offsets
//   3. scatter: inside a chunk, 8 warps take 256 slots each; per-warp
//               histograms give each warp its first row per expert, and
//               __match_any_sync ranks equal experts inside each 32-slot step.
// An index >= E is never dispatched; its inv entry is INVALID_ROW.
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int SCATTER_WARPS = 8;
constexpr int SLOTS_PER_WARP = DISPATCH_CHUNK / SCATTER_WARPS;  // 256

__global__ void __launch_bounds__(512) dispatch_count_kernel(const uint32_t* __restrict__ indices,
                                                             int64_t n, int E,
                                                             uint32_t* __restrict__ hist) {
  __shared__ uint32_t h[ROUTE_MAX_E];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * DISPATCH_CHUNK;
  for (int i = threadIdx.x; i < DISPATCH_CHUNK; i += blockDim.x) {
    const int64_t f = base + i;
    if (f < n) {
      const uint32_t e = indices[f];
      if (e < static_cast<uint32_t>(E)) atomicAdd(&h[e], 1u);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(blockIdx.x) * E + e] = h[e];
}

// One block of 1024 threads. hist[c][e] becomes the first dispatched row of
// chunk c's slots for expert e.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(uint32_t* __restrict__ hist,
                                                             int nchunks, int E,
                                                             uint32_t* __restrict__ counts,
                                                             uint32_t* __restrict__ offsets) {
  __shared__ uint32_t tot[ROUTE_MAX_E];
  __shared__ uint32_t warp_sums[32];
  const int tid = threadIdx.x;
  // per-expert prefix over chunks (one expert per thread, E <= 1024)
  uint32_t run = 0;
  if (tid < E) {
    for (int c = 0; c < nchunks; ++c) {
      const uint32_t v = hist[static_cast<int64_t>(c) * E + tid];
      hist[static_cast<int64_t>(c) * E + tid] = run;
      run += v;
    }
  }
  // exclusive scan of the per-expert totals across the block
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t incl = (tid < E) ? run : 0;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_up_sync(FULL_MASK, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t ws = warp_sums[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL_MASK, ws, off);
      if (lane >= off) ws += o;
    }
    warp_sums[lane] = ws;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t before_warp = warp > 0 ? warp_sums[warp - 1] : 0u;
  const uint32_t excl = before_warp + incl - ((tid < E) ? run : 0u);
  if (tid < E) {
    tot[tid] = excl;
    counts[tid] = run;
    offsets[tid] = excl;
  }
  if (tid == 0) offsets[E] = warp_sums[31];
  __syncthreads();
  if (tid < E) {
    for (int c = 0; c < nchunks; ++c) hist[static_cast<int64_t>(c) * E + tid] += tot[tid];
  }
}

__global__ void __launch_bounds__(SCATTER_WARPS * 32) dispatch_scatter_kernel(
    const uint32_t* __restrict__ indices, int64_t n, int E, const uint32_t* __restrict__ first_row,
    uint32_t* __restrict__ row_src, uint32_t* __restrict__ inv) {
  __shared__ uint32_t wh[SCATTER_WARPS][ROUTE_MAX_E];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t chunk0 = static_cast<int64_t>(blockIdx.x) * DISPATCH_CHUNK;
  const int64_t w0 = chunk0 + static_cast<int64_t>(warp) * SLOTS_PER_WARP;
  for (int e = lane; e < E; e += 32) wh[warp][e] = 0;
  __syncwarp();
  for (int i = lane; i < SLOTS_PER_WARP; i += 32) {
    const int64_t f = w0 + i;
    if (f < n) {
      const uint32_t e = indices[f];
      if (e < static_cast<uint32_t>(E)) atomicAdd(&wh[warp][e], 1u);
    }
  }
  __syncthreads();
  // turn per-warp counts into each warp's first row per expert
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    uint32_t run = first_row[static_cast<int64_t>(blockIdx.x) * E + e];
#pragma unroll
    for (int w = 0; w < SCATTER_WARPS; ++w) {
      const uint32_t v = wh[w][e];
      wh[w][e] = run;
      run += v;
    }
  }
  __syncthreads();
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int step = 0; step < SLOTS_PER_WARP; step += 32) {
    const int64_t f = w0 + step + lane;
    const bool in_range = f < n;
    uint32_t e = in_range ? indices[f] : 0xFFFFFFFFu;
    const bool valid = in_range && e < static_cast<uint32_t>(E);
    if (!valid) e = 0xFFFFFFFFu;
    const uint32_t peers = __match_any_sync(FULL_MASK, e);
    uint32_t row = 0;
    if (valid) row = wh[warp][e] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && lane == 31 - __clz(peers)) wh[warp][e] += __popc(peers);
    __syncwarp();
    if (valid) {
      row_src[row] = static_cast<uint32_t>(f);
      inv[f] = row;
    } else if (in_range) {
      inv[f] = INVALID_ROW;
    }
  }
}

// x_dispatched[r] = x[row_src[r] / k] for r < offsets[E]; one warp per row.
template <typename VecT>
__global__ void __launch_bounds__(256) dispatch_gather_kernel(const VecT* __restrict__ x,
                                                              const uint32_t* __restrict__ row_src,
                                                              const uint32_t* __restrict__ offsets,
                                                              int E, int k, int64_t vec_per_row,
                                                              VecT* __restrict__ xd) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = offsets[E];
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = warp0; r < rows; r += nwarps) {
    const int64_t t = row_src[r] / static_cast<uint32_t>(k);
    const VecT* src = x + t * vec_per_row;
    VecT* dst = xd + r * vec_per_row;
    for (int64_t i = lane; i < vec_per_row; i += 32) dst[i] = src[i];
  }
}

// Fixed scratch of moe_dispatch_noalloc. Every GPU that loads this library
// holds this array (1 MiB) in its device image until the process exits; all
// calls on a device share it.
static __device__ __align__(256) uint32_t g_noalloc_dispatch_scratch[NOALLOC_DISPATCH_SCRATCH_BYTES / 4];

}  // namespace

cudaError_t noalloc_dispatch_scratch(void** ptr) {
  // In host code the array's name is only a stand-in for the device symbol;
  // the device address comes from cudaGetSymbolAddress, looked up once per
  // device with that device current and cached.
  constexpr int kMaxDevices = 256;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_dispatch_scratch);
    if (err != cudaSuccess) return err;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

size_t dispatch_scratch_bytes(int64_t T, int64_t E, int top_k) {
  const int64_t n = T * top_k;
  const int64_t nchunks = (n + DISPATCH_CHUNK - 1) / DISPATCH_CHUNK;
  return align_up(static_cast<size_t>(nchunks > 0 ? nchunks : 1) * static_cast<size_t>(E) * 4, 256);
}

cudaError_t launch_dispatch(const uint32_t* indices, int64_t T, int E, int top_k, const void* x,
                            moe_dtype dtype, int64_t H, uint32_t* counts, uint32_t* offsets,
                            uint32_t* row_src, uint32_t* inv, void* x_dispatched, void* scratch,
                            cudaStream_t stream) {
  const int64_t n = T * top_k;
  const int nchunks = static_cast<int>((n + DISPATCH_CHUNK - 1) / DISPATCH_CHUNK);
  uint32_t* hist = static_cast<uint32_t*>(scratch);
  if (nchunks > 0) {
    dispatch_count_kernel<<<nchunks, 512, 0, stream>>>(indices, n, E, hist);
  }
  // The scan also writes counts/offsets when there are no slots at all.
  dispatch_scan_kernel<<<1, 1024, 0, stream>>>(hist, nchunks, E, counts, offsets);
  if (nchunks > 0) {
    dispatch_scatter_kernel<<<nchunks, SCATTER_WARPS * 32, 0, stream>>>(indices, n, E, hist,
                                                                        row_src, inv);
  }
  if (x_dispatched != nullptr && n > 0) {
    const int64_t row_bytes = H * static_cast<int64_t>(dtype_size(dtype));
    const int64_t blocks64 = (n + 7) / 8;
    const int blocks = static_cast<int>(blocks64 < 16384 ? blocks64 : 16384);
    const bool vec16 = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(x_dispatched) % 16 == 0;
    if (vec16) {
      dispatch_gather_kernel<uint4><<<blocks, 256, 0, stream>>>(
          static_cast<const uint4*>(x), row_src, offsets, E, top_k, row_bytes / 16,
          static_cast<uint4*>(x_dispatched));
    } else if (dtype == MOE_F32) {
      dispatch_gather_kernel<float><<<blocks, 256, 0, stream>>>(
          static_cast<const float*>(x), row_src, offsets, E, top_k, H,
          static_cast<float*>(x_dispatched));
    } else {
      dispatch_gather_kernel<uint16_t><<<blocks, 256, 0, stream>>>(
          static_cast<const uint16_t*>(x), row_src, offsets, E, top_k, H,
          static_cast<uint16_t*>(x_dispatched));
    }
  }
  return cudaGetLastError();
}

}  // namespace moe
