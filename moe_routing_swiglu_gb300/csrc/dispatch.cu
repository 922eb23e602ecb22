// K2: compact per-expert dispatch (ruDNN user guide, section 5 "Expert
// weights and dispatch": no capacity dropping; a saved mapping restores
// token order). "PyTorch general ops", section 4 (gather/scatter), motivates
// handing the index table to the compute kernels instead of pre-gathering;
// the optional x_dispatched copy below serves the split API.
//
// The flat slots f = t*k + j are cut into chunks of DISPATCH_CHUNK; two
// launches (one when a single chunk holds every slot) make the layout stable
// (row order inside an expert = ascending f) without atomics on the output:
//   1. count:   per-chunk expert histogram          -> scratch[c][e]
//   2. scatter: every chunk block re-derives what it needs from all chunks'
//               histograms (expert totals -> exclusive scan -> offsets; the
//               sum over earlier chunks -> its first row per expert); block 0
//               writes counts and offsets. Inside a chunk, 8 warps take 256
//               slots each: per-warp histograms give each warp its first row
//               per expert, and __match_any_sync ranks equal experts inside
//               each 32-slot step. Indices are loaded once into registers.
// An index >= E is never dispatched; its inv entry is INVALID_ROW.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int SCATTER_WARPS = 8;
constexpr int SLOTS_PER_WARP = DISPATCH_CHUNK / SCATTER_WARPS;  // 256

__global__ void __launch_bounds__(256) dispatch_count_kernel(const uint32_t* __restrict__ indices,
                                                             int64_t n, int E,
                                                             uint32_t* __restrict__ hist) {
  __shared__ uint32_t h[ROUTE_MAX_E];
  grid_dependency_wait();
  launch_dependents();
  constexpr int PER = DISPATCH_CHUNK / 256;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * DISPATCH_CHUNK;
  uint32_t e_reg[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int64_t f = base + threadIdx.x + 256 * i;
    e_reg[i] = f < n ? indices[f] : 0xFFFFFFFFu;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (e_reg[i] < static_cast<uint32_t>(E)) atomicAdd(&h[e_reg[i]], 1u);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(blockIdx.x) * E + e] = h[e];
}

// SINGLE: one chunk holds every slot (n <= DISPATCH_CHUNK, decode-sized
// batches): the block counts its own slots, so no count launch is needed.
template <bool SINGLE>
__global__ void __launch_bounds__(SCATTER_WARPS * 32) dispatch_scatter_kernel(
    const uint32_t* __restrict__ indices, int64_t n, int E, int nchunks,
    const uint32_t* __restrict__ hist, uint32_t* __restrict__ counts, uint32_t* __restrict__ offsets,
    uint32_t* __restrict__ row_src, uint32_t* __restrict__ inv, uint32_t* __restrict__ zero_words, int64_t n_zero) {
  __shared__ uint32_t wh[SCATTER_WARPS][ROUTE_MAX_E];
  __shared__ uint32_t first[ROUTE_MAX_E];   // first row of this chunk per expert
  __shared__ uint32_t tot[ROUTE_MAX_E];
  __shared__ uint32_t warp_sums[SCATTER_WARPS];
  constexpr int STEPS = SLOTS_PER_WARP / 32;
  grid_dependency_wait();
  launch_dependents();
  // The counters of the expert GEMMs that follow in moe_forward (tile
  // counter and per-expert ready counters), 16 bytes per store, spread over
  // the grid.
  if (zero_words != nullptr) {
    const int64_t n4 = n_zero >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    uint4* z4 = reinterpret_cast<uint4*>(zero_words);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride)
      z4[i] = make_uint4(0u, 0u, 0u, 0u);
    if (blockIdx.x == 0 && threadIdx.x < (n_zero & 3)) zero_words[(n4 << 2) + threadIdx.x] = 0u;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t w0 = static_cast<int64_t>(blockIdx.x) * DISPATCH_CHUNK +
                     static_cast<int64_t>(warp) * SLOTS_PER_WARP;
  uint32_t e_reg[STEPS];
#pragma unroll
  for (int i = 0; i < STEPS; ++i) {
    const int64_t f = w0 + 32 * i + lane;
    e_reg[i] = f < n ? indices[f] : 0xFFFFFFFFu;
  }
  for (int e = lane; e < E; e += 32) wh[warp][e] = 0;
  if constexpr (SINGLE) {
    // this block's own histogram is the total; nothing comes before it
    __syncthreads();
#pragma unroll
    for (int i = 0; i < STEPS; ++i)
      if (e_reg[i] < static_cast<uint32_t>(E)) atomicAdd(&wh[warp][e_reg[i]], 1u);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      uint32_t all = 0;
#pragma unroll
      for (int w = 0; w < SCATTER_WARPS; ++w) all += wh[w][e];
      first[e] = 0;
      tot[e] = all;
      counts[e] = all;
    }
  } else {
    // expert totals over all chunks and this chunk's offset from earlier chunks
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      uint32_t before = 0, all = 0;
      for (int c = 0; c < nchunks; ++c) {
        const uint32_t v = hist[static_cast<int64_t>(c) * E + e];
        before += c < static_cast<int>(blockIdx.x) ? v : 0u;
        all += v;
      }
      first[e] = before;
      tot[e] = all;
    }
  }
  __syncthreads();
  // exclusive scan of the totals over experts: warp w scans experts [w*E/8 ...)
  {
    const int per = (E + SCATTER_WARPS - 1) / SCATTER_WARPS;
    const int e_lo = warp * per, e_hi = min(E, e_lo + per);
    uint32_t carry = 0;
    for (int b = e_lo; b < e_hi; b += 32) {
      const int e = b + lane;
      const uint32_t v = e < e_hi ? tot[e] : 0u;
      uint32_t incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL_MASK, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < e_hi) tot[e] = carry + incl - v;   // exclusive within the warp's range
      carry += __shfl_sync(FULL_MASK, incl, 31);
    }
    if (lane == 0) warp_sums[warp] = carry;
  }
  if constexpr (!SINGLE) {
#pragma unroll
    for (int i = 0; i < STEPS; ++i)
      if (e_reg[i] < static_cast<uint32_t>(E)) atomicAdd(&wh[warp][e_reg[i]], 1u);
  }
  __syncthreads();
  {
    const int per = (E + SCATTER_WARPS - 1) / SCATTER_WARPS;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      uint32_t off = tot[e];
      for (int w = 0; w < e / per; ++w) off += warp_sums[w];
      if (blockIdx.x == 0) offsets[e] = off;
      uint32_t run = off + first[e];
#pragma unroll
      for (int w = 0; w < SCATTER_WARPS; ++w) {
        const uint32_t v = wh[w][e];
        wh[w][e] = run;
        run += v;
      }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      uint32_t all = 0;
      for (int w = 0; w < SCATTER_WARPS; ++w) all += warp_sums[w];
      offsets[E] = all;
    }
  }
  if (!SINGLE && blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      uint32_t all = 0;
      for (int c = 0; c < nchunks; ++c) all += hist[static_cast<int64_t>(c) * E + e];
      counts[e] = all;
    }
  }
  __syncthreads();
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < STEPS; ++i) {
    const int64_t f = w0 + 32 * i + lane;
    const bool in_range = f < n;
    const bool valid = e_reg[i] < static_cast<uint32_t>(E);
    const uint32_t e = valid ? e_reg[i] : 0xFFFFFFFFu;
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

// With no slots at all the scatter kernel has no blocks: write zero counts/offsets.
__global__ void dispatch_empty_kernel(int E, uint32_t* __restrict__ counts, uint32_t* __restrict__ offsets) {
  grid_dependency_wait();
  launch_dependents();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    if (e < E) counts[e] = 0;
    offsets[e] = 0;
  }
}

// x_dispatched[r] = x[row_src[r] / k] for r < offsets[E]; one warp per row.
template <typename VecT>
__global__ void __launch_bounds__(256) dispatch_gather_kernel(const VecT* __restrict__ x,
                                                              const uint32_t* __restrict__ row_src,
                                                              const uint32_t* __restrict__ offsets,
                                                              int E, int k, int64_t vec_per_row,
                                                              VecT* __restrict__ xd) {
  grid_dependency_wait();
  launch_dependents();
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

// Row moves by an index, warp per row: gather dst[r] = src[index[r]]
// (a row whose index is outside src is written as zeros), or scatter
// dst[index[r]] = src[r] (a row whose index is outside dst is skipped).
template <typename VecT, bool SCATTER>
__global__ void __launch_bounds__(256) permute_rows_kernel(const VecT* __restrict__ src, int64_t src_rows,
                                                           VecT* __restrict__ dst, int64_t dst_rows,
                                                           const int64_t* __restrict__ index, int64_t rows,
                                                           int64_t vec_per_row) {
  grid_dependency_wait();
  launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = warp0; r < rows; r += nwarps) {
    const int64_t i = index[r];
    if constexpr (SCATTER) {
      if (i < 0 || i >= dst_rows) continue;
      const VecT* s = src + r * vec_per_row;
      VecT* d = dst + i * vec_per_row;
      for (int64_t c = lane; c < vec_per_row; c += 32) d[c] = s[c];
    } else {
      VecT* d = dst + r * vec_per_row;
      if (i < 0 || i >= src_rows) {
        for (int64_t c = lane; c < vec_per_row; c += 32) d[c] = VecT{};
        continue;
      }
      const VecT* s = src + i * vec_per_row;
      for (int64_t c = lane; c < vec_per_row; c += 32) d[c] = s[c];
    }
  }
}

template <typename VecT>
cudaError_t launch_permute_t(const void* src, int64_t src_rows, void* dst, int64_t dst_rows, const int64_t* index,
                             int64_t rows, int64_t vec_per_row, bool scatter, cudaStream_t stream) {
  const int64_t blocks64 = (rows + 7) / 8;
  const int blocks = static_cast<int>(blocks64 < 16384 ? blocks64 : 16384);
  const VecT* s = static_cast<const VecT*>(src);
  VecT* d = static_cast<VecT*>(dst);
  return scatter ? launch_dependent(permute_rows_kernel<VecT, true>, dim3(blocks), dim3(256), 0, stream, s, src_rows,
                                    d, dst_rows, index, rows, vec_per_row)
                 : launch_dependent(permute_rows_kernel<VecT, false>, dim3(blocks), dim3(256), 0, stream, s, src_rows,
                                    d, dst_rows, index, rows, vec_per_row);
}

// Fixed scratch of moe_dispatch_noalloc. Every GPU that loads this library
// holds this array (1 MiB) in its device image until the process exits; all
// calls on a device share it.
static __device__ __align__(256) uint32_t g_noalloc_dispatch_scratch[NOALLOC_DISPATCH_SCRATCH_BYTES / 4];

}  // namespace

cudaError_t noalloc_dispatch_scratch(void** ptr) {
  // In host code the array's name is only a stand-in for the device symbol;
  // its device address comes from cudaGetSymbolAddress with the device
  // current. It is looked up again on every call (a host-side table lookup
  // once the module is loaded): an address kept from an earlier call would be
  // stale after cudaDeviceReset, which unloads the module and drops the array.
  *ptr = nullptr;
  return cudaGetSymbolAddress(ptr, g_noalloc_dispatch_scratch);
}

cudaError_t launch_permute_rows(const void* src, int64_t src_rows, void* dst, int64_t dst_rows,
                                const int64_t* index, int64_t rows, int64_t row_bytes, bool scatter,
                                cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const bool v16 = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(dst) % 16 == 0;
  const bool v4 = row_bytes % 4 == 0 && reinterpret_cast<uintptr_t>(src) % 4 == 0 &&
                  reinterpret_cast<uintptr_t>(dst) % 4 == 0;
  if (v16) return launch_permute_t<uint4>(src, src_rows, dst, dst_rows, index, rows, row_bytes / 16, scatter, stream);
  if (v4) return launch_permute_t<uint32_t>(src, src_rows, dst, dst_rows, index, rows, row_bytes / 4, scatter, stream);
  return launch_permute_t<uint8_t>(src, src_rows, dst, dst_rows, index, rows, row_bytes, scatter, stream);
}

size_t dispatch_scratch_bytes(int64_t T, int64_t E, int top_k) {
  const int64_t n = T * top_k;
  const int64_t nchunks = (n + DISPATCH_CHUNK - 1) / DISPATCH_CHUNK;
  return align_up(static_cast<size_t>(nchunks > 0 ? nchunks : 1) * static_cast<size_t>(E) * 4, 256);
}

cudaError_t launch_dispatch(const uint32_t* indices, int64_t T, int E, int top_k, const void* x,
                            moe_dtype dtype, int64_t H, uint32_t* counts, uint32_t* offsets,
                            uint32_t* row_src, uint32_t* inv, void* x_dispatched, void* scratch,
                            cudaStream_t stream, uint32_t* zero_words, int64_t n_zero) {
  const int64_t n = T * top_k;
  const int nchunks = static_cast<int>((n + DISPATCH_CHUNK - 1) / DISPATCH_CHUNK);
  uint32_t* hist = static_cast<uint32_t*>(scratch);
  cudaError_t err = cudaSuccess;
  if (nchunks == 1) {
    err = launch_dependent(dispatch_scatter_kernel<true>, dim3(1), dim3(SCATTER_WARPS * 32), 0, stream, indices, n, E,
                           1, hist, counts, offsets, row_src, inv, zero_words, n_zero);
  } else if (nchunks > 1) {
    err = launch_dependent(dispatch_count_kernel, dim3(nchunks), dim3(256), 0, stream, indices, n, E, hist);
    if (err == cudaSuccess)
      err = launch_dependent(dispatch_scatter_kernel<false>, dim3(nchunks), dim3(SCATTER_WARPS * 32), 0, stream,
                             indices, n, E, nchunks, hist, counts, offsets, row_src, inv, zero_words, n_zero);
  } else {
    dispatch_empty_kernel<<<1, 256, 0, stream>>>(E, counts, offsets);
  }
  if (err != cudaSuccess) return err;
  if (x_dispatched != nullptr && n > 0) {
    const int64_t row_bytes = H * static_cast<int64_t>(dtype_size(dtype));
    const int64_t blocks64 = (n + 7) / 8;
    const int blocks = static_cast<int>(blocks64 < 16384 ? blocks64 : 16384);
    const bool vec16 = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(x_dispatched) % 16 == 0;
    if (vec16) {
      err = launch_dependent(dispatch_gather_kernel<uint4>, dim3(blocks), dim3(256), 0, stream,
                             static_cast<const uint4*>(x), row_src, offsets, E, top_k, row_bytes / 16,
                             static_cast<uint4*>(x_dispatched));
    } else if (dtype == MOE_F32) {
      err = launch_dependent(dispatch_gather_kernel<float>, dim3(blocks), dim3(256), 0, stream,
                             static_cast<const float*>(x), row_src, offsets, E, top_k, H,
                             static_cast<float*>(x_dispatched));
    } else {
      err = launch_dependent(dispatch_gather_kernel<uint16_t>, dim3(blocks), dim3(256), 0, stream,
                             static_cast<const uint16_t*>(x), row_src, offsets, E, top_k, H,
                             static_cast<uint16_t*>(x_dispatched));
    }
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

}  // namespace moe
