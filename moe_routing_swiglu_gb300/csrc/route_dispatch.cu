// K1 + K2 in one cooperative launch: softmax / top-k routing (ruDNN user
// guide, section 4 "Routing contract") or the grouped, bias-corrected sigmoid
// routing (section 10), then the compact per-expert dispatch (section 5
// "Expert weights and dispatch": no capacity dropping; a saved mapping
// restores token order), with the same outputs, bit for bit, as the routing
// kernel followed by the dispatch kernels.
//
// Block b owns the contiguous tokens [b*tpb, (b+1)*tpb), so the blocks'
// slots f = t*k + j come in block order, and the stable layout (rows of an
// expert in ascending f) is:
//   row(f) = offsets[e] + (slots of expert e in blocks before b)
//            + (slots of expert e in block b before f).
//   1. Route: warp w routes token b*tpb + r*W + w in round r (route_softmax.cuh
//      or route_grouped.cuh, the routing kernels' own code). The top-k
//      experts of one token are distinct, so each warp marks one bit per
//      chosen expert in a 32-bit per-expert mask; a chosen slot's rank inside
//      the block is the block's running count of the expert plus the marks
//      of the lower warps. The rank goes to inv[f] for now; the block's
//      histogram goes to hist[b].
//   2. Grid barrier (one arrival counter, zeroed on the stream before the
//      launch; the wait is bounded like the GEMMs' waits and records 0x1B).
//      A grid of one block (batches of up to one block's warps) skips it.
//   3. Every block sums all blocks' histograms (the totals give counts and,
//      by an exclusive scan over experts, offsets; the blocks before it give
//      its first row per expert), then turns its ranks into rows: inv[f],
//      row_src[row], and (prefill) the copy of x[t] into the k rows of its
//      slots — each x row read once and written top_k times.
// The cooperative launch keeps every block resident, so the barrier cannot
// wait on a block that has not started.
#include <algorithm>
#include <atomic>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "route_grouped.cuh"
#include "route_softmax.cuh"

namespace moe {
namespace {

constexpr uint32_t ST_RD_BARRIER = 0x1B;
constexpr uint64_t RD_WAIT_LIMIT_NS = 1000000000ull;  // about a second

// Warps per block: one token each per round; fewer for large E, whose
// per-lane logits and keys take more registers (a 32-warp block leaves 64
// registers a thread).
template <int V> struct RdWarps { static constexpr int value = V <= 4 ? 32 : (V == 8 ? 16 : 8); };
// Batches of at most this many tokens run as one block of this many warps:
// no grid barrier, and twice the registers of a 32-warp block for the
// routing chain of each token.
constexpr int RD_SMALL_T = 16;

struct RdArgs {
  const void* logits;
  int64_t T;
  int E, k, renorm;
  const float* bias;    // grouped routing: [E] or NULL
  GroupRouteParams gp;  // grouped routing
  uint32_t* indices;
  void* weights;
  float* weights32;
  const void* x;       // [T, H] (NULL: no x_dispatched)
  void* xd;            // [T*k, H]
  int64_t row_units;   // one x row in copy units (16 bytes, else 2 bytes)
  int vec16;           // rows copied in 16-byte units
  uint32_t* counts;
  uint32_t* offsets;
  uint32_t* row_src;
  uint32_t* inv;
  uint32_t* hist;      // [gridDim.x, E]
  uint32_t* barrier;   // [1], zero at launch
  uint32_t* zero_words;
  int64_t n_zero;
  int64_t tpb;         // tokens per block
  uint32_t* status;
};

// Routing policies: the per-token routing of phase 1, the number of slot
// registers per lane it returns the chosen experts in (slot j on lane j % 32,
// register j / 32), and what the block loads once before routing.
template <typename TL_, int V>
struct SoftmaxRouter {
  using TL = TL_;
  static constexpr int S = V;  // top_k <= E <= 32 * V
  struct Shared {};
  __device__ static bool prepare(const RdArgs&, Shared&) { return false; }
  __device__ static void route(const RdArgs& a, const Shared&, bool, int64_t t, int lane, float* buf,
                               uint32_t (&sid)[S]) {
    route_token<TL, V>(static_cast<const TL*>(a.logits), t, a.E, a.k, a.renorm, lane, buf, a.indices,
                       static_cast<TL*>(a.weights), a.weights32, sid);
  }
};

template <typename TL_, int V>
struct GroupedRouter {
  using TL = TL_;
  static constexpr int S = 2;  // top_k <= 64
  struct Shared {
    float bias[ROUTE_MAX_E];
    uint8_t grp[ROUTE_MAX_E];
  };
  // The bias (0 without one) and every expert's group id in shared memory;
  // returns whether any bias is NaN. Called by the whole block.
  __device__ static bool prepare(const RdArgs& a, Shared& sh) {
    bool nan = false;
    for (int i = threadIdx.x; i < a.E; i += blockDim.x) {
      const float b = a.bias != nullptr ? a.bias[i] : 0.0f;
      sh.bias[i] = b;
      nan |= isnan(b);
      sh.grp[i] = static_cast<uint8_t>(i / a.gp.group_size);
    }
    return __syncthreads_or(nan) != 0;
  }
  __device__ static void route(const RdArgs& a, const Shared& sh, bool bias_nan, int64_t t, int lane, float* buf,
                               uint32_t (&sid)[S]) {
    route_token_grouped<TL, V>(static_cast<const TL*>(a.logits), t, a.E, a.gp, sh.bias, sh.grp, bias_nan, lane, buf,
                               a.indices, static_cast<TL*>(a.weights), a.weights32, sid);
  }
};

// Copies x[t] into the dispatched rows of its k slots (slot j's row held on
// lane j % 32, register j / 32): U units per lane in flight, then k stores.
// (Stores do not hold registers once issued, so the loads in flight are the
// only register cost; eight per lane spilled under the 64-register limit of
// a 32-warp block.)
template <typename U_T, int S>
__device__ __forceinline__ void copy_token(const U_T* __restrict__ x, U_T* __restrict__ xd, int64_t units,
                                           int64_t t, int k, int lane, const uint32_t (&row)[S]) {
  constexpr int U = 4;
  const U_T* src = x + t * units;
  for (int64_t c0 = 0; c0 < units; c0 += 32 * U) {
    U_T v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = c0 + u * 32 + lane;
      if (i < units) v[u] = src[i];
    }
    for (int j = 0; j < k; ++j) {
      uint32_t rj = 0;
#pragma unroll
      for (int q = 0; q < S; ++q)
        if (q == (j >> 5)) rj = row[q];
      rj = __shfl_sync(FULL_MASK, rj, j & 31);
      U_T* dst = xd + static_cast<int64_t>(rj) * units;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = c0 + u * 32 + lane;
        if (i < units) dst[i] = v[u];
      }
    }
  }
}

template <typename R, int V, int W>
__global__ void __launch_bounds__(W * 32, 1) route_dispatch_kernel(const RdArgs a) {
  constexpr int S = R::S;
  __shared__ __align__(16) float e_sm[W * 32 * V];   // phase 1: the warps' exp buffers
  __shared__ uint32_t cnt[ROUTE_MAX_E];              // the block's running count per expert
  __shared__ uint32_t mark[ROUTE_MAX_E];             // phase 1: this round's warp marks; phase 3: first rows
  __shared__ uint32_t warp_sums[32];
  __shared__ int s_abort;
  __shared__ typename R::Shared router_sm;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = a.E, k = a.k;
  const int nthreads = blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * a.tpb;
  const int64_t t1 = min(a.T, t0 + a.tpb);
  const int rounds = static_cast<int>((a.tpb + W - 1) / W);  // the same in every block

  // A one-block grid is launched as a programmatic dependent of the previous
  // kernel in the stream: wait for it before touching memory it may use.
  grid_dependency_wait();
  for (int e = threadIdx.x; e < E; e += nthreads) {
    cnt[e] = 0;
    mark[e] = 0;
  }
  if (threadIdx.x == 0) s_abort = 0;
  // The counters of the expert GEMMs that follow in moe_forward.
  if (a.zero_words != nullptr) {
    const int64_t n4 = a.n_zero >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * nthreads;
    uint4* z4 = reinterpret_cast<uint4*>(a.zero_words);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * nthreads + threadIdx.x; i < n4; i += stride)
      z4[i] = make_uint4(0u, 0u, 0u, 0u);
    if (blockIdx.x == 0 && threadIdx.x < (a.n_zero & 3)) a.zero_words[(n4 << 2) + threadIdx.x] = 0u;
  }
  const bool router_flag = R::prepare(a, router_sm);  // syncs the block if it loads anything
  __syncthreads();

  // ---- 1. route; ranks inside the block
  float* my_e = e_sm + warp * 32 * V;
  const uint32_t lower_warps = (1u << warp) - 1u;
  for (int r = 0; r < rounds; ++r) {
    const int64_t t = t0 + static_cast<int64_t>(r) * W + warp;
    const bool active = t < t1;
    uint32_t sid[S];
    if (active) {
      R::route(a, router_sm, router_flag, t, lane, my_e, sid);
#pragma unroll
      for (int q = 0; q < S; ++q)
        if (q * 32 + lane < k) atomicOr(&mark[sid[q]], 1u << warp);
    }
    __syncthreads();
    if (active) {
#pragma unroll
      for (int q = 0; q < S; ++q) {
        const int j = q * 32 + lane;
        if (j < k) a.inv[t * k + j] = cnt[sid[q]] + __popc(mark[sid[q]] & lower_warps);
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += nthreads) {
      cnt[e] += __popc(mark[e]);
      mark[e] = 0;
    }
    __syncthreads();
  }
  // The histogram goes out only if another block reads it. Thread 0's
  // release at the barrier, after the block-wide sync, orders the block's
  // histogram stores before its arrival.
  if (gridDim.x > 1)
    for (int e = threadIdx.x; e < E; e += nthreads) a.hist[static_cast<int64_t>(blockIdx.x) * E + e] = cnt[e];
  __syncthreads();

  // ---- 2. grid barrier
  if (gridDim.x > 1) {
    if (threadIdx.x == 0) {
      counter_release_add(a.barrier);
      if (!counter_wait_bounded(a.barrier, gridDim.x, nullptr, a.status, ST_RD_BARRIER, RD_WAIT_LIMIT_NS))
        s_abort = 1;
    }
    __syncthreads();
    if (s_abort) return;
  }
  launch_dependents();

  // ---- 3. totals, offsets, this block's first rows; then rows and the x copy
  uint32_t* tot = reinterpret_cast<uint32_t*>(e_sm);  // e_sm holds >= 8*E words
  uint32_t* before = tot + E;
  for (int e = threadIdx.x; e < E; e += nthreads) {
    tot[e] = 0;
    before[e] = 0;
  }
  __syncthreads();
  if (gridDim.x == 1) {
    for (int e = threadIdx.x; e < E; e += nthreads) tot[e] = cnt[e];
  } else if ((E & 3) == 0 && nthreads % (E >> 2) == 0) {
    // 16-byte vectors of four experts: consecutive threads read consecutive
    // vectors of a histogram row (coalesced), each thread every
    // (nthreads / (E/4))-th row, all its loads in flight at once; the sums
    // meet in shared memory.
    const int G = gridDim.x, b = blockIdx.x, E4 = E >> 2;
    const uint4* hist4 = reinterpret_cast<const uint4*>(a.hist);
    const int e4 = threadIdx.x % E4, rstep = nthreads / E4;
    constexpr int U = 8;
    uint32_t all[4] = {0u, 0u, 0u, 0u}, bef[4] = {0u, 0u, 0u, 0u};
    for (int c = threadIdx.x / E4; c < G; c += U * rstep) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        v[u] = c + u * rstep < G ? __ldcg(hist4 + static_cast<int64_t>(c + u * rstep) * E4 + e4)
                                 : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool early = c + u * rstep < b;
        all[0] += v[u].x;
        all[1] += v[u].y;
        all[2] += v[u].z;
        all[3] += v[u].w;
        bef[0] += early ? v[u].x : 0u;
        bef[1] += early ? v[u].y : 0u;
        bef[2] += early ? v[u].z : 0u;
        bef[3] += early ? v[u].w : 0u;
      }
    }
    if (threadIdx.x / E4 < G) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        atomicAdd(&tot[4 * e4 + i], all[i]);
        atomicAdd(&before[4 * e4 + i], bef[i]);
      }
    }
  } else {
    const int G = gridDim.x, b = blockIdx.x;
    const int S = nthreads >= 2 * E ? nthreads / E : 1;  // segments of the histogram rows per expert
    constexpr int U = 8;                                   // loads in flight per thread
    for (int idx = threadIdx.x; idx < E * S; idx += nthreads) {
      const int e = idx % E, sg = idx / E;
      uint32_t all = 0, bef = 0;
      for (int c = sg; c < G; c += U * S) {
        uint32_t v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          v[u] = c + u * S < G ? __ldcg(a.hist + static_cast<int64_t>(c + u * S) * E + e) : 0u;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          all += v[u];
          bef += c + u * S < b ? v[u] : 0u;
        }
      }
      atomicAdd(&tot[e], all);
      atomicAdd(&before[e], bef);
    }
  }
  __syncthreads();
  // exclusive scan of the totals over experts, blockDim experts at a time
  const int nwarps = nthreads >> 5;
  uint32_t carry = 0;
  for (int c0 = 0; c0 < E; c0 += nthreads) {
    const int e = c0 + threadIdx.x;
    const uint32_t v = e < E ? tot[e] : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL_MASK, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      uint32_t ws = lane < nwarps ? warp_sums[lane] : 0u;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL_MASK, ws, off);
        if (lane >= off) ws += o;
      }
      if (lane < nwarps) warp_sums[lane] = ws;
    }
    __syncthreads();
    if (e < E) {
      const uint32_t off_e = carry + (warp > 0 ? warp_sums[warp - 1] : 0u) + incl - v;
      if (blockIdx.x == 0) {
        a.counts[e] = v;
        a.offsets[e] = off_e;
      }
      mark[e] = off_e + before[e];
    }
    carry += warp_sums[nwarps - 1];
    __syncthreads();
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) a.offsets[E] = carry;

  for (int r = 0; r < rounds; ++r) {
    const int64_t t = t0 + static_cast<int64_t>(r) * W + warp;
    if (t >= t1) break;
    uint32_t row[S];
#pragma unroll
    for (int q = 0; q < S; ++q) {
      const int j = q * 32 + lane;
      row[q] = 0;
      if (j < k) {
        const int64_t f = t * k + j;
        row[q] = mark[a.indices[f]] + a.inv[f];
        a.inv[f] = row[q];
        a.row_src[row[q]] = static_cast<uint32_t>(f);
      }
    }
    if (a.x != nullptr) {
      if (a.vec16)
        copy_token<uint4, S>(static_cast<const uint4*>(a.x), static_cast<uint4*>(a.xd), a.row_units, t, k, lane, row);
      else
        copy_token<uint16_t, S>(static_cast<const uint16_t*>(a.x), static_cast<uint16_t*>(a.xd), a.row_units, t, k,
                                lane, row);
    }
  }
}

template <typename R, int V, int W>
cudaError_t launch_rd_v(RdArgs a, int num_sms, cudaStream_t stream) {
  auto kern = route_dispatch_kernel<R, V, W>;
  static std::atomic<int> occ_cache{0};  // resident blocks per SM (per kernel; one GPU architecture)
  int occ = occ_cache.load(std::memory_order_relaxed);
  if (occ == 0) {
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, W * 32, 0);
    if (err != cudaSuccess) return err;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    occ_cache.store(occ, std::memory_order_relaxed);
  }
  const int64_t gmax = std::min<int64_t>(static_cast<int64_t>(occ) * num_sms, RD_MAX_BLOCKS);
  // One block while the batch fits its warps; else the batch spread evenly
  // over every resident block.
  a.tpb = a.T <= W ? W : (a.T + gmax - 1) / gmax;
  const int64_t grid = (a.T + a.tpb - 1) / a.tpb;
  if (grid == 1)  // no barrier: an ordinary launch, overlapping the previous kernel's tail
    return launch_dependent(kern, dim3(1), dim3(W * 32), 0, stream, a);
  cudaError_t err = cudaMemsetAsync(a.barrier, 0, 4, stream);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <template <typename, int> class Router, typename TL, int V>
cudaError_t launch_rd_w(const RdArgs& a, int num_sms, cudaStream_t stream) {
  using R = Router<TL, V>;
  constexpr int W = RdWarps<V>::value;
  if constexpr (W > RD_SMALL_T) {
    if (a.T <= RD_SMALL_T) return launch_rd_v<R, V, RD_SMALL_T>(a, num_sms, stream);
  }
  return launch_rd_v<R, V, W>(a, num_sms, stream);
}

template <template <typename, int> class Router, typename TL>
cudaError_t launch_rd_t(const RdArgs& a, int num_sms, cudaStream_t stream) {
  if (a.E <= 32) return launch_rd_w<Router, TL, 1>(a, num_sms, stream);
  if (a.E <= 64) return launch_rd_w<Router, TL, 2>(a, num_sms, stream);
  if (a.E <= 128) return launch_rd_w<Router, TL, 4>(a, num_sms, stream);
  if (a.E <= 256) return launch_rd_w<Router, TL, 8>(a, num_sms, stream);
  if (a.E <= 512) return launch_rd_w<Router, TL, 16>(a, num_sms, stream);
  return launch_rd_w<Router, TL, 32>(a, num_sms, stream);
}

template <template <typename, int> class Router>
cudaError_t launch_rd_dtype(const RdArgs& a, moe_dtype logits_dtype, int num_sms, cudaStream_t stream) {
  switch (logits_dtype) {
    case MOE_F32: return launch_rd_t<Router, float>(a, num_sms, stream);
    case MOE_F16: return launch_rd_t<Router, __half>(a, num_sms, stream);
    default: return launch_rd_t<Router, __nv_bfloat16>(a, num_sms, stream);
  }
}

// The arguments both routings share: outputs, x copy, scratch, counters.
cudaError_t fill_common(RdArgs& a, int64_t T, int E, int top_k, uint32_t* indices, void* weights,
                        float* weights_fp32, const void* x, moe_dtype x_dtype, int64_t H, uint32_t* counts,
                        uint32_t* offsets, uint32_t* row_src, uint32_t* inv, void* x_dispatched, void* scratch,
                        uint32_t* zero_words, int64_t n_zero) {
  uint32_t* status = nullptr;
  cudaError_t err = device_status_ptr(&status);
  if (err != cudaSuccess) return err;
  a.T = T;
  a.E = E;
  a.k = top_k;
  a.indices = indices;
  a.weights = weights;
  a.weights32 = weights_fp32;
  const bool copy = x_dispatched != nullptr;
  a.x = copy ? x : nullptr;
  a.xd = copy ? x_dispatched : nullptr;
  if (copy) {
    const int64_t row_bytes = H * static_cast<int64_t>(dtype_size(x_dtype));
    a.vec16 = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
              reinterpret_cast<uintptr_t>(x_dispatched) % 16 == 0;
    a.row_units = a.vec16 ? row_bytes / 16 : row_bytes / 2;
  }
  a.counts = counts;
  a.offsets = offsets;
  a.row_src = row_src;
  a.inv = inv;
  a.hist = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(scratch) + RD_BARRIER_BYTES);
  a.barrier = static_cast<uint32_t*>(scratch);
  a.zero_words = zero_words;
  a.n_zero = n_zero;
  a.status = status;
  return cudaSuccess;
}

}  // namespace

size_t route_dispatch_scratch_bytes(int64_t T, int64_t E) {
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(T, RD_MAX_BLOCKS));
  return RD_BARRIER_BYTES + align_up(static_cast<size_t>(blocks) * static_cast<size_t>(E) * 4, 256);
}

cudaError_t launch_route_dispatch(const void* logits, moe_dtype logits_dtype, int64_t T, int E, int top_k,
                                  bool renormalize, uint32_t* indices, void* weights, float* weights_fp32,
                                  const void* x, moe_dtype x_dtype, int64_t H, uint32_t* counts, uint32_t* offsets,
                                  uint32_t* row_src, uint32_t* inv, void* x_dispatched, void* scratch,
                                  int num_sms, cudaStream_t stream, uint32_t* zero_words, int64_t n_zero) {
  if (T == 0) return cudaSuccess;
  RdArgs a{};
  cudaError_t err = fill_common(a, T, E, top_k, indices, weights, weights_fp32, x, x_dtype, H, counts, offsets,
                                row_src, inv, x_dispatched, scratch, zero_words, n_zero);
  if (err != cudaSuccess) return err;
  a.logits = logits;
  a.renorm = renormalize ? 1 : 0;
  return launch_rd_dtype<SoftmaxRouter>(a, logits_dtype, num_sms, stream);
}

cudaError_t launch_route_dispatch_grouped(const void* logits, moe_dtype logits_dtype, int64_t T, int E,
                                          const float* bias, const GroupRouteParams& p, uint32_t* indices,
                                          void* weights, float* weights_fp32, const void* x, moe_dtype x_dtype,
                                          int64_t H, uint32_t* counts, uint32_t* offsets, uint32_t* row_src,
                                          uint32_t* inv, void* x_dispatched, void* scratch, int num_sms,
                                          cudaStream_t stream, uint32_t* zero_words, int64_t n_zero) {
  if (T == 0) return cudaSuccess;
  RdArgs a{};
  cudaError_t err = fill_common(a, T, E, p.k, indices, weights, weights_fp32, x, x_dtype, H, counts, offsets,
                                row_src, inv, x_dispatched, scratch, zero_words, n_zero);
  if (err != cudaSuccess) return err;
  a.logits = logits;
  a.bias = bias;
  a.gp = p;
  return launch_rd_dtype<GroupedRouter>(a, logits_dtype, num_sms, stream);
}

}  // namespace moe
