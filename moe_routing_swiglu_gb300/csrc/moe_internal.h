// Host-side launchers shared between the C-ABI layer (api.cu) and the kernel
// translation units. Every launcher only enqueues work on `stream`; argument
// checks have already been done by the caller.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "moe.h"

namespace moe {

// Launch `kernel` with programmatic stream serialization: its blocks may be
// scheduled (and run their prologue) while the previous kernel in the stream
// finishes; the kernel calls grid_dependency_wait() before touching that
// kernel's data.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- K1 routing (route.cu)
constexpr int ROUTE_MAX_E = 1024;
cudaError_t launch_route(const void* logits, moe_dtype dtype, int64_t T, int E, int top_k,
                         bool renormalize, uint32_t* indices, void* weights, float* weights_fp32,
                         cudaStream_t stream);

// ---- grouped, bias-corrected sigmoid routing (route_grouped.cu)
struct GroupRouteParams {
  int k;            // top_k, 1..64
  int groups;       // 1..128, divides E
  int group_size;   // E / groups
  int selected;     // selected groups, 1..groups
  int top_two;      // group score: sum of the two largest corrected scores
  int renormalize;  // divide the chosen weights by their sum
  float scale;      // finite, > 0
};
cudaError_t launch_route_sigmoid_grouped(const void* logits, moe_dtype dtype, int64_t T, int E,
                                         const float* bias, const GroupRouteParams& p, uint32_t* indices,
                                         void* weights, float* weights_fp32, cudaStream_t stream);

// ---- K2 dispatch (dispatch.cu)
constexpr int DISPATCH_CHUNK = 2048;  // flat slots per counting/scatter block
size_t dispatch_scratch_bytes(int64_t T, int64_t E, int top_k);
// Device address of the fixed scratch array used by moe_dispatch_noalloc on
// the current device (set up on first use per device).
constexpr size_t NOALLOC_DISPATCH_SCRATCH_BYTES = size_t{1} << 20;
cudaError_t noalloc_dispatch_scratch(void** ptr);
// zero_words (optional, 16-byte aligned): n_zero uint32 the scatter kernel
// sets to 0 (moe_forward's GEMM tile and ready counters, so the GEMMs need
// no memset).
cudaError_t launch_dispatch(const uint32_t* indices, int64_t T, int E, int top_k, const void* x,
                            moe_dtype dtype, int64_t H, uint32_t* counts, uint32_t* offsets,
                            uint32_t* row_src, uint32_t* inv, void* x_dispatched, void* scratch,
                            cudaStream_t stream, uint32_t* zero_words = nullptr, int64_t n_zero = 0);

// Row moves by an int64 index (the expert-parallel exchange's reorders):
// gather dst[r] = src[index[r]] (out-of-range index: zero row) or scatter
// dst[index[r]] = src[r] (out-of-range index: skipped).
cudaError_t launch_permute_rows(const void* src, int64_t src_rows, void* dst, int64_t dst_rows,
                                const int64_t* index, int64_t rows, int64_t row_bytes, bool scatter,
                                cudaStream_t stream);

// ---- K1 + K2 in one cooperative launch (route_dispatch.cu): softmax routing,
// then the dispatch maps and (x_dispatched != NULL) the x copy; the same bits
// as launch_route followed by launch_dispatch. scratch: RD_BARRIER_BYTES for
// the grid barrier (zeroed on the stream by the launcher), then the blocks'
// expert histograms.
constexpr int64_t RD_MAX_BLOCKS = 2048;
constexpr size_t RD_BARRIER_BYTES = 256;
size_t route_dispatch_scratch_bytes(int64_t T, int64_t E);
cudaError_t launch_route_dispatch(const void* logits, moe_dtype logits_dtype, int64_t T, int E, int top_k,
                                  bool renormalize, uint32_t* indices, void* weights, float* weights_fp32,
                                  const void* x, moe_dtype x_dtype, int64_t H, uint32_t* counts, uint32_t* offsets,
                                  uint32_t* row_src, uint32_t* inv, void* x_dispatched, void* scratch,
                                  int num_sms, cudaStream_t stream, uint32_t* zero_words = nullptr,
                                  int64_t n_zero = 0);
// The same with the grouped, bias-corrected sigmoid routing (the same bits as
// launch_route_sigmoid_grouped followed by launch_dispatch).
cudaError_t launch_route_dispatch_grouped(const void* logits, moe_dtype logits_dtype, int64_t T, int E,
                                          const float* bias, const GroupRouteParams& p, uint32_t* indices,
                                          void* weights, float* weights_fp32, const void* x, moe_dtype x_dtype,
                                          int64_t H, uint32_t* counts, uint32_t* offsets, uint32_t* row_src,
                                          uint32_t* inv, void* x_dispatched, void* scratch, int num_sms,
                                          cudaStream_t stream, uint32_t* zero_words = nullptr, int64_t n_zero = 0);

// ---- K5 combine (combine.cu)
cudaError_t launch_combine(const void* y_dispatched, moe_dtype dtype, const uint32_t* inv,
                           const void* weights, moe_dtype weights_dtype, int64_t T, int top_k,
                           int64_t H, void* out, cudaStream_t stream);

// ---- K7 FP32 experts on CUDA cores (experts_simt.cu). gate_up: a = x_dispatched
// [rows, H], w0/w1 = gate/up, out = h [rows, I]; else a = h, w0 = down, out = y [rows, H].
// Gather mode of the gate/up stage (both expert paths): dispatched row r reads x[row_src[r] / top_k]
// instead of row r of a materialised x_dispatched.
struct TcGather {
  const void* x;            // [x_rows, H]
  const uint32_t* row_src;  // [rows]
  int top_k;
  int64_t x_rows;
};
// Training forward: the gate/up stage also writes the pre-activations.
struct TcCache {
  void* g;  // [rows, I]
  void* u;  // [rows, I]
};
cudaError_t launch_experts_simt_f32(bool gate_up, const float* a, const TcGather* gather, const TcCache* cache,
                                    const uint32_t* offsets, int E, int64_t rows, const float* w0,
                                    const float* w1, int64_t H, int64_t I, float* out, cudaStream_t stream);

// ---- K3/K4 F16/BF16 experts on tcgen05 tensor cores (experts_tc.cu)
struct TcWeights {
  CUtensorMap gate, up, down;  // 3-D maps over [E, rows, K] with 64 x 128 x 1 boxes
};
bool tc_encode_weights(const void* gate, const void* up, const void* down, moe_dtype dtype,
                       int64_t E, int64_t H, int64_t I, TcWeights* out, const char** why);
// moe_forward gathers x rows in the gate/up stage for decode-sized batches
// (at most 8 dispatched rows per expert on average, where the 32-token tiles
// run) and materialises x_dispatched for larger ones.
inline bool forward_gathers_rows(int64_t rows, int64_t E) { return rows <= 8 * E; }
// gate_up: K3, a = x_dispatched [rows, H] (or gather != NULL) -> out = h [rows, I];
// else K4, a = h -> out = y [rows, H].
// sched: one uint32 of device memory for the tile counter (zeroed on the stream before the launch).
constexpr size_t TC_SCHED_BYTES = 256;
cudaError_t launch_experts_tc(const TcWeights& w, moe_dtype dtype, bool gate_up, const void* a,
                              const TcGather* gather, const TcCache* cache, const uint32_t* offsets, int E,
                              int64_t rows, int64_t H, int64_t I, void* out, uint32_t* sched, int num_sms,
                              cudaStream_t stream, const char** why, bool sched_zeroed = false);
// Fused combine of the chained launch: once every down tile has stored its
// y rows (one done counter), the epilogue warps of all CTAs write
// out[t] = sum_j w[t, j] * y[inv[t*top_k + j]] (FP32, slot order), each warp
// a fixed stripe of the tokens.
struct TcCombine {
  const uint32_t* inv;      // [T * top_k] flat slot -> dispatched row (from the dispatch)
  const void* weights;      // [T, top_k], weights_dtype
  moe_dtype weights_dtype;
  int top_k;                // 1 .. COMB_MAX_TOP_K
  int64_t T;
  uint32_t* done;           // [1] counter, zero on the stream before the launch
  void* out;                // [T, H]
};
// Largest top_k of the fused combine (a warp stages the (row, weight) pairs
// of four tokens in its 2 KB shared buffer); larger top_k combine in their
// own launch.
constexpr int COMB_MAX_TOP_K = 64;
// K3 and K4 in one launch (moe_forward): gate/up tiles (x_dispatched, or x
// gathered through row_src for decode-sized batches -> h), then down tiles
// (h -> y), each waiting for its expert's h rows. sched[0] and ready[0..E)
// must be zero on the stream before the launch (the dispatch zeroes them).
// cache (optional): the gate/up tiles also store the pre-activations g, u.
// comb (optional): the fused combine (y is still written, in dispatched order).
cudaError_t launch_experts_tc_chain(const TcWeights& w, moe_dtype dtype, const void* xd, const TcGather* gather,
                                    const TcCache* cache, const uint32_t* offsets, int E, int64_t rows, int64_t H,
                                    int64_t I, void* h, void* y, uint32_t* sched, uint32_t* ready, int num_sms,
                                    cudaStream_t stream, const char** why, const TcCombine* comb = nullptr);
cudaError_t read_device_status(uint32_t* code, bool clear);
// Device address of the status word the bounded waits report into.
cudaError_t device_status_ptr(uint32_t** p);

// ---- first-order training (train_router.cu, train_experts.cu, combine.cu)
struct RouterParams {
  int scoring;      // 0 softmax, 1 sigmoid
  int renormalize;
  float scale;
};
// index_type: 0 uint32, 1 int32, 2 int64
cudaError_t launch_router_weights(const void* logits, moe_dtype dtype, int64_t T, int E, const void* indices,
                                  int index_type, int top_k, const RouterParams& p, float* weights,
                                  cudaStream_t stream);
cudaError_t launch_router_backward(const void* logits, moe_dtype dtype, int64_t T, int E, const void* indices,
                                   int index_type, int top_k, const RouterParams& p, const float* grad_weights,
                                   void* dlogits, cudaStream_t stream);
cudaError_t launch_combine_backward(const void* y_dispatched, moe_dtype dtype, const uint32_t* inv,
                                    const uint32_t* row_src, const void* weights, moe_dtype weights_dtype,
                                    const void* grad_out, int64_t T, int top_k, int64_t H, void* dexpert,
                                    float* dweights, cudaStream_t stream);
cudaError_t launch_dispatch_backward(const void* dinput, moe_dtype dtype, const uint32_t* inv, int64_t T,
                                     int top_k, int64_t H, void* dx, cudaStream_t stream);
struct TrainBuffers {
  const void* x;     // x_dispatched [rows, H]
  const void* h;     // [rows, I]
  const void* g;     // [rows, I]
  const void* u;     // [rows, I]
  const void* dy;    // dexpert [rows, H]
  const void* gate;  // [E, I, H]
  const void* up;    // [E, I, H]
  const void* down;  // [E, H, I]
  float* dh;         // scratch [rows, I]
  void* dg;          // scratch [rows, I]
  void* du;          // scratch [rows, I]
  void* dx;          // out [rows, H]
  float* dgate;      // out [E, I, H]
  float* dup;        // out [E, I, H]
  float* ddown;      // out [E, H, I]
};
// CUDA-core backward (every dtype; the F32 path).
cudaError_t launch_experts_backward(moe_dtype dtype, const TrainBuffers& b, const uint32_t* offsets, int E,
                                    int64_t rows, int64_t H, int64_t I, cudaStream_t stream);
// Tensor-core backward (F16/BF16): dgrad and wgrad grouped GEMMs on tcgen05
// (experts_bwd_tc.cu); sched is one uint32 of device memory.
cudaError_t launch_experts_backward_tc(moe_dtype dtype, const TrainBuffers& b, const uint32_t* offsets, int E,
                                       int64_t rows, int64_t H, int64_t I, uint32_t* sched, int num_sms,
                                       cudaStream_t stream, const char** why);
cudaError_t launch_bounded_wait_selftest(uint32_t limit_us, cudaStream_t stream);

}  // namespace moe
