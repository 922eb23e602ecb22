// C ABI of the local MoE forward chain: argument checks on the host, then
// kernel launches on the caller's stream. See include/moe.h for the contract
// of every entry point. No entry point allocates device memory or waits for
// the device (moe_device_status excepted, which exists to read a result).
#include <stdio.h>

#include <algorithm>
#include <limits>
#include <string>

#include "moe_common.cuh"
#include "moe_internal.h"

using moe::align_up;
using moe::dtype_size;
using moe::dtype_valid;

struct moe_experts {
  int device;
  int num_sms;
  moe_dtype dtype;
  int64_t E, H, I;
  const void* gate;
  const void* up;
  const void* down;
  moe::TcWeights tc;  // TMA descriptors of gate/up/down (F16/BF16 only)
};

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status st, const std::string& why) {
  g_last_error = why;
  return st;
}

moe_status cuda_fail(cudaError_t err, const char* where, const char* why = nullptr) {
  std::string msg = std::string(where) + ": " + cudaGetErrorString(err);
  if (why != nullptr) msg += std::string(" (") + why + ")";
  return fail(MOE_ERR_CUDA, msg);
}

moe_status ok() {
  g_last_error.clear();
  return MOE_OK;
}

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }
bool aligned256(const void* p) { return reinterpret_cast<uintptr_t>(p) % 256 == 0; }

// Flat slot numbers t*k+j and dispatched row numbers are uint32 and
// 0xFFFFFFFF marks an undispatched slot, so T*k must stay below it.
bool slots_fit(int64_t T, int64_t k) {
  return T >= 0 && k >= 1 && T <= (int64_t{0xFFFFFFFE} / k);
}

moe_status check_route_args(const void* logits, int dtype, int64_t T, int64_t E, int64_t top_k,
                            const void* indices, const void* weights) {
  if (!dtype_valid(dtype)) return fail(MOE_ERR_DTYPE, "logits dtype must be MOE_F32, MOE_F16 or MOE_BF16");
  if (E < 1 || E > moe::ROUTE_MAX_E) return fail(MOE_ERR_SHAPE, "E must satisfy 1 <= E <= 1024");
  if (top_k < 1 || top_k > E) return fail(MOE_ERR_TOP_K, "top_k must satisfy 1 <= top_k <= E");
  if (T < 0 || !slots_fit(T, top_k)) return fail(MOE_ERR_SHAPE, "T must be >= 0 and T*top_k < 2^32-1");
  if (T > 0 && (logits == nullptr || indices == nullptr || weights == nullptr))
    return fail(MOE_ERR_NULL, "logits, indices and weights must be non-NULL");
  return MOE_OK;
}

// GroupRoutingOptions ranges (ruDNN user guide, section 10).
moe_status check_group_options(const moe_group_routing_options* o, int64_t E, moe::GroupRouteParams* p) {
  if (o == nullptr) return fail(MOE_ERR_NULL, "options must be non-NULL");
  if (o->groups < 1 || o->groups > 128) return fail(MOE_ERR_SHAPE, "groups must satisfy 1 <= groups <= 128");
  if (E % o->groups != 0) return fail(MOE_ERR_SHAPE, "the expert count must be divisible by groups");
  if (o->selected_groups < 1 || o->selected_groups > o->groups)
    return fail(MOE_ERR_SHAPE, "selected_groups must satisfy 1 <= selected_groups <= groups");
  const int64_t G = E / o->groups;
  if (o->top_k < 1 || o->top_k > 64) return fail(MOE_ERR_TOP_K, "top_k must satisfy 1 <= top_k <= 64");
  if (o->top_k > o->selected_groups * G)
    return fail(MOE_ERR_TOP_K, "top_k exceeds the experts of the selected groups");
  if (o->group_top_two != 0 && G < 2)
    return fail(MOE_ERR_SHAPE, "group_top_two needs at least two experts per group");
  if (!(o->scale > 0.0f) || !(o->scale <= std::numeric_limits<float>::max()))
    return fail(MOE_ERR_SHAPE, "scale must be finite and positive");
  if (p != nullptr) {
    p->k = o->top_k;
    p->groups = o->groups;
    p->group_size = static_cast<int>(G);
    p->selected = o->selected_groups;
    p->top_two = o->group_top_two != 0;
    p->renormalize = o->renormalize != 0;
    p->scale = o->scale;
  }
  return MOE_OK;
}

moe_status check_bias(const float* bias) {
  if (reinterpret_cast<uintptr_t>(bias) % 4 != 0) return fail(MOE_ERR_ALIGNMENT, "bias must be 4-byte aligned");
  return MOE_OK;
}

// The fused combine (moe_experts_forward_combine) runs for F16/BF16 and
// top_k <= 64 (a warp stages the (row, weight) pairs of four tokens in a
// 2 KB buffer).
bool combine_can_fuse(const moe_experts* ex, int64_t top_k) {
  return ex->dtype != MOE_F32 && top_k <= moe::COMB_MAX_TOP_K;
}

struct ForwardLayout {
  size_t indices, weights, counts, offsets, row_src, inv, scratch, sched, xd, h, yd, total;
};

ForwardLayout forward_layout(const moe_experts* ex, int64_t T, int top_k) {
  const size_t n = static_cast<size_t>(T) * static_cast<size_t>(top_k);
  const size_t es = dtype_size(ex->dtype);
  ForwardLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return at;
  };
  L.indices = take(n * 4);
  L.weights = take(n * 4);  // room for any logits dtype
  L.counts = take(static_cast<size_t>(ex->E) * 4);
  L.offsets = take(static_cast<size_t>(ex->E + 1) * 4);
  L.row_src = take(n * 4);
  L.inv = take(n * 4);
  L.scratch = take(std::max(moe::dispatch_scratch_bytes(T, ex->E, top_k), moe::route_dispatch_scratch_bytes(T, ex->E)));
  // Tile counters, then (from word 64) one ready counter per expert for the
  // chained gate/up + down kernel; the dispatch zeroes them.
  L.sched = take(moe::TC_SCHED_BYTES + static_cast<size_t>(ex->E) * 4);
  L.xd = take(moe::forward_gathers_rows(static_cast<int64_t>(n), ex->E) ? 0 : n * static_cast<size_t>(ex->H) * es);
  L.h = take(n * static_cast<size_t>(ex->I) * es);
  L.yd = take(n * static_cast<size_t>(ex->H) * es);
  L.total = off;
  return L;
}

moe_status check_current_device(const moe_experts* ex) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (dev != ex->device)
    return fail(MOE_ERR_UNSUPPORTED, "the current device is not the device the experts were created on");
  return MOE_OK;
}

// One expert GEMM stage: gate_up (x_dispatched, or x gathered through
// row_src, -> h) or down (h -> y).
moe_status run_stage(const moe_experts* ex, bool gate_up, const void* a, const moe::TcGather* gather,
                     const uint32_t* offsets, int64_t rows, void* out, void* sched, cudaStream_t s,
                     const moe::TcCache* cache = nullptr, bool sched_zeroed = false) {
  cudaError_t err;
  const char* why = nullptr;
  if (ex->dtype == MOE_F32) {
    err = moe::launch_experts_simt_f32(gate_up, static_cast<const float*>(a), gather, cache, offsets,
                                       static_cast<int>(ex->E), rows,
                                       static_cast<const float*>(gate_up ? ex->gate : ex->down),
                                       static_cast<const float*>(gate_up ? ex->up : nullptr), ex->H,
                                       ex->I, static_cast<float*>(out), s);
  } else {
    err = moe::launch_experts_tc(ex->tc, ex->dtype, gate_up, a, gather, cache, offsets, static_cast<int>(ex->E),
                                 rows, ex->H, ex->I, out, static_cast<uint32_t*>(sched), ex->num_sms, s, &why,
                                 sched_zeroed);
  }
  if (err != cudaSuccess) return cuda_fail(err, gate_up ? "gate/up GEMM launch" : "down GEMM launch", why);
  return MOE_OK;
}

moe_status run_experts(const moe_experts* ex, const void* xd, const uint32_t* offsets, int64_t rows,
                       void* h, void* y, void* sched, cudaStream_t s) {
  moe_status st = run_stage(ex, true, xd, nullptr, offsets, rows, h, sched, s);
  if (st != MOE_OK) return st;
  return run_stage(ex, false, h, nullptr, offsets, rows, y, sched, s);
}

moe_status check_stage_args(const moe_experts* ex, const void* a, const uint32_t* offsets, int64_t rows,
                            const void* out, const void* ws, size_t ws_bytes) {
  if (ex == nullptr || offsets == nullptr) return fail(MOE_ERR_NULL, "experts and offsets must be non-NULL");
  if (ws == nullptr || ws_bytes < moe::TC_SCHED_BYTES)
    return fail(MOE_ERR_WORKSPACE, "workspace must hold at least 256 bytes");
  if (!aligned256(ws)) return fail(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (rows < 0 || rows >= int64_t{0xFFFFFFFF}) return fail(MOE_ERR_SHAPE, "rows must be in 0 .. 2^32-2");
  if (rows > 0 && (a == nullptr || out == nullptr)) return fail(MOE_ERR_NULL, "input and output must be non-NULL");
  if (ex->dtype != MOE_F32 && (!aligned16(a) || !aligned16(out)))
    return fail(MOE_ERR_ALIGNMENT, "input and output must be 16-byte aligned");
  return check_current_device(ex);
}

// The routing of a forward call: softmax / top-k (grouped == NULL) or the
// grouped, bias-corrected sigmoid routing. Either runs with the dispatch as
// one launch.
struct ForwardRouting {
  const void* logits;
  bool renormalize;                      // softmax routing
  const float* bias;                     // grouped routing: [E] or NULL
  const moe::GroupRouteParams* grouped;  // NULL: softmax routing
};

// Route + dispatch (one launch), experts, combine: the body of moe_forward
// and moe_forward_sigmoid_grouped once the routing arguments are checked.
moe_status forward_chain(const moe_experts* ex, const void* x, moe_dtype logits_dtype, int64_t T, int top_k,
                         void* out, uint32_t* indices_opt, void* weights_opt, void* workspace,
                         size_t workspace_bytes, cudaStream_t s, const ForwardRouting& routing) {
  if (T > 0 && (x == nullptr || out == nullptr)) return fail(MOE_ERR_NULL, "x and out must be non-NULL");
  const ForwardLayout L = forward_layout(ex, T, top_k);
  if (workspace == nullptr || workspace_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_forward_workspace_size()");
  if (!aligned256(workspace)) return fail(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  moe_status st = check_current_device(ex);
  if (st != MOE_OK) return st;
  if (T == 0) return ok();

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* indices = indices_opt ? indices_opt : reinterpret_cast<uint32_t*>(ws + L.indices);
  void* weights = weights_opt ? weights_opt : static_cast<void*>(ws + L.weights);
  uint32_t* counts = reinterpret_cast<uint32_t*>(ws + L.counts);
  uint32_t* offsets = reinterpret_cast<uint32_t*>(ws + L.offsets);
  uint32_t* row_src = reinterpret_cast<uint32_t*>(ws + L.row_src);
  uint32_t* inv = reinterpret_cast<uint32_t*>(ws + L.inv);
  void* h = ws + L.h;
  void* yd = ws + L.yd;
  const int64_t rows = T * top_k;
  const bool gather_rows = moe::forward_gathers_rows(rows, ex->E);
  void* xd = gather_rows ? nullptr : ws + L.xd;

  // Decode-sized batches: dispatch writes the maps only and the gate/up GEMM
  // gathers each dispatched row straight from x through row_src (TMA row
  // gathers). Larger batches: dispatch also writes x_dispatched, which the
  // GEMM streams with 128-row TMA boxes (a row gather costs about as much
  // TMA time as a whole box, so gathering every weight tile's 256 rows is
  // slower there than the extra copy).
  // The dispatch (the fused route + dispatch launch, or the scatter kernel)
  // zeroes the GEMMs' tile counter and the per-expert ready counters, so the
  // GEMMs need no memset (each kernel after the dispatch is launched as a
  // dependent of the previous). F16/BF16: gate/up and down run as one
  // launch whose down tiles start on each expert as soon as its h rows are
  // stored; F32: two launches.
  uint32_t* sched = reinterpret_cast<uint32_t*>(ws + L.sched);
  uint32_t* ready = sched + moe::TC_SCHED_BYTES / 4;
  const int64_t n_zero = static_cast<int64_t>(moe::TC_SCHED_BYTES / 4 + ex->E);
  const void* xg = gather_rows ? nullptr : x;
  cudaError_t err =
      routing.grouped != nullptr
          ? moe::launch_route_dispatch_grouped(routing.logits, logits_dtype, T, static_cast<int>(ex->E), routing.bias,
                                               *routing.grouped, indices, weights, nullptr, xg, ex->dtype, ex->H,
                                               counts, offsets, row_src, inv, xd, ws + L.scratch, ex->num_sms, s,
                                               sched, n_zero)
          : moe::launch_route_dispatch(routing.logits, logits_dtype, T, static_cast<int>(ex->E), top_k,
                                       routing.renormalize, indices, weights, nullptr, xg, ex->dtype, ex->H, counts,
                                       offsets, row_src, inv, xd, ws + L.scratch, ex->num_sms, s, sched, n_zero);
  if (err != cudaSuccess) return cuda_fail(err, "forward route + dispatch launch");
  const moe::TcGather gather{x, row_src, top_k, T};
  if (ex->dtype == MOE_F32) {
    st = run_stage(ex, true, xd, gather_rows ? &gather : nullptr, offsets, rows, h, sched, s, nullptr, true);
    if (st != MOE_OK) return st;
    st = run_stage(ex, false, h, nullptr, offsets, rows, yd, sched + 1, s, nullptr, true);
    if (st != MOE_OK) return st;
  } else {
    // F16/BF16: gate/up and down in one launch. The combine stays a launch
    // of its own: with the combine inside the experts' launch
    // (moe_experts_forward_combine) every measured workload ran slower.
    const char* why = nullptr;
    err = moe::launch_experts_tc_chain(ex->tc, ex->dtype, xd, gather_rows ? &gather : nullptr, nullptr, offsets,
                                       static_cast<int>(ex->E), rows, ex->H, ex->I, h, yd, sched, ready, ex->num_sms,
                                       s, &why);
    if (err != cudaSuccess) return cuda_fail(err, "gate/up + down GEMM launch", why);
  }
  err = moe::launch_combine(yd, ex->dtype, inv, weights, logits_dtype, T, top_k, ex->H, out, s);
  if (err != cudaSuccess) return cuda_fail(err, "forward combine launch");
  return ok();
}

// moe_forward_host's workspace: moe_forward's, then device staging for x,
// logits and out, each 256-byte aligned.
struct HostLayout {
  size_t fwd, x, logits, out, total;
  size_t x_bytes, logits_bytes, out_bytes;
};

HostLayout host_layout(const moe_experts* ex, int64_t T, int top_k, moe_dtype logits_dtype) {
  HostLayout h{};
  h.fwd = forward_layout(ex, T, top_k).total;
  const size_t t = static_cast<size_t>(T);
  h.x_bytes = t * static_cast<size_t>(ex->H) * dtype_size(ex->dtype);
  h.logits_bytes = t * static_cast<size_t>(ex->E) * dtype_size(logits_dtype);
  h.out_bytes = h.x_bytes;
  size_t off = align_up(h.fwd, 256);
  h.x = off;
  off += align_up(h.x_bytes + 1, 256);
  h.logits = off;
  off += align_up(h.logits_bytes + 1, 256);
  h.out = off;
  off += align_up(h.out_bytes + 1, 256);
  h.total = off;
  return h;
}

// FP32 dh scratch of moe_experts_backward: the F32 path's dgrad writes it;
// the tensor-core path turns dh into dg and du in the dgrad epilogue.
size_t backward_dh_bytes(const moe_experts* ex, size_t n) {
  return ex->dtype == MOE_F32 ? align_up(n * 4 + 1, 256) : 0;
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_NULL: return "MOE_ERR_NULL";
    case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE";
    case MOE_ERR_DTYPE: return "MOE_ERR_DTYPE";
    case MOE_ERR_TOP_K: return "MOE_ERR_TOP_K";
    case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
    default: return "MOE_ERR_UNKNOWN";
  }
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

int moe_version(void) { return 10100; }

moe_status moe_route(const void* logits, moe_dtype dtype, int64_t T, int64_t E, int32_t top_k,
                     int32_t renormalize, uint32_t* indices, void* weights, float* weights_fp32,
                     void* stream) {
  moe_status st = check_route_args(logits, dtype, T, E, top_k, indices, weights);
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  cudaError_t err = moe::launch_route(logits, dtype, T, static_cast<int>(E), top_k, renormalize != 0,
                                      indices, weights, weights_fp32, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_route launch");
  return ok();
}

size_t moe_dispatch_workspace_size(int64_t T, int64_t E, int32_t top_k) {
  if (T < 0 || E < 1 || top_k < 1) return 0;
  return moe::dispatch_scratch_bytes(T, E, top_k);
}

moe_status moe_dispatch(const uint32_t* indices, int64_t T, int64_t E, int32_t top_k,
                        const void* x, moe_dtype dtype, int64_t H, uint32_t* counts,
                        uint32_t* offsets, uint32_t* row_src, uint32_t* inv, void* x_dispatched,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (E < 1 || E > moe::ROUTE_MAX_E) return fail(MOE_ERR_SHAPE, "E must satisfy 1 <= E <= 1024");
  if (top_k < 1 || top_k > E) return fail(MOE_ERR_TOP_K, "top_k must satisfy 1 <= top_k <= E");
  if (T < 0 || !slots_fit(T, top_k)) return fail(MOE_ERR_SHAPE, "T must be >= 0 and T*top_k < 2^32-1");
  if (counts == nullptr || offsets == nullptr) return fail(MOE_ERR_NULL, "counts and offsets must be non-NULL");
  if (T > 0 && (indices == nullptr || row_src == nullptr || inv == nullptr))
    return fail(MOE_ERR_NULL, "indices, row_src and inv must be non-NULL");
  if (x_dispatched != nullptr) {
    if (x == nullptr) return fail(MOE_ERR_NULL, "x_dispatched needs x");
    if (!dtype_valid(dtype)) return fail(MOE_ERR_DTYPE, "x dtype must be MOE_F32, MOE_F16 or MOE_BF16");
    if (H < 1) return fail(MOE_ERR_SHAPE, "H must be >= 1");
  }
  const size_t need = moe::dispatch_scratch_bytes(T, E, top_k);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_dispatch_workspace_size()");
  if (!aligned256(workspace)) return fail(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  cudaError_t err = moe::launch_dispatch(indices, T, static_cast<int>(E), top_k, x, dtype, H, counts,
                                         offsets, row_src, inv, x_dispatched, workspace,
                                         static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_dispatch launch");
  return ok();
}

moe_status moe_dispatch_noalloc(const uint32_t* indices, int64_t T, int64_t E, int32_t top_k,
                                const void* x, moe_dtype dtype, int64_t H, uint32_t* counts,
                                uint32_t* offsets, uint32_t* row_src, uint32_t* inv,
                                void* x_dispatched, void* stream) {
  if (E < 1 || E > moe::ROUTE_MAX_E) return fail(MOE_ERR_SHAPE, "E must satisfy 1 <= E <= 1024");
  if (top_k < 1 || top_k > E) return fail(MOE_ERR_TOP_K, "top_k must satisfy 1 <= top_k <= E");
  if (T < 0 || !slots_fit(T, top_k)) return fail(MOE_ERR_SHAPE, "T must be >= 0 and T*top_k < 2^32-1");
  if (counts == nullptr || offsets == nullptr) return fail(MOE_ERR_NULL, "counts and offsets must be non-NULL");
  if (T > 0 && (indices == nullptr || row_src == nullptr || inv == nullptr))
    return fail(MOE_ERR_NULL, "indices, row_src and inv must be non-NULL");
  if (x_dispatched != nullptr) {
    if (x == nullptr) return fail(MOE_ERR_NULL, "x_dispatched needs x");
    if (!dtype_valid(dtype)) return fail(MOE_ERR_DTYPE, "x dtype must be MOE_F32, MOE_F16 or MOE_BF16");
    if (H < 1) return fail(MOE_ERR_SHAPE, "H must be >= 1");
  }
  const size_t need = moe::dispatch_scratch_bytes(T, E, top_k);
  if (need > moe::NOALLOC_DISPATCH_SCRATCH_BYTES)
    return fail(MOE_ERR_SHAPE, "moe_dispatch_noalloc: ceil(T*top_k/2048)*E*4 = " + std::to_string(need) +
                                   " bytes exceeds its fixed 1 MiB scratch; use moe_dispatch with a workspace");
  void* scratch = nullptr;
  cudaError_t err = moe::noalloc_dispatch_scratch(&scratch);
  if (err != cudaSuccess) return cuda_fail(err, "moe_dispatch_noalloc scratch set-up");
  err = moe::launch_dispatch(indices, T, static_cast<int>(E), top_k, x, dtype, H, counts, offsets, row_src,
                             inv, x_dispatched, scratch, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_dispatch_noalloc launch");
  return ok();
}

// The checks moe_route_dispatch and moe_route_sigmoid_grouped_dispatch share
// beyond the routing's own: maps, x copy, workspace.
static moe_status check_route_dispatch_maps(int64_t T, int64_t E, const void* x, moe_dtype x_dtype, int64_t H,
                                            const uint32_t* counts, const uint32_t* offsets,
                                            const uint32_t* row_src, const uint32_t* inv,
                                            const void* x_dispatched, const void* workspace,
                                            size_t workspace_bytes) {
  if (counts == nullptr || offsets == nullptr) return fail(MOE_ERR_NULL, "counts and offsets must be non-NULL");
  if (T > 0 && (row_src == nullptr || inv == nullptr)) return fail(MOE_ERR_NULL, "row_src and inv must be non-NULL");
  if (x_dispatched != nullptr) {
    if (x == nullptr) return fail(MOE_ERR_NULL, "x_dispatched needs x");
    if (!dtype_valid(x_dtype)) return fail(MOE_ERR_DTYPE, "x dtype must be MOE_F32, MOE_F16 or MOE_BF16");
    if (H < 1) return fail(MOE_ERR_SHAPE, "H must be >= 1");
  }
  const size_t need = moe::route_dispatch_scratch_bytes(T, E);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_route_dispatch_workspace_size()");
  if (!aligned256(workspace)) return fail(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  return MOE_OK;
}

// No slots: zero counts and offsets, as moe_dispatch writes them.
static moe_status zero_maps(int64_t E, uint32_t* counts, uint32_t* offsets, cudaStream_t s, const char* what) {
  cudaError_t err = cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * 4, s);
  if (err == cudaSuccess) err = cudaMemsetAsync(offsets, 0, static_cast<size_t>(E + 1) * 4, s);
  if (err != cudaSuccess) return cuda_fail(err, what);
  return ok();
}

static moe_status current_sm_count(int* sms) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return cuda_fail(err, "device query");
  return MOE_OK;
}

size_t moe_route_dispatch_workspace_size(int64_t T, int64_t E) {
  if (T < 0 || E < 1 || E > moe::ROUTE_MAX_E) return 0;
  return moe::route_dispatch_scratch_bytes(T, E);
}

moe_status moe_route_dispatch(const void* logits, moe_dtype logits_dtype, int64_t T, int64_t E, int32_t top_k,
                              int32_t renormalize, uint32_t* indices, void* weights, float* weights_fp32,
                              const void* x, moe_dtype x_dtype, int64_t H, uint32_t* counts, uint32_t* offsets,
                              uint32_t* row_src, uint32_t* inv, void* x_dispatched, void* workspace,
                              size_t workspace_bytes, void* stream) {
  moe_status st = check_route_args(logits, logits_dtype, T, E, top_k, indices, weights);
  if (st != MOE_OK) return st;
  st = check_route_dispatch_maps(T, E, x, x_dtype, H, counts, offsets, row_src, inv, x_dispatched, workspace,
                                 workspace_bytes);
  if (st != MOE_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) return zero_maps(E, counts, offsets, s, "moe_route_dispatch: zero counts and offsets");
  int sms = 0;
  st = current_sm_count(&sms);
  if (st != MOE_OK) return st;
  cudaError_t err = moe::launch_route_dispatch(logits, logits_dtype, T, static_cast<int>(E), top_k, renormalize != 0,
                                               indices, weights, weights_fp32, x, x_dtype, H, counts, offsets, row_src,
                                               inv, x_dispatched, workspace, sms, s);
  if (err != cudaSuccess) return cuda_fail(err, "moe_route_dispatch launch");
  return ok();
}

moe_status moe_permute_rows(const void* src, int64_t src_rows, void* dst, int64_t dst_rows, const int64_t* index,
                            int64_t rows, int64_t row_bytes, int32_t scatter, void* stream) {
  if (src_rows < 0 || dst_rows < 0 || rows < 0 || row_bytes < 1)
    return fail(MOE_ERR_SHAPE, "row counts must be >= 0 and row_bytes >= 1");
  if (rows > (scatter != 0 ? src_rows : dst_rows))
    return fail(MOE_ERR_SHAPE, "rows exceeds the rows of the side read or written in order");
  if (rows == 0) return ok();
  if (src == nullptr || dst == nullptr || index == nullptr)
    return fail(MOE_ERR_NULL, "src, dst and index must be non-NULL");
  cudaError_t err = moe::launch_permute_rows(src, src_rows, dst, dst_rows, index, rows, row_bytes, scatter != 0,
                                             static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_permute_rows launch");
  return ok();
}

moe_status moe_experts_create(const void* gate, const void* up, const void* down, moe_dtype dtype,
                              int64_t E, int64_t H, int64_t I, moe_experts** out) {
  if (out == nullptr) return fail(MOE_ERR_NULL, "out must be non-NULL");
  *out = nullptr;
  if (gate == nullptr || up == nullptr || down == nullptr)
    return fail(MOE_ERR_NULL, "gate, up and down must be non-NULL");
  if (!dtype_valid(dtype)) return fail(MOE_ERR_DTYPE, "expert dtype must be MOE_F32, MOE_F16 or MOE_BF16");
  if (E < 1 || E > moe::ROUTE_MAX_E) return fail(MOE_ERR_SHAPE, "E must satisfy 1 <= E <= 1024");
  if (H < 1 || I < 1 || H > (int64_t{1} << 30) || I > (int64_t{1} << 30))
    return fail(MOE_ERR_SHAPE, "H and I must be in 1 .. 2^30");
  if (dtype != MOE_F32) {
    if (H % 8 != 0 || I % 8 != 0)
      return fail(MOE_ERR_ALIGNMENT, "F16/BF16 experts need H and I to be multiples of 8 (16-byte rows)");
    if (!aligned16(gate) || !aligned16(up) || !aligned16(down))
      return fail(MOE_ERR_ALIGNMENT, "expert weights must be 16-byte aligned");
  }
  moe_experts* ex = new moe_experts{};
  ex->dtype = dtype;
  ex->E = E;
  ex->H = H;
  ex->I = I;
  ex->gate = gate;
  ex->up = up;
  ex->down = down;
  cudaError_t err = cudaGetDevice(&ex->device);
  if (err == cudaSuccess)
    err = cudaDeviceGetAttribute(&ex->num_sms, cudaDevAttrMultiProcessorCount, ex->device);
  if (err != cudaSuccess) {
    delete ex;
    return cuda_fail(err, "moe_experts_create device query");
  }
  if (dtype != MOE_F32) {
    const char* why = nullptr;
    if (!moe::tc_encode_weights(gate, up, down, dtype, E, H, I, &ex->tc, &why)) {
      delete ex;
      return fail(MOE_ERR_CUDA, why ? why : "tensor map encoding failed");
    }
  }
  *out = ex;
  return ok();
}

void moe_experts_destroy(moe_experts* experts) { delete experts; }

// h, then the tile counter (and, from word 64, one ready counter per expert
// for the chained gate/up + down launch).
size_t moe_experts_forward_dispatched_workspace_size(const moe_experts* ex, int64_t rows) {
  if (ex == nullptr || rows < 0) return 0;
  return align_up(static_cast<size_t>(rows) * static_cast<size_t>(ex->I) * dtype_size(ex->dtype) + 1, 256) +
         moe::TC_SCHED_BYTES + static_cast<size_t>(ex->E) * 4;
}

moe_status moe_experts_forward_dispatched(const moe_experts* ex, const void* x_dispatched,
                                          const uint32_t* offsets, int64_t rows,
                                          void* y_dispatched, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  if (ex == nullptr || offsets == nullptr) return fail(MOE_ERR_NULL, "experts and offsets must be non-NULL");
  if (rows < 0 || rows >= int64_t{0xFFFFFFFF}) return fail(MOE_ERR_SHAPE, "rows must be in 0 .. 2^32-2");
  if (rows > 0 && (x_dispatched == nullptr || y_dispatched == nullptr))
    return fail(MOE_ERR_NULL, "x_dispatched and y_dispatched must be non-NULL");
  const size_t need = moe_experts_forward_dispatched_workspace_size(ex, rows);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_experts_forward_dispatched_workspace_size()");
  if (!aligned256(workspace)) return fail(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (ex->dtype != MOE_F32 && (!aligned16(x_dispatched) || !aligned16(y_dispatched)))
    return fail(MOE_ERR_ALIGNMENT, "x_dispatched and y_dispatched must be 16-byte aligned");
  moe_status st = check_current_device(ex);
  if (st != MOE_OK) return st;
  if (rows == 0) return ok();
  const size_t cnt_bytes = moe::TC_SCHED_BYTES + static_cast<size_t>(ex->E) * 4;
  uint8_t* counters = static_cast<uint8_t*>(workspace) + (need - cnt_bytes);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ex->dtype == MOE_F32) {
    st = run_experts(ex, x_dispatched, offsets, rows, workspace, y_dispatched, counters, s);
    if (st != MOE_OK) return st;
    return ok();
  }
  // F16/BF16: one chained launch (as in moe_forward); its counters start at 0.
  cudaError_t err = cudaMemsetAsync(counters, 0, cnt_bytes, s);
  if (err != cudaSuccess) return cuda_fail(err, "counter reset");
  const char* why = nullptr;
  uint32_t* sched = reinterpret_cast<uint32_t*>(counters);
  err = moe::launch_experts_tc_chain(ex->tc, ex->dtype, x_dispatched, nullptr, nullptr, offsets, static_cast<int>(ex->E), rows,
                                     ex->H, ex->I, workspace, y_dispatched, sched, sched + moe::TC_SCHED_BYTES / 4,
                                     ex->num_sms, s, &why);
  if (err != cudaSuccess) return cuda_fail(err, "gate/up + down GEMM launch", why);
  return ok();
}

// h, then y_dispatched, then the tile counter, the per-expert ready counters
// and the combine's done counter.
size_t moe_experts_forward_combine_workspace_size(const moe_experts* ex, int64_t T, int32_t top_k) {
  if (ex == nullptr || T < 0 || top_k < 1 || !slots_fit(T, top_k)) return 0;
  const size_t n = static_cast<size_t>(T) * static_cast<size_t>(top_k);
  const size_t es = dtype_size(ex->dtype);
  return align_up(n * static_cast<size_t>(ex->I) * es + 1, 256) + align_up(n * static_cast<size_t>(ex->H) * es + 1, 256) +
         moe::TC_SCHED_BYTES + static_cast<size_t>(ex->E) * 4 + 16;
}

moe_status moe_experts_forward_combine(const moe_experts* ex, const void* x_dispatched, const uint32_t* offsets,
                                       const uint32_t* inv, const void* weights, moe_dtype weights_dtype, int64_t T,
                                       int32_t top_k, void* out, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  if (ex == nullptr || offsets == nullptr) return fail(MOE_ERR_NULL, "experts and offsets must be non-NULL");
  if (!dtype_valid(weights_dtype)) return fail(MOE_ERR_DTYPE, "weights dtype must be MOE_F32, MOE_F16 or MOE_BF16");
  if (T < 0 || top_k < 1 || top_k > ex->E) return fail(MOE_ERR_TOP_K, "top_k must satisfy 1 <= top_k <= E");
  if (!slots_fit(T, top_k)) return fail(MOE_ERR_SHAPE, "T * top_k must be below 2^32 - 1");
  if (!combine_can_fuse(ex, top_k))
    return fail(MOE_ERR_UNSUPPORTED, "the fused combine runs on the F16/BF16 tensor-core path with top_k <= 64; "
                                     "otherwise use moe_experts_forward_dispatched and moe_combine");
  if (T > 0 && (x_dispatched == nullptr || inv == nullptr || weights == nullptr || out == nullptr))
    return fail(MOE_ERR_NULL, "x_dispatched, inv, weights and out must be non-NULL");
  if (T > 0 && (!aligned16(x_dispatched) || !aligned16(out)))
    return fail(MOE_ERR_ALIGNMENT, "x_dispatched and out must be 16-byte aligned");
  if (T > 0 && reinterpret_cast<uintptr_t>(weights) % dtype_size(weights_dtype) != 0)
    return fail(MOE_ERR_ALIGNMENT, "weights must be aligned to their element size");
  const size_t need = moe_experts_forward_combine_workspace_size(ex, T, top_k);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_experts_forward_combine_workspace_size()");
  if (!aligned256(workspace)) return fail(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  moe_status st = check_current_device(ex);
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  const int64_t rows = T * top_k;
  const size_t n = static_cast<size_t>(rows);
  const size_t es = dtype_size(ex->dtype);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* h = ws;
  const size_t h_bytes = align_up(n * static_cast<size_t>(ex->I) * es + 1, 256);
  void* yd = ws + h_bytes;
  uint8_t* counters = ws + h_bytes + align_up(n * static_cast<size_t>(ex->H) * es + 1, 256);
  const size_t cnt_bytes = moe::TC_SCHED_BYTES + static_cast<size_t>(ex->E) * 4 + 16;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemsetAsync(counters, 0, cnt_bytes, s);
  if (err != cudaSuccess) return cuda_fail(err, "counter reset");
  uint32_t* sched = reinterpret_cast<uint32_t*>(counters);
  uint32_t* ready = sched + moe::TC_SCHED_BYTES / 4;
  const moe::TcCombine comb{inv, weights, weights_dtype, top_k, T, ready + ex->E, out};
  const char* why = nullptr;
  err = moe::launch_experts_tc_chain(ex->tc, ex->dtype, x_dispatched, nullptr, nullptr, offsets,
                                     static_cast<int>(ex->E), rows, ex->H, ex->I, h, yd, sched, ready, ex->num_sms, s,
                                     &why, &comb);
  if (err != cudaSuccess) return cuda_fail(err, "gate/up + down + combine GEMM launch", why);
  return ok();
}

moe_status moe_experts_gate_up(const moe_experts* ex, const void* x_dispatched,
                               const uint32_t* offsets, int64_t rows, void* h, void* workspace,
                               size_t workspace_bytes, void* stream) {
  moe_status st = check_stage_args(ex, x_dispatched, offsets, rows, h, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if (rows == 0) return ok();
  st = run_stage(ex, true, x_dispatched, nullptr, offsets, rows, h, workspace, static_cast<cudaStream_t>(stream));
  return st != MOE_OK ? st : ok();
}

moe_status moe_experts_gate_up_gather(const moe_experts* ex, const void* x, int64_t T, const uint32_t* row_src,
                                      int32_t top_k, const uint32_t* offsets, int64_t rows, void* h,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  moe_status st = check_stage_args(ex, x, offsets, rows, h, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if (top_k < 1 || T < 0 || !slots_fit(T, top_k)) return fail(MOE_ERR_SHAPE, "need top_k >= 1, T >= 0, T*top_k < 2^32-1");
  if (rows > T * top_k) return fail(MOE_ERR_SHAPE, "rows must not exceed T * top_k");
  if (rows > 0 && row_src == nullptr) return fail(MOE_ERR_NULL, "row_src must be non-NULL");
  if (rows == 0) return ok();
  const moe::TcGather gather{x, row_src, top_k, T};
  st = run_stage(ex, true, nullptr, &gather, offsets, rows, h, workspace, static_cast<cudaStream_t>(stream));
  return st != MOE_OK ? st : ok();
}

moe_status moe_experts_down(const moe_experts* ex, const void* h, const uint32_t* offsets, int64_t rows,
                            void* y_dispatched, void* workspace, size_t workspace_bytes, void* stream) {
  moe_status st = check_stage_args(ex, h, offsets, rows, y_dispatched, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if (rows == 0) return ok();
  st = run_stage(ex, false, h, nullptr, offsets, rows, y_dispatched, workspace, static_cast<cudaStream_t>(stream));
  return st != MOE_OK ? st : ok();
}

moe_status moe_combine(const void* y_dispatched, moe_dtype dtype, const uint32_t* inv,
                       const void* weights, moe_dtype weights_dtype, int64_t T, int32_t top_k,
                       int64_t H, void* out, void* stream) {
  if (!dtype_valid(dtype) || !dtype_valid(weights_dtype))
    return fail(MOE_ERR_DTYPE, "dtypes must be MOE_F32, MOE_F16 or MOE_BF16");
  if (top_k < 1) return fail(MOE_ERR_TOP_K, "top_k must be >= 1");
  if (T < 0 || !slots_fit(T, top_k) || H < 1) return fail(MOE_ERR_SHAPE, "need T >= 0, H >= 1, T*top_k < 2^32-1");
  if (T > 0 && (y_dispatched == nullptr || inv == nullptr || weights == nullptr || out == nullptr))
    return fail(MOE_ERR_NULL, "y_dispatched, inv, weights and out must be non-NULL");
  if (T == 0) return ok();
  cudaError_t err = moe::launch_combine(y_dispatched, dtype, inv, weights, weights_dtype, T, top_k, H,
                                        out, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_combine launch");
  return ok();
}

size_t moe_forward_workspace_size(const moe_experts* ex, int64_t T, int32_t top_k) {
  if (ex == nullptr || T < 0 || top_k < 1 || !slots_fit(T, top_k)) return 0;
  return forward_layout(ex, T, top_k).total;
}

moe_status moe_forward(const moe_experts* ex, const void* x, const void* logits,
                       moe_dtype logits_dtype, int64_t T, int32_t top_k, int32_t renormalize,
                       void* out, uint32_t* indices_opt, void* weights_opt, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (ex == nullptr) return fail(MOE_ERR_NULL, "experts must be non-NULL");
  moe_status st = check_route_args(logits, logits_dtype, T, ex->E, top_k, logits, logits);
  if (st != MOE_OK) return st;
  const ForwardRouting routing{logits, renormalize != 0, nullptr, nullptr};
  return forward_chain(ex, x, logits_dtype, T, top_k, out, indices_opt, weights_opt, workspace,
                       workspace_bytes, static_cast<cudaStream_t>(stream), routing);
}

size_t moe_forward_host_workspace_size(const moe_experts* ex, int64_t T, int32_t top_k, moe_dtype logits_dtype) {
  if (ex == nullptr || T < 0 || top_k < 1 || !slots_fit(T, top_k) || !dtype_valid(logits_dtype)) return 0;
  return host_layout(ex, T, top_k, logits_dtype).total;
}

moe_status moe_forward_host(const moe_experts* ex, const void* x_host, const void* logits_host,
                            moe_dtype logits_dtype, int64_t T, int32_t top_k, int32_t renormalize, void* out_host,
                            uint32_t* indices_opt, void* weights_opt, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (ex == nullptr) return fail(MOE_ERR_NULL, "experts must be non-NULL");
  if (!dtype_valid(logits_dtype)) return fail(MOE_ERR_DTYPE, "logits dtype must be MOE_F32, MOE_F16 or MOE_BF16");
  if (top_k < 1 || top_k > ex->E) return fail(MOE_ERR_TOP_K, "top_k must satisfy 1 <= top_k <= E");
  if (T < 0 || !slots_fit(T, top_k)) return fail(MOE_ERR_SHAPE, "T must be >= 0 and T*top_k < 2^32-1");
  if (T > 0 && (x_host == nullptr || logits_host == nullptr || out_host == nullptr))
    return fail(MOE_ERR_NULL, "x_host, logits_host and out_host must be non-NULL");
  const HostLayout h = host_layout(ex, T, top_k, logits_dtype);
  if (workspace == nullptr || workspace_bytes < h.total)
    return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_forward_host_workspace_size()");
  if (!aligned256(workspace)) return fail(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  moe_status st = check_current_device(ex);
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* dx = ws + h.x;
  void* dl = ws + h.logits;
  void* dout = ws + h.out;
  st = check_route_args(dl, logits_dtype, T, ex->E, top_k, dl, dl);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemcpyAsync(dx, x_host, h.x_bytes, cudaMemcpyHostToDevice, s);
  if (err != cudaSuccess) return cuda_fail(err, "moe_forward_host: copy of x to the device");
  err = cudaMemcpyAsync(dl, logits_host, h.logits_bytes, cudaMemcpyHostToDevice, s);
  if (err != cudaSuccess) return cuda_fail(err, "moe_forward_host: copy of the logits to the device");
  const ForwardRouting routing{dl, renormalize != 0, nullptr, nullptr};
  st = forward_chain(ex, dx, logits_dtype, T, top_k, dout, indices_opt, weights_opt, ws, h.fwd, s, routing);
  if (st != MOE_OK) return st;
  err = cudaMemcpyAsync(out_host, dout, h.out_bytes, cudaMemcpyDeviceToHost, s);
  if (err != cudaSuccess) return cuda_fail(err, "moe_forward_host: copy of out to the host");
  return ok();
}

moe_status moe_route_sigmoid_grouped(const void* logits, moe_dtype dtype, int64_t T, int64_t E,
                                     const float* bias, const moe_group_routing_options* options,
                                     uint32_t* indices, void* weights, float* weights_fp32, void* stream) {
  if (!dtype_valid(dtype)) return fail(MOE_ERR_DTYPE, "logits dtype must be MOE_F32, MOE_F16 or MOE_BF16");
  if (E < 1 || E > moe::ROUTE_MAX_E) return fail(MOE_ERR_SHAPE, "E must satisfy 1 <= E <= 1024");
  moe::GroupRouteParams p{};
  moe_status st = check_group_options(options, E, &p);
  if (st != MOE_OK) return st;
  if (T < 0 || !slots_fit(T, p.k)) return fail(MOE_ERR_SHAPE, "T must be >= 0 and T*top_k < 2^32-1");
  if (T > 0 && (logits == nullptr || indices == nullptr || weights == nullptr))
    return fail(MOE_ERR_NULL, "logits, indices and weights must be non-NULL");
  st = check_bias(bias);
  if (st != MOE_OK) return st;
  if (T == 0) return ok();
  cudaError_t err = moe::launch_route_sigmoid_grouped(logits, dtype, T, static_cast<int>(E), bias, p, indices,
                                                      weights, weights_fp32, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_route_sigmoid_grouped launch");
  return ok();
}

moe_status moe_route_sigmoid_grouped_dispatch(const void* logits, moe_dtype logits_dtype, int64_t T, int64_t E,
                                              const float* bias, const moe_group_routing_options* options,
                                              uint32_t* indices, void* weights, float* weights_fp32, const void* x,
                                              moe_dtype x_dtype, int64_t H, uint32_t* counts, uint32_t* offsets,
                                              uint32_t* row_src, uint32_t* inv, void* x_dispatched, void* workspace,
                                              size_t workspace_bytes, void* stream) {
  if (!dtype_valid(logits_dtype)) return fail(MOE_ERR_DTYPE, "logits dtype must be MOE_F32, MOE_F16 or MOE_BF16");
  if (E < 1 || E > moe::ROUTE_MAX_E) return fail(MOE_ERR_SHAPE, "E must satisfy 1 <= E <= 1024");
  moe::GroupRouteParams p{};
  moe_status st = check_group_options(options, E, &p);
  if (st != MOE_OK) return st;
  if (T < 0 || !slots_fit(T, p.k)) return fail(MOE_ERR_SHAPE, "T must be >= 0 and T*top_k < 2^32-1");
  if (T > 0 && (logits == nullptr || indices == nullptr || weights == nullptr))
    return fail(MOE_ERR_NULL, "logits, indices and weights must be non-NULL");
  st = check_bias(bias);
  if (st != MOE_OK) return st;
  st = check_route_dispatch_maps(T, E, x, x_dtype, H, counts, offsets, row_src, inv, x_dispatched, workspace,
                                 workspace_bytes);
  if (st != MOE_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) return zero_maps(E, counts, offsets, s, "moe_route_sigmoid_grouped_dispatch: zero counts and offsets");
  int sms = 0;
  st = current_sm_count(&sms);
  if (st != MOE_OK) return st;
  cudaError_t err = moe::launch_route_dispatch_grouped(logits, logits_dtype, T, static_cast<int>(E), bias, p, indices,
                                                       weights, weights_fp32, x, x_dtype, H, counts, offsets, row_src,
                                                       inv, x_dispatched, workspace, sms, s);
  if (err != cudaSuccess) return cuda_fail(err, "moe_route_sigmoid_grouped_dispatch launch");
  return ok();
}

moe_status moe_forward_sigmoid_grouped(const moe_experts* ex, const void* x, const void* logits,
                                       moe_dtype logits_dtype, int64_t T, const float* bias,
                                       const moe_group_routing_options* options, void* out,
                                       uint32_t* indices_opt, void* weights_opt, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  if (ex == nullptr || options == nullptr) return fail(MOE_ERR_NULL, "experts and options must be non-NULL");
  if (!dtype_valid(logits_dtype))
    return fail(MOE_ERR_DTYPE, "logits dtype must be MOE_F32, MOE_F16 or MOE_BF16");
  moe::GroupRouteParams p{};
  moe_status st = check_group_options(options, ex->E, &p);
  if (st != MOE_OK) return st;
  if (T < 0 || !slots_fit(T, p.k)) return fail(MOE_ERR_SHAPE, "T must be >= 0 and T*top_k < 2^32-1");
  if (T > 0 && logits == nullptr) return fail(MOE_ERR_NULL, "logits must be non-NULL");
  st = check_bias(bias);
  if (st != MOE_OK) return st;
  const ForwardRouting routing{logits, false, bias, &p};
  return forward_chain(ex, x, logits_dtype, T, p.k, out, indices_opt, weights_opt, workspace,
                       workspace_bytes, static_cast<cudaStream_t>(stream), routing);
}

// ---------------------------------------------------------------- first-order training

static moe_status check_router_weight_args(const void* logits, int dtype, int64_t T, int64_t E,
                                           const void* indices, int index_type, int32_t top_k,
                                           const moe_router_weight_options* o, moe::RouterParams* p) {
  if (!dtype_valid(dtype)) return fail(MOE_ERR_DTYPE, "logits dtype must be MOE_F32, MOE_F16 or MOE_BF16");
  if (index_type < MOE_INDEX_U32 || index_type > MOE_INDEX_I64)
    return fail(MOE_ERR_DTYPE, "index type must be MOE_INDEX_U32, MOE_INDEX_I32 or MOE_INDEX_I64");
  if (E < 1 || E > moe::ROUTE_MAX_E) return fail(MOE_ERR_SHAPE, "E must satisfy 1 <= E <= 1024");
  if (top_k < 1 || top_k > E || top_k > 64) return fail(MOE_ERR_TOP_K, "top_k must satisfy 1 <= top_k <= min(E, 64)");
  if (o == nullptr) return fail(MOE_ERR_NULL, "options must be non-NULL");
  if (o->scoring != MOE_ROUTER_SOFTMAX && o->scoring != MOE_ROUTER_SIGMOID)
    return fail(MOE_ERR_SHAPE, "scoring must be MOE_ROUTER_SOFTMAX or MOE_ROUTER_SIGMOID");
  if (!(o->scale > 0.0f) || !(o->scale <= std::numeric_limits<float>::max()))
    return fail(MOE_ERR_SHAPE, "scale must be finite and positive");
  if (T < 0 || !slots_fit(T, top_k)) return fail(MOE_ERR_SHAPE, "T must be >= 0 and T*top_k < 2^32-1");
  if (T > 0 && (logits == nullptr || indices == nullptr)) return fail(MOE_ERR_NULL, "logits and indices must be non-NULL");
  p->scoring = o->scoring;
  p->renormalize = o->renormalize != 0;
  p->scale = o->scale;
  return MOE_OK;
}

moe_status moe_router_weights(const void* logits, moe_dtype dtype, int64_t T, int64_t E, const void* indices,
                              moe_index_type index_type, int32_t top_k, const moe_router_weight_options* options,
                              float* weights, void* stream) {
  moe::RouterParams p{};
  moe_status st = check_router_weight_args(logits, dtype, T, E, indices, index_type, top_k, options, &p);
  if (st != MOE_OK) return st;
  if (T > 0 && weights == nullptr) return fail(MOE_ERR_NULL, "weights must be non-NULL");
  if (T == 0) return ok();
  cudaError_t err = moe::launch_router_weights(logits, dtype, T, static_cast<int>(E), indices, index_type, top_k, p,
                                               weights, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_router_weights launch");
  return ok();
}

moe_status moe_router_backward(const void* logits, moe_dtype dtype, int64_t T, int64_t E, const void* indices,
                               moe_index_type index_type, int32_t top_k, const moe_router_weight_options* options,
                               const float* grad_weights, void* dlogits, void* stream) {
  moe::RouterParams p{};
  moe_status st = check_router_weight_args(logits, dtype, T, E, indices, index_type, top_k, options, &p);
  if (st != MOE_OK) return st;
  if (T > 0 && (grad_weights == nullptr || dlogits == nullptr))
    return fail(MOE_ERR_NULL, "grad_weights and dlogits must be non-NULL");
  if (T == 0) return ok();
  cudaError_t err = moe::launch_router_backward(logits, dtype, T, static_cast<int>(E), indices, index_type, top_k,
                                                p, grad_weights, dlogits, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_router_backward launch");
  return ok();
}

moe_status moe_combine_backward(const void* y_dispatched, moe_dtype dtype, const uint32_t* inv,
                                const uint32_t* row_src, const void* weights, moe_dtype weights_dtype,
                                const void* grad_out, int64_t T, int32_t top_k, int64_t H, void* dexpert,
                                float* dweights, void* stream) {
  if (!dtype_valid(dtype) || !dtype_valid(weights_dtype)) return fail(MOE_ERR_DTYPE, "unknown dtype");
  if (top_k < 1) return fail(MOE_ERR_TOP_K, "top_k must be >= 1");
  if (H < 1 || T < 0 || !slots_fit(T, top_k)) return fail(MOE_ERR_SHAPE, "need H >= 1, T >= 0, T*top_k < 2^32-1");
  if (T > 0 && (y_dispatched == nullptr || inv == nullptr || row_src == nullptr || weights == nullptr ||
                grad_out == nullptr || dexpert == nullptr || dweights == nullptr))
    return fail(MOE_ERR_NULL, "every buffer must be non-NULL");
  if (T == 0) return ok();
  cudaError_t err = moe::launch_combine_backward(y_dispatched, dtype, inv, row_src, weights, weights_dtype, grad_out,
                                                 T, top_k, H, dexpert, dweights, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_combine_backward launch");
  return ok();
}

moe_status moe_dispatch_backward(const void* dinput, moe_dtype dtype, const uint32_t* inv, int64_t T, int32_t top_k,
                                 int64_t H, void* dx, void* stream) {
  if (!dtype_valid(dtype)) return fail(MOE_ERR_DTYPE, "unknown dtype");
  if (top_k < 1) return fail(MOE_ERR_TOP_K, "top_k must be >= 1");
  if (H < 1 || T < 0 || !slots_fit(T, top_k)) return fail(MOE_ERR_SHAPE, "need H >= 1, T >= 0, T*top_k < 2^32-1");
  if (T > 0 && (dinput == nullptr || inv == nullptr || dx == nullptr))
    return fail(MOE_ERR_NULL, "dinput, inv and dx must be non-NULL");
  if (T == 0) return ok();
  cudaError_t err = moe::launch_dispatch_backward(dinput, dtype, inv, T, top_k, H, dx, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_dispatch_backward launch");
  return ok();
}

size_t moe_experts_forward_training_workspace_size(const moe_experts* ex) {
  if (ex == nullptr) return 0;
  return moe::TC_SCHED_BYTES + static_cast<size_t>(ex->E) * 4;
}

moe_status moe_experts_forward_training(const moe_experts* ex, const void* x_dispatched, const uint32_t* offsets,
                                        int64_t rows, void* h, void* y_dispatched, void* cache_g, void* cache_u,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  moe_status st = check_stage_args(ex, x_dispatched, offsets, rows, y_dispatched, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if (workspace_bytes < moe_experts_forward_training_workspace_size(ex))
    return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_experts_forward_training_workspace_size()");
  if (rows > 0 && (h == nullptr || cache_g == nullptr || cache_u == nullptr))
    return fail(MOE_ERR_NULL, "h, cache_g and cache_u must be non-NULL");
  if (ex->dtype != MOE_F32 && (!aligned16(h) || !aligned16(cache_g) || !aligned16(cache_u)))
    return fail(MOE_ERR_ALIGNMENT, "h, cache_g and cache_u must be 16-byte aligned");
  if (rows == 0) return ok();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const moe::TcCache cache{cache_g, cache_u};
  if (ex->dtype == MOE_F32) {
    st = run_stage(ex, true, x_dispatched, nullptr, offsets, rows, h, workspace, s, &cache);
    if (st != MOE_OK) return st;
    st = run_stage(ex, false, h, nullptr, offsets, rows, y_dispatched, workspace, s);
    return st != MOE_OK ? st : ok();
  }
  // F16/BF16: the chained launch, its counters reset first.
  const size_t cnt_bytes = moe_experts_forward_training_workspace_size(ex);
  cudaError_t err = cudaMemsetAsync(workspace, 0, cnt_bytes, s);
  if (err != cudaSuccess) return cuda_fail(err, "counter reset");
  const char* why = nullptr;
  uint32_t* sched = static_cast<uint32_t*>(workspace);
  err = moe::launch_experts_tc_chain(ex->tc, ex->dtype, x_dispatched, nullptr, &cache, offsets, static_cast<int>(ex->E),
                                     rows, ex->H, ex->I, h, y_dispatched, sched, sched + moe::TC_SCHED_BYTES / 4,
                                     ex->num_sms, s, &why);
  if (err != cudaSuccess) return cuda_fail(err, "gate/up + down GEMM launch", why);
  return ok();
}

size_t moe_experts_backward_workspace_size(const moe_experts* ex, int64_t rows) {
  if (ex == nullptr || rows < 0) return 0;
  const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(ex->I);
  return backward_dh_bytes(ex, n) + 2 * align_up(n * dtype_size(ex->dtype) + 1, 256) + moe::TC_SCHED_BYTES;
}

moe_status moe_experts_backward(const moe_experts* ex, const void* x_dispatched, const uint32_t* offsets, int64_t rows,
                                const void* h, const void* cache_g, const void* cache_u, const void* dexpert,
                                void* dx_dispatched, float* dgate, float* dup, float* ddown, void* workspace,
                                size_t workspace_bytes, void* stream) {
  moe_status st = check_stage_args(ex, x_dispatched, offsets, rows, dx_dispatched, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if (dgate == nullptr || dup == nullptr || ddown == nullptr)
    return fail(MOE_ERR_NULL, "dgate, dup and ddown must be non-NULL");
  if (rows > 0 && (h == nullptr || cache_g == nullptr || cache_u == nullptr || dexpert == nullptr))
    return fail(MOE_ERR_NULL, "h, cache_g, cache_u and dexpert must be non-NULL");
  if (workspace_bytes < moe_experts_backward_workspace_size(ex, rows))
    return fail(MOE_ERR_WORKSPACE, "workspace smaller than moe_experts_backward_workspace_size()");
  const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(ex->I);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t dh_bytes = backward_dh_bytes(ex, n);
  const size_t d_bytes = align_up(n * dtype_size(ex->dtype) + 1, 256);
  moe::TrainBuffers b{x_dispatched, h, cache_g, cache_u, dexpert, ex->gate, ex->up, ex->down,
                      dh_bytes > 0 ? reinterpret_cast<float*>(ws) : nullptr, ws + dh_bytes, ws + dh_bytes + d_bytes,
                      dx_dispatched, dgate, dup, ddown};
  cudaError_t err;
  const char* why = nullptr;
  if (ex->dtype == MOE_F32 || rows == 0) {
    err = moe::launch_experts_backward(ex->dtype, b, offsets, static_cast<int>(ex->E), rows, ex->H, ex->I,
                                       static_cast<cudaStream_t>(stream));
  } else {
    uint32_t* sched = reinterpret_cast<uint32_t*>(ws + dh_bytes + 2 * d_bytes);
    err = moe::launch_experts_backward_tc(ex->dtype, b, offsets, static_cast<int>(ex->E), rows, ex->H, ex->I, sched,
                                          ex->num_sms, static_cast<cudaStream_t>(stream), &why);
  }
  if (err != cudaSuccess) return cuda_fail(err, "moe_experts_backward launch", why);
  return ok();
}

moe_status moe_device_status(uint32_t* code, int32_t clear) {
  if (code == nullptr) return fail(MOE_ERR_NULL, "code must be non-NULL");
  cudaError_t err = moe::read_device_status(code, clear != 0);
  if (err != cudaSuccess) return cuda_fail(err, "moe_device_status");
  return ok();
}

moe_status moe_selftest_bounded_wait(uint32_t limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 10u * 1000u * 1000u)
    return fail(MOE_ERR_SHAPE, "limit_us must be in 1 .. 10^7");
  cudaError_t err = moe::launch_bounded_wait_selftest(limit_us, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "moe_selftest_bounded_wait launch");
  return ok();
}

}  // extern "C"
