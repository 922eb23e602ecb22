/*
 * moe.h - C ABI of the GB300 (sm_103a) local Mixture-of-Experts forward chain.
 *
 * The chain (ruDNN user guide, section 3 "MoE workflow"):
 *
 *     logits [T,E] -> softmax/top-k routing -> compact per-expert dispatch
 *                  -> SwiGLU experts -> routing-weighted combine -> out [T,H]
 *
 * Conventions shared by every entry point
 *   - All pointers named "device" are CUDA device pointers on the current
 *     device; the caller allocates and owns every buffer, including the
 *     workspaces. The library allocates no device memory on any call below.
 *   - Tensors are dense and row-major (C order) with the shapes given.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Every call only enqueues work on that stream and returns; no
 *     call waits for the device. Results are ready when the stream is.
 *   - Every argument check runs on the host before anything is launched; a
 *     failed check returns its status and enqueues nothing. MOE_ERR_CUDA
 *     means a launch was rejected by the CUDA runtime (the message is in
 *     moe_last_error()).
 *   - Dtypes: MOE_F32, MOE_F16, MOE_BF16 (non-quantised floats, ruDNN user
 *     guide section 4). Arithmetic: routing in FP32; expert projections
 *     accumulate in FP32 (tensor cores for F16/BF16, FP32 FMA for F32, never
 *     TF32); combine accumulates in FP32.
 *   - Indices are uint32 (ruDNN user guide section 4: "indices use U32").
 *   - Thread safety: calls on different streams may run concurrently when
 *     their buffers do not overlap. A moe_experts handle is read-only after
 *     creation and may be shared.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { MOE_F32 = 0, MOE_F16 = 1, MOE_BF16 = 2 } moe_dtype;

/* Status codes: the C counterpart of MoeError (ruDNN user guide section 3:
 * "computation entry points return Result with MoeError for invalid shapes,
 * dtypes, or other arguments"). */
typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULL = 1,          /* a required pointer is NULL                          */
  MOE_ERR_SHAPE = 2,         /* a size is out of range or sizes disagree             */
  MOE_ERR_DTYPE = 3,         /* unknown dtype, or dtypes that must agree do not      */
  MOE_ERR_TOP_K = 4,         /* top_k outside 1 <= top_k <= E (section 4)            */
  MOE_ERR_ALIGNMENT = 5,     /* a pointer or row pitch is not 16-byte aligned        */
  MOE_ERR_WORKSPACE = 6,     /* workspace pointer NULL or smaller than required      */
  MOE_ERR_UNSUPPORTED = 7,   /* a valid request this build does not implement        */
  MOE_ERR_CUDA = 8,          /* the CUDA runtime rejected a launch or query          */
  MOE_ERR_DEVICE_CHECK = 9   /* a device-side wait ran out of time (see moe_device_status) */
} moe_status;

/* Opaque expert-weight handle (SwiGluExperts::new, ruDNN user guide section 3). */
typedef struct moe_experts moe_experts;

/* Human-readable name of a status code; never NULL. */
const char* moe_status_string(int status);

/* Detail of the last failed call on this host thread (empty if none). */
const char* moe_last_error(void);

/* ABI version of this library (major * 10000 + minor * 100 + patch): 1.1.0
 * adds moe_experts_forward_combine, moe_route_dispatch,
 * moe_route_sigmoid_grouped_dispatch and moe_permute_rows to 1.0.0; nothing
 * was removed or changed. */
int moe_version(void);

/*
 * moe_route - softmax/top-k routing (RoutingPlan, ruDNN user guide section 4
 * "Routing contract"; restated in the Japanese guide section 4 and the
 * ruDNN 0.1.5 User Guide section 4).
 *
 *   logits        device, [T, E] in `dtype`.
 *   T, E          1 <= E <= 1024, T >= 0 (T = 0 enqueues nothing).
 *   top_k         1 <= top_k <= E, else MOE_ERR_TOP_K.
 *   renormalize   nonzero: divide the selected weights by their sum.
 *   indices       device, [T, top_k] uint32 out: selected experts, slot 0 the
 *                 largest logit, ties to the lower expert id.
 *   weights       device, [T, top_k] out in `dtype`: FP32 softmax over all E
 *                 experts, gathered, optionally renormalized, then rounded to
 *                 `dtype` (round to nearest even).
 *   weights_fp32  device, [T, top_k] float out before that rounding, or NULL.
 *
 * A row holding a NaN or +inf, or only -inf, gets NaN weights (no uniform
 * fallback) and indices 0..top_k-1. Selection compares the logits
 * themselves (softmax is strictly increasing, so this is "softmax then
 * top-k" without ties added by exp rounding).
 */
moe_status moe_route(const void* logits, moe_dtype dtype, int64_t T, int64_t E, int32_t top_k,
                     int32_t renormalize, uint32_t* indices, void* weights, float* weights_fp32,
                     void* stream);

/*
 * moe_dispatch - compact per-expert token layout with no capacity dropping
 * (RoutingPlan::dispatch; ruDNN user guide section 5 "Expert weights and
 * dispatch": tokens are never dropped, a saved mapping restores token order).
 *
 *   indices       device, [T, top_k] uint32 (from moe_route or the caller).
 *   x             device, [T, H] in `dtype`, or NULL to skip x_dispatched.
 *   counts        device, [E] uint32 out: rows per expert.
 *   offsets       device, [E + 1] uint32 out: exclusive prefix of counts.
 *   row_src       device, [T * top_k] uint32 out: dispatched row r holds slot
 *                 row_src[r] = t * top_k + j.
 *   inv           device, [T * top_k] uint32 out: slot t * top_k + j sits in
 *                 dispatched row inv[t * top_k + j].
 *   x_dispatched  device, [T * top_k, H] out (row r = x[row_src[r] / top_k]),
 *                 or NULL. Needs x.
 *   workspace     device scratch of moe_dispatch_workspace_size(T, E, top_k)
 *                 bytes (256-byte aligned); contents need not be initialised.
 *
 * Order within an expert is ascending t * top_k + j, so the maps are the
 * same on every run (the pages leave that order free). An index >= E is not
 * dispatched: its inv entry is 0xFFFFFFFF, counts exclude it, and
 * moe_combine writes a NaN row for that token. No out-of-range access, no
 * host synchronisation.
 */
size_t moe_dispatch_workspace_size(int64_t T, int64_t E, int32_t top_k);
moe_status moe_dispatch(const uint32_t* indices, int64_t T, int64_t E, int32_t top_k,
                        const void* x, moe_dtype dtype, int64_t H, uint32_t* counts,
                        uint32_t* offsets, uint32_t* row_src, uint32_t* inv, void* x_dispatched,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_dispatch_noalloc - moe_dispatch without a workspace argument, for
 * callers that cannot allocate device memory when they dispatch: a plugin
 * that reaches the library through this C ABI from a host framework owning
 * every device allocation, or a serving loop whose memory budget is fixed at
 * start-up and may not grow afterwards. The pages have no counterpart; the
 * outputs are the same as moe_dispatch's, bit for bit.
 *
 * Arguments and outputs are those of moe_dispatch. The scratch instead lives
 * in a fixed 1 MiB (MOE_DISPATCH_NOALLOC_SCRATCH_BYTES) array inside the
 * library's device image; every GPU that loads the library holds it until the
 * process exits. Requests whose scratch, ceil(T*top_k/2048)*E*4 bytes, exceeds
 * it are rejected with MOE_ERR_SHAPE before anything is launched. No call
 * allocates or frees device memory. Every call looks up the array's device
 * address (cudaGetSymbolAddress) with the calling device current, so the
 * address stays right after a cudaDeviceReset; the first call on a device
 * also loads the library's device code there, so make it before any stream
 * capture. All calls on a device share
 * the array and it keeps the last call's contents (each call writes every
 * entry it reads, so nothing needs clearing): calls that may overlap on the
 * GPU, such as calls on different streams without ordering between them, race
 * on it and must not be issued.
 */
#define MOE_DISPATCH_NOALLOC_SCRATCH_BYTES (1u << 20)
moe_status moe_dispatch_noalloc(const uint32_t* indices, int64_t T, int64_t E, int32_t top_k,
                                const void* x, moe_dtype dtype, int64_t H, uint32_t* counts,
                                uint32_t* offsets, uint32_t* row_src, uint32_t* inv,
                                void* x_dispatched, void* stream);

/*
 * moe_route_dispatch - moe_route followed by moe_dispatch as one cooperative
 * launch (ruDNN user guide sections 4 "Routing contract" and 5 "Expert
 * weights and dispatch"): every output is the same, bit for bit, as those two
 * calls give. moe_forward runs this launch for its routing and dispatch.
 *
 *   logits, logits_dtype, T, E, top_k, renormalize, indices, weights,
 *   weights_fp32      as moe_route.
 *   x, x_dtype, H, counts, offsets, row_src, inv, x_dispatched
 *                     as moe_dispatch (x_dtype is x's dtype; x_dispatched
 *                     NULL writes the maps only).
 *   workspace         device scratch of moe_route_dispatch_workspace_size(T, E)
 *                     bytes (256-byte aligned); contents need not be
 *                     initialised (the call zeroes what it needs on the
 *                     stream).
 *
 * The blocks of the launch meet once at a grid-wide barrier (all of them are
 * resident: the launch is cooperative). Its wait is bounded (about one
 * second); a wait that runs out records 0x1B in the device status word
 * (moe_device_status) and the launch returns with its outputs incomplete.
 */
size_t moe_route_dispatch_workspace_size(int64_t T, int64_t E);
moe_status moe_route_dispatch(const void* logits, moe_dtype logits_dtype, int64_t T, int64_t E, int32_t top_k,
                              int32_t renormalize, uint32_t* indices, void* weights, float* weights_fp32,
                              const void* x, moe_dtype x_dtype, int64_t H, uint32_t* counts, uint32_t* offsets,
                              uint32_t* row_src, uint32_t* inv, void* x_dispatched, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * moe_permute_rows - move whole rows by an index: the reorders of the
 * expert-parallel exchange (the received rows into expert-major order, the
 * experts' outputs back into the received order); the exchange itself is the
 * caller's collective. Not on the pages: they run every expert on one device.
 *
 *   src           device, [src_rows, row_bytes] (rows contiguous).
 *   dst           device, [dst_rows, row_bytes]; must not overlap src.
 *   index         device, [rows] int64.
 *   scatter       zero: gather, dst[r] = src[index[r]] for r < rows
 *                 (rows <= dst_rows); a row whose index is outside
 *                 0..src_rows-1 is written as zeros. Nonzero: scatter,
 *                 dst[index[r]] = src[r] for r < rows (rows <= src_rows); a
 *                 row whose index is outside 0..dst_rows-1 is skipped, and
 *                 repeated indexes leave one of their rows (unspecified).
 *   row_bytes     > 0; 16-byte rows and pointers move as 16-byte vectors.
 *
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE (negative sizes, row_bytes < 1, rows
 * beyond the written or read side). Enqueued on the stream, no host sync.
 */
moe_status moe_permute_rows(const void* src, int64_t src_rows, void* dst, int64_t dst_rows, const int64_t* index,
                            int64_t rows, int64_t row_bytes, int32_t scatter, void* stream);

/*
 * moe_experts_create - validate and wrap bias-free SwiGLU expert weights
 * (SwiGluExperts::new; ruDNN user guide section 5: gate and up [E, I, H],
 * down [E, H, I], one float dtype, one device).
 *
 *   gate, up      device, [E, I, H] in `dtype`.
 *   down          device, [E, H, I] in `dtype`.
 *   E, H, I       1 <= E <= 1024; H, I >= 1. F16/BF16 need H and I to be
 *                 multiples of 8 (16-byte row pitch), else MOE_ERR_ALIGNMENT.
 *   out           receives the handle.
 *
 * The handle records the pointers (the caller keeps the weights alive and
 * unchanged while it is in use) and the prebuilt TMA descriptors. It is
 * reusable across batches and read-only; free it with moe_experts_destroy.
 * Device is the current device at creation.
 */
moe_status moe_experts_create(const void* gate, const void* up, const void* down, moe_dtype dtype,
                              int64_t E, int64_t H, int64_t I, moe_experts** out);
void moe_experts_destroy(moe_experts* experts);

/*
 * moe_experts_forward_dispatched - SwiGLU experts on dispatched rows
 * (SwiGluExperts::forward_dispatched; "tiny-llm deep dive 5: ops.rs",
 * section on SiLU: FFN(x) = W_down (SiLU(W_gate x) * W_up x)).
 *
 *   x_dispatched  device, [rows, H] in the experts' dtype (from moe_dispatch).
 *   offsets       device, [E + 1] uint32 (from moe_dispatch); expert e owns
 *                 rows offsets[e] .. offsets[e+1]-1; offsets[E] must equal
 *                 rows. The host never reads the counts.
 *   rows          T * top_k.
 *   y_dispatched  device, [rows, H] out in the experts' dtype:
 *                 y = W_down[e] h, h = SiLU(W_gate[e] x) * (W_up[e] x), FP32
 *                 accumulation, h rounded to the dtype before the down
 *                 projection.
 *   workspace     device scratch of
 *                 moe_experts_forward_dispatched_workspace_size(experts, rows)
 *                 bytes (holds h, the GEMMs' tile counter and one counter per
 *                 expert), 256-byte aligned.
 *
 * F16/BF16 run both GEMMs as one launch (after a reset of the counters):
 * tiles of the gate/up GEMM first, then tiles of the down GEMM, each of
 * which waits (bounded, about a second; on timeout the device status word
 * records 0x19) until every gate/up tile of its expert has stored its h
 * rows. The results are bit-identical to moe_experts_gate_up followed by
 * moe_experts_down.
 */
size_t moe_experts_forward_dispatched_workspace_size(const moe_experts* experts, int64_t rows);
moe_status moe_experts_forward_dispatched(const moe_experts* experts, const void* x_dispatched,
                                          const uint32_t* offsets, int64_t rows,
                                          void* y_dispatched, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * moe_experts_forward_combine - the experts and the weighted combine in one
 * launch: SwiGluExperts::forward_dispatched followed by
 * DispatchedTokens::combine (ruDNN user guide section 6), the combine run by
 * the down GEMM's epilogue warps ("PyTorch general ops", section "two ways
 * to write a contraction": the routing-weighted sum over a token's top_k
 * expert outputs is part of the expert contraction).
 *
 *   x_dispatched, offsets   as in moe_experts_forward_dispatched.
 *   inv           device, [T * top_k] uint32 (from moe_dispatch).
 *   weights       device, [T, top_k] in `weights_dtype` (from moe_route),
 *                 aligned to its element size.
 *   T, top_k      1 <= top_k <= min(E, 64); rows = T * top_k.
 *   out           device, [T, H] out in the experts' dtype, 16-byte aligned:
 *                 out[t] = sum over j = 0..top_k-1, in that order, of
 *                 w[t, j] * y[inv[t * top_k + j]], FP32 accumulation, then
 *                 rounded to the dtype, y being the expert outputs rounded to
 *                 the dtype. The bits equal moe_experts_forward_dispatched
 *                 followed by moe_combine.
 *   workspace     device scratch of
 *                 moe_experts_forward_combine_workspace_size(experts, T,
 *                 top_k) bytes (h, y_dispatched, the tile counter, one
 *                 counter per expert and the combine's counter), 256-byte
 *                 aligned.
 *
 * How: every epilogue warp of every down tile raises one done counter once
 * its y rows are stored; a CTA that has run out of tiles waits (bounded,
 * about a second: on timeout the device status word records 0x1A) until the
 * counter shows every down tile done, then its epilogue warps combine a
 * fixed stripe of the tokens, four tokens' slot rows in one stream of loads
 * per warp. It waits only on tiles already claimed by running CTAs, so it
 * cannot deadlock. The counters are reset on the stream first. F16/BF16
 * experts and top_k <= 64 only (else MOE_ERR_UNSUPPORTED; use
 * moe_experts_forward_dispatched and moe_combine). An inv entry >= rows
 * makes its token's row NaN, as in moe_combine.
 */
size_t moe_experts_forward_combine_workspace_size(const moe_experts* experts, int64_t T, int32_t top_k);
moe_status moe_experts_forward_combine(const moe_experts* experts, const void* x_dispatched,
                                       const uint32_t* offsets, const uint32_t* inv, const void* weights,
                                       moe_dtype weights_dtype, int64_t T, int32_t top_k, void* out,
                                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_experts_gate_up / moe_experts_down - the two grouped-GEMM stages of
 * moe_experts_forward_dispatched, for callers that want h or want to time or
 * schedule the stages apart. Same arguments and checks as above.
 *
 *   gate_up:  x_dispatched [rows, H] -> h [rows, I],
 *             h = SiLU(W_gate[e] x) * (W_up[e] x), FP32 accumulation, rounded
 *             to the experts' dtype.
 *   down:     h [rows, I] -> y_dispatched [rows, H], y = W_down[e] h.
 *   workspace at least 256 bytes, 256-byte aligned (the tensor-core kernels'
 *             tile counter, reset on the stream by each call); two calls
 *             that may run at the same time need separate workspaces.
 */
moe_status moe_experts_gate_up(const moe_experts* experts, const void* x_dispatched,
                               const uint32_t* offsets, int64_t rows, void* h, void* workspace,
                               size_t workspace_bytes, void* stream);
moe_status moe_experts_down(const moe_experts* experts, const void* h, const uint32_t* offsets,
                            int64_t rows, void* y_dispatched, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * moe_experts_gate_up_gather - the gate/up stage reading each dispatched row
 * straight from x: row r is x[row_src[r] / top_k] (row_src from
 * moe_dispatch), so no x_dispatched copy is needed. This is the stage
 * moe_forward runs; the pages have no separate entry for it (their split API
 * materialises x_dispatched). h is bit-identical to moe_experts_gate_up on
 * the x_dispatched that moe_dispatch would write.
 *
 *   x         device, [T, H] in the experts' dtype (16-byte aligned for F16/BF16).
 *   row_src   device, [rows] uint32 from moe_dispatch; an entry >= T * top_k
 *             reads as a zero row.
 *   top_k     >= 1; rows <= T * top_k.
 *   offsets, rows, h, workspace   as in moe_experts_gate_up.
 */
moe_status moe_experts_gate_up_gather(const moe_experts* experts, const void* x, int64_t T,
                                      const uint32_t* row_src, int32_t top_k, const uint32_t* offsets,
                                      int64_t rows, void* h, void* workspace, size_t workspace_bytes,
                                      void* stream);

/*
 * moe_combine - restore token order and take the routing-weighted sum
 * (DispatchedTokens::combine; ruDNN user guide section 6: combine uses the
 * dispatch mapping to restore token order and merges the expert outputs with
 * the routing weights).
 *
 *   y_dispatched  device, [T * top_k, H] in `dtype`.
 *   inv           device, [T * top_k] uint32 (from moe_dispatch).
 *   weights       device, [T, top_k] in `weights_dtype` (from moe_route).
 *   out           device, [T, H] out in `dtype`:
 *                 out[t] = sum over j = 0..top_k-1, in that order, of
 *                 w[t, j] * y[inv[t * top_k + j]], FP32 accumulation, then
 *                 rounded to `dtype`. Deterministic: no atomics.
 */
moe_status moe_combine(const void* y_dispatched, moe_dtype dtype, const uint32_t* inv,
                       const void* weights, moe_dtype weights_dtype, int64_t T, int32_t top_k,
                       int64_t H, void* out, void* stream);

/*
 * moe_forward - the whole local chain in one call (SwiGluExperts::forward;
 * ruDNN user guide section 6): route, dispatch, SwiGLU experts, combine.
 *
 *   experts       handle from moe_experts_create (its dtype is x's and out's).
 *   x             device, [T, H] in the experts' dtype.
 *   logits        device, [T, E] in `logits_dtype` (E from the handle).
 *   top_k, renormalize   as in moe_route.
 *   out           device, [T, H] out in the experts' dtype.
 *   indices_opt   device [T, top_k] uint32 out, or NULL (kept in workspace).
 *   weights_opt   device [T, top_k] out in `logits_dtype`, or NULL.
 *   workspace     device scratch of moe_forward_workspace_size(experts, T,
 *                 top_k) bytes, 256-byte aligned, uninitialised is fine.
 *
 * Same numerics as calling moe_route, moe_dispatch,
 * moe_experts_forward_dispatched and moe_combine in turn: the outputs are
 * bit-identical to that sequence. F16/BF16 run the two expert GEMMs as one
 * launch (as moe_experts_forward_dispatched does; the dispatch zeroes its
 * counters), then the combine as its own launch (measured faster than the
 * combine inside the experts' launch, moe_experts_forward_combine). For
 * decode-sized batches (T * top_k <= 8 * E) it dispatches the maps only and
 * the gate/up tiles gather x rows through row_src (as
 * moe_experts_gate_up_gather), so x_dispatched is never written.
 */
size_t moe_forward_workspace_size(const moe_experts* experts, int64_t T, int32_t top_k);
moe_status moe_forward(const moe_experts* experts, const void* x, const void* logits,
                       moe_dtype logits_dtype, int64_t T, int32_t top_k, int32_t renormalize,
                       void* out, uint32_t* indices_opt, void* weights_opt, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * moe_forward_host - moe_forward on host buffers: the inputs are copied from
 * host memory into device staging in the workspace, the chain runs, and out
 * is copied back to host memory. Every step is enqueued on `stream` (one
 * cudaMemcpyAsync per copy, then the kernels); nothing synchronises the host.
 *
 *   x_host       host, [T, H] in the experts' dtype.
 *   logits_host  host, [T, E] in `logits_dtype`.
 *   out_host     host, [T, H] out in the experts' dtype.
 *   indices_opt, weights_opt   device outputs as in moe_forward, or NULL.
 *   workspace    device scratch of moe_forward_host_workspace_size(experts,
 *                T, top_k, logits_dtype) bytes, 256-byte aligned.
 *
 * Same outputs as moe_forward on device copies of x and logits (bit for bit).
 * With page-locked host buffers the copies are asynchronous: a caller that
 * runs consecutive batches on two streams with two workspaces overlaps one
 * batch's copies with the other's kernels. Pageable host memory works, but
 * each copy then completes before the call returns. The host buffers stay
 * owned by the caller; they must not be changed (x_host, logits_host) or read
 * (out_host) until the stream has passed the call's work.
 */
size_t moe_forward_host_workspace_size(const moe_experts* experts, int64_t T, int32_t top_k,
                                       moe_dtype logits_dtype);
moe_status moe_forward_host(const moe_experts* experts, const void* x_host, const void* logits_host,
                            moe_dtype logits_dtype, int64_t T, int32_t top_k, int32_t renormalize,
                            void* out_host, uint32_t* indices_opt, void* weights_opt, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * moe_group_routing_options - GroupRoutingOptions of the group-limited
 * sigmoid routing (ruDNN user guide, section 10).
 *
 *   top_k            1..64, at most selected_groups * (E / groups).
 *   groups           1..128 and divides E.
 *   selected_groups  1..groups: groups whose experts may be chosen.
 *   group_top_two    nonzero: a group scores the sum of its two largest
 *                    corrected scores (needs E / groups >= 2); zero: its
 *                    largest corrected score.
 *   renormalize      nonzero: divide the chosen weights by their sum.
 *   scale            finite and > 0: multiplies the weights last.
 */
typedef struct {
  int32_t top_k;
  int32_t groups;
  int32_t selected_groups;
  int32_t group_top_two;
  int32_t renormalize;
  float scale;
} moe_group_routing_options;

/*
 * moe_route_sigmoid_grouped - group-limited, bias-corrected sigmoid routing
 * (route_sigmoid_grouped, ruDNN user guide section 10; the group steps
 * follow the DeepSeek-style routing of "PyTorch general ops").
 *
 *   logits        device, [T, E] in `dtype` (MOE_F32, MOE_F16, MOE_BF16),
 *                 1 <= E <= 1024, T >= 0 (T = 0 enqueues nothing).
 *   bias          device, [E] float (FP32), or NULL for no correction; it
 *                 steers the selection only. 4-byte aligned.
 *   options       host pointer, read during the call only.
 *   indices       device, [T, top_k] uint32 out: slot 0 the largest
 *                 corrected score; ties to the lower id (groups too).
 *   weights       device, [T, top_k] out in `dtype`: the uncorrected sigmoid
 *                 scores of the chosen experts, optionally renormalized,
 *                 times scale, rounded to `dtype` (round to nearest even).
 *   weights_fp32  device, [T, top_k] float out before that rounding, or NULL.
 *
 * Scores are FP32: s = 1 / (1 + exp(-l)), c = s + bias. A row with a NaN
 * logit (or any NaN bias) gets NaN weights and indices 0..top_k-1. A group
 * whose two largest corrected scores are +inf and -inf has a NaN score and
 * ranks below every other group. Errors: MOE_ERR_TOP_K for top_k outside
 * 1..64 or above the selected groups' experts, MOE_ERR_SHAPE for any other
 * option or size out of range, MOE_ERR_DTYPE, MOE_ERR_NULL, MOE_ERR_ALIGNMENT.
 */
moe_status moe_route_sigmoid_grouped(const void* logits, moe_dtype dtype, int64_t T, int64_t E,
                                     const float* bias, const moe_group_routing_options* options,
                                     uint32_t* indices, void* weights, float* weights_fp32, void* stream);

/*
 * moe_route_sigmoid_grouped_dispatch - moe_route_sigmoid_grouped followed by
 * moe_dispatch as one cooperative launch, as moe_route_dispatch is for the
 * softmax routing: every output is the same, bit for bit, as those two calls
 * give. Routing arguments as moe_route_sigmoid_grouped; x, x_dtype, H, the
 * maps and x_dispatched as moe_dispatch; the workspace is
 * moe_route_dispatch_workspace_size(T, E) bytes (256-byte aligned, contents
 * need not be initialised). The grid barrier's wait is bounded as in
 * moe_route_dispatch (status 0x1B).
 */
moe_status moe_route_sigmoid_grouped_dispatch(const void* logits, moe_dtype logits_dtype, int64_t T, int64_t E,
                                              const float* bias, const moe_group_routing_options* options,
                                              uint32_t* indices, void* weights, float* weights_fp32, const void* x,
                                              moe_dtype x_dtype, int64_t H, uint32_t* counts, uint32_t* offsets,
                                              uint32_t* row_src, uint32_t* inv, void* x_dispatched, void* workspace,
                                              size_t workspace_bytes, void* stream);

/*
 * moe_forward_sigmoid_grouped - the whole local chain with grouped sigmoid
 * routing (SwiGluExperts::forward_sigmoid_grouped, ruDNN user guide section
 * 10): the grouped routing and the dispatch (one launch, as
 * moe_route_sigmoid_grouped_dispatch), then SwiGLU experts and combine
 * exactly as moe_forward does. Arguments as in moe_forward, with `bias` and
 * `options` as in moe_route_sigmoid_grouped; the workspace is
 * moe_forward_workspace_size(experts, T, options->top_k) bytes.
 */
moe_status moe_forward_sigmoid_grouped(const moe_experts* experts, const void* x, const void* logits,
                                       moe_dtype logits_dtype, int64_t T, const float* bias,
                                       const moe_group_routing_options* options, void* out,
                                       uint32_t* indices_opt, void* weights_opt, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * First-order training (ruDNN user guide, section 12). The backward runs in
 * the order the guide gives: combine_backward -> experts backward (the
 * forward cache's backward) -> dispatch_backward, and the FP32 dweights go
 * to moe_router_backward for the logits gradient.
 * ---------------------------------------------------------------------- */

typedef enum { MOE_ROUTER_SOFTMAX = 0, MOE_ROUTER_SIGMOID = 1 } moe_router_scoring;
typedef enum { MOE_INDEX_U32 = 0, MOE_INDEX_I32 = 1, MOE_INDEX_I64 = 2 } moe_index_type;

/* RouterWeightOptions: scoring, renormalize over the selected slots, and a
 * finite positive scale applied last. */
typedef struct {
  int32_t scoring;      /* moe_router_scoring */
  int32_t renormalize;  /* nonzero: divide by the sum over the slots */
  float scale;
} moe_router_weight_options;

/*
 * moe_router_weights - selected_router_weights: FP32 weights of a fixed
 * selection. Softmax: the FP32 softmax over all E experts (as moe_route
 * computes it) at each selected index; sigmoid: 1 / (1 + exp(-l)) of each
 * selected logit. Then optional renormalize (slot-ordered FP32 sum), then
 * times scale.
 *
 *   logits    device [T, E] in `dtype` (1 <= E <= 1024).
 *   indices   device [T, top_k] in `index_type` (uint32, int32 or int64),
 *             1 <= top_k <= min(E, 64). Repeated indices gather; any index
 *             outside 0..E-1 makes the token's whole row NaN (no out-of-range
 *             access, no host synchronisation).
 *   weights   device [T, top_k] float out.
 */
moe_status moe_router_weights(const void* logits, moe_dtype dtype, int64_t T, int64_t E, const void* indices,
                              moe_index_type index_type, int32_t top_k, const moe_router_weight_options* options,
                              float* weights, void* stream);

/*
 * moe_router_backward - selected_router_backward: dlogits [T, E] in the
 * logits dtype, the gradient of the moe_router_weights output (given as
 * FP32 grad_weights [T, top_k]) with respect to the logits, for the fixed
 * selection (the top-k itself, group choice and correction bias are not
 * differentiated). Every entry of dlogits is written. Same checks as
 * moe_router_weights; an invalid index makes the row of dlogits NaN.
 */
moe_status moe_router_backward(const void* logits, moe_dtype dtype, int64_t T, int64_t E, const void* indices,
                               moe_index_type index_type, int32_t top_k, const moe_router_weight_options* options,
                               const float* grad_weights, void* dlogits, void* stream);

/*
 * moe_experts_forward_training - forward_dispatched_training: the experts'
 * forward that also keeps the cache the backward needs.
 *
 *   x_dispatched, offsets, rows   as in moe_experts_forward_dispatched.
 *   h             device [rows, I] out: SiLU(g) * u in the dtype.
 *   y_dispatched  device [rows, H] out.
 *   cache_g, cache_u  device [rows, I] out: the pre-activations g = W_gate x
 *                 and u = W_up x, rounded to the dtype.
 *   workspace     device scratch of
 *                 moe_experts_forward_training_workspace_size(experts) bytes
 *                 (the GEMMs' counters), 256-byte aligned.
 * y_dispatched and h are bit-identical to moe_experts_forward_dispatched's
 * (F16/BF16: the same chained launch, whose gate/up tiles also store g, u).
 */
size_t moe_experts_forward_training_workspace_size(const moe_experts* experts);
moe_status moe_experts_forward_training(const moe_experts* experts, const void* x_dispatched,
                                        const uint32_t* offsets, int64_t rows, void* h, void* y_dispatched,
                                        void* cache_g, void* cache_u, void* workspace, size_t workspace_bytes,
                                        void* stream);

/*
 * moe_combine_backward - combine_backward: for each token t and slot j with
 * r = inv[t * top_k + j]: dexpert[r] = w[t, j] * grad_out[t] (rounded to the
 * dtype) and dweights[t, j] = <grad_out[t], y[r]> (FP32). A slot whose inv
 * entry is >= T * top_k gets a NaN dweight and writes no dexpert row;
 * dexpert rows no slot points at are not written.
 *
 *   y_dispatched  device [T * top_k, H] in `dtype` (the forward's expert output).
 *   inv, row_src  device [T * top_k] uint32, the two maps of moe_dispatch
 *                 (slot -> row and row -> slot). The work runs in row order;
 *                 a row r counts only when inv[row_src[r]] == r, so the
 *                 entries of row_src past the dispatched rows may hold
 *                 anything.
 *   weights       device [T, top_k] in `weights_dtype` (the forward's weights).
 *   grad_out      device [T, H] in `dtype`.
 *   dexpert       device [T * top_k, H] out in `dtype`.
 *   dweights      device [T, top_k] float out.
 */
moe_status moe_combine_backward(const void* y_dispatched, moe_dtype dtype, const uint32_t* inv,
                                const uint32_t* row_src, const void* weights, moe_dtype weights_dtype,
                                const void* grad_out, int64_t T, int32_t top_k, int64_t H, void* dexpert,
                                float* dweights, void* stream);

/*
 * moe_experts_backward - the forward cache's backward: from dexpert [rows, H]
 * (dy), the dispatched input gradient dx_dispatched [rows, H] (dtype) and the
 * FP32 weight gradients dgate, dup [E, I, H] and ddown [E, H, I] (every
 * entry written; experts without rows get zeros):
 *   dh = W_down^T dy; dg = dh * u * SiLU'(g); du = dh * SiLU(g);
 *   dx = W_gate^T dg + W_up^T du; ddown = dy h^T; dgate = dg x^T; dup = du x^T.
 *   workspace  moe_experts_backward_workspace_size(experts, rows) bytes,
 *              256-byte aligned (dg and du in the dtype; F32 experts also
 *              keep dh there in FP32, F16/BF16 experts turn dh into dg and du
 *              inside the dgrad GEMM).
 */
size_t moe_experts_backward_workspace_size(const moe_experts* experts, int64_t rows);
moe_status moe_experts_backward(const moe_experts* experts, const void* x_dispatched, const uint32_t* offsets,
                                int64_t rows, const void* h, const void* cache_g, const void* cache_u,
                                const void* dexpert, void* dx_dispatched, float* dgate, float* dup, float* ddown,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_dispatch_backward - dispatch_backward: dx[t] = sum over slots j of
 * dinput[inv[t * top_k + j]], added in slot order in FP32 and rounded to the
 * dtype; the routing weight is not applied again. A token with an inv entry
 * >= T * top_k gets a NaN row.
 */
moe_status moe_dispatch_backward(const void* dinput, moe_dtype dtype, const uint32_t* inv, int64_t T, int32_t top_k,
                                 int64_t H, void* dx, void* stream);

/*
 * moe_device_status - read (and clear, if `clear` is nonzero) the device
 * status word. The expert GEMM kernels bound every pipeline wait (about one
 * second); a wait that runs out stops its kernel's remaining work, lets the
 * copies and MMAs already issued finish, frees its tensor memory, returns,
 * and records a code here instead of hanging the GPU. Codes (first one
 * wins): 0x11 producer waiting for a free stage, 0x12 MMA waiting for a
 * loaded stage, 0x13 MMA waiting for a drained accumulator, 0x14 epilogue
 * waiting for a finished accumulator, 0x15 / 0x16 teardown drains, 0x17 a
 * wait on the shared-memory tile ring of the tile scheduler, 0x18 a gather
 * loader waiting for a free stage, 0x19 a down tile of the chained gate/up +
 * down launch waiting for its expert's h rows, 0x1A the combine of
 * moe_experts_forward_combine waiting for the last down tile, 0x1B the grid
 * barrier of moe_route_dispatch and moe_route_sigmoid_grouped_dispatch (and
 * of the forward calls' routing), 0x100
 * moe_selftest_bounded_wait. Synchronises the current device; *code = 0 when
 * no wait has timed out.
 */
moe_status moe_device_status(uint32_t* code, int32_t clear);

/*
 * moe_selftest_bounded_wait - launch one thread that waits on an mbarrier
 * nothing ever arrives on, with a limit of `limit_us` microseconds
 * (1 .. 10^7). The wait gives up, records 0x100 in the device status word
 * and the kernel returns; the CUDA context stays usable. Exercises the same
 * bounded-wait routine the expert GEMMs use.
 */
moe_status moe_selftest_bounded_wait(uint32_t limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
