// Shared device helpers for the MoE kernels: dtype conversion, warp helpers,
// and thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor) and
// the 5th-generation tensor core (tcgen05.*) on sm_103a.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr unsigned FULL_MASK = 0xFFFFFFFFu;
constexpr uint32_t INVALID_ROW = 0xFFFFFFFFu;

// ---------------------------------------------------------------- dtype conversion

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// Round-to-nearest-even conversion from FP32.
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Backward of h = SiLU(g) * u for one element, given d = dL/dh (ruDNN user
// guide, section 12, cache.backward; the textbook derivative SiLU'(g) =
// s (1 + g (1 - s)), s = sigmoid(g)): dg = d * u * SiLU'(g), du = d * SiLU(g),
// in FP32.
__device__ __forceinline__ void silu_mul_backward(float d, float g, float u, float* dg, float* du) {
  const float s = 1.0f / (1.0f + expf(-g));
  const float silu = g * s;
  const float dsilu = s * (1.0f + g * (1.0f - s));
  *dg = d * u * dsilu;
  *du = d * silu;
}

// Two FP32 values packed as one 32-bit pair of 16-bit floats (low half first).
template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

inline size_t dtype_size(moe_dtype d) { return d == MOE_F32 ? 4 : 2; }
inline bool dtype_valid(int d) { return d == MOE_F32 || d == MOE_F16 || d == MOE_BF16; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------- time and status

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// First nonzero code wins; later timeouts do not overwrite it.
__device__ __forceinline__ void record_status(uint32_t* status, uint32_t code) {
  if (status != nullptr) atomicCAS(status, 0u, code);
}

// ---------------------------------------------------------------- dependent launches

// Wait until the kernel this one depends on (the previous kernel in the
// stream) has completed and its writes are visible. Kernels launched with
// programmatic stream serialization (launch_dependent below) may start before
// their predecessor finishes: they call this before reading anything it
// wrote or writing anything it reads. Returns at once otherwise.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the kernel launched after this one as a programmatic dependent start
// once every block of this grid has reached this point (or exited): its blocks
// then run their prologue while this grid finishes, and they still wait in
// grid_dependency_wait for this grid's completion before touching its data.
// Every block of this grid has started by then, so the dependent's blocks can
// never hold resources that one of this grid's blocks still needs.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- grouped-GEMM tile plan

// Tiles of a grouped GEMM: expert e owns ceil(count_e / bm) row tiles times
// n_tiles column tiles, numbered after all tiles of experts 0..e-1. Warp 0
// writes the exclusive prefix tile_start[0..E] (E+1 entries) into shared
// memory; the caller synchronises the block afterwards.
__device__ __forceinline__ void build_tile_prefix(const uint32_t* __restrict__ offsets, int E,
                                                  int bm, int n_tiles, uint32_t* tile_start) {
  const int lane = threadIdx.x & 31;
  uint32_t carry = 0;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    const uint32_t cnt = e < E ? offsets[e + 1] - offsets[e] : 0u;
    const uint32_t tiles = (cnt + bm - 1) / bm * static_cast<uint32_t>(n_tiles);
    uint32_t incl = tiles;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL_MASK, incl, off);
      if (lane >= off) incl += o;
    }
    if (e < E) tile_start[e] = carry + incl - tiles;
    carry += __shfl_sync(FULL_MASK, incl, 31);
  }
  if (lane == 0) tile_start[E] = carry;
}

struct TileCoord {
  int e;          // expert
  int m;          // row tile inside the expert
  int n;          // column tile
  uint32_t row0;  // first dispatched row of the tile
  int rows;       // valid rows in the tile (1..bm)
};

// Tile -> (expert, row tile, column tile). Row tiles vary fastest so that
// consecutive tiles share one weight tile (it is read from HBM once and then
// hit in L2). Requires tile < tile_start[E].
__device__ __forceinline__ TileCoord decode_tile(uint32_t tile, const uint32_t* tile_start, int E,
                                                 const uint32_t* __restrict__ offsets, int bm,
                                                 int n_tiles) {
  int lo = 0, hi = E;  // find the last e with tile_start[e] <= tile
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid;
  }
  TileCoord c;
  c.e = lo;
  const uint32_t local = tile - tile_start[lo];
  const uint32_t m_tiles = (tile_start[lo + 1] - tile_start[lo]) / static_cast<uint32_t>(n_tiles);
  c.n = static_cast<int>(local / m_tiles);
  c.m = static_cast<int>(local % m_tiles);
  const uint32_t o0 = offsets[lo], o1 = offsets[lo + 1];
  c.row0 = o0 + static_cast<uint32_t>(c.m) * bm;
  const uint32_t left = o1 - c.row0;
  c.rows = static_cast<int>(left < static_cast<uint32_t>(bm) ? left : static_cast<uint32_t>(bm));
  return c;
}

// ---------------------------------------------------------------- shared memory / mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte global -> shared copy without registers (cp.async); src_bytes < 16
// zero-fills the rest (0: nothing is read, the destination gets zeros).
__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "r"(src_bytes)
               : "memory");
}

// Arrive on the mbarrier once every cp.async this thread issued so far has
// landed; the arrival counts against the barrier's expected count.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity, for at most `limit_ns`. Returns
// false (and raises *abort, recording `code` in *status) when the time runs
// out, or false at once when another role has raised *abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, uint32_t* status,
                                                  uint32_t code, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        if (abort_flag != nullptr) *abort_flag = 1;
        record_status(status, code);
        return false;
      }
    }
  }
}

// Waits (bounded, like mbar_wait_bounded) until the device counter *ctr,
// read with acquire semantics at GPU scope, reaches `need`; then orders the
// data that the counter's writers stored (generic proxy) before this
// thread's later TMA reads of it (async proxy).
__device__ __forceinline__ bool counter_wait_bounded(const uint32_t* ctr, uint32_t need, volatile int* abort_flag,
                                                     uint32_t* status, uint32_t code, uint64_t limit_ns) {
  auto ready = [&]() {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    return v >= need;
  };
  bool ok = ready();
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; !ok; ++it) {
      __nanosleep(64);
      ok = ready();
      if (!ok && (it & 15u) == 0) {
        if (abort_flag != nullptr && *abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
          if (abort_flag != nullptr) *abort_flag = 1;
          record_status(status, code);
          return false;
        }
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// Raises the device counter *ctr by one with release semantics at GPU scope
// (the calling thread's earlier stores, and those it observed, become
// visible to an acquiring reader first).
__device__ __forceinline__ void counter_release_add(uint32_t* ctr) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
}

// Adds one to the device counter *ctr with acquire-release semantics at GPU
// scope and returns the value it held: stores the caller made (or observed)
// before the add are visible to whoever later reads the counter, and stores
// that earlier adders released are visible to the caller after it.
__device__ __forceinline__ uint32_t counter_acq_rel_add(uint32_t* ctr) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(ctr) : "memory");
  return old;
}

// Asynchronous prefetch of `bytes` of global memory into L2 (one bulk request,
// no registers, nothing to wait for). Address and size must be multiples of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- TMA (bulk tensor copies)

__device__ __forceinline__ void tma_prefetch_desc(const void* desc) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(desc) : "memory");
}

// 2-D tiled load global -> shared, completion counted on `bar` in bytes.
// c0 is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* desc, uint64_t* bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(desc), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// Row gather: four rows r0..r3 of a 2-D tensor map whose box is one row high,
// columns c0.. (the box width), landing as four consecutive box rows at
// smem_dst. The swizzle follows the shared-memory address, so a destination
// 512 bytes into a 1024-byte swizzle atom holds atom rows 4..7.
__device__ __forceinline__ void tma_gather4(void* smem_dst, const void* desc, uint64_t* bar, int c0, int r0,
                                            int r1, int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(desc), "r"(smem_u32(bar)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* smem_dst, const void* desc, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(desc), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Tensor store shared -> global of one box at (c0, c1, c2) of a 3-D map, in
// the issuing thread's current bulk async-group.
__device__ __forceinline__ void tma_store_3d(const void* desc, uint32_t smem_src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(desc),
               "r"(c0), "r"(c1), "r"(c2), "r"(smem_src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store of this thread has read its shared
// source (the buffer may be rewritten), or has completed (all).
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* desc, uint64_t* bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(desc), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05 (TMEM + UMMA)

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (F16 or BF16 inputs, FP32 accumulate).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive FP32 columns of this warp's 32 TMEM lanes (lane i of the warp
// reads TMEM lane base_lane + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes (64 16-bit elements of K), groups of 8
// rows 1024 bytes apart. Fields: start address >> 4 in bits 0-13, leading
// byte offset >> 4 in bits 16-29 (unused for swizzled K-major), stride byte
// offset >> 4 in bits 32-45, descriptor version 1 in bits 46-47, base offset
// 0 (tiles are 1024-byte aligned), swizzle mode 2 (128B) in bits 61-63.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// MN-major operand with 128-byte swizzle: atoms of 8 K-rows x 128 B (64
// 16-bit MN elements), as a TMA box {64 (MN, inner), rows (K)} lays them out;
// `lbo` is the byte distance between MN-adjacent atoms (the next 64 MN
// elements), `sbo` between K-adjacent atoms (the next 8 K-rows).
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor for tcgen05.mma kind::f16: FP32 accumulator (bits 4-5
// = 1), A and B format (bits 7-9 and 10-12: 0 = F16, 1 = BF16), both operands
// K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// The same with A (bit 15) and / or B (bit 16) MN-major.
__host__ __device__ constexpr uint32_t idesc_f16_major(bool bf16, int M, int N, bool a_mn, bool b_mn) {
  return idesc_f16(bf16, M, N) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16);
}

}  // namespace moe
