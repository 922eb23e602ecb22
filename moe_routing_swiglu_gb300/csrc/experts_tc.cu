// K3 / K4: F16/BF16 SwiGLU experts as grouped GEMMs on the sm_103a tensor
// cores (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// Per dispatched row r of expert e ("tiny-llm deep dive 5: ops.rs", section
// on SiLU, FFN(x) = W_down (SiLU(W_gate x) * W_up x); shapes from the ruDNN
// user guide, section 5):
//   K3  acc = x_r [gate[e]; up[e]]^T      (K = H), epilogue h = SiLU(g) * u
//   K4  acc = h_r down[e]^T               (K = I), epilogue y = acc
// The SiLU-and-multiply is fused into K3's epilogue, so the gate and up
// projections never reach HBM ("PyTorch general ops", section on RMSNorm
// and SiLU x Mul).
//
// One persistent CTA per SM, 192 threads in three roles:
//   warp 0 lane 0   TMA producer: A tile (128 rows x 64 K) + B tile (256 rows x 64 K)
//                   per stage, 4 stages of 48 KB, 128-byte swizzle.
//   warp 1 lane 0   MMA issuer: 4 x tcgen05.mma (M=128, N=256, K=16) per stage into
//                   one of two 256-column TMEM accumulators; also allocates TMEM.
//   warps 2..5      epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//                   lanes 32*(w%4)..), FP32 math, rounding, masked global stores.
// Tiles: for K3 a tile is 128 rows x (128 gate + 128 up) columns, so gate and
// up columns of the same i meet in one accumulator; for K4 it is 128 rows x
// 256 output columns. The tile plan comes from the device offsets (the host
// never learns per-expert counts); row tiles vary fastest so CTAs running at
// the same time share each weight tile through L2.
//
// Every mbarrier wait is bounded (about a second). A wait that runs out
// records a code in the device status word, raises the CTA's abort flag so
// the other roles stop, drains the copies and MMAs already issued, frees
// TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

// Device status word (see moe_device_status in moe.h).
__device__ uint32_t g_moe_device_status = 0;

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int UMMA_K = 16;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BYTES = BN * BK * 2;             // 32 KB
constexpr uint32_t STAGE_TX = A_BYTES + B_BYTES;  // bytes landing per stage
constexpr uint32_t TMEM_COLS = 2 * BN;            // two accumulators
constexpr int NUM_THREADS = 192;
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

constexpr int SMEM_A = 0;
constexpr int SMEM_B = SMEM_A + STAGES * A_BYTES;
constexpr int SMEM_BAR = SMEM_B + STAGES * B_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr int SMEM_MISC = SMEM_BAR + 128;
constexpr int SMEM_TILES = SMEM_MISC + 16;
constexpr int SMEM_BYTES = 1024 + SMEM_TILES + 4 * (ROUTE_MAX_E + 1);
static_assert(NUM_BARS * 8 <= 128, "barrier area");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// Status codes recorded by a wait that timed out.
constexpr uint32_t ST_PRODUCER_EMPTY = 0x11;
constexpr uint32_t ST_MMA_FULL = 0x12;
constexpr uint32_t ST_MMA_TMEM_EMPTY = 0x13;
constexpr uint32_t ST_EPI_TMEM_FULL = 0x14;
constexpr uint32_t ST_MMA_DRAIN = 0x15;
constexpr uint32_t ST_PRODUCER_DRAIN = 0x16;
constexpr uint32_t ST_SELFTEST = 0x100;

struct TcArgs {
  const uint32_t* offsets;  // [E + 1]
  void* out;                // [rows, n_out]: h for K3, y for K4
  int E;
  int n_tiles;              // column tiles per expert
  int k_blocks;             // ceil(K / BK)
  int n_out;                // output columns (I for K3, H for K4)
  uint32_t rows_total;      // rows of the activation and output matrices
  uint32_t tile_cap;        // host bound on the tile count
  uint32_t* status;
};

template <typename T>
__device__ __forceinline__ void store_row_chunk(T* dst, int64_t col0, int64_t n_out,
                                                const uint32_t (&packed)[16]) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    if (col0 + v * 8 + 8 <= n_out) {
      *reinterpret_cast<uint4*>(dst + col0 + v * 8) =
          make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
    }
  }
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + __expf(-g)); }

template <typename T, bool GATE_UP>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    experts_tc_kernel(const __grid_constant__ CUtensorMap tm_a,
                      const __grid_constant__ CUtensorMap tm_b0,
                      const __grid_constant__ CUtensorMap tm_b1, const TcArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem + SMEM_A;
  uint8_t* sB = smem + SMEM_B;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SMEM_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + SMEM_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SMEM_MISC + 4);
  uint32_t* tile_start = reinterpret_cast<uint32_t*>(smem + SMEM_TILES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b0);
    tma_prefetch_desc(&tm_b1);
  }
  __syncwarp();
  if (warp == 0) build_tile_prefix(args.offsets, args.E, BM, args.n_tiles, tile_start);
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // The cap keeps a corrupt offsets array from producing an endless tile loop.
  const uint32_t total = min(tile_start[args.E], args.tile_cap);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (uint32_t tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileCoord tc = decode_tile(tile, tile_start, args.E, args.offsets, BM, args.n_tiles);
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status,
                                 ST_PRODUCER_EMPTY, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = sA + stage * A_BYTES;
          uint8_t* b_dst = sB + stage * B_BYTES;
          mbar_arrive_expect_tx(&full[stage], STAGE_TX);
          tma_load_2d(a_dst, &tm_a, &full[stage], kb * BK, static_cast<int>(tc.row0));
          if (GATE_UP) {
            tma_load_3d(b_dst, &tm_b0, &full[stage], kb * BK, tc.n * (BN / 2), tc.e);
            tma_load_3d(b_dst + B_BYTES / 2, &tm_b1, &full[stage], kb * BK, tc.n * (BN / 2), tc.e);
          } else {
            tma_load_3d(b_dst, &tm_b0, &full[stage], kb * BK, tc.n * BN, tc.e);
            tma_load_3d(b_dst + B_BYTES / 2, &tm_b0, &full[stage], kb * BK, tc.n * BN + BN / 2, tc.e);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the block can exit.
        const uint32_t n_back = issued < STAGES ? issued : STAGES;
        for (uint32_t i = 1; i <= n_back; ++i) {
          const uint32_t n = issued - i;
          mbar_wait_bounded(&full[n % STAGES], (n / STAGES) & 1u, nullptr, args.status,
                            ST_PRODUCER_DRAIN, WAIT_LIMIT_NS);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
      constexpr uint32_t IDESC = idesc_f16(kBF16, BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (uint32_t tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, args.status,
                               ST_MMA_TMEM_EMPTY, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.status, ST_MMA_FULL,
                                 WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_addr = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            umma_f16(d_tmem, sdesc_kmajor_sw128(a_addr + k * UMMA_K * 2),
                     sdesc_kmajor_sw128(b_addr + k * UMMA_K * 2), IDESC,
                     (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Every MMA issued above completes before TMEM is released.
      umma_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr, args.status, ST_MMA_DRAIN, WAIT_LIMIT_NS);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (uint32_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileCoord tc = decode_tile(tile, tile_start, args.E, args.offsets, BM, args.n_tiles);
      const bool ready = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, args.status,
                                           ST_EPI_TMEM_FULL, WAIT_LIMIT_NS);
      // The tcgen05.ld below is warp-collective: the whole warp goes on or stops.
      if (!__all_sync(FULL_MASK, ready)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      const bool row_ok = r < tc.rows && tc.row0 + static_cast<uint32_t>(r) < args.rows_total;
      T* dst = static_cast<T*>(args.out) + (static_cast<int64_t>(tc.row0) + r) * args.n_out;
      if (GATE_UP) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(t_row + c * 32, g);
          tmem_ld_32x32b_x32(t_row + BN / 2 + c * 32, u);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float h0 = silu_f32(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
            const float h1 = silu_f32(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
            packed[i] = pack2<T>(h0, h1);
          }
          if (row_ok) store_row_chunk<T>(dst, static_cast<int64_t>(tc.n) * (BN / 2) + c * 32, args.n_out, packed);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t d[32];
          tmem_ld_32x32b_x32(t_row + c * 32, d);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            packed[i] = pack2<T>(__uint_as_float(d[2 * i]), __uint_as_float(d[2 * i + 1]));
          }
          if (row_ok) store_row_chunk<T>(dst, static_cast<int64_t>(tc.n) * BN + c * 32, args.n_out, packed);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
    // Nothing ever arrives on this barrier: the wait has to give up, record
    // its code and return.
    mbar_wait_bounded(&bar, 0, nullptr, &g_moe_device_status, ST_SELFTEST, limit_ns);
  }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  });
  return fn;
}

CUtensorMapDataType tmap_dtype(moe_dtype d) {
  return d == MOE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// [outer, inner] row-major 16-bit matrix, box 64 (inner) x 128 (outer).
bool encode_2d(CUtensorMap* m, moe_dtype dt, const void* ptr, uint64_t inner, uint64_t outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {BK, BM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, tmap_dtype(dt), 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [E, rows, inner] row-major 16-bit tensor, box 64 x 128 x 1.
bool encode_3d(CUtensorMap* m, moe_dtype dt, const void* ptr, uint64_t inner, uint64_t rows,
               uint64_t E) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {inner, rows, E};
  const cuuint64_t strides[2] = {inner * 2, rows * inner * 2};
  const cuuint32_t box[3] = {BK, BN / 2, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, tmap_dtype(dt), 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t tile_bound(int64_t rows, int E, int64_t n_tiles) {
  const int64_t m_tiles = rows / BM + (rows < E ? rows : E);
  return m_tiles * n_tiles;
}

template <typename T, bool GATE_UP>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                       const TcArgs& args, int64_t rows, int num_sms, cudaStream_t stream) {
  auto kern = experts_tc_kernel<T, GATE_UP>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (err != cudaSuccess) return err;
  const int64_t bound = tile_bound(rows, args.E, args.n_tiles);
  const int grid = static_cast<int>(bound < num_sms ? bound : num_sms);
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(a, b0, b1, args);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_stage(const TcWeights& w, moe_dtype dtype, bool gate_up, const void* a,
                         const uint32_t* offsets, int E, int64_t rows, int64_t H, int64_t I,
                         void* out, int num_sms, cudaStream_t stream, const char** why) {
  uint32_t* status = nullptr;
  cudaError_t err = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_moe_device_status);
  if (err != cudaSuccess) return err;
  const int64_t K = gate_up ? H : I;
  const int64_t n_out = gate_up ? I : H;
  CUtensorMap ta;
  if (!encode_2d(&ta, dtype, a, static_cast<uint64_t>(K), static_cast<uint64_t>(rows))) {
    *why = "cuTensorMapEncodeTiled rejected the activation tensor map";
    return cudaErrorInvalidValue;
  }
  const int nt = static_cast<int>(gate_up ? (I + BN / 2 - 1) / (BN / 2) : (H + BN - 1) / BN);
  TcArgs args{offsets, out, E, nt, static_cast<int>((K + BK - 1) / BK), static_cast<int>(n_out),
              static_cast<uint32_t>(rows), static_cast<uint32_t>(tile_bound(rows, E, nt)), status};
  if (gate_up) return launch_one<T, true>(ta, w.gate, w.up, args, rows, num_sms, stream);
  return launch_one<T, false>(ta, w.down, w.down, args, rows, num_sms, stream);
}

}  // namespace

bool tc_encode_weights(const void* gate, const void* up, const void* down, moe_dtype dtype,
                       int64_t E, int64_t H, int64_t I, TcWeights* out, const char** why) {
  if (encode_fn() == nullptr) {
    *why = "the CUDA driver does not provide cuTensorMapEncodeTiled";
    return false;
  }
  if (!encode_3d(&out->gate, dtype, gate, H, I, E) || !encode_3d(&out->up, dtype, up, H, I, E) ||
      !encode_3d(&out->down, dtype, down, I, H, E)) {
    *why = "cuTensorMapEncodeTiled rejected an expert weight tensor map";
    return false;
  }
  return true;
}

cudaError_t launch_experts_tc(const TcWeights& w, moe_dtype dtype, bool gate_up, const void* a,
                              const uint32_t* offsets, int E, int64_t rows, int64_t H, int64_t I,
                              void* out, int num_sms, cudaStream_t stream, const char** why) {
  if (rows == 0) return cudaSuccess;
  if (dtype == MOE_BF16)
    return launch_stage<__nv_bfloat16>(w, dtype, gate_up, a, offsets, E, rows, H, I, out, num_sms, stream, why);
  return launch_stage<__half>(w, dtype, gate_up, a, offsets, E, rows, H, I, out, num_sms, stream, why);
}

cudaError_t read_device_status(uint32_t* code, bool clear) {
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return err;
  err = cudaMemcpyFromSymbol(code, g_moe_device_status, sizeof(uint32_t));
  if (err != cudaSuccess || !clear) return err;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_moe_device_status, &zero, sizeof(uint32_t));
}

cudaError_t launch_bounded_wait_selftest(uint32_t limit_us, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(limit_us) * 1000ull);
  return cudaGetLastError();
}

}  // namespace moe
