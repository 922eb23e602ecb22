// Backward grouped GEMMs of the SwiGLU experts on the tensor cores (F16/BF16):
// tcgen05.mma with FP32 accumulators in TMEM, operands staged by TMA.
//
// With dy the gradient of the dispatched rows' outputs (ruDNN user guide,
// section 12, cache.backward):
//   DGRAD_H   dh[r, i] = sum_h W_down[e][h][i] dy[r][h] (FP32, in TMEM), then
//             in the epilogue dg = dh * u * SiLU'(g), du = dh * SiLU(g)
//             from the cached g and u                           -> dtype [rows, I] x 2
//   DGRAD_X   dx[r, h] = sum_i W_gate[e][i][h] dg[r][i]
//                      + sum_i W_up[e][i][h]   du[r][i]        -> dtype [rows, H]
//   WGRAD_D   ddown[e][h][i] = sum_{r in e} dy[r][h] h[r][i]   -> FP32 [E, H, I]
//   WGRAD_GU  dgate[e][i][h] = sum_{r in e} dg[r][i] x[r][h],
//             dup[e][i][h]   = sum_{r in e} du[r][i] x[r][h]   -> FP32 [E, I, H] x 2
//
// Operand layouts. DGRAD reads the weights as they are stored: the output
// channel (the MMA's M, 128 TMEM lanes) is the contiguous dimension of
// W[e] = [K][M], so A is MN-major, loaded as TMA boxes of 64 M-elements x 64
// K-rows (two boxes per 128-row MMA); the token rows are K-major B tiles as
// in the forward. WGRAD reads activations [rows, M] and [rows, N]: K is the
// row index, so both operands are MN-major boxes of 64 elements x 64 rows,
// and a k-block of an expert's rows may run into the next expert's rows: the
// MMA warp zeroes those rows in shared memory before the MMAs. An expert
// without rows gets zero weight gradients.
//
// Structure as the forward (experts_tc.cu): one persistent CTA per SM; warp 0
// lane 0 claims tiles and issues the TMA copies, warp 1 issues the MMAs, warps
// 2..9 drain TMEM. Every mbarrier wait is bounded; a wait that runs out
// records a code in the device status word and the CTA winds down.
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

enum BwdMode { DGRAD_H = 0, DGRAD_X = 1, WGRAD_D = 2, WGRAD_GU = 3 };

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int RING = 4;
constexpr int BOX = 64 * 128;                 // one 64 x 64 MN-major box: 8 KB
constexpr int A_BYTES = 2 * BOX;              // a 128-row MMA operand
constexpr uint32_t TMEM_COLS = 512;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 32 * (2 + NUM_EPI_WARPS);
constexpr int XPOSE_BYTES = 32 * 32 * 2;
constexpr int DH_PITCH = 36;                  // DGRAD_H: FP32 [16 tokens][36] staging rows
constexpr int STAGE_SMEM = 192 * 1024;
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;
constexpr uint32_t TILE_END = 0xFFFFFFFFu;
// DGRAD token block (N of the MMAs). dh: 128, so that its two accumulators
// (2 x 128 channels x 128 tokens) fit TMEM twice and the heavy SiLU-backward
// epilogue of one tile overlaps the MMAs of the next (193 -> 146 us at the
// prefill workload); dx: 256 (its light epilogue gains nothing from the
// overlap and 128-token tiles re-stream its weights: 193 -> 215 us).
template <int MODE>
constexpr int dgrad_tbm() { return MODE == DGRAD_H ? 128 : 256; }
// WGRAD output columns per tile (N). 128 for dgate/dup would let their two
// accumulators fit TMEM twice (epilogue overlapping the next tile's MMAs),
// but the tiles double and each re-loads its dg/du operand: measured slower
// at the prefill workload (463 vs 444 us).
constexpr int WN = 256;

constexpr uint32_t ST_PRODUCER_EMPTY = 0x21;
constexpr uint32_t ST_MMA_FULL = 0x22;
constexpr uint32_t ST_MMA_TMEM_EMPTY = 0x23;
constexpr uint32_t ST_EPI_TMEM_FULL = 0x24;
constexpr uint32_t ST_MMA_DRAIN = 0x25;
constexpr uint32_t ST_PRODUCER_DRAIN = 0x26;
constexpr uint32_t ST_TILE_RING = 0x27;

template <int MODE>
struct BwdCfg {
  static constexpr bool DGRAD = MODE == DGRAD_H || MODE == DGRAD_X;
  static constexpr int N_A = (MODE == WGRAD_D) ? 1 : 2;                // MMAs per k-step
  static constexpr int TBM = dgrad_tbm<MODE>();
  static constexpr int B_BYTES = DGRAD ? TBM * 128 : (WN / 64) * BOX;  // B operand per stage
  static constexpr int STAGE_BYTES = N_A * A_BYTES + B_BYTES;
  // WGRAD keeps 32 KB for its FP32 output transposes.
  static constexpr int STAGES = (DGRAD ? STAGE_SMEM : STAGE_SMEM - 32 * 1024) / STAGE_BYTES >= 3
                                    ? (DGRAD ? STAGE_SMEM : STAGE_SMEM - 32 * 1024) / STAGE_BYTES
                                    : 3;
  static constexpr int ACC_N = DGRAD ? TBM : WN;                       // accumulator columns per MMA
  static constexpr int ACC = (N_A * ACC_N * 2 <= static_cast<int>(TMEM_COLS)) ? 2 : 1;
  static constexpr uint32_t ACC_COLS = TMEM_COLS / ACC;
  static constexpr uint32_t D1 = ACC_N;                                // second accumulator
  static constexpr int SMEM_STAGES = 0;
  static constexpr int XPOSE_WARP =                                      // per epilogue warp
      MODE == DGRAD_H ? 16 * DH_PITCH * 4 : (DGRAD ? XPOSE_BYTES : 32 * 32 * 4);
  static constexpr int SMEM_XPOSE = STAGES * STAGE_BYTES;
  static constexpr int SMEM_BAR = SMEM_XPOSE + NUM_EPI_WARPS * XPOSE_WARP;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * RING + 5;
  static constexpr int SMEM_RING = SMEM_BAR + 8 * NUM_BARS;
  static constexpr int SMEM_MISC = SMEM_RING + 4 * RING;
  static constexpr int SMEM_TILES = SMEM_MISC + 16;
  static constexpr int SMEM_BYTES = 1024 + SMEM_TILES + (DGRAD ? 4 * (ROUTE_MAX_E + 1) : 0);
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(STAGES >= 3, "pipeline depth");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(N_A * ACC_N <= static_cast<int>(ACC_COLS), "accumulators fit a buffer");
};

struct BwdArgs {
  const uint32_t* offsets;  // [E + 1]
  void* out0;               // DGRAD: [rows, n_out] (DGRAD_H: dg); WGRAD: [E, M, N] FP32
  void* out1;               // DGRAD_H: du; WGRAD_GU: dup
  uint32_t* sched;
  int E;
  int n_wblocks;            // DGRAD: output-channel blocks of 256; WGRAD: N blocks of 256
  int m_blocks;             // WGRAD: M blocks of 128
  int k_blocks;             // DGRAD: k-blocks of the first term (DGRAD_X has two terms)
  int n_out;                // DGRAD: output channels; WGRAD: N
  int m_out;                // WGRAD: M
  uint32_t rows_total;
  uint32_t tile_cap;
  uint32_t* status;
  const void* in_g;         // DGRAD_H: cached pre-activations g, u [rows, n_out]
  const void* in_u;
  // Nonzero: the A (B) maps view their 64-element atoms as one more dimension
  // and one copy brings every atom of a k-block (DGRAD A: 4, WGRAD A: 2,
  // WGRAD B: 4) instead of one copy per atom.
  int merged_a;
  int merged_b;
};

template <typename T, int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                  const __grid_constant__ CUtensorMap tm_b0, const __grid_constant__ CUtensorMap tm_b0s,
                  const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_b1s,
                  const __grid_constant__ CUtensorMap tm_o0, const __grid_constant__ CUtensorMap tm_o1,
                  const BwdArgs args) {
  using C = BwdCfg<MODE>;
  constexpr bool DGRAD = C::DGRAD;
  constexpr int STAGES = C::STAGES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::SMEM_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tile_full = empty + STAGES;
  uint64_t* tile_empty = tile_full + RING;
  uint64_t* tfull = tile_empty + RING;  // [2]
  uint64_t* tempty = tfull + 2;         // [2]
  uint64_t* drain = tempty + 2;
  volatile uint32_t* ring = reinterpret_cast<volatile uint32_t*>(smem + C::SMEM_RING);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::SMEM_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::SMEM_MISC + 4);
  uint32_t* tile_start = reinterpret_cast<uint32_t*>(smem + C::SMEM_TILES);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int r = 0; r < RING; ++r) {
      mbar_init(&tile_full[r], 1);
      mbar_init(&tile_empty[r], NUM_EPI_WARPS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], NUM_EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_a0);
    tma_prefetch_desc(&tm_a1);
    tma_prefetch_desc(&tm_b0);
    tma_prefetch_desc(&tm_b1);
  }
  __syncwarp();
  if (DGRAD && warp == 0) build_tile_prefix(args.offsets, args.E, C::TBM, args.n_wblocks, tile_start);
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint32_t total = DGRAD ? min(tile_start[args.E], args.tile_cap)
                               : static_cast<uint32_t>(args.E) * args.m_blocks * args.n_wblocks;

  // Tile -> work: DGRAD (expert, token block, 256-channel block); WGRAD
  // (expert, 128-row M block, 256-column N block) with the expert's rows.
  struct Work {
    int e, mb, nb;
    uint32_t row0;
    int rows;       // DGRAD: tokens in the block; WGRAD: the expert's rows
    int kb_count;   // k-blocks
  };
  auto decode = [&](uint32_t tile) {
    Work w;
    if (DGRAD) {
      const TileCoord tc = decode_tile(tile, tile_start, args.E, args.offsets, C::TBM, args.n_wblocks);
      w.e = tc.e;
      w.mb = tc.m;
      w.nb = tc.n;
      w.row0 = tc.row0;
      w.rows = tc.rows;
      w.kb_count = (MODE == DGRAD_X ? 2 : 1) * args.k_blocks;
    } else {
      const uint32_t per_e = static_cast<uint32_t>(args.m_blocks) * args.n_wblocks;
      w.e = static_cast<int>(tile / per_e);
      const uint32_t rem = tile % per_e;
      w.mb = static_cast<int>(rem / args.n_wblocks);
      w.nb = static_cast<int>(rem % args.n_wblocks);
      uint32_t lo = args.offsets[w.e], hi = args.offsets[w.e + 1];
      if (hi > args.rows_total) hi = args.rows_total;
      if (lo > hi) lo = hi;
      w.row0 = lo;
      w.rows = static_cast<int>(hi - lo);
      w.kb_count = (w.rows + BK - 1) / BK;
    }
    return w;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ scheduler + TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (uint32_t it = 0;; ++it) {
        const uint32_t slot = it % RING;
        if (!mbar_wait_bounded(&tile_empty[slot], ((it / RING) & 1u) ^ 1u, abort_flag, args.status, ST_TILE_RING,
                               WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        const uint32_t claimed = atomicAdd(args.sched, 1u);
        const uint32_t tile = claimed < total ? claimed : TILE_END;
        ring[slot] = tile;
        mbar_arrive(&tile_full[slot]);
        if (tile == TILE_END) break;
        const Work w = decode(tile);
        const int n_tok = (w.rows + 15) & ~15;
        uint32_t tx;
        if (DGRAD) tx = static_cast<uint32_t>(2 * A_BYTES + n_tok * 128);
        else tx = static_cast<uint32_t>(C::N_A * A_BYTES + C::B_BYTES);
        for (int kb = 0; kb < w.kb_count; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status, ST_PRODUCER_EMPTY,
                                 WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + C::SMEM_STAGES + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], tx);
          if (DGRAD) {
            // A: the weights [E][K][M] as 3-D boxes {64 channels, 64 k, 1};
            // B: the token rows [rows][K] in 128- and 16-row boxes.
            const bool second = MODE == DGRAD_X && kb >= args.k_blocks;
            const int k0 = (second ? kb - args.k_blocks : kb) * BK;
            const CUtensorMap* am = second ? &tm_a1 : &tm_a0;
            const int c0 = w.nb * (2 * BM);
            if (args.merged_a) {
              tma_load_4d(st, am, &full[stage], 0, k0, c0 / 64, w.e);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q) tma_load_3d(st + q * BOX, am, &full[stage], c0 + 64 * q, k0, w.e);
            }
            const CUtensorMap* b128 = second ? &tm_b1 : &tm_b0;
            const CUtensorMap* b16 = second ? &tm_b1s : &tm_b0s;
            uint8_t* b_dst = st + 2 * A_BYTES;
            int r = 0;
            for (; r + 128 <= n_tok; r += 128)
              tma_load_2d(b_dst + r * 128, b128, &full[stage], k0, static_cast<int>(w.row0) + r);
            for (; r < n_tok; r += 16)
              tma_load_2d(b_dst + r * 128, b16, &full[stage], k0, static_cast<int>(w.row0) + r);
          } else {
            // A (and A1): activations [rows][M] as boxes {64 elements, 64 rows};
            // B: activations [rows][N], four boxes for 256 columns.
            const int r0 = static_cast<int>(w.row0) + kb * BK;
            const int m0 = w.mb * BM, n0 = w.nb * WN;
            uint8_t* b_dst = st + C::N_A * A_BYTES;
            if (args.merged_a) {
              tma_load_3d(st, &tm_a0, &full[stage], 0, r0, m0 / 64);
              if (C::N_A == 2) tma_load_3d(st + A_BYTES, &tm_a1, &full[stage], 0, r0, m0 / 64);
            } else {
              for (int q = 0; q < 2; ++q) tma_load_2d(st + q * BOX, &tm_a0, &full[stage], m0 + 64 * q, r0);
              if (C::N_A == 2)
                for (int q = 0; q < 2; ++q)
                  tma_load_2d(st + A_BYTES + q * BOX, &tm_a1, &full[stage], m0 + 64 * q, r0);
            }
            if (args.merged_b) {
              tma_load_3d(b_dst, &tm_b0, &full[stage], 0, r0, n0 / 64);
            } else {
              for (int q = 0; q < WN / 64; ++q) tma_load_2d(b_dst + q * BOX, &tm_b0, &full[stage], n0 + 64 * q, r0);
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (!ok) {
        const uint32_t n_back = issued < STAGES ? issued : STAGES;
        for (uint32_t i = 1; i <= n_back; ++i) {
          const uint32_t n = issued - i;
          mbar_wait_bounded(&full[n % STAGES], (n / STAGES) & 1u, nullptr, args.status, ST_PRODUCER_DRAIN,
                            WAIT_LIMIT_NS);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (+ WGRAD tail zeroing)
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (uint32_t it = 0;; ++it) {
      const uint32_t slot = it % RING;
      bool w_ok = mbar_wait_bounded(&tile_full[slot], (it / RING) & 1u, abort_flag, args.status, ST_TILE_RING,
                                    WAIT_LIMIT_NS);
      if (!__all_sync(FULL_MASK, w_ok)) {
        ok = false;
        break;
      }
      const uint32_t tile = ring[slot];
      if (tile == TILE_END) break;
      const Work w = decode(tile);
      const int n_tok = (w.rows + 15) & ~15;
      const uint32_t idesc = DGRAD ? idesc_f16_major(kBF16, BM, n_tok, true, false)
                                   : idesc_f16_major(kBF16, BM, WN, true, true);
      const uint32_t acc = it % C::ACC;
      const uint32_t acc_use = it / C::ACC;
      w_ok = mbar_wait_bounded(&tempty[acc], (acc_use & 1u) ^ 1u, abort_flag, args.status, ST_MMA_TMEM_EMPTY,
                               WAIT_LIMIT_NS);
      if (!__all_sync(FULL_MASK, w_ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d0 = tmem_base + acc * C::ACC_COLS;
      for (int kb = 0; kb < w.kb_count; ++kb) {
        w_ok = mbar_wait_bounded(&full[stage], phase, abort_flag, args.status, ST_MMA_FULL, WAIT_LIMIT_NS);
        if (!__all_sync(FULL_MASK, w_ok)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + C::SMEM_STAGES + stage * STAGE_BYTES;
        // MMAs (16 K-rows each) of this stage: all 4, except in WGRAD's last
        // k-block, where those wholly past the expert's end are skipped.
        int n_sub = BK / UMMA_K;
        if (!DGRAD) {
          // Rows past the expert's end belong to the next expert (or are the
          // tensor's zero fill). Inside the last MMA that runs they are zeroed
          // in every box before the MMAs read the stage: at most 15 rows, each
          // a 128-byte line of its box, four rows per warp store.
          const int valid = w.rows - kb * BK;
          if (valid < BK) {
            n_sub = (valid + UMMA_K - 1) / UMMA_K;
            const int end = n_sub * UMMA_K;
            if (valid < end) {
              constexpr int boxes = C::N_A * 2 + WN / 64;
              const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
              for (int bx = 0; bx < boxes; ++bx)
                for (int rr = valid + (lane >> 3); rr < end; rr += 4)
                  *reinterpret_cast<uint4*>(st + bx * BOX + rr * 128 + (lane & 7) * 16) = z;
              fence_proxy_async_smem();
            }
            __syncwarp();
          }
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(st);
          const uint32_t a1 = a0 + A_BYTES;
          const uint32_t b = a0 + C::N_A * A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            if (k >= n_sub) break;
            const uint32_t accum = (kb > 0 || k > 0) ? 1u : 0u;
            // A: MN-major, 16 K-rows per MMA = 2 atoms of 8 rows (2 KB).
            const uint64_t ad0 = sdesc_mnmajor_sw128(a0 + k * 2048, BOX, 1024);
            const uint64_t ad1 = sdesc_mnmajor_sw128(a1 + k * 2048, BOX, 1024);
            const uint64_t bd = DGRAD ? sdesc_kmajor_sw128(b + k * UMMA_K * 2)
                                      : sdesc_mnmajor_sw128(b + k * 2048, BOX, 1024);
            umma_f16(d0, ad0, bd, idesc, accum);
            if (C::N_A == 2) umma_f16(d0 + C::D1, ad1, bd, idesc, accum);
          }
          umma_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(&tfull[acc]);
      __syncwarp();
    }
    if (lane == 0) {
      umma_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr, args.status, ST_MMA_DRAIN, WAIT_LIMIT_NS);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    uint16_t* xp = reinterpret_cast<uint16_t*>(smem + C::SMEM_XPOSE + ew * C::XPOSE_WARP);
    float* xf = reinterpret_cast<float*>(smem + C::SMEM_XPOSE + ew * C::XPOSE_WARP);
    const int rd_tok = lane >> 2;
    const int rd_part = lane & 3;
    for (uint32_t it = 0;; ++it) {
      const uint32_t slot = it % RING;
      bool ok = mbar_wait_bounded(&tile_full[slot], (it / RING) & 1u, abort_flag, args.status, ST_TILE_RING,
                                  WAIT_LIMIT_NS);
      const uint32_t tile = ok ? static_cast<uint32_t>(ring[slot]) : static_cast<uint32_t>(TILE_END);
      if (!__all_sync(FULL_MASK, ok) || tile == TILE_END) break;
      const Work w = decode(tile);
      const uint32_t acc = it % C::ACC;
      ok = mbar_wait_bounded(&tfull[acc], (it / C::ACC) & 1u, abort_flag, args.status, ST_EPI_TMEM_FULL,
                             WAIT_LIMIT_NS);
      if (!__all_sync(FULL_MASK, ok)) break;
      tc_fence_after();
      const uint32_t t_lane = tmem_base + acc * C::ACC_COLS + (static_cast<uint32_t>(quad * 32) << 16);
      if (MODE == DGRAD_H) {
        // lane = channel, TMEM column = token. Each 16-token half of a
        // 32 x 32 block of dh goes through a padded FP32 staging tile (row j
        // at j * 36 floats: conflict-free both ways); then lane (tok, part)
        // takes 8 channels of one token, reads g and u with 16-byte loads and
        // writes dg and du with 16-byte stores.
        const int n_tok = (w.rows + 15) & ~15;
        const int64_t chan0 = static_cast<int64_t>(w.nb) * (2 * BM) + quad * 32;
        for (int c0 = 32 * half; c0 < n_tok; c0 += 64) {
          for (int blk = 0; blk < 2; ++blk) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_lane + blk * C::D1 + static_cast<uint32_t>(c0), v);
            const int64_t col = chan0 + blk * BM + rd_part * 8;
            // This lane's four (token, 8 channels) groups of g and u, loaded
            // while the accumulator load is in flight.
            uint4 gq[4], uq[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int t_in = c0 + (i >> 1) * 16 + (i & 1) * 8 + rd_tok;
              gq[i] = uq[i] = make_uint4(0u, 0u, 0u, 0u);
              if (t_in < w.rows && col + 8 <= args.n_out) {
                const int64_t off = (static_cast<int64_t>(w.row0) + t_in) * args.n_out + col;
                gq[i] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(args.in_g) + off));
                uq[i] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(args.in_u) + off));
              }
            }
            tmem_ld_wait();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
              for (int j = 0; j < 16; ++j) xf[j * DH_PITCH + lane] = __uint_as_float(v[hh * 16 + j]);
              __syncwarp();
#pragma unroll
              for (int p = 0; p < 2; ++p) {
                const int j = p * 8 + rd_tok;
                const int t_in = c0 + hh * 16 + j;
                if (t_in < w.rows && col + 8 <= args.n_out) {
                  const int64_t off = (static_cast<int64_t>(w.row0) + t_in) * args.n_out + col;
                  const float4 d0 = *reinterpret_cast<const float4*>(xf + j * DH_PITCH + rd_part * 8);
                  const float4 d1 = *reinterpret_cast<const float4*>(xf + j * DH_PITCH + rd_part * 8 + 4);
                  const uint4 gv4 = gq[hh * 2 + p];
                  const uint4 uv4 = uq[hh * 2 + p];
                  const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
                  const T* gv = reinterpret_cast<const T*>(&gv4);
                  const T* uv = reinterpret_cast<const T*>(&uv4);
                  uint32_t dgw[4], duw[4];
#pragma unroll
                  for (int q = 0; q < 4; ++q) {
                    float g0, g1, u0, u1;
                    silu_mul_backward(d[2 * q], to_f32(gv[2 * q]), to_f32(uv[2 * q]), &g0, &u0);
                    silu_mul_backward(d[2 * q + 1], to_f32(gv[2 * q + 1]), to_f32(uv[2 * q + 1]), &g1, &u1);
                    dgw[q] = pack2<T>(g0, g1);
                    duw[q] = pack2<T>(u0, u1);
                  }
                  *reinterpret_cast<uint4*>(static_cast<T*>(args.out0) + off) =
                      make_uint4(dgw[0], dgw[1], dgw[2], dgw[3]);
                  *reinterpret_cast<uint4*>(static_cast<T*>(args.out1) + off) =
                      make_uint4(duw[0], duw[1], duw[2], duw[3]);
                }
              }
              __syncwarp();
            }
          }
        }
      } else if (DGRAD) {
        // lane = output channel, TMEM column = token of the block.
        const int n_tok = (w.rows + 15) & ~15;
        const int64_t chan0 = static_cast<int64_t>(w.nb) * (2 * BM) + quad * 32;
        for (int c0 = 32 * half; c0 < n_tok; c0 += 64) {
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(c0), v0);
          tmem_ld_32x32b_x32(t_lane + C::D1 + static_cast<uint32_t>(c0), v1);
          tmem_ld_wait();
          for (int blk = 0; blk < 2; ++blk) {
            const int64_t chan = chan0 + blk * BM;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const T hv = from_f32<T>(__uint_as_float(blk == 0 ? v0[j] : v1[j]));
              xp[j * 32 + lane] = *reinterpret_cast<const uint16_t*>(&hv);
            }
            __syncwarp();
            const int64_t col = chan + rd_part * 8;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const int j = p * 8 + rd_tok;
              const uint4 row = *reinterpret_cast<const uint4*>(xp + j * 32 + rd_part * 8);
              const int t_in = c0 + j;
              if (t_in < w.rows && col + 8 <= args.n_out) {
                T* dst = static_cast<T*>(args.out0) + (static_cast<int64_t>(w.row0) + t_in) * args.n_out + col;
                *reinterpret_cast<uint4*>(dst) = row;
              }
            }
            __syncwarp();
          }
        }
      } else {
        // TMEM lane = output row m, column = output n; FP32 [E, M, N]. Each
        // 32 x 32 block is staged in the warp's 4 KB tile with the 128-byte
        // swizzle (16-byte chunk q of row r at chunk q ^ (r % 8): conflict-
        // free stores) and written by one TMA tensor store, which clips rows
        // and columns past the expert's [M, N]. Lane 0 waits for the previous
        // store to have read the tile before the warp rewrites it.
        const int m_base = w.mb * BM + quad * 32;
        const bool empty_expert = w.kb_count == 0;
        for (int c0 = 32 * half; c0 < WN; c0 += 64) {
          for (int blk = 0; blk < C::N_A; ++blk) {
            uint32_t v[32];
            if (!empty_expert) {
              tmem_ld_32x32b_x32(t_lane + blk * C::D1 + static_cast<uint32_t>(c0), v);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0u;
            }
            // One staging tile per warp: the previous store must have read it
            // (a second tile, letting two stores per warp be in flight, was
            // slower: the stores then crowd the stage loads on the TMA unit).
            const uint32_t xbuf = smem_u32(xf);
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_shared_v4(xbuf + lane * 128 + ((q ^ (lane & 7)) << 4), v[4 * q], v[4 * q + 1], v[4 * q + 2],
                           v[4 * q + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(blk == 0 ? &tm_o0 : &tm_o1, xbuf, w.nb * WN + c0, m_base, w.e);
              bulk_commit_group();
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[acc]);
        mbar_arrive(&tile_empty[slot]);
      }
    }
    // The tensor stores read shared memory and write the gradients: both end
    // before the block exits.
    if (!DGRAD && lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_bwd() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool enc(CUtensorMap* m, moe_dtype dt, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
         const cuuint32_t* box) {
  auto fn = encode_fn_bwd();
  if (fn == nullptr) return false;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, dt == MOE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank,
            const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [E][K][M] weights as boxes {64 (M), 64 (K), 1}.
bool enc_weights_mn(CUtensorMap* m, moe_dtype dt, const void* w, int64_t E, int64_t K, int64_t M) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(E)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(M) * 2, static_cast<cuuint64_t>(K * M) * 2};
  const cuuint32_t box[3] = {64, 64, 1};
  return enc(m, dt, w, 3, dims, strides, box);
}

// FP32 weight gradient [E][M][N] as boxes {32 (N), 32 (M), 1}, 128-byte
// swizzle (the epilogue's staging layout); rows and columns past [M, N] of an
// expert are clipped by the store.
bool enc_grad_out(CUtensorMap* m, const float* p, int64_t E, int64_t M, int64_t N) {
  auto fn = encode_fn_bwd();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(E)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 4, static_cast<cuuint64_t>(M * N) * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(p), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [E][K][M] weights viewed as {64, K, M / 64, E} (the 64-element atoms of M
// as a dimension of stride 128 B): box {64, 64, 4, 1} brings the four atoms
// of a 256-channel block in one copy. Needs M % 64 == 0.
bool enc_weights_mn_merged(CUtensorMap* m, moe_dtype dt, const void* w, int64_t E, int64_t K, int64_t M) {
  if (M % 64 != 0) return false;
  const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M / 64),
                              static_cast<cuuint64_t>(E)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(M) * 2, 128, static_cast<cuuint64_t>(K * M) * 2};
  const cuuint32_t box[4] = {64, 64, 4, 1};
  return enc(m, dt, w, 4, dims, strides, box);
}

// [rows][C] activations viewed as {64, rows, C / 64}: box {64, 64, atoms}
// brings `atoms` consecutive 64-element atoms of 64 rows in one copy. Needs
// C % 64 == 0.
bool enc_rows_merged(CUtensorMap* m, moe_dtype dt, const void* p, int64_t rows, int64_t C, uint32_t atoms) {
  if (C % 64 != 0) return false;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(C / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 2, 128};
  const cuuint32_t box[3] = {64, 64, atoms};
  return enc(m, dt, p, 3, dims, strides, box);
}

// [rows][C] activations as boxes {64 (C), box_rows}.
bool enc_rows(CUtensorMap* m, moe_dtype dt, const void* p, int64_t rows, int64_t C, uint32_t box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(C) * 2};
  const cuuint32_t box[2] = {64, box_rows};
  return enc(m, dt, p, 2, dims, strides, box);
}

template <typename T, int MODE>
cudaError_t launch_mode(const CUtensorMap* maps, const BwdArgs& args, int num_sms, cudaStream_t s) {
  auto kern = bwd_tc_kernel<T, MODE>;
  constexpr int SMEM = BwdCfg<MODE>::SMEM_BYTES;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (err != cudaSuccess) return err;
  const int grid = static_cast<int>(args.tile_cap < static_cast<uint32_t>(num_sms) ? args.tile_cap : num_sms);
  if (grid <= 0) return cudaSuccess;
  err = cudaMemsetAsync(args.sched, 0, sizeof(uint32_t), s);
  if (err != cudaSuccess) return err;
  kern<<<grid, NUM_THREADS, SMEM, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], args);
  return cudaGetLastError();
}

template <typename T>
cudaError_t backward_tc_t(moe_dtype dt, const TrainBuffers& b, const uint32_t* offsets, int E, int64_t rows,
                          int64_t H, int64_t I, uint32_t* sched, int num_sms, cudaStream_t s, const char** why) {
  uint32_t* status = nullptr;
  cudaError_t err = device_status_ptr(&status);
  if (err != cudaSuccess) return err;
  CUtensorMap maps[8];  // a0, a1, b0, b0s, b1, b1s, and the WGRAD outputs o0, o1
  auto fail_enc = [&]() {
    *why = "cuTensorMapEncodeTiled rejected a backward tensor map";
    return cudaErrorInvalidValue;
  };
  auto tok_blocks = [&](int tbm) { return rows / tbm + (rows < E ? rows : E); };
  const uint32_t srows = static_cast<uint32_t>(rows);
  // dh = dy W_down: A = W_down [E][H][I] (K = H, M = I), B = dy [rows][H];
  // the epilogue turns dh into dg and du with the cached g and u.
  {
    const bool merged = enc_weights_mn_merged(&maps[0], dt, b.down, E, H, I);
    if ((!merged && !enc_weights_mn(&maps[0], dt, b.down, E, H, I)) || !enc_rows(&maps[2], dt, b.dy, rows, H, 128) ||
        !enc_rows(&maps[3], dt, b.dy, rows, H, 16))
      return fail_enc();
    maps[1] = maps[0];
    maps[4] = maps[2];
    maps[5] = maps[3];
    maps[6] = maps[7] = maps[0];
    const int nw = static_cast<int>((I + 2 * BM - 1) / (2 * BM));
    BwdArgs a{offsets, b.dg, b.du, sched, E, nw, 0, static_cast<int>((H + BK - 1) / BK), static_cast<int>(I),
              0, srows, static_cast<uint32_t>(tok_blocks(dgrad_tbm<DGRAD_H>()) * nw), status, b.g, b.u,
              merged ? 1 : 0, 0};
    err = launch_mode<T, DGRAD_H>(maps, a, num_sms, s);
    if (err != cudaSuccess) return err;
  }
  // dx = dg W_gate + du W_up: A = W_gate / W_up [E][I][H] (K = I, M = H), B = dg / du [rows][I]
  {
    const bool merged =
        enc_weights_mn_merged(&maps[0], dt, b.gate, E, I, H) && enc_weights_mn_merged(&maps[1], dt, b.up, E, I, H);
    if ((!merged && (!enc_weights_mn(&maps[0], dt, b.gate, E, I, H) || !enc_weights_mn(&maps[1], dt, b.up, E, I, H))) ||
        !enc_rows(&maps[2], dt, b.dg, rows, I, 128) || !enc_rows(&maps[3], dt, b.dg, rows, I, 16) ||
        !enc_rows(&maps[4], dt, b.du, rows, I, 128) || !enc_rows(&maps[5], dt, b.du, rows, I, 16))
      return fail_enc();
    maps[6] = maps[7] = maps[0];
    const int nw = static_cast<int>((H + 2 * BM - 1) / (2 * BM));
    BwdArgs a{offsets, b.dx, nullptr, sched, E, nw, 0, static_cast<int>((I + BK - 1) / BK), static_cast<int>(H),
              0, srows, static_cast<uint32_t>(tok_blocks(dgrad_tbm<DGRAD_X>()) * nw), status, nullptr, nullptr,
              merged ? 1 : 0, 0};
    err = launch_mode<T, DGRAD_X>(maps, a, num_sms, s);
    if (err != cudaSuccess) return err;
  }
  // ddown[e] = dy^T h: A = dy [rows][H] (M = H), B = h [rows][I] (N = I)
  {
    const bool ma = enc_rows_merged(&maps[0], dt, b.dy, rows, H, 2);
    const bool mb_ = enc_rows_merged(&maps[2], dt, b.h, rows, I, WN / 64);
    if ((!ma && !enc_rows(&maps[0], dt, b.dy, rows, H, 64)) || (!mb_ && !enc_rows(&maps[2], dt, b.h, rows, I, 64)) ||
        !enc_grad_out(&maps[6], b.ddown, E, H, I))
      return fail_enc();
    maps[1] = maps[0];
    maps[3] = maps[4] = maps[5] = maps[2];
    maps[7] = maps[6];
    const int mb = static_cast<int>((H + BM - 1) / BM), nb = static_cast<int>((I + WN - 1) / WN);
    BwdArgs a{offsets, b.ddown, nullptr, sched, E, nb, mb, 0, static_cast<int>(I), static_cast<int>(H), srows,
              static_cast<uint32_t>(static_cast<int64_t>(E) * mb * nb), status, nullptr, nullptr, ma ? 1 : 0,
              mb_ ? 1 : 0};
    err = launch_mode<T, WGRAD_D>(maps, a, num_sms, s);
    if (err != cudaSuccess) return err;
  }
  // dgate[e], dup[e] = dg^T x, du^T x: A0 = dg, A1 = du [rows][I] (M = I), B = x [rows][H] (N = H)
  {
    const bool ma = enc_rows_merged(&maps[0], dt, b.dg, rows, I, 2) && enc_rows_merged(&maps[1], dt, b.du, rows, I, 2);
    const bool mb_ = enc_rows_merged(&maps[2], dt, b.x, rows, H, WN / 64);
    if ((!ma && (!enc_rows(&maps[0], dt, b.dg, rows, I, 64) || !enc_rows(&maps[1], dt, b.du, rows, I, 64))) ||
        (!mb_ && !enc_rows(&maps[2], dt, b.x, rows, H, 64)) || !enc_grad_out(&maps[6], b.dgate, E, I, H) ||
        !enc_grad_out(&maps[7], b.dup, E, I, H))
      return fail_enc();
    maps[3] = maps[4] = maps[5] = maps[2];
    const int mb = static_cast<int>((I + BM - 1) / BM), nb = static_cast<int>((H + WN - 1) / WN);
    BwdArgs a{offsets, b.dgate, b.dup, sched, E, nb, mb, 0, static_cast<int>(H), static_cast<int>(I), srows,
              static_cast<uint32_t>(static_cast<int64_t>(E) * mb * nb), status, nullptr, nullptr, ma ? 1 : 0,
              mb_ ? 1 : 0};
    err = launch_mode<T, WGRAD_GU>(maps, a, num_sms, s);
  }
  return err;
}

}  // namespace

cudaError_t launch_experts_backward_tc(moe_dtype dtype, const TrainBuffers& b, const uint32_t* offsets, int E,
                                       int64_t rows, int64_t H, int64_t I, uint32_t* sched, int num_sms,
                                       cudaStream_t stream, const char** why) {
  if (dtype == MOE_BF16)
    return backward_tc_t<__nv_bfloat16>(dtype, b, offsets, E, rows, H, I, sched, num_sms, stream, why);
  return backward_tc_t<__half>(dtype, b, offsets, E, rows, H, I, sched, num_sms, stream, why);
}

}  // namespace moe
