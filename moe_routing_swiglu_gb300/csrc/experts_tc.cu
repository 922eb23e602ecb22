// K3 / K4: F16/BF16 SwiGLU experts as grouped GEMMs on the sm_103a tensor
// cores (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// Per dispatched row r of expert e ("tiny-llm deep dive 5: ops.rs", section
// on SiLU, FFN(x) = W_down (SiLU(W_gate x) * W_up x); shapes from the ruDNN
// user guide, section 5):
//   K3  h_r = SiLU(W_gate[e] x_r) * (W_up[e] x_r)    (K = H)
//   K4  y_r = W_down[e] h_r                          (K = I)
// The SiLU-and-multiply is fused into K3's epilogue, so the gate and up
// projections never reach HBM ("PyTorch general ops", section on RMSNorm
// and SiLU x Mul).
//
// Operand roles. The MMA's M side (128 TMEM lanes) holds expert weight rows
// and its N side holds the expert's tokens, N = the tile's token count
// rounded up to 16 (at most 256): an expert with 270 rows is one 256-token
// tile plus one 16-token tile, and a decode expert with 1-2 tokens costs
// N = 16. Each k-step issues two MMAs that share the token tile:
//   K3 tile: A0 = gate rows c0..c0+127, A1 = up rows c0..c0+127  -> D0, D1
//   K4 tile: A0 = down rows n0..n0+127, A1 = down rows n0+128..n0+255
// so one token tile feeds 256 weight rows (the token rows are re-read from
// L2 half as often as with one MMA), and TMEM lane i of D0 and D1 holds the
// gate and up values of the same channel in the same thread.
//
// One persistent CTA per SM, 320 threads in three roles:
//   warp 0 lane 0   scheduler + TMA producer: claims tiles from a global
//                   counter (atomicAdd), publishes them in a 4-deep ring in
//                   shared memory, and streams 3 stages of (2 x 16 KB weights
//                   + N x 128 B tokens), 128-byte swizzle; token rows come
//                   in 128-row and 16-row boxes so a short tile moves only
//                   its rows.
//   warp 1 lane 0   MMA issuer: 2 x 4 tcgen05.mma (M=128, N, K=16) per stage
//                   into D0 (TMEM columns 0..N-1) and D1 (256..256+N-1); the
//                   instruction descriptor carries the tile's N. Warp 1 also
//                   allocates the 512 TMEM columns.
//   warps 2..9      epilogue: warp w reads TMEM lanes 32*(w%4).. and takes
//                   every other 32-token chunk; it computes the outputs in
//                   FP32 (K3: SiLU(g)*u), transposes its 32 x 32 block
//                   through a warp-private shared buffer and writes each
//                   token's 64-byte runs with 16-byte stores.
// Token rows reach shared memory in one of three ways (the template's LOAD):
//   TOK_DENSE    TMA boxes of 128 and 16 rows over x_dispatched;
//   TOK_GATHER4  TMA row gathers straight from x: row r of a tile is
//                x[row_src[r] / top_k], four rows per tile::gather4 copy,
//                issued by the lanes of warp 0 (decode-sized tiles of at
//                most 32 rows; the dispatch then writes no x_dispatched);
//   TOK_CPASYNC  the same gather by four extra loader warps with 16-byte
//                cp.async copies into the swizzled layout (256-row tiles,
//                where 64 row gathers per stage would keep the TMA unit
//                busy far longer than one 128-row box).
// Tiles: expert e has ceil(count_e / 256) token blocks times the weight
// blocks; token blocks vary fastest and tiles are claimed in order, so the
// CTAs that share a weight tile run together and read it from L2. The plan
// comes from the device offsets (the host never learns per-expert counts).
//
// Chained mode (what moe_forward runs for F16/BF16): one launch takes K3's
// tiles and then K4's from one counter; a K4 tile waits for its expert's h
// rows through a per-expert counter that K3's epilogue warps raise (see the
// kernel's comment). CTAs that run out of K3 tiles start K4 tiles instead of
// idling through K3's last wave.
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

constexpr int BM = 128;            // weight rows per MMA (TMEM lanes)
constexpr int BK = 64;             // one 128-byte swizzle atom of 16-bit elements
constexpr int UMMA_K = 16;
constexpr int RING = 4;            // tile ring depth
constexpr int ROW_BYTES = BK * 2;             // 128 B per row per stage
constexpr int A_BYTES = BM * ROW_BYTES;       // 16 KB per weight tile
constexpr uint32_t TMEM_COLS = 512;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_LOAD_WARPS = 4;             // token-row loaders of the cp.async gather
constexpr int FIRST_LOAD_WARP = 2 + NUM_EPI_WARPS;
enum TokenLoad { TOK_DENSE = 0, TOK_CPASYNC = 1, TOK_GATHER4 = 2 };
template <int LOAD>
constexpr int num_threads() { return 32 * (2 + NUM_EPI_WARPS + (LOAD == TOK_CPASYNC ? NUM_LOAD_WARPS : 0)); }
constexpr int BAD_WORDS = 8;                  // per ring slot: one flag bit per token row (256)
constexpr int XPOSE_BYTES = 32 * 32 * 2;      // per-warp transpose buffer
constexpr int STAGE_SMEM = 192 * 1024;        // shared memory given to pipeline stages
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;
constexpr uint32_t TILE_END = 0xFFFFFFFFu;

// Layout for a token-block cap TBM (the largest N of a tile): 256 for
// prefill; 32 for decode, where the smaller token tile leaves room for more
// stages (more weight bytes in flight).
template <int TBM>
struct TcCfg {
  static constexpr int B_BYTES = TBM * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;
  static constexpr int STAGES = STAGE_SMEM / STAGE_BYTES;
  // Accumulator buffers in TMEM: one tile needs D0 and D1 of TBM columns
  // each, so tiles of up to 128 tokens get two buffers and the MMAs of the
  // next tile run while the epilogue drains the previous one.
  static constexpr int ACC = (2 * 2 * TBM <= static_cast<int>(TMEM_COLS)) ? 2 : 1;
  static constexpr uint32_t ACC_COLS = TMEM_COLS / ACC;  // columns per buffer
  static constexpr uint32_t D1 = ACC_COLS / 2;           // D1 offset within a buffer
  static constexpr int SMEM_STAGES = 0;
  static constexpr int SMEM_XPOSE = SMEM_STAGES + STAGES * STAGE_BYTES;
  static constexpr int SMEM_BAR = SMEM_XPOSE + NUM_EPI_WARPS * XPOSE_BYTES;
  // full[S], empty[S], tile_full[R], tile_empty[R], tfull[2], tempty[2], drain
  static constexpr int NUM_BARS = 2 * STAGES + 2 * RING + 5;
  static constexpr int SMEM_RING = SMEM_BAR + 8 * NUM_BARS;
  static constexpr int SMEM_MISC = SMEM_RING + 4 * RING;          // TMEM address, abort flag, combine flag
  static constexpr int SMEM_BAD = SMEM_MISC + 16;                  // [RING][BAD_WORDS]
  static constexpr int SMEM_TILES = SMEM_BAD + 4 * RING * BAD_WORDS;
  static constexpr int SMEM_BYTES = 1024 + SMEM_TILES + 4 * (ROUTE_MAX_E + 1);
  // The chained gate/up + down kernel keeps a second tile prefix (the down
  // tiles') after the first.
  static constexpr int SMEM_TILES2 = SMEM_TILES + 4 * (ROUTE_MAX_E + 1);
  static constexpr int SMEM_BYTES_CHAIN = SMEM_BYTES + 4 * (ROUTE_MAX_E + 1);
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(STAGES >= 3, "pipeline depth");
  static_assert(SMEM_BYTES_CHAIN <= 227 * 1024, "shared memory budget");
  static_assert(TBM % 32 == 0 && TBM <= 256, "token block");
  static_assert(2 * TBM <= static_cast<int>(ACC_COLS), "D0 and D1 fit one accumulator buffer");
};

// Status codes recorded by a wait that timed out.
constexpr uint32_t ST_PRODUCER_EMPTY = 0x11;
constexpr uint32_t ST_MMA_FULL = 0x12;
constexpr uint32_t ST_MMA_TMEM_EMPTY = 0x13;
constexpr uint32_t ST_EPI_TMEM_FULL = 0x14;
constexpr uint32_t ST_MMA_DRAIN = 0x15;
constexpr uint32_t ST_PRODUCER_DRAIN = 0x16;
constexpr uint32_t ST_TILE_RING = 0x17;
constexpr uint32_t ST_LOADER_EMPTY = 0x18;
constexpr uint32_t ST_CHAIN_READY = 0x19;
constexpr uint32_t ST_SELFTEST = 0x100;

struct TcArgs {
  const uint32_t* offsets;  // [E + 1]
  void* out;                // [rows, n_out]: h for K3, y for K4
  uint32_t* sched;          // tile counter, zero at launch
  int E;
  int n_wblocks;            // weight blocks per expert (I/128 for K3, H/256 for K4)
  int k_blocks;             // ceil(K / BK)
  int n_out;                // output columns (I for K3, H for K4)
  uint32_t rows_total;      // rows of the token and output matrices
  uint32_t tile_cap;        // host bound on the tile count
  uint32_t* status;
  // Gather modes (K3 only): token row r of a tile is x[row_src[r] / top_k].
  const uint8_t* gx;        // x [x_rows, K], 16-bit, rows of k_bytes
  const uint32_t* row_src;  // [rows_total]
  int top_k;
  uint32_t x_rows;
  int k_bytes;              // K * 2
  // Training mode (K3 only): the pre-activations g and u, [rows, I] each.
  void* out_g;
  void* out_u;
  // Chained mode (K3 then K4 in one launch): the down tiles' output y
  // [rows, n_out2], their weight blocks per expert and k-blocks, and one
  // counter per expert (zero at launch) that each gate/up epilogue warp
  // raises once its h rows are stored.
  void* out2;
  int n_wblocks2;
  int k_blocks2;
  int n_out2;
  uint32_t* ready;
  // Fused combine (chained mode): every epilogue warp of every down tile
  // raises one done counter once its y rows are stored. A CTA whose tiles
  // are all done waits until the counter shows every down tile done, then
  // its epilogue warps write out[t] = sum_{j=0..k-1} w[t, j] * y[inv[t*k + j]]
  // (FP32, slot order) for a fixed stripe of the tokens.
  const uint32_t* comb_inv;  // [T * top_k] flat slot -> dispatched row
  const void* comb_w;        // [T, top_k] routing weights, dtype comb_wdt
  int comb_wdt;              // moe_dtype of the weights
  int comb_k;                // top_k, 1 .. COMB_MAX_K
  uint32_t comb_T;           // tokens
  uint32_t* comb_done;       // [1] down-tile epilogue arrivals, zero at launch
  void* comb_out;            // [T, n_out2]
};

constexpr int COMB_TOKENS_PER_PASS = 4;  // tokens a warp combines in one stream of loads
// A warp stages the (row, weight) pairs of COMB_TOKENS_PER_PASS tokens in
// its 2 KB buffer: top_k is at most 2048 / (8 * COMB_TOKENS_PER_PASS).
constexpr int COMB_PAIRS = XPOSE_BYTES / 8;
constexpr int COMB_MAX_K = COMB_PAIRS / COMB_TOKENS_PER_PASS;
static_assert(COMB_MAX_K == COMB_MAX_TOP_K, "the host's top_k bound matches the staging buffer");
constexpr uint32_t ST_COMB_WAIT = 0x1A;

__device__ __forceinline__ float comb_weight(const void* w, int wdt, int64_t i) {
  if (wdt == MOE_F32) return static_cast<const float*>(w)[i];
  if (wdt == MOE_F16) return __half2float(static_cast<const __half*>(w)[i]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(w)[i]);
}

// The combine of n tokens (tok[0..n)) by one warp from their staged (row,
// weight) pairs rows[i*k + j], wts[i*k + j] (bad[i]: a slot of token i is
// undispatched, its row becomes NaN as in the separate combine): lane l takes
// the 8-column chunks q = l, l + 32, ... and computes
//   out[t, c] = sum_{j=0..k-1} w[t, j] * y[row_j, c]
// with FP32 FMAs in slot order (the order and arithmetic of the separate
// combine kernel, so the two give the same bits), then rounds to T. The
// (token, chunk, slot) triples are visited in that order, G row loads in
// flight per lane across tokens.
template <typename T, int NMAX>
__device__ __forceinline__ void comb_tokens(int n, const uint32_t (&tok)[NMAX], const bool (&bad)[NMAX],
                                            const TcArgs& a, const uint32_t* rows, const float* wts, int lane) {
  constexpr int G = 16;
  const int k = a.comb_k;
  const int64_t H = a.n_out2;
  const int nq = static_cast<int>((H / 8 + 31) / 32);  // chunks per lane (H is a multiple of 8)
  const T* y = static_cast<const T*>(a.out2);
  const float qnan = __int_as_float(0x7FC00000);
  int b = 0, i = 0, j = 0;  // token, chunk, slot of the next triple
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
  while (b < n) {
    uint4 v[G];
    float wv[G];
    int pb[G], pi[G], pj[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      pb[g] = b;
      pi[g] = i;
      pj[g] = j;
      wv[g] = 0.0f;
      v[g] = make_uint4(0u, 0u, 0u, 0u);
      if (b < n) {
        const int64_t col = static_cast<int64_t>(lane + 32 * i) * 8;
        wv[g] = wts[b * k + j];
        if (col < H) v[g] = __ldcg(reinterpret_cast<const uint4*>(y + static_cast<int64_t>(rows[b * k + j]) * H + col));
        if (++j == k) {
          j = 0;
          if (++i == nq) {
            i = 0;
            ++b;
          }
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (pb[g] < n) {
        if (pj[g] == 0) {
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
        }
        const T* e8 = reinterpret_cast<const T*>(&v[g]);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(wv[g], to_f32(e8[e]), acc[e]);
        const int64_t col = static_cast<int64_t>(lane + 32 * pi[g]) * 8;
        if (pj[g] == k - 1 && col < H) {
          bool badb = false;
          uint32_t t = 0;
#pragma unroll
          for (int x = 0; x < NMAX; ++x)
            if (x == pb[g]) {
              badb = bad[x];
              t = tok[x];
            }
          uint4 raw;
          T* r = reinterpret_cast<T*>(&raw);
#pragma unroll
          for (int e = 0; e < 8; ++e) r[e] = from_f32<T>(badb ? qnan : acc[e]);
          *reinterpret_cast<uint4*>(static_cast<T*>(a.comb_out) + static_cast<int64_t>(t) * H + col) = raw;
        }
      }
    }
  }
}

// SiLU(g) = g * sigmoid(g), sigmoid(g) = 0.5 + 0.5 tanh(g / 2): one
// tanh.approx (relative error about 2^-11, below the 16-bit output's rounding).
__device__ __forceinline__ float silu_f32(float g) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * g));
  return g * fmaf(0.5f, t, 0.5f);
}

// Tensor maps: a0/a1 weight tiles (128-row boxes: K3 gate/up, K4 down rows
// n0 and n0+128), b128/b16 token rows in 128-row and 16-row boxes
// (TOK_GATHER4: b128 is x with a one-row box).
// CHAIN: one launch runs K3's tiles and then K4's from one tile counter
// (GATE_UP is then ignored): tiles [0, n_gu) are gate/up tiles over a0/a1
// (gate, up) and b128/b16 (x rows), the rest down tiles over a2 (down) and
// c128/c16 (h rows, written by this launch's gate/up tiles). A down tile of
// expert e waits until every gate/up tile of e has stored its h rows (a
// per-expert counter, bounded wait): CTAs that run out of gate/up tiles
// start the down GEMM of the experts already done instead of idling until
// the last gate/up tile ends. Every gate/up tile is claimed before any down
// tile, by a running CTA, so every wait ends.
// COMB (chained mode only): the down tiles combine into out (see TcArgs).
template <typename T, bool GATE_UP, int TBM, int LOAD, bool CHAIN = false, bool COMB = false>
__global__ void __launch_bounds__(num_threads<LOAD>(), 1)
    experts_tc_kernel(const __grid_constant__ CUtensorMap tm_a0,
                      const __grid_constant__ CUtensorMap tm_a1,
                      const __grid_constant__ CUtensorMap tm_b128,
                      const __grid_constant__ CUtensorMap tm_b16,
                      const __grid_constant__ CUtensorMap tm_a2,
                      const __grid_constant__ CUtensorMap tm_c128,
                      const __grid_constant__ CUtensorMap tm_c16, const TcArgs args) {
  static_assert(!CHAIN || LOAD != TOK_CPASYNC, "the chained kernel streams dense or row-gathered tokens");
  static_assert(!COMB || CHAIN, "the fused combine belongs to the chained kernel");
  using C = TcCfg<TBM>;
  constexpr int STAGES = C::STAGES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  constexpr int TB = TBM;
  constexpr bool GATHER = LOAD == TOK_CPASYNC;  // loader warps
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::SMEM_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tile_full = empty + STAGES;
  uint64_t* tile_empty = tile_full + RING;
  uint64_t* tfull = tile_empty + RING;   // [2]
  uint64_t* tempty = tfull + 2;          // [2]
  uint64_t* drain = tempty + 2;
  volatile uint32_t* ring = reinterpret_cast<volatile uint32_t*>(smem + C::SMEM_RING);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::SMEM_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::SMEM_MISC + 4);
  volatile uint32_t* tile_bad = reinterpret_cast<volatile uint32_t*>(smem + C::SMEM_BAD);
  uint32_t* tile_start = reinterpret_cast<uint32_t*>(smem + C::SMEM_TILES);
  uint32_t* tile_start2 = reinterpret_cast<uint32_t*>(smem + C::SMEM_TILES2);  // CHAIN: down tiles

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // Gather mode: the producer's expect_tx arrival plus one cp.async
      // arrival per loader thread.
      mbar_init(&full[s], GATHER ? 1 + 32 * NUM_LOAD_WARPS : 1);
      mbar_init(&empty[s], 1);
    }
    for (int r = 0; r < RING; ++r) {
      mbar_init(&tile_full[r], 1);
      mbar_init(&tile_empty[r], NUM_EPI_WARPS + (GATHER ? NUM_LOAD_WARPS : 0));
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], NUM_EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    abort_flag[1] = 0;  // the fused combine's go flag
    fence_mbarrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_a0);
    tma_prefetch_desc(&tm_a1);
    tma_prefetch_desc(&tm_b128);
    tma_prefetch_desc(&tm_b16);
    if (CHAIN) {
      tma_prefetch_desc(&tm_a2);
      tma_prefetch_desc(&tm_c128);
      tma_prefetch_desc(&tm_c16);
    }
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  // Everything above touches only this CTA's shared memory and TMEM; from
  // here on the kernel reads what earlier kernels wrote (offsets, rows).
  grid_dependency_wait();
  if (warp == 0) build_tile_prefix(args.offsets, args.E, TB, args.n_wblocks, tile_start);
  if (CHAIN && warp == 2) build_tile_prefix(args.offsets, args.E, TB, args.n_wblocks2, tile_start2);

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // The cap keeps a corrupt offsets array from producing an endless tile loop.
  const uint32_t n_gu = CHAIN ? tile_start[args.E] : 0u;
  const uint32_t total = min(CHAIN ? n_gu + tile_start2[args.E] : tile_start[args.E], args.tile_cap);
  // Tile -> coordinates, and whether it is a gate/up tile (GEMM tiles only).
  auto tile_coord = [&](uint32_t tile, bool& gu) -> TileCoord {
    if (!CHAIN || tile < n_gu) {
      gu = CHAIN ? true : GATE_UP;
      return decode_tile(tile, tile_start, args.E, args.offsets, TB, args.n_wblocks);
    }
    gu = false;
    return decode_tile(tile - n_gu, tile_start2, args.E, args.offsets, TB, args.n_wblocks2);
  };

  if (warp == 0 && LOAD == TOK_GATHER4) {
    // ------------------------------------------------------------ scheduler + TMA producer, row gathers
    // Lane 0 claims tiles and issues the weight copies; lane l gathers the
    // tile's rows 4 (l + 32 g) .. 4 (l + 32 g) + 3 for g < G4.
    constexpr int G4 = (TBM / 4 + 31) / 32;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;
    bool ok = true;
    for (uint32_t it = 0;; ++it) {
      const uint32_t slot = it % RING;
      uint32_t tile = TILE_END;
      if (lane == 0) {
        ok = mbar_wait_bounded(&tile_empty[slot], ((it / RING) & 1u) ^ 1u, abort_flag, args.status, ST_TILE_RING,
                               WAIT_LIMIT_NS);
        if (ok) {
          const uint32_t claimed = atomicAdd(args.sched, 1u);
          tile = claimed < total ? claimed : TILE_END;
        }
      }
      ok = __shfl_sync(FULL_MASK, ok ? 1 : 0, 0) != 0;
      tile = __shfl_sync(FULL_MASK, tile, 0);
      if (!ok) break;
      if (tile == TILE_END) {
        if (lane == 0) {
          ring[slot] = TILE_END;
          mbar_arrive(&tile_full[slot]);
          launch_dependents();  // this CTA claims no more tiles
        }
        break;
      }
      bool gu;
      const TileCoord tc = tile_coord(tile, gu);
      const int n_tok = (tc.rows + 15) & ~15;
      // Rows past the tile's rows (up to its 16-row N) read x row 0: their
      // outputs are never written. A row whose token is out of range reads
      // row 0 too and is flagged, and the epilogue writes zeros for it (the
      // outputs of a zero x row). Down tiles (CHAIN) read h densely: no flags.
      int tok[G4][4];
      uint32_t nib[G4];
#pragma unroll
      for (int g = 0; g < G4; ++g) {
        nib[g] = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * (lane + 32 * g) + i;
          uint32_t t = 0;
          if (gu && r < tc.rows && tc.row0 + static_cast<uint32_t>(r) < args.rows_total) {
            t = args.row_src[tc.row0 + r] / static_cast<uint32_t>(args.top_k);
            if (t >= args.x_rows) {
              nib[g] |= 1u << i;
              t = 0;
            }
          }
          tok[g][i] = static_cast<int>(t);
        }
      }
      // Flag word w holds rows 32 w .. 32 w + 31: lanes 8q .. 8q + 7 of
      // gather g fill word 4 g + q, lane l at bits 4 (l % 8) ...
#pragma unroll
      for (int g = 0; g < G4; ++g) {
        uint32_t wv = nib[g] << (4 * (lane & 7));
        wv |= __shfl_xor_sync(FULL_MASK, wv, 1);
        wv |= __shfl_xor_sync(FULL_MASK, wv, 2);
        wv |= __shfl_xor_sync(FULL_MASK, wv, 4);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t word = __shfl_sync(FULL_MASK, wv, 8 * q);
          if (lane == 0 && 4 * g + q < BAD_WORDS) tile_bad[slot * BAD_WORDS + 4 * g + q] = word;
        }
      }
      if (CHAIN && !gu) {
        // The expert's h rows: every gate/up tile of it has stored them.
        // Waited for before the tile is published, so that the MMA and
        // epilogue waits of a down tile start only once its inputs exist.
        bool ready = true;
        if (lane == 0) {
          const uint32_t need = static_cast<uint32_t>(NUM_EPI_WARPS) * (tile_start[tc.e + 1] - tile_start[tc.e]);
          ready = counter_wait_bounded(args.ready + tc.e, need, abort_flag, args.status, ST_CHAIN_READY,
                                       WAIT_LIMIT_NS);
        }
        if (__shfl_sync(FULL_MASK, ready ? 1 : 0, 0) == 0) {
          ok = false;
          break;
        }
      }
      if (lane == 0) {
        ring[slot] = tile;
        mbar_arrive(&tile_full[slot]);  // release: the ring entry and flags are visible to the waiters
      }
      const uint32_t tx = static_cast<uint32_t>(2 * A_BYTES + n_tok * ROW_BYTES);
      const int n_gather = n_tok >> 2;
      const int wrow0 = gu ? tc.n * BM : tc.n * (2 * BM);
      const int wrow1 = gu ? tc.n * BM : tc.n * (2 * BM) + BM;
      const int k_blocks = CHAIN && !gu ? args.k_blocks2 : args.k_blocks;
      for (int kb = 0; kb < k_blocks; ++kb) {
        uint8_t* st = smem + C::SMEM_STAGES + stage * STAGE_BYTES;
        const int k0 = kb * BK;
        uint8_t* b_dst = st + 2 * A_BYTES;
        bool got = true;
        if (lane == 0) {
          got = mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status, ST_PRODUCER_EMPTY,
                                  WAIT_LIMIT_NS);
          if (got) {
            mbar_arrive_expect_tx(&full[stage], tx);
            tma_load_3d(st, CHAIN && !gu ? &tm_a2 : &tm_a0, &full[stage], k0, wrow0, tc.e);
            tma_load_3d(st + A_BYTES, CHAIN && !gu ? &tm_a2 : &tm_a1, &full[stage], k0, wrow1, tc.e);
            if (CHAIN && !gu) {
              // h rows in 16-row boxes (a decode tile has at most TBM = 32).
              for (int r = 0; r < n_tok; r += 16)
                tma_load_2d(b_dst + r * ROW_BYTES, &tm_c16, &full[stage], k0, static_cast<int>(tc.row0) + r);
            }
          }
        }
        if (__shfl_sync(FULL_MASK, got ? 1 : 0, 0) == 0) {
          ok = false;
          break;
        }
        if (gu) {
#pragma unroll
          for (int g = 0; g < G4; ++g) {
            const int gi = lane + 32 * g;
            if (gi < n_gather)
              tma_gather4(b_dst + gi * 4 * ROW_BYTES, &tm_b128, &full[stage], k0, tok[g][0], tok[g][1], tok[g][2],
                          tok[g][3]);
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
    if (!ok && lane == 0) {
      // Let the copies already in flight land before the block can exit.
      const uint32_t n_back = issued < STAGES ? issued : STAGES;
      for (uint32_t i = 1; i <= n_back; ++i) {
        const uint32_t n = issued - i;
        mbar_wait_bounded(&full[n % STAGES], (n / STAGES) & 1u, nullptr, args.status, ST_PRODUCER_DRAIN,
                          WAIT_LIMIT_NS);
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------------ scheduler + TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (uint32_t it = 0;; ++it) {
        const uint32_t slot = it % RING;
        if (!mbar_wait_bounded(&tile_empty[slot], ((it / RING) & 1u) ^ 1u, abort_flag, args.status,
                               ST_TILE_RING, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        const uint32_t claimed = atomicAdd(args.sched, 1u);
        const uint32_t tile = claimed < total ? claimed : TILE_END;
        if (tile == TILE_END) {
          ring[slot] = tile;
          mbar_arrive(&tile_full[slot]);  // release: the ring entry is visible to the waiters
          launch_dependents();  // this CTA claims no more tiles
          break;
        }
        bool gu;
        const TileCoord tc = tile_coord(tile, gu);
        const int n_tok = (tc.rows + 15) & ~15;        // N of this tile
        const int n128 = n_tok >> 7;                   // 128-row boxes
        const int n16 = (n_tok & 127) >> 4;            // then 16-row boxes
        const uint32_t tx = static_cast<uint32_t>(2 * A_BYTES + (GATHER ? 0 : n_tok * ROW_BYTES));
        const int wrow0 = gu ? tc.n * BM : tc.n * (2 * BM);
        const int wrow1 = gu ? tc.n * BM : tc.n * (2 * BM) + BM;
        const int k_blocks = CHAIN && !gu ? args.k_blocks2 : args.k_blocks;
        // Down tile (CHAIN): the expert's h rows, once every gate/up tile of
        // it has stored them; waited for before the tile is published, so
        // that the MMA and epilogue waits of a down tile start only once its
        // inputs exist.
        if (CHAIN && !gu &&
            !counter_wait_bounded(args.ready + tc.e,
                                  static_cast<uint32_t>(NUM_EPI_WARPS) * (tile_start[tc.e + 1] - tile_start[tc.e]),
                                  abort_flag, args.status, ST_CHAIN_READY, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        ring[slot] = tile;
        mbar_arrive(&tile_full[slot]);  // release: the ring entry is visible to the waiters
        const CUtensorMap* ma0 = CHAIN && !gu ? &tm_a2 : &tm_a0;
        const CUtensorMap* ma1 = CHAIN && !gu ? &tm_a2 : &tm_a1;
        const CUtensorMap* mb128 = CHAIN && !gu ? &tm_c128 : &tm_b128;
        const CUtensorMap* mb16 = CHAIN && !gu ? &tm_c16 : &tm_b16;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status,
                                 ST_PRODUCER_EMPTY, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + C::SMEM_STAGES + stage * STAGE_BYTES;
          const int k0 = kb * BK;
          mbar_arrive_expect_tx(&full[stage], tx);
          tma_load_3d(st, ma0, &full[stage], k0, wrow0, tc.e);
          tma_load_3d(st + A_BYTES, ma1, &full[stage], k0, wrow1, tc.e);
          if (!GATHER) {
            uint8_t* b_dst = st + 2 * A_BYTES;
            int r = 0;
            for (int b = 0; b < n128; ++b, r += 128)
              tma_load_2d(b_dst + r * ROW_BYTES, mb128, &full[stage], k0, static_cast<int>(tc.row0) + r);
            for (int b = 0; b < n16; ++b, r += 16)
              tma_load_2d(b_dst + r * ROW_BYTES, mb16, &full[stage], k0, static_cast<int>(tc.row0) + r);
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
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (uint32_t it = 0;; ++it) {
        const uint32_t slot = it % RING;
        if (!mbar_wait_bounded(&tile_full[slot], (it / RING) & 1u, abort_flag, args.status,
                               ST_TILE_RING, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        const uint32_t tile = ring[slot];
        if (tile == TILE_END) break;
        bool gu;
        const TileCoord tc = tile_coord(tile, gu);
        const int n_tok = (tc.rows + 15) & ~15;
        const int k_blocks = CHAIN && !gu ? args.k_blocks2 : args.k_blocks;
        const uint32_t idesc = idesc_f16(kBF16, BM, n_tok);
        const uint32_t acc = it % C::ACC;             // accumulator buffer of this tile
        const uint32_t acc_use = it / C::ACC;         // earlier tiles on this buffer
        if (!mbar_wait_bounded(&tempty[acc], (acc_use & 1u) ^ 1u, abort_flag, args.status, ST_MMA_TMEM_EMPTY,
                               WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + acc * C::ACC_COLS;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.status, ST_MMA_FULL,
                                 WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          // Token rows written by the loaders' cp.async (generic proxy) are
          // read by the tensor cores (async proxy).
          if (GATHER) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + C::SMEM_STAGES + stage * STAGE_BYTES);
          const uint32_t a1 = a0 + A_BYTES;
          const uint32_t b = a0 + 2 * A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint32_t accum = (kb > 0 || k > 0) ? 1u : 0u;
            const uint64_t bd = sdesc_kmajor_sw128(b + k * UMMA_K * 2);
            umma_f16(d0, sdesc_kmajor_sw128(a0 + k * UMMA_K * 2), bd, idesc, accum);
            umma_f16(d0 + C::D1, sdesc_kmajor_sw128(a1 + k * UMMA_K * 2), bd, idesc, accum);
          }
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
      }
      // Every MMA issued above completes before TMEM is released.
      umma_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr, args.status, ST_MMA_DRAIN, WAIT_LIMIT_NS);
    }
    __syncwarp();
  } else if (warp < FIRST_LOAD_WARP) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                    // 0..7
    const int quad = warp & 3;                  // TMEM lanes 32*quad .. 32*quad+31
    const int half = ew >> 2;                   // takes chunks half, half+2, ...
    uint16_t* xp = reinterpret_cast<uint16_t*>(smem + C::SMEM_XPOSE + ew * XPOSE_BYTES);
    const int rd_tok = lane >> 2;               // transpose read-back: token within 8
    const int rd_part = lane & 3;               // 16-byte run within the 64-byte row
    bool tiles_done = false;  // the tile loop ended at the scheduler's end mark, not on a failure
    for (uint32_t it = 0;; ++it) {
      const uint32_t slot = it % RING;
      bool ok = mbar_wait_bounded(&tile_full[slot], (it / RING) & 1u, abort_flag, args.status,
                                  ST_TILE_RING, WAIT_LIMIT_NS);
      const uint32_t tile = ok ? static_cast<uint32_t>(ring[slot]) : static_cast<uint32_t>(TILE_END);
      const bool all_ok = __all_sync(FULL_MASK, ok);
      if (!all_ok || tile == TILE_END) {
        tiles_done = all_ok;
        break;
      }
      bool gu;
      const TileCoord tc = tile_coord(tile, gu);
      const uint32_t acc = it % C::ACC;
      ok = mbar_wait_bounded(&tfull[acc], (it / C::ACC) & 1u, abort_flag, args.status, ST_EPI_TMEM_FULL,
                             WAIT_LIMIT_NS);
      // tcgen05.ld is warp-collective: the whole warp goes on or stops.
      if (!__all_sync(FULL_MASK, ok)) break;
      tc_fence_after();
      const int n_tok = (tc.rows + 15) & ~15;
      const uint32_t t_lane = tmem_base + acc * C::ACC_COLS + (static_cast<uint32_t>(quad * 32) << 16);
      const volatile uint32_t* bad = tile_bad + slot * BAD_WORDS;  // TOK_GATHER4: rows to write as zeros
      // The tile's outputs, compiled once per tile kind (G: gate/up).
      auto drain = [&](auto g_tag) {
      constexpr bool G = decltype(g_tag)::value;
      // Output columns of this warp's 32 lanes (two blocks for K4).
      const int64_t colA = G ? static_cast<int64_t>(tc.n) * BM + quad * 32
                              : static_cast<int64_t>(tc.n) * (2 * BM) + quad * 32;
      void* const out_main = CHAIN && !G ? args.out2 : args.out;
      const int n_out = CHAIN && !G ? args.n_out2 : args.n_out;
      for (int c0 = 32 * half; c0 < n_tok; c0 += 64) {
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(c0), v0);
        tmem_ld_32x32b_x32(t_lane + C::D1 + static_cast<uint32_t>(c0), v1);
        tmem_ld_wait();
        // K3 writes h, and in training mode also the pre-activations g and u
        // (the forward cache); K4 writes its two 128-column blocks.
        const int n_blk = G ? (args.out_g != nullptr ? 3 : 1) : 2;
        for (int blk = 0; blk < n_blk; ++blk) {
          // Lane = output column, j = token: write column-major, read token rows.
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float val;
            if (G) {
              const float gv = __uint_as_float(v0[j]), uv = __uint_as_float(v1[j]);
              val = blk == 0 ? silu_f32(gv) * uv : (blk == 1 ? gv : uv);
            } else {
              val = __uint_as_float(blk == 0 ? v0[j] : v1[j]);
            }
            const T hv = from_f32<T>(val);
            xp[j * 32 + lane] = *reinterpret_cast<const uint16_t*>(&hv);
          }
          __syncwarp();
          const int64_t col = colA + ((G || blk == 0) ? 0 : BM) + rd_part * 8;
          void* out_base = !G || blk == 0 ? out_main : (blk == 1 ? args.out_g : args.out_u);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int j = p * 8 + rd_tok;
            const uint4 row = *reinterpret_cast<const uint4*>(xp + j * 32 + rd_part * 8);
            const int t_in = c0 + j;
            if (t_in < tc.rows && tc.row0 + static_cast<uint32_t>(t_in) < args.rows_total &&
                col + 8 <= n_out) {
              T* dst = static_cast<T*>(out_base) + (static_cast<int64_t>(tc.row0) + t_in) * n_out + col;
              const bool zero = LOAD == TOK_GATHER4 && G && ((bad[t_in >> 5] >> (t_in & 31)) & 1u) != 0;
              *reinterpret_cast<uint4*>(dst) = zero ? make_uint4(0u, 0u, 0u, 0u) : row;
            }
          }
          __syncwarp();
        }
      }
      };
      if (!CHAIN) drain(std::integral_constant<bool, GATE_UP>{});
      else if (gu) drain(std::true_type{});
      else drain(std::false_type{});
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[acc]);
        mbar_arrive(&tile_empty[slot]);
      }
      if (CHAIN && gu) {
        // Publish this warp's h rows of the tile to the down tiles (other
        // CTAs' TMA reads): each lane's stores, then one release per warp.
        // After the accumulator is released, so that waiting for the stores
        // to drain overlaps the next tile's MMAs.
        __threadfence();
        __syncwarp();
        if (lane == 0) counter_release_add(args.ready + tc.e);
      }
      if (COMB && !gu) {
        // Publish this warp's y rows of the tile to the combine (other CTAs'
        // reads): each lane's stores, then one release per warp on the done
        // counter, after the accumulator is released.
        __threadfence();
        __syncwarp();
        if (lane == 0) counter_release_add(args.comb_done);
      }
    }
    if (COMB && tiles_done) {
      // Every tile was claimed by a running CTA before this one saw the end
      // mark, so the done counter reaches its total and the wait ends. One
      // warp per CTA polls it (bounded) and raises a shared flag for the
      // others (whose wait is bounded too).
      volatile int* go = abort_flag + 1;
      bool ok = true;
      if (ew == 0) {
        if (lane == 0)
          ok = counter_wait_bounded(args.comb_done, static_cast<uint32_t>(NUM_EPI_WARPS) * tile_start2[args.E],
                                    abort_flag, args.status, ST_COMB_WAIT, WAIT_LIMIT_NS);
        ok = __shfl_sync(FULL_MASK, ok ? 1 : 0, 0) != 0;
        if (ok && lane == 0) {
          __threadfence_block();
          *go = 1;
        }
      } else {
        if (lane == 0) {
          const uint64_t t0 = globaltimer_ns();
          for (uint32_t poll = 0; *go == 0; ++poll) {
            __nanosleep(128);
            if ((poll & 15u) == 15u && (*abort_flag != 0 || globaltimer_ns() - t0 > WAIT_LIMIT_NS)) {
              if (*abort_flag == 0) {
                *abort_flag = 1;
                record_status(args.status, ST_COMB_WAIT);
              }
              ok = false;
              break;
            }
          }
          __threadfence();  // the flag's writer had acquired the counter at GPU scope
        }
        ok = __shfl_sync(FULL_MASK, ok ? 1 : 0, 0) != 0;
      }
      __syncwarp();
      if (ok) {
        // Tokens gw, gw + nw, gw + 2 nw, ... of the global warp gw, up to
        // COMB_TOKENS_PER_PASS per pass: stage their (row, weight) pairs,
        // then combine them in one stream of loads.
        constexpr int P = COMB_TOKENS_PER_PASS;
        uint32_t* rows = reinterpret_cast<uint32_t*>(xp);
        float* wts = reinterpret_cast<float*>(xp) + COMB_PAIRS;
        const int k = args.comb_k;
        const uint32_t nw = gridDim.x * NUM_EPI_WARPS;
        const uint32_t gw = blockIdx.x * NUM_EPI_WARPS + ew;
        for (uint32_t t0 = gw; t0 < args.comb_T; t0 += P * nw) {
          uint32_t tok[P];
          bool bad[P];
          int n = 0;
#pragma unroll
          for (int i = 0; i < P; ++i) {
            tok[i] = t0 + static_cast<uint32_t>(i) * nw;
            bad[i] = false;
            if (tok[i] < args.comb_T) n = i + 1;
          }
          for (int p0 = 0; p0 < n * k; p0 += 32) {
            const int p = p0 + lane;
            const int pi = p / k, pj = p - pi * k;
            bool inval = false;
            if (p < n * k) {
              uint32_t t = 0;
#pragma unroll
              for (int i = 0; i < P; ++i)
                if (i == pi) t = tok[i];
              const int64_t sidx = static_cast<int64_t>(t) * k + pj;
              const uint32_t r = args.comb_inv[sidx];
              inval = r >= args.rows_total;
              rows[p] = inval ? 0u : r;
              wts[p] = comb_weight(args.comb_w, args.comb_wdt, sidx);
            }
#pragma unroll
            for (int i = 0; i < P; ++i) bad[i] |= __any_sync(FULL_MASK, inval && pi == i);
          }
          __syncwarp();
          comb_tokens<T, P>(n, tok, bad, args, rows, wts, lane);
          __syncwarp();  // the staged pairs are rewritten by the next pass
        }
      }
    }
  } else if (GATHER) {
    // ------------------------------------------------------------ token-row loaders (gather mode)
    // Row r of a tile's token block is x[row_src[row0 + r] / top_k]. In each
    // copy instruction lanes 8i..8i+7 move the eight 16-byte chunks of one
    // 128-byte row slice (four whole rows per instruction), each chunk to its
    // 128-byte-swizzle position (chunk ^ (row & 7)), the layout a TMA copy
    // with 128-byte swizzle produces. Rows past the tile's rows up to its
    // 16-row N are zero-filled.
    constexpr int RPT = TBM / (4 * NUM_LOAD_WARPS);  // rows per thread per stage
    const int lw = warp - FIRST_LOAD_WARP;
    const int q = lane & 7;
    const int rsub = lw * 4 + (lane >> 3);           // row = rsub + 16 * j
    int stage = 0;
    uint32_t phase = 0;
    for (uint32_t it = 0;; ++it) {
      const uint32_t slot = it % RING;
      bool ok = mbar_wait_bounded(&tile_full[slot], (it / RING) & 1u, abort_flag, args.status,
                                  ST_TILE_RING, WAIT_LIMIT_NS);
      const uint32_t tile = ok ? static_cast<uint32_t>(ring[slot]) : static_cast<uint32_t>(TILE_END);
      if (!__all_sync(FULL_MASK, ok) || tile == TILE_END) break;
      const TileCoord tc = decode_tile(tile, tile_start, args.E, args.offsets, TB, args.n_wblocks);
      const int n_tok = (tc.rows + 15) & ~15;
      const uint8_t* src[RPT];
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        const int r = rsub + 16 * j;
        src[j] = nullptr;
        if (r < tc.rows && tc.row0 + static_cast<uint32_t>(r) < args.rows_total) {
          const uint32_t tok = args.row_src[tc.row0 + r] / static_cast<uint32_t>(args.top_k);
          if (tok < args.x_rows) src[j] = args.gx + static_cast<int64_t>(tok) * args.k_bytes;
        }
      }
      for (int kb = 0; kb < args.k_blocks; ++kb) {
        ok = mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, args.status, ST_LOADER_EMPTY,
                               WAIT_LIMIT_NS);
        if (!__all_sync(FULL_MASK, ok)) break;
        const uint32_t b = smem_u32(smem + C::SMEM_STAGES + stage * STAGE_BYTES + 2 * A_BYTES);
        const int kbyte = kb * (BK * 2) + q * 16;
        const bool kin = kbyte < args.k_bytes;
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
          const int r = rsub + 16 * j;
          if (r < n_tok) {
            const uint32_t dst = b + static_cast<uint32_t>(r * ROW_BYTES + ((q ^ (r & 7)) << 4));
            if (src[j] != nullptr && kin) cp_async_16(dst, src[j] + kbyte, 16);
            else cp_async_16(dst, args.gx, 0);
          }
        }
        cp_async_mbar_arrive_noinc(&full[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&tile_empty[slot]);
    }
    // No copy may land after the block has exited.
    cp_async_wait_all();
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

// [outer, inner] row-major 16-bit matrix, box 64 (inner) x box_rows (outer).
bool encode_2d(CUtensorMap* m, moe_dtype dt, const void* ptr, uint64_t inner, uint64_t outer,
               uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, tmap_dtype(dt), 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [E, rows, inner] row-major 16-bit tensor, box 64 x box_rows x 1.
bool encode_3d(CUtensorMap* m, moe_dtype dt, const void* ptr, uint64_t inner, uint64_t rows,
               uint64_t E, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {inner, rows, E};
  const cuuint64_t strides[2] = {inner * 2, rows * inner * 2};
  const cuuint32_t box[3] = {BK, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, tmap_dtype(dt), 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Upper bound on the tile count: token blocks of at most tbm rows per expert.
int64_t tile_bound(int64_t rows, int E, int64_t n_wblocks, int tbm) {
  const int64_t t_blocks = rows / tbm + (rows < E ? rows : E);
  return t_blocks * n_wblocks;
}

template <typename T, bool GATE_UP, int TBM, int LOAD = TOK_DENSE>
cudaError_t launch_one(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b128,
                       const CUtensorMap& b16, const TcArgs& args, int num_sms, cudaStream_t stream,
                       bool sched_zeroed) {
  auto kern = experts_tc_kernel<T, GATE_UP, TBM, LOAD>;
  constexpr int SMEM_BYTES = TcCfg<TBM>::SMEM_BYTES;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (err != cudaSuccess) return err;
  const int grid = static_cast<int>(args.tile_cap < static_cast<uint32_t>(num_sms) ? args.tile_cap : num_sms);
  if (grid <= 0) return cudaSuccess;
  if (!sched_zeroed) {
    err = cudaMemsetAsync(args.sched, 0, sizeof(uint32_t), stream);
    if (err != cudaSuccess) return err;
  }
  return launch_dependent(kern, dim3(grid), dim3(num_threads<LOAD>()), SMEM_BYTES, stream, a0, a1, b128, b16, a0,
                          b128, b16, args);
}

// K3 and K4 in one launch (CHAIN): gate/up tiles, then down tiles that wait
// for their expert's h rows. args carries both stages' sizes, y in out2 and
// the per-expert ready counters (zero at launch, like the tile counter).
template <typename T, int TBM, int LOAD, bool COMB>
cudaError_t launch_chain(const TcWeights& w, const CUtensorMap& x128, const CUtensorMap& x16,
                         const CUtensorMap& h128, const CUtensorMap& h16, const TcArgs& args, int num_sms,
                         cudaStream_t stream) {
  auto kern = experts_tc_kernel<T, true, TBM, LOAD, true, COMB>;
  constexpr int SMEM_BYTES = TcCfg<TBM>::SMEM_BYTES_CHAIN;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (err != cudaSuccess) return err;
  const int grid = static_cast<int>(args.tile_cap < static_cast<uint32_t>(num_sms) ? args.tile_cap : num_sms);
  if (grid <= 0) return cudaSuccess;
  return launch_dependent(kern, dim3(grid), dim3(num_threads<LOAD>()), SMEM_BYTES, stream, w.gate, w.up, x128, x16,
                          w.down, h128, h16, args);
}

template <typename T>
cudaError_t launch_stage(const TcWeights& w, moe_dtype dtype, bool gate_up, const void* a,
                         const TcGather* gather, const TcCache* cache, const uint32_t* offsets, int E, int64_t rows,
                         int64_t H, int64_t I, void* out, uint32_t* sched, int num_sms, cudaStream_t stream,
                         const char** why, bool sz) {
  uint32_t* status = nullptr;
  cudaError_t err = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_moe_device_status);
  if (err != cudaSuccess) return err;
  const int64_t K = gate_up ? H : I;
  const int64_t n_out = gate_up ? I : H;
  // Token maps: 128- and 16-row boxes over the dense rows, or x with a
  // one-row box for the row gathers (t16 is then never dereferenced).
  CUtensorMap t128 = w.gate, t16 = w.gate;
  const bool maps_ok =
      gather == nullptr
          ? encode_2d(&t128, dtype, a, static_cast<uint64_t>(K), static_cast<uint64_t>(rows), 128) &&
                encode_2d(&t16, dtype, a, static_cast<uint64_t>(K), static_cast<uint64_t>(rows), 16)
          : encode_2d(&t128, dtype, gather->x, static_cast<uint64_t>(K), static_cast<uint64_t>(gather->x_rows), 1);
  if (!maps_ok) {
    *why = "cuTensorMapEncodeTiled rejected the token tensor map";
    return cudaErrorInvalidValue;
  }
  const int nw = static_cast<int>(gate_up ? (I + BM - 1) / BM : (H + 2 * BM - 1) / (2 * BM));
  // Decode-sized batches (at most 8 rows per expert on average) stream
  // weights with 32-token blocks, deeper pipelines and double-buffered
  // accumulators; prefill uses 256-token blocks (each weight tile feeds
  // twice the tokens; measured faster than 128 with double buffering).
  const bool small = rows <= 8 * static_cast<int64_t>(E);
  const int64_t cap = tile_bound(rows, E, nw, small ? 32 : 256);
  TcArgs args{offsets, out, sched, E, nw, static_cast<int>((K + BK - 1) / BK), static_cast<int>(n_out),
              static_cast<uint32_t>(rows), static_cast<uint32_t>(cap), status,
              nullptr, nullptr, 1, 0, static_cast<int>(K * 2), nullptr, nullptr};
  if (cache != nullptr) {
    if (!gate_up) {
      *why = "the pre-activation cache belongs to the gate/up stage";
      return cudaErrorInvalidValue;
    }
    args.out_g = cache->g;
    args.out_u = cache->u;
  }
  if (gather != nullptr) {
    if (!gate_up) {
      *why = "the gather mode applies to the gate/up stage only";
      return cudaErrorInvalidValue;
    }
    args.gx = static_cast<const uint8_t*>(gather->x);
    args.row_src = gather->row_src;
    args.top_k = gather->top_k;
    args.x_rows = static_cast<uint32_t>(gather->x_rows);
    // Decode-sized tiles (at most 32 rows): TMA row gathers, a few per
    // stage. Prefill-sized tiles: 256 rows per stage are 64 row gathers,
    // and the TMA unit spends about as long on one 4-row gather as on a
    // whole 128-row box (gate/up at the prefill workload: 466 us with row
    // gathers, 253 us with the cp.async loader warps).
    if (small) return launch_one<T, true, 32, TOK_GATHER4>(w.gate, w.up, t128, t16, args, num_sms, stream, sz);
    return launch_one<T, true, 256, TOK_CPASYNC>(w.gate, w.up, t128, t16, args, num_sms, stream, sz);
  }
  if (small) {
    if (gate_up) return launch_one<T, true, 32>(w.gate, w.up, t128, t16, args, num_sms, stream, sz);
    return launch_one<T, false, 32>(w.down, w.down, t128, t16, args, num_sms, stream, sz);
  }
  if (gate_up) return launch_one<T, true, 256>(w.gate, w.up, t128, t16, args, num_sms, stream, sz);
  return launch_one<T, false, 256>(w.down, w.down, t128, t16, args, num_sms, stream, sz);
}

template <typename T, int TBM, int LOAD>
cudaError_t launch_chain_comb(const TcWeights& w, const CUtensorMap& x128, const CUtensorMap& x16,
                              const CUtensorMap& h128, const CUtensorMap& h16, const TcArgs& args, int num_sms,
                              cudaStream_t stream, bool comb) {
  if (comb) return launch_chain<T, TBM, LOAD, true>(w, x128, x16, h128, h16, args, num_sms, stream);
  return launch_chain<T, TBM, LOAD, false>(w, x128, x16, h128, h16, args, num_sms, stream);
}

template <typename T>
cudaError_t chain_stage(const TcWeights& w, moe_dtype dtype, const void* xd, const TcGather* gather,
                        const TcCache* cache, const uint32_t* offsets, int E, int64_t rows, int64_t H, int64_t I, void* h, void* y,
                        uint32_t* sched, uint32_t* ready, int num_sms, cudaStream_t stream, const char** why,
                        const TcCombine* comb) {
  uint32_t* status = nullptr;
  cudaError_t err = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_moe_device_status);
  if (err != cudaSuccess) return err;
  const bool small = rows <= 8 * static_cast<int64_t>(E);
  if (gather != nullptr && !small) {
    *why = "the chained experts gather x rows only for decode-sized batches";
    return cudaErrorInvalidValue;
  }
  CUtensorMap x128 = w.gate, x16 = w.gate, h128 = w.gate, h16 = w.gate;
  const bool maps_ok =
      (gather == nullptr
           ? encode_2d(&x128, dtype, xd, static_cast<uint64_t>(H), static_cast<uint64_t>(rows), 128) &&
                 encode_2d(&x16, dtype, xd, static_cast<uint64_t>(H), static_cast<uint64_t>(rows), 16)
           : encode_2d(&x128, dtype, gather->x, static_cast<uint64_t>(H), static_cast<uint64_t>(gather->x_rows), 1)) &&
      encode_2d(&h128, dtype, h, static_cast<uint64_t>(I), static_cast<uint64_t>(rows), 128) &&
      encode_2d(&h16, dtype, h, static_cast<uint64_t>(I), static_cast<uint64_t>(rows), 16);
  if (!maps_ok) {
    *why = "cuTensorMapEncodeTiled rejected a token tensor map";
    return cudaErrorInvalidValue;
  }
  const int nw3 = static_cast<int>((I + BM - 1) / BM);
  const int nw4 = static_cast<int>((H + 2 * BM - 1) / (2 * BM));
  const int tbm = small ? 32 : 256;
  const int64_t cap = tile_bound(rows, E, nw3, tbm) + tile_bound(rows, E, nw4, tbm);
  TcArgs args{offsets, h, sched, E, nw3, static_cast<int>((H + BK - 1) / BK), static_cast<int>(I),
              static_cast<uint32_t>(rows), static_cast<uint32_t>(cap), status,
              nullptr, nullptr, 1, 0, static_cast<int>(H * 2), nullptr, nullptr,
              y, nw4, static_cast<int>((I + BK - 1) / BK), static_cast<int>(H), ready};
  if (cache != nullptr) {
    args.out_g = cache->g;
    args.out_u = cache->u;
  }
  if (comb != nullptr) {
    if (cache != nullptr || comb->T * static_cast<int64_t>(comb->top_k) != rows || comb->top_k < 1 ||
        comb->top_k > COMB_MAX_K) {
      *why = "the fused combine needs rows == T * top_k, top_k <= 256 and no training cache";
      return cudaErrorInvalidValue;
    }
    args.comb_inv = comb->inv;
    args.comb_w = comb->weights;
    args.comb_wdt = static_cast<int>(comb->weights_dtype);
    args.comb_k = comb->top_k;
    args.comb_T = static_cast<uint32_t>(comb->T);
    args.comb_done = comb->done;
    args.comb_out = comb->out;
  }
  const bool cb = comb != nullptr;
  if (gather != nullptr) {
    args.gx = static_cast<const uint8_t*>(gather->x);
    args.row_src = gather->row_src;
    args.top_k = gather->top_k;
    args.x_rows = static_cast<uint32_t>(gather->x_rows);
    return launch_chain_comb<T, 32, TOK_GATHER4>(w, x128, x16, h128, h16, args, num_sms, stream, cb);
  }
  if (small) return launch_chain_comb<T, 32, TOK_DENSE>(w, x128, x16, h128, h16, args, num_sms, stream, cb);
  return launch_chain_comb<T, 256, TOK_DENSE>(w, x128, x16, h128, h16, args, num_sms, stream, cb);
}

}  // namespace

cudaError_t launch_experts_tc_chain(const TcWeights& w, moe_dtype dtype, const void* xd, const TcGather* gather,
                                    const TcCache* cache, const uint32_t* offsets, int E, int64_t rows, int64_t H,
                                    int64_t I, void* h, void* y, uint32_t* sched, uint32_t* ready, int num_sms,
                                    cudaStream_t stream, const char** why, const TcCombine* comb) {
  if (rows == 0) return cudaSuccess;
  if (dtype == MOE_BF16)
    return chain_stage<__nv_bfloat16>(w, dtype, xd, gather, cache, offsets, E, rows, H, I, h, y, sched, ready,
                                      num_sms, stream, why, comb);
  return chain_stage<__half>(w, dtype, xd, gather, cache, offsets, E, rows, H, I, h, y, sched, ready, num_sms,
                             stream, why, comb);
}

bool tc_encode_weights(const void* gate, const void* up, const void* down, moe_dtype dtype,
                       int64_t E, int64_t H, int64_t I, TcWeights* out, const char** why) {
  if (encode_fn() == nullptr) {
    *why = "the CUDA driver does not provide cuTensorMapEncodeTiled";
    return false;
  }
  if (!encode_3d(&out->gate, dtype, gate, H, I, E, BM) || !encode_3d(&out->up, dtype, up, H, I, E, BM) ||
      !encode_3d(&out->down, dtype, down, I, H, E, BM)) {
    *why = "cuTensorMapEncodeTiled rejected an expert weight tensor map";
    return false;
  }
  return true;
}

cudaError_t launch_experts_tc(const TcWeights& w, moe_dtype dtype, bool gate_up, const void* a,
                              const TcGather* gather, const TcCache* cache, const uint32_t* offsets, int E,
                              int64_t rows, int64_t H, int64_t I, void* out, uint32_t* sched, int num_sms,
                              cudaStream_t stream, const char** why, bool sched_zeroed) {
  if (rows == 0) return cudaSuccess;
  if (dtype == MOE_BF16)
    return launch_stage<__nv_bfloat16>(w, dtype, gate_up, a, gather, cache, offsets, E, rows, H, I, out, sched,
                                       num_sms, stream, why, sched_zeroed);
  return launch_stage<__half>(w, dtype, gate_up, a, gather, cache, offsets, E, rows, H, I, out, sched, num_sms,
                              stream, why, sched_zeroed);
}

cudaError_t device_status_ptr(uint32_t** p) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(p), g_moe_device_status);
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
