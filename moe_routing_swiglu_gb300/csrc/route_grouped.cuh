// Grouped, bias-corrected sigmoid routing of one token by one warp: the body
// of the grouped routing kernel (route_grouped.cu) and of the routing phase
// of the fused route + dispatch kernel (route_dispatch.cu), so both give the
// same bits.
//
// ruDNN user guide, section 10 "Group-limited sigmoid MoE routing": FP32
// scores s_i = 1 / (1 + exp(-l_i)); corrected scores c_i = s_i + bias_i steer
// the selection only; a group's score is its largest c, or the sum of its two
// largest c (group_top_two); the selected_groups best groups are kept, then
// the top_k largest c among their experts, ties to the lower id (groups and
// experts alike); weights are the uncorrected s of the chosen experts,
// optionally divided by their sum, times scale, cast to the logits dtype.
// The group-max / top-groups / mask / top-k order is the DeepSeek-style
// routing of "PyTorch general ops", section "MoE routing: topk, scatter and
// masked_fill".
//
// Exactness. Every value is rounded the way a plain FP32 evaluation rounds it
// (exp rounded once to FP32, then 1 + e, then 1 / d, then s + b; group sums
// as one FP32 add), so equal inputs give equal keys and ties resolve by id.
// The one step CUDA has no correctly rounded FP32 form of is exp. The first
// pass uses expf (within 2 ulp): its s is within 5 FP32 ulps of 1.0 of the
// correctly rounded s, hence c within 6 * 2^-23 * max(1, |c|) and a group
// sum within 14 * 2^-23 * max(1, max|c|). The pass checks every comparison
// the result depends on (adjacent selected slots, the best unselected expert,
// the last selected against the best unselected group); if any margin is
// within tau = 2^-16 * max(1, max|c|) of a tie, the row is redone from the
// double-precision exp rounded to FP32 (a correctly rounded FP32 exp except
// where the double result sits within an ulp of an FP32 rounding boundary).
// Weights always come from that double-based s, so they do not depend on
// which pass decided the selection.
//
// Layout: lane l holds experts l*V .. l*V+V-1 (V = ceil(E/32) rounded to a
// power of two). The block keeps the bias and every expert's group id in
// shared memory; each warp has a buffer of its row's c in id order, which the
// group scores are read from.
#pragma once

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace grouped_detail {

constexpr int GR_MAX_GROUPS = 128;

__device__ __forceinline__ uint32_t order_bits(float v) {
  const uint32_t b = __float_as_uint(v + 0.0f);  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float from_order_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// Larger key = larger value, then smaller id. Key 0 means "none".
__device__ __forceinline__ uint64_t value_key(float v, uint32_t id) {
  return (static_cast<uint64_t>(order_bits(v)) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - id);
}

// A NaN group score (+inf and -inf in one group's top two) ranks below every
// number, ties to the lower group id.
__device__ __forceinline__ uint64_t group_key(float v, uint32_t g) {
  return isnan(v) ? static_cast<uint64_t>(0xFFFFFFFFu - g) : value_key(v, g);
}

__device__ __forceinline__ float key_value(uint64_t key) {
  const uint32_t hi = static_cast<uint32_t>(key >> 32);
  return hi == 0 ? __int_as_float(0x7FC00000) : from_order_bits(hi);
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const uint64_t o = __shfl_xor_sync(FULL_MASK, v, off);
    v = v > o ? v : o;
  }
  return v;
}

__device__ __forceinline__ float sigmoid_fast(float l) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l)));
}

__device__ __forceinline__ float sigmoid_exact(float l) {
  const float e = __double2float_rn(exp(-static_cast<double>(l)));
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

// Insert x into a descending top-two (m1 >= m2).
__device__ __forceinline__ void top2_insert(float& m1, float& m2, float x) {
  if (x > m1) {
    m2 = m1;
    m1 = x;
  } else {
    m2 = fmaxf(m2, x);
  }
}

// The selected-group bitmask lives in four warp-uniform words.
__device__ __forceinline__ bool group_selected(const uint32_t (&gm)[4], uint32_t g) {
  uint32_t w = gm[0];
  if (g >= 32) w = gm[1];
  if (g >= 64) w = gm[2];
  if (g >= 96) w = gm[3];
  return (w >> (g & 31)) & 1u;
}

// One selection pass over a row held as logits l[V] (blocked layout). With
// EXACT = false, s comes from expf and the return value says whether any
// comparison the result depends on lies within tau of a tie (the caller then
// runs the EXACT pass). With EXACT = true, s comes from the double-precision
// exp rounded to FP32 and the result is final. Chosen ids land in keep_id
// (slot j on lane j % 32, word j / 32).
template <bool EXACT, int V>
__device__ __forceinline__ bool select_pass(const float (&l)[V], const float* __restrict__ bias_sm,
                                            const uint8_t* __restrict__ grp_sm, float* __restrict__ my_c,
                                            int E, const GroupRouteParams& p, int lane, uint32_t (&keep_id)[2]) {
  const int G = p.group_size;
  __syncwarp();  // earlier readers of my_c are done
  float cmax = 0.0f;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int id = lane * V + v;
    if (id < E) {
      const float s = EXACT ? sigmoid_exact(l[v]) : sigmoid_fast(l[v]);
      const float c = __fadd_rn(s, bias_sm[id]);
      my_c[id] = c;
      cmax = fmaxf(cmax, fabsf(c));
    }
  }
  float tau = 0.0f;
  if (!EXACT) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(FULL_MASK, cmax, off));
    tau = fmaxf(1.0f, cmax) * 0x1p-16f;
  }
  __syncwarp();

  // Group scores: lane g (+32 r) ends with group g's score in gs[r].
  float gs[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (G >= 32) {  // then groups <= 32: the warp scans one group at a time
    for (int g = 0; g < p.groups; ++g) {
      float m1 = -INFINITY, m2 = -INFINITY;
      for (int i = lane; i < G; i += 32) top2_insert(m1, m2, my_c[g * G + i]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float o1 = __shfl_xor_sync(FULL_MASK, m1, off);
        const float o2 = __shfl_xor_sync(FULL_MASK, m2, off);
        const float n2 = fmaxf(fminf(m1, o1), fmaxf(m2, o2));
        m1 = fmaxf(m1, o1);
        m2 = n2;
      }
      if (lane == g) gs[0] = p.top_two ? __fadd_rn(m1, m2) : m1;
    }
  } else {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int g = r * 32 + lane;
      if (g < p.groups) {
        float m1 = -INFINITY, m2 = -INFINITY;
        for (int i = 0; i < G; ++i) top2_insert(m1, m2, my_c[g * G + i]);
        gs[r] = p.top_two ? __fadd_rn(m1, m2) : m1;
      }
    }
  }

  uint64_t gkey[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int g = r * 32 + lane;
    gkey[r] = g < p.groups ? group_key(gs[r], static_cast<uint32_t>(g)) : 0ull;
  }
  uint32_t gm[4] = {0u, 0u, 0u, 0u};
  bool near = false;
  float last = 0.0f;
  for (int j = 0; j < p.selected; ++j) {
    uint64_t best = gkey[0];
#pragma unroll
    for (int r = 1; r < 4; ++r) best = best > gkey[r] ? best : gkey[r];
    best = warp_max_u64(best);
    const uint32_t g = 0xFFFFFFFFu - static_cast<uint32_t>(best);
    if (lane == static_cast<int>(g & 31)) {
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (r == static_cast<int>(g >> 5)) gkey[r] = 0ull;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
      if (r == static_cast<int>(g >> 5)) gm[r] |= 1u << (g & 31);
    if (!EXACT) last = key_value(best);
  }
  if (!EXACT && p.selected < p.groups) {
    uint64_t best = gkey[0];
#pragma unroll
    for (int r = 1; r < 4; ++r) best = best > gkey[r] ? best : gkey[r];
    best = warp_max_u64(best);
    if (!(__fsub_rn(last, key_value(best)) > tau)) near = true;
  }

  // Expert keys: only experts of the selected groups take part.
  uint64_t key[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int id = lane * V + v;
    key[v] = (id < E && group_selected(gm, grp_sm[id])) ? value_key(my_c[id], static_cast<uint32_t>(id)) : 0ull;
  }
  float prev = 0.0f;
  for (int j = 0; j < p.k; ++j) {
    uint64_t best = key[0];
#pragma unroll
    for (int v = 1; v < V; ++v) best = best > key[v] ? best : key[v];
    best = warp_max_u64(best);
    const uint32_t id = 0xFFFFFFFFu - static_cast<uint32_t>(best);
    if (lane == static_cast<int>(id / V)) {
      const int slot = static_cast<int>(id % V);
#pragma unroll
      for (int v = 0; v < V; ++v)
        if (v == slot) key[v] = 0ull;
    }
    if (lane == (j & 31)) {
      if (j < 32) keep_id[0] = id;
      else keep_id[1] = id;
    }
    if (!EXACT) {
      const float cv = key_value(best);
      if (j > 0 && !(__fsub_rn(prev, cv) > tau)) near = true;
      prev = cv;
    }
  }
  if (!EXACT) {
    uint64_t best = key[0];
#pragma unroll
    for (int v = 1; v < V; ++v) best = best > key[v] ? best : key[v];
    best = warp_max_u64(best);
    if (best != 0ull && !(__fsub_rn(prev, key_value(best)) > tau)) near = true;
  }
  return near;
}


}  // namespace grouped_detail

// Routes token t (the whole warp calls it). bias_sm and grp_sm are the
// block's shared copies of the bias (0 without one) and of every expert's
// group id; bias_nan says whether any bias is NaN; my_c is the warp's
// private shared buffer of 32*V floats. Writes indices[t*k + j],
// weights[t*k + j] and, if weights32 is not NULL, the FP32 weight. On return
// keep_id[q] holds, on lane l, the expert of slot j = q*32 + l (j < k <= 64).
template <typename TL, int V>
__device__ __forceinline__ void route_token_grouped(const TL* __restrict__ logits, int64_t t, int E,
                                                    const GroupRouteParams& p, const float* __restrict__ bias_sm,
                                                    const uint8_t* __restrict__ grp_sm, bool bias_nan, int lane,
                                                    float* my_c, uint32_t* __restrict__ indices,
                                                    TL* __restrict__ weights, float* __restrict__ weights32,
                                                    uint32_t (&keep_id)[2]) {
  using namespace grouped_detail;
  const int k = p.k;
  const float qnan = __int_as_float(0x7FC00000);
  const TL* row = logits + t * E;
  uint32_t* idx_row = indices + t * k;
  float l[V];
  bool has_nan = bias_nan;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int id = lane * V + v;
    l[v] = id < E ? to_f32(row[id]) : 0.0f;
    has_nan |= id < E && isnan(l[v]);
  }
  if (__any_sync(FULL_MASK, has_nan)) {
    keep_id[0] = static_cast<uint32_t>(lane);
    keep_id[1] = static_cast<uint32_t>(lane + 32);
    for (int j = lane; j < k; j += 32) {
      idx_row[j] = static_cast<uint32_t>(j);
      weights[t * k + j] = from_f32<TL>(qnan);
      if (weights32 != nullptr) weights32[t * k + j] = qnan;
    }
    return;
  }

  keep_id[0] = 0u;
  keep_id[1] = 0u;
  if (select_pass<false>(l, bias_sm, grp_sm, my_c, E, p, lane, keep_id))
    select_pass<true>(l, bias_sm, grp_sm, my_c, E, p, lane, keep_id);

  // Weights from the double-based s of the chosen experts (warp-uniform
  // branches, so the second word costs nothing unless top_k > 32).
  float w[2] = {0.0f, 0.0f};
  if (lane < k) w[0] = sigmoid_exact(to_f32(row[keep_id[0]]));
  if (k > 32 && lane + 32 < k) w[1] = sigmoid_exact(to_f32(row[keep_id[1]]));
  if (p.renormalize) {
    float z = 0.0f;
    for (int j = 0; j < k; ++j) {
      const float wj = __shfl_sync(FULL_MASK, j < 32 ? w[0] : w[1], j & 31);
      z = __fadd_rn(z, wj);
    }
    w[0] = __fdiv_rn(w[0], z);
    w[1] = __fdiv_rn(w[1], z);
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int j = q * 32 + lane;
    if (j < k) {
      const float wj = __fmul_rn(w[q], p.scale);
      idx_row[j] = keep_id[q];
      weights[t * k + j] = from_f32<TL>(wj);
      if (weights32 != nullptr) weights32[t * k + j] = wj;
    }
  }
}

}  // namespace moe
