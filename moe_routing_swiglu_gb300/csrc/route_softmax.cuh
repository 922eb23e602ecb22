// Softmax / top-k routing of one token by one warp: the body of the routing
// kernel (route.cu) and of the routing phase of the fused route + dispatch
// kernel (route_dispatch.cu), so both give the same bits.
//
// ruDNN user guide, section 4 "Routing contract": softmax over all E experts
// in FP32, then top-k with ties to the lower expert id, optional renormalize,
// then a cast to the logits dtype; rows with a NaN, a +inf or only -inf keep
// NaN weights. The max-shifted softmax follows "tiny-llm deep dive 5: ops.rs"
// (section on softmax).
//
// Layout: lane l of the warp holds experts l*V .. l*V+V-1 (V = ceil(E/32)
// rounded up to a power of two), so walking lanes then registers visits the
// experts in id order.
//  * The denominator s = e_0 + e_1 + ... + e_{E-1} is a left-to-right FP32
//    sum (the order the oracle uses, so FP32 weights differ only by expf's
//    ulps): the lanes store their e_i to a warp-private shared buffer in id
//    order and every lane adds them back in that order (broadcast reads).
//  * Selection is k rounds of a warp arg-max. Every expert has a key that
//    orders it by logit, then by the complement of its id, so the largest
//    key is the largest logit with ties to the smaller id. 16-bit logits
//    (F16/BF16): one 32-bit key (order-preserving bits of the 16-bit value,
//    then 0xFFFF - id) and one warp max reduction (redux.sync) per round.
//    F32 logits: the order-preserving 32-bit value first (one reduction),
//    then, among the experts holding it, 0xFFFF - id (a second one). The
//    owner lane zeroes a taken key (every real key is above zero).
//  * Slot j's lane then reads its e_j back from that buffer (the value the sum
//    used), divides by s, and the renormalizing sum is taken over slots
//    0..k-1 in order.
#pragma once

#include "moe_common.cuh"

namespace moe {
namespace route_detail {

// Order-preserving unsigned images of a float: a larger image is a larger
// value; -0 is folded into +0 first, so the two compare equal, as floats do.
__device__ __forceinline__ uint32_t ord32(float v) {
  const uint32_t b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ uint32_t ord16(uint16_t raw) {
  const uint32_t b = raw == 0x8000u ? 0u : raw;  // -0 -> +0
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}
template <typename TL>
__device__ __forceinline__ uint16_t bits16(TL v) {
  return *reinterpret_cast<const uint16_t*>(&v);
}

// The V logits of lane `lane` (experts lane*V .. lane*V+V-1, -inf past E)
// and their raw 16-bit patterns (16-bit dtypes), with one vector load when
// the row allows it.
template <typename TL, int V>
__device__ __forceinline__ void load_row(const TL* row, int E, int lane, float (&l)[V], uint16_t (&raw)[V]) {
  constexpr int BYTES = V * static_cast<int>(sizeof(TL));
  const int first = lane * V;
  const bool vec = (BYTES == 4 || BYTES == 8 || BYTES == 16) && first + V <= E &&
                   (reinterpret_cast<uintptr_t>(row + first) % (BYTES >= 16 ? 16 : BYTES)) == 0;
  TL v[V];
  if (vec) {
    if constexpr (BYTES == 16) *reinterpret_cast<uint4*>(v) = *reinterpret_cast<const uint4*>(row + first);
    else if constexpr (BYTES == 8) *reinterpret_cast<uint2*>(v) = *reinterpret_cast<const uint2*>(row + first);
    else if constexpr (BYTES == 4) *reinterpret_cast<uint32_t*>(v) = *reinterpret_cast<const uint32_t*>(row + first);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) v[i] = first + i < E ? row[first + i] : from_f32<TL>(-INFINITY);
  }
#pragma unroll
  for (int i = 0; i < V; ++i) {
    l[i] = first + i < E ? to_f32(v[i]) : -INFINITY;
    if constexpr (sizeof(TL) == 2) raw[i] = bits16(v[i]);
    else raw[i] = 0;
  }
}

}  // namespace route_detail

// Routes token t (the whole warp calls it; `my_e` is the warp's private
// shared buffer of 32*V floats). Writes indices[t*k + j], weights[t*k + j]
// and, if weights32 is not NULL, the FP32 weight. On return slot_id[q] holds,
// on lane l, the expert of slot j = q*32 + l (for j < k).
template <typename TL, int V>
__device__ __forceinline__ void route_token(const TL* __restrict__ logits, int64_t t, int E, int k, int renormalize,
                                            int lane, float* my_e, uint32_t* __restrict__ indices,
                                            TL* __restrict__ weights, float* __restrict__ weights32,
                                            uint32_t (&slot_id)[V]) {
  using namespace route_detail;
  constexpr bool K16 = sizeof(TL) == 2;  // one 32-bit key per expert
  const float qnan = __int_as_float(0x7FC00000);
  float l[V];
  uint16_t raw[V];
  load_row<TL, V>(logits + t * E, E, lane, l, raw);
  bool nonfinite = false, all_neg_inf = true;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    if (lane * V + v < E) {
      nonfinite |= isnan(l[v]) || l[v] == INFINITY;
      all_neg_inf &= l[v] == -INFINITY;
    }
  }
  nonfinite = __any_sync(FULL_MASK, nonfinite);
  all_neg_inf = __all_sync(FULL_MASK, all_neg_inf);
  uint32_t* idx_row = indices + t * k;
  if (nonfinite || all_neg_inf) {
    // All probabilities of such a row are NaN: NaN weights, and the tie
    // rule over all-equal keys picks ids 0..k-1.
#pragma unroll
    for (int q = 0; q < V; ++q) slot_id[q] = static_cast<uint32_t>(q * 32 + lane);
    for (int j = lane; j < k; j += 32) {
      idx_row[j] = static_cast<uint32_t>(j);
      weights[t * k + j] = from_f32<TL>(qnan);
      if (weights32 != nullptr) weights32[t * k + j] = qnan;
    }
    return;
  }

  // m = max_i l_i (exact, order-free); absent slots hold -inf.
  float m = -INFINITY;
#pragma unroll
  for (int v = 0; v < V; ++v) m = fmaxf(m, l[v]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, off));

  // e_i = exp(l_i - m), stored in id order; s = e_0 + ... + e_{E-1}.
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int id = lane * V + v;
    my_e[id] = id < E ? expf(__fsub_rn(l[v], m)) : 0.0f;
  }
  __syncwarp();
  float s = 0.0f;
  const int e4 = E & ~3;
  for (int i = 0; i < e4; i += 4) {
    const float4 q = *reinterpret_cast<const float4*>(my_e + i);
    s = __fadd_rn(s, q.x);
    s = __fadd_rn(s, q.y);
    s = __fadd_rn(s, q.z);
    s = __fadd_rn(s, q.w);
  }
  for (int i = e4; i < E; ++i) s = __fadd_rn(s, my_e[i]);
  __syncwarp();

  // Keys (0 marks an absent or taken expert; every real key is above 0).
  uint32_t kh[V], kl[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const uint32_t id = static_cast<uint32_t>(lane * V + v);
    const bool real = id < static_cast<uint32_t>(E);
    if constexpr (K16) {
      kh[v] = real ? (ord16(raw[v]) << 16) | (0xFFFFu - id) : 0u;
      kl[v] = 0u;
    } else {
      kh[v] = real ? ord32(l[v]) : 0u;
      kl[v] = real ? 0xFFFFu - id : 0u;
    }
  }
  // k rounds of arg-max; slot j's id ends on lane j % 32, register j / 32
  // (while k <= 32, the usual case, every slot sits in register 0).
#pragma unroll
  for (int q = 0; q < V; ++q) slot_id[q] = 0;
  auto arg_max_round = [&]() -> uint32_t {
    uint32_t bh = kh[0];
#pragma unroll
    for (int v = 1; v < V; ++v) bh = max(bh, kh[v]);
    bh = __reduce_max_sync(FULL_MASK, bh);
    uint32_t id;
    if constexpr (K16) {
      id = 0xFFFFu - (bh & 0xFFFFu);
    } else {
      uint32_t bl = 0;
#pragma unroll
      for (int v = 0; v < V; ++v) bl = kh[v] == bh ? max(bl, kl[v]) : bl;
      bl = __reduce_max_sync(FULL_MASK, bl);
      id = 0xFFFFu - bl;
    }
    // The owner lane zeroes the taken key (selects, no divergent branch).
    const bool mine = lane == static_cast<int>(id / V);
    const uint32_t slot = id % V;
#pragma unroll
    for (int v = 0; v < V; ++v) kh[v] = (mine && static_cast<uint32_t>(v) == slot) ? 0u : kh[v];
    return id;
  };
  if (k <= 32) {
    for (int j = 0; j < k; ++j) {
      const uint32_t id = arg_max_round();
      slot_id[0] = lane == j ? id : slot_id[0];
    }
  } else {
    for (int j = 0; j < k; ++j) {
      const uint32_t id = arg_max_round();
      if (lane == (j & 31)) {
#pragma unroll
        for (int q = 0; q < V; ++q)
          if (q == (j >> 5)) slot_id[q] = id;
      }
    }
  }

  // p_j = e_j / s on slot j's lane; renormalize by the slot-ordered sum.
  float p[V];
#pragma unroll
  for (int q = 0; q < V; ++q) {
    const int j = q * 32 + lane;
    p[q] = 0.0f;
    if (q * 32 < k && j < k) p[q] = __fdiv_rn(my_e[slot_id[q]], s);  // registers holding slots only
  }
  float z = 0.0f;
  if (renormalize && k <= 32) {
#pragma unroll 4
    for (int j = 0; j < k; ++j) z = __fadd_rn(z, __shfl_sync(FULL_MASK, p[0], j));
  } else if (renormalize) {
    for (int j = 0; j < k; ++j) {
      float pj = 0.0f;
#pragma unroll
      for (int q = 0; q < V; ++q)
        if (q == (j >> 5)) pj = p[q];
      z = __fadd_rn(z, __shfl_sync(FULL_MASK, pj, j & 31));
    }
  }
#pragma unroll
  for (int q = 0; q < V; ++q) {
    const int j = q * 32 + lane;
    if (q * 32 < k && j < k) {
      const float w = renormalize ? __fdiv_rn(p[q], z) : p[q];
      idx_row[j] = slot_id[q];
      weights[t * k + j] = from_f32<TL>(w);
      if (weights32 != nullptr) weights32[t * k + j] = w;
    }
  }
  __syncwarp();
}

}  // namespace moe
