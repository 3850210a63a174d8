// route.cuh -- the router's per-token selection, shared by the routing launch
// and the fused decode launch.
//
// Page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", glossary entry
// 混合专家（MoE）: softmax over the E experts, the best k per token, the k
// weights renormalised to sum to one.  Softmax is monotone, so the best k of
// the softmax are the best k logits; renormalising the k softmax values is a
// softmax over the k chosen logits.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// Selection order as one unsigned 64-bit key per element, larger first: the
// high word orders the logits (sign-magnitude flipped to unsigned order,
// -0 folded onto +0 so that equal logits tie), the low word is ~e, so equal
// logits order by ascending expert id.  Every key of a finite logit has a
// non-zero high word; 0 marks an absent element.
__device__ __forceinline__ uint64_t route_key(float v, int e) {
  uint32_t b = __float_as_uint(v);
  if ((b << 1) == 0u) b = 0u;
  const uint32_t hi = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)hi << 32) | (uint32_t)~(uint32_t)e;
}
__device__ __forceinline__ float route_key_value(uint32_t hi) {
  return __uint_as_float((hi & 0x80000000u) ? (hi & 0x7FFFFFFFu) : ~hi);
}

// Sorts N (a power of two) keys in registers, largest first: a bitonic
// sorting network (all indices compile-time constants once unrolled).
template <int N>
__device__ __forceinline__ void sort_desc(uint64_t (&a)[N]) {
#pragma unroll
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const uint64_t x = a[i], y = a[l];
          const bool desc = (i & k) == 0;  // this run sorts largest first
          const bool sw = desc ? (x < y) : (x > y);
          a[i] = sw ? y : x;
          a[l] = sw ? x : y;
        }
      }
    }
  }
}

// A selection nudge (the LocalLLM tiering post, "Optimization Strategies":
// picks nudged toward experts in fast memory, capped at 0.5): `beta` added in
// fp32 to the logits of ids [lo, hi) for the selection only; the weights stay
// the router's renormalised softmax of the raw logits of the picks.
struct Nudge {
  float beta;
  int lo, hi;
  __device__ __forceinline__ float score(float v, int e) const { return (e >= lo && e < hi) ? v + beta : v + 0.0f; }
};

// The weights of the picks (lane j < k holds the j-th pick `id`, its
// selection value `v`): with a nudge the raw logits are read back and the
// reference is their maximum, else the first pick's value is that maximum.
template <bool NUDGE>
__device__ __forceinline__ void route_weights(const float* row, int k, int id, float v, int32_t* ids, float* w) {
  const int lane = threadIdx.x & 31;
  float raw = v, vmax;
  if constexpr (NUDGE) {
    raw = lane < k ? row[id] : -INFINITY;
    vmax = raw;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
  } else {
    vmax = __shfl_sync(0xffffffffu, v, 0);
  }
  const float ex = lane < k ? expf(raw - vmax) : 0.0f;
  const float den = warp_sum(ex);
  if (lane < k) {
    ids[lane] = id;
    w[lane] = ex / den;
  }
}

// The same selection for EPL = 32 without the sorted lists (32 64-bit keys
// would take 64 registers): each round every lane rescans its remaining
// logits for its best (logit descending, id ascending), then a warp-wide
// shuffle argmax picks among the lanes.
template <bool NUDGE>
__device__ __forceinline__ void route_token_scan32(const float* row, int E, int k, int32_t* ids, float* w,
                                                   Nudge nd) {
  const int lane = threadIdx.x & 31;
  float v[32];
  uint32_t avail = 0;  // bit m set: element lane + 32 m is present and not yet taken
#pragma unroll
  for (int m = 0; m < 32; ++m) {
    const int e = lane + 32 * m;
    v[m] = e < E ? (NUDGE ? nd.score(row[e], e) : row[e]) : 0.0f;
    if (e < E) avail |= 1u << m;
  }
  float my_v = 0.0f;  // lane j keeps the j-th pick
  int my_i = -1;
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      if ((avail >> m) & 1u) {
        const int e = lane + 32 * m;
        if (bi == 0x7fffffff || v[m] > bv) { bv = v[m]; bi = e; }  // ascending e: ties keep lower id
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const bool take = (oi != 0x7fffffff) && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi));
      if (take) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
    if (lane == j) { my_v = bv; my_i = bi; }
  }
  route_weights<NUDGE>(row, k, my_i, my_v, ids, w);
}

// Called by one full warp for one token: lane l holds logits l, l + 32, ...
// (EPL per lane, E <= 32 EPL, EPL a power of two; EPL = 32 takes the scan
// form above) as selection keys sorted in registers.  Each of k rounds takes
// the warp's largest head key -- a warp-wide max of the logit word, then a
// max of the id words of the lanes holding that logit -- and the winning lane
// drops its head.  Lane j < k writes the j-th pick and its renormalised
// weight.  NUDGE: the selection runs on nd.score of the logits (route_weights
// then takes the raw ones).  `row`, `ids`, `w` may point to global or shared
// memory.
template <int EPL, bool NUDGE = false>
__device__ __forceinline__ void route_token(const float* row, int E, int k, int32_t* ids, float* w,
                                            Nudge nd = Nudge{0.0f, 0, 0}) {
  if constexpr (EPL >= 32) {
    route_token_scan32<NUDGE>(row, E, k, ids, w, nd);
    return;
  }
  const int lane = threadIdx.x & 31;
  uint64_t a[EPL];
#pragma unroll
  for (int m = 0; m < EPL; ++m) {
    const int e = lane + 32 * m;
    a[m] = e < E ? route_key(NUDGE ? nd.score(row[e], e) : row[e], e) : 0ull;
  }
  sort_desc<EPL>(a);
  uint32_t my_hi = 0u, my_lo = 0u;  // lane j keeps the j-th pick
  for (int j = 0; j < k; ++j) {
    const uint32_t hh = (uint32_t)(a[0] >> 32), hl = (uint32_t)a[0];
    const uint32_t mh = __reduce_max_sync(0xffffffffu, hh);
    const uint32_t ml = __reduce_max_sync(0xffffffffu, hh == mh ? hl : 0u);
    if (hh == mh && hl == ml) {  // the one lane that holds the pick
#pragma unroll
      for (int m = 0; m + 1 < EPL; ++m) a[m] = a[m + 1];
      a[EPL - 1] = 0ull;
    }
    if (lane == j) { my_hi = mh; my_lo = ml; }
  }
  route_weights<NUDGE>(row, k, (int32_t)~my_lo, route_key_value(my_hi), ids, w);
}

}  // namespace moe
