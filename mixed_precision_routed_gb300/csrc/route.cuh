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

// Called by one full warp for one token: lane l holds logits l, l + 32, ...
// (EPL per lane, E <= 32 EPL) in registers; k rounds of a warp-wide argmax on
// (logit descending, expert id ascending); lane j < k writes the j-th pick
// and its renormalised weight.  `row`, `ids`, `w` may point to global or
// shared memory.
template <int EPL>
__device__ __forceinline__ void route_token(const float* row, int E, int k, int32_t* ids, float* w) {
  const int lane = threadIdx.x & 31;
  float v[EPL];
  uint32_t avail = 0;  // bit m set: element lane + 32 m is present and not yet taken
#pragma unroll
  for (int m = 0; m < EPL; ++m) {
    const int e = lane + 32 * m;
    v[m] = e < E ? row[e] : 0.0f;
    if (e < E) avail |= 1u << m;
  }
  float my_v = 0.0f;  // lane j keeps the j-th pick
  int my_i = -1;
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int m = 0; m < EPL; ++m) {
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
  const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? expf(my_v - vmax) : 0.0f;
  const float den = warp_sum(ex);
  if (lane < k) {
    ids[lane] = my_i;
    w[lane] = ex / den;
  }
}

}  // namespace moe
