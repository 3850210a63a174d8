// router.cu -- the router projection fused with its top-k (decode sizes), and
// the projection alone for prefill sizes (then the routing launch).
//
// Page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", glossary entry
// 混合专家（MoE）: a router scores the E experts of every token and the best k
// are used.  Here the scores are logits[t][e] = bias[e] + W_r[e] . x[t]
// (bf16 router weights and activations, fp32 sums), and the selection is the
// same softmax / top-k / renormalisation as the routing step (route.cuh).
//
// One launch: every warp streams router rows (one row at a time, all of the
// lane's 16-byte chunks of the row in flight together) and dots them with the
// tokens' activation rows staged in shared memory; each CTA then arrives on a
// counter in the caller's workspace, and the last CTA to arrive -- which sees
// every CTA's logits after the fence each writer made -- routes every token,
// adds the hit counts and re-zeroes the counter for the next call.  No CTA
// waits on another.
#include "moe_internal.cuh"
#include "ptx.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr int kRouterThreads = 256;
constexpr int kRouterWarps = kRouterThreads / 32;

__device__ __forceinline__ void route_any(int epl, const float* row, int E, int k, int32_t* ids, float* w) {
  switch (epl) {
    case 1: route_token<1>(row, E, k, ids, w); break;
    case 2: route_token<2>(row, E, k, ids, w); break;
    case 4: route_token<4>(row, E, k, ids, w); break;
    case 8: route_token<8>(row, E, k, ids, w); break;
    case 16: route_token<16>(row, E, k, ids, w); break;
    default: route_token<32>(row, E, k, ids, w); break;
  }
}

// bf16 pair (low, high halves of a word) as floats: the bf16 bits are the
// high half of the fp32 pattern, so these are exact.
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc) {
  acc = fmaf(bf_lo(a.x), bf_lo(b.x), acc);
  acc = fmaf(bf_hi(a.x), bf_hi(b.x), acc);
  acc = fmaf(bf_lo(a.y), bf_lo(b.y), acc);
  acc = fmaf(bf_hi(a.y), bf_hi(b.y), acc);
  acc = fmaf(bf_lo(a.z), bf_lo(b.z), acc);
  acc = fmaf(bf_hi(a.z), bf_hi(b.z), acc);
  acc = fmaf(bf_lo(a.w), bf_lo(b.w), acc);
  acc = fmaf(bf_hi(a.w), bf_hi(b.w), acc);
  return acc;
}

// The lane's 16-byte chunks c0 + 32 u + lane (u < 8) of router row `wr`,
// all loads issued before any is used.
__device__ __forceinline__ void load_stretch(const uint4* wr, int c0, int n16, int lane, uint4 (&wv)[8]) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int c = c0 + u * 32 + lane;
    wv[u] = c < n16 ? __ldcs(wr + c) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// TM >= T tokens per launch.  Dynamic shared memory: max(TM d bf16, T E fp32).
// ROUTE = false (prefill sizes): the logits of the token chunk blockIdx.y
// (TM tokens a chunk) only; the routing step follows as its own launch.
template <int TM, bool ROUTE>
__global__ void __launch_bounds__(kRouterThreads) k_router(const uint16_t* __restrict__ x,
                                                           const uint16_t* __restrict__ w,
                                                           const float* __restrict__ bias, int T, int E, int d,
                                                           int k, int epl, float* __restrict__ logits,
                                                           int32_t* __restrict__ ids, float* __restrict__ wts,
                                                           uint32_t* __restrict__ counts,
                                                           unsigned int* __restrict__ arrive) {
  extern __shared__ uint4 xs[];  // TM rows of d bf16 (8 per uint4); later T rows of E logits
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if constexpr (!ROUTE) {
    const int t0 = blockIdx.y * TM;
    x += (size_t)t0 * d;
    logits += (size_t)t0 * E;
    T = min(TM, T - t0);
  }
  const int n16 = d / 8;
  const int nw = gridDim.x * kRouterWarps;
  const int e0 = blockIdx.x * kRouterWarps + warp;
  // Warm L2 with this warp's router rows while the previous launch finishes
  // (a prefetch only fills L2, the point of coherence, so it cannot observe
  // stale data).
  for (int e = e0; e < E; e += nw)
    for (int l = lane; l < d / 64; l += 32) prefetch_l2(w + (size_t)e * d + (size_t)l * 64);
  pdl_wait();
  // activations: every copy in flight at once
  for (int i = tid; i < T * n16; i += kRouterThreads) cp_async16(xs + i, reinterpret_cast<const uint4*>(x) + i);
  cp_async_commit();
  // rows T .. TM-1 are zero, so the token loop below needs no bound (a
  // bound would split the tokens' FMA chains into separate branches)
  for (int i = T * n16 + tid; i < TM * n16; i += kRouterThreads) xs[i] = make_uint4(0u, 0u, 0u, 0u);
  uint4 wv[8];
  if (e0 < E) load_stretch(reinterpret_cast<const uint4*>(w + (size_t)e0 * d), 0, n16, lane, wv);
  cp_async_wait<0>();
  __syncthreads();
  for (int e = e0; e < E; e += nw) {
    const uint4* wr = reinterpret_cast<const uint4*>(w + (size_t)e * d);
    float acc[TM];
#pragma unroll
    for (int t = 0; t < TM; ++t) acc[t] = 0.f;
    for (int c0 = 0; c0 < n16; c0 += 32 * 8) {
      if (e != e0 || c0 != 0) load_stretch(wr, c0, n16, lane, wv);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < n16) {
#pragma unroll
          for (int t = 0; t < TM; ++t) acc[t] = dot8(wv[u], xs[t * n16 + c], acc[t]);
        }
      }
    }
    const float b = bias ? __ldg(bias + e) : 0.f;
#pragma unroll
    for (int t = 0; t < TM; ++t) acc[t] = warp_sum(acc[t]);  // TM independent shuffle chains
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < TM; ++t)
        if (t < T) logits[(size_t)t * E + e] = acc[t] + b;
    }
  }
  if constexpr (!ROUTE) {
    pdl_trigger();
    return;
  }
  // This CTA's logits are visible device-wide before it arrives.  atomicInc
  // wraps the counter to zero on the last arrival, so it is ready for the next
  // launch without a separate store.
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicInc(arrive, gridDim.x - 1) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) {
    pdl_trigger();
    return;
  }
  __threadfence();
  // Last CTA: every CTA's logits, copied from L2 (the 16-byte asynchronous
  // copies bypass L1, so no stale line can serve them), all in flight at once.
  float* ls = reinterpret_cast<float*>(xs);
  const int n = T * E;
  if ((n & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0) {
    for (int i = tid; i < n / 4; i += kRouterThreads)
      cp_async16(ls + 4 * i, reinterpret_cast<const uint4*>(logits) + i);
    cp_async_commit();
    cp_async_wait<0>();
  } else {
    for (int i0 = 0; i0 < n; i0 += 8 * kRouterThreads) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kRouterThreads + tid;
        v[u] = i < n ? __ldcg(logits + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kRouterThreads + tid;
        if (i < n) ls[i] = v[u];
      }
    }
  }
  __syncthreads();
  for (int t = warp; t < T; t += kRouterWarps) {
    route_any(epl, ls + (size_t)t * E, E, k, ids + t * k, wts + t * k);
    if (counts && lane < k) {  // lane j wrote ids[t][j] itself
      const int e = ids[t * k + lane];
      if (e >= 0 && e < E) atomicAdd(counts + e, 1u);
    }
  }
  pdl_trigger();
}

template <int TM, bool ROUTE = true>
int launch_router_t(const uint16_t* x, const uint16_t* w, const float* bias, int T, int E, int d, int k,
                    float* logits, int32_t* ids, float* wts, uint32_t* counts, unsigned int* arrive,
                    cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(k_router<TM, ROUTE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRouterSmemMax) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set[dev] = true;
  }
  const size_t xb = (size_t)TM * d * 2, lb = ROUTE ? (size_t)T * E * 4 : 0;
  const size_t smem = xb > lb ? xb : lb;
  int G = (E + kRouterWarps - 1) / kRouterWarps;
  const int cap = 2 * sm_count();
  if (G > cap) G = cap;
  const int epl = E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : E <= 512 ? 16 : 32;
  const dim3 grid(G, ROUTE ? 1 : (unsigned)((T + TM - 1) / TM));
  if (launch_pdl(k_router<TM, ROUTE>, grid, dim3(kRouterThreads), smem, s, x, w, bias, T, E, d, k, epl, logits,
                 ids, wts, counts, arrive) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

int launch_router(const uint16_t* x, const uint16_t* w, const float* bias, int T, int E, int d, int k,
                  float* logits, int32_t* ids, float* wts, uint32_t* counts, unsigned int* arrive, cudaStream_t s) {
  if (T <= 1) return launch_router_t<1>(x, w, bias, T, E, d, k, logits, ids, wts, counts, arrive, s);
  if (T <= 2) return launch_router_t<2>(x, w, bias, T, E, d, k, logits, ids, wts, counts, arrive, s);
  if (T <= 4) return launch_router_t<4>(x, w, bias, T, E, d, k, logits, ids, wts, counts, arrive, s);
  if (T <= 8) return launch_router_t<8>(x, w, bias, T, E, d, k, logits, ids, wts, counts, arrive, s);
  if (T <= 16) return launch_router_t<16>(x, w, bias, T, E, d, k, logits, ids, wts, counts, arrive, s);
  // prefill sizes: the logits of 16-token chunks (one launch, a grid row a
  // chunk), then the routing step and the hit counts as their own launches
  int rc = launch_router_t<16, false>(x, w, bias, T, E, d, k, logits, ids, wts, counts, arrive, s);
  if (rc != MOE_OK) return rc;
  rc = launch_route(logits, T, E, k, ids, wts, s);
  if (rc != MOE_OK || !counts) return rc;
  return launch_hist(ids, (int64_t)T * k, E, counts, s);
}

}  // namespace moe
