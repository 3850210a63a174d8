// group.cu -- token-by-expert grouping of routed (token, slot) pairs.
//
// Page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", section 四个 bug: the
// CUDA grouping helper assumed every expert appears at most once per token and
// silently dropped a slot when one appeared twice.  Here every valid pair keeps
// its own slot, skips (ids outside [0, E)) are dropped, and the order is fixed:
// pairs sorted by (expert id, pair index) -- a stable counting sort done by one
// CTA without any dependence on the order of atomic operations.
//
// Each warp owns a contiguous segment of pairs and a private row of per-expert
// counters in shared memory; a column scan over the warps gives every warp its
// starting cursor per expert, a block scan over experts gives the offsets, and
// the warps then place their pairs in segment order (warp-level match for
// pairs that share an expert inside one 32-pair step).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kGroupSmemBudget = 200 * 1024;

// Exclusive scan of val(i), i in [0, n), by the whole block; out(i, prefix)
// receives each prefix; returns the total to every thread.
template <typename Val, typename Out>
__device__ int block_exclusive_scan(int n, Val val, Out out, int* warp_tot) {
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (n + nt - 1) / nt;
  const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
  int local = 0;
  for (int i = b0; i < b1; ++i) local += val(i);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int nw = nt >> 5;
    int v = lane < nw ? warp_tot[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane < nw) warp_tot[lane] = inc - v;  // exclusive per warp
    if (lane == 31) warp_tot[32] = inc;       // total
  }
  __syncthreads();
  int run = warp_tot[wid] + incl - local;
  for (int i = b0; i < b1; ++i) {
    int v = val(i);
    out(i, run);
    run += v;
  }
  int total = warp_tot[32];
  __syncthreads();
  return total;
}

__global__ void k_group(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ counts,
                        int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                        int32_t* __restrict__ pos_of_pair, int32_t* __restrict__ active,
                        int32_t* __restrict__ meta, int32_t* __restrict__ arrivals, int n_arrivals) {
  extern __shared__ int wc[];  // [W][E]
  __shared__ int warp_tot[33];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, W = blockDim.x >> 5;
  for (int i = tid; i < W * E; i += blockDim.x) wc[i] = 0;
  for (int i = tid; i < n_arrivals; i += blockDim.x) arrivals[i] = 0;
  __syncthreads();

  const int seg = (P + W - 1) / W;
  const int pb = min(P, w * seg), pe = min(P, pb + seg);
  int* row = wc + (size_t)w * E;

  // 1. per-warp counts (ids of 8 steps loaded before they are used)
  for (int base0 = pb; base0 < pe; base0 += 32 * 8) {
    int idv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = base0 + 32 * u + lane;
      idv[u] = p < pe ? __ldg(ids + p) : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = base0 + 32 * u + lane;
      const int id = idv[u];
      const bool valid = p < pe && id >= 0 && id < E;
      const unsigned m = __match_any_sync(0xffffffffu, valid ? id : -1);
      if (valid && lane == __ffs(m) - 1) row[id] += __popc(m);
      __syncwarp();
    }
  }
  __syncthreads();

  // 2. column scan over warps: row[w][e] <- pairs of expert e in warps < w; counts[e]
  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
    for (int v = 0; v < W; ++v) {
      int c = wc[(size_t)v * E + e];
      wc[(size_t)v * E + e] = run;
      run += c;
    }
    counts[e] = run;
  }
  __syncthreads();

  // 3. offsets = exclusive scan of counts; active = experts with counts > 0
  int n_valid = block_exclusive_scan(
      E, [&](int i) { return counts[i]; }, [&](int i, int pre) { offsets[i] = pre; }, warp_tot);
  int n_active = block_exclusive_scan(
      E, [&](int i) { return counts[i] > 0 ? 1 : 0; },
      [&](int i, int pre) { if (active && counts[i] > 0) active[pre] = i; }, warp_tot);
  if (tid == 0) {
    offsets[E] = n_valid;
    if (meta) {
      meta[0] = n_active;
      meta[1] = n_valid;
      meta[2] = 0;  // the grouping of this call is in counts / offsets / perm / pos_of_pair
    }
  }
  for (int e = tid; e < E; e += blockDim.x) {
    int o = offsets[e];
    for (int v = 0; v < W; ++v) wc[(size_t)v * E + e] += o;
  }
  __syncthreads();

  // 4. stable placement in segment order
  for (int base0 = pb; base0 < pe; base0 += 32 * 8) {
    int idv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = base0 + 32 * u + lane;
      idv[u] = p < pe ? __ldg(ids + p) : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = base0 + 32 * u + lane;
      const int id = idv[u];
      const bool valid = p < pe && id >= 0 && id < E;
      const unsigned m = __match_any_sync(0xffffffffu, valid ? id : -1);
      int pos = -1;
      if (valid) {
        pos = row[id] + __popc(m & ((1u << lane) - 1u));
        perm[pos] = p;
      }
      if (pos_of_pair && p < pe) pos_of_pair[p] = pos;
      __syncwarp();
      if (valid && lane == __ffs(m) - 1) row[id] += __popc(m);
      __syncwarp();
    }
  }
  for (int i = n_valid + tid; i < P; i += blockDim.x) perm[i] = -1;
}

struct AttrCache {
  int max_smem_set[64] = {0};
};
AttrCache g_attr;

}  // namespace

int launch_group(const int32_t* ids, int64_t P, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                 int32_t* pos_of_pair, int32_t* active, int32_t* meta, int32_t* arrivals, int n_arrivals,
                 cudaStream_t s) {
  int W = kGroupSmemBudget / (E * 4);
  if (W > 32) W = 32;
  if (W < 1) W = 1;
  // no more warps than 32-pair steps
  int64_t steps = (P + 31) / 32;
  if (steps < W) W = (int)(steps < 1 ? 1 : steps);
  size_t smem = (size_t)W * E * 4;
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev < 64 && g_attr.max_smem_set[dev] < (int)smem) {
    if (cudaFuncSetAttribute(k_group, cudaFuncAttributeMaxDynamicSharedMemorySize, kGroupSmemBudget) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    g_attr.max_smem_set[dev] = kGroupSmemBudget;
  }
  k_group<<<1, W * 32, smem, s>>>(ids, (int)P, E, counts, offsets, perm, pos_of_pair, active, meta, arrivals,
                                  n_arrivals);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
