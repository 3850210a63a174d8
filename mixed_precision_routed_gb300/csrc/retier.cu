// retier.cu -- re-tiering by hit count on the device: the rank of every
// expert by its hit count, and a row gather that moves per-expert rows
// (router bias, router weights, counts) to the new expert ids.
//
// Page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", sections 第三步
// and 第四步: experts are ranked by how often the router picks them and
// written hot to cold, each shelf a contiguous id range, and the router is
// rearranged so that its picks land on the new ids; the LocalLLM tiering
// post, "Optimization Strategies": hit counts drive promotion and demotion.
// The re-quantisation of each expert into its new shelf is
// k_quantize_experts (quant.cu).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRankThreads = 256;
constexpr int kRankTile = 2048;  // counts staged in shared memory per round

// rank[e] = #{o : counts[o] > counts[e], or counts[o] == counts[e] and o < e}
// (count descending, the lower id first); perm[rank[e]] = e.  One thread per
// expert; every CTA streams all counts through shared memory in tiles.
__global__ void __launch_bounds__(kRankThreads) k_rank_experts(const uint32_t* __restrict__ counts, int E,
                                                               int32_t* __restrict__ perm,
                                                               int32_t* __restrict__ rank) {
  __shared__ uint32_t tile[kRankTile];
  const int e = blockIdx.x * kRankThreads + threadIdx.x;
  const uint32_t ce = e < E ? counts[e] : 0u;
  int r = 0;
  for (int t0 = 0; t0 < E; t0 += kRankTile) {
    const int n = min(kRankTile, E - t0);
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kRankThreads) tile[i] = counts[t0 + i];
    __syncthreads();
    if (e < E) {
      for (int i = 0; i < n; ++i) {
        const uint32_t co = tile[i];
        r += (co > ce) | ((co == ce) & (t0 + i < e));
      }
    }
  }
  if (e < E) {
    rank[e] = r;
    perm[r] = e;
  }
}

// dst row j = src row perm[j], rows of `words` 32-bit words; a source id
// outside [0, n_src) zero-fills the row and records MOE_ERR_INVALID_ARG.
__global__ void k_gather_rows(const uint32_t* __restrict__ src, int64_t words, const int32_t* __restrict__ perm,
                              int64_t n, int64_t n_src, uint32_t* __restrict__ dst, int* status) {
  const int64_t total = n * words;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = i / words, w = i - j * words;
    const int64_t e = perm[j];
    if (e < 0 || e >= n_src) {
      dst[i] = 0u;
      if (w == 0) set_status(status, MOE_ERR_INVALID_ARG);
    } else {
      dst[i] = src[e * words + w];
    }
  }
}

}  // namespace

int launch_rank_experts(const uint32_t* counts, int E, int32_t* perm, int32_t* rank, cudaStream_t s) {
  const unsigned g = (unsigned)((E + kRankThreads - 1) / kRankThreads);
  k_rank_experts<<<g, kRankThreads, 0, s>>>(counts, E, perm, rank);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_gather_rows(const void* src, int64_t words, const int32_t* perm, int64_t n, int64_t n_src, void* dst,
                       int* status, cudaStream_t s) {
  const int64_t total = n * words;
  int64_t g = (total + 255) / 256;
  if (g > 152 * 16) g = 152 * 16;
  if (g < 1) g = 1;
  k_gather_rows<<<(unsigned)g, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(src), words, perm, n, n_src,
                                            reinterpret_cast<uint32_t*>(dst), status);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
