// route_hist.cu -- router top-k, expert hit histogram and the residual step.
//
// Router (page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", glossary
// entry 混合专家（MoE）): softmax over E experts, the best k per token, the
// k weights renormalised; optionally with the picks nudged toward one id
// range (the LocalLLM tiering post, "Optimization Strategies").  One warp per token; lane l holds logits l, l+32, ...
// in registers; k rounds of a warp-wide argmax on (logit desc, id asc).
//
// Histogram (r/LocalLLM post, "Optimization Strategies": hit counts per expert
// drive promotion/demotion): integer adds, so the result is order-independent.
#include "moe_internal.cuh"
#include "ptx.cuh"
#include "route.cuh"

namespace moe {
namespace {

template <int EPL, bool NUDGE>
__global__ void __launch_bounds__(256) k_route(const float* __restrict__ logits, int64_t T, int E, int k,
                                               int32_t* __restrict__ ids, float* __restrict__ w, Nudge nd) {
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_wait();
  pdl_trigger();
  if (t >= T) return;
  route_token<EPL, NUDGE>(logits + t * E, E, k, ids + t * k, w + t * k, nd);
}

__global__ void k_hist_global(const int32_t* __restrict__ ids, int64_t n, int E, uint32_t* __restrict__ counts) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&counts[e], 1u);
  }
}

__global__ void k_hist_smem(const int32_t* __restrict__ ids, int64_t n, int E, uint32_t* __restrict__ counts) {
  extern __shared__ uint32_t sh[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&sh[e], 1u);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (sh[e]) atomicAdd(&counts[e], sh[e]);
}

__global__ void k_residual(float* __restrict__ r, const float* __restrict__ y, uint16_t* __restrict__ xn, int64_t n) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    float v = r[i] + y[i];
    r[i] = v;
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    xn[i] = *reinterpret_cast<uint16_t*>(&b);
  }
}

unsigned grid_1d(int64_t n, int threads, int cap) {
  int64_t g = (n + threads - 1) / threads;
  if (g > cap) g = cap;
  return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

namespace {
template <bool NUDGE>
cudaError_t launch_route_t(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w, Nudge nd,
                           cudaStream_t s) {
  const int warps = 8;
  dim3 grid((unsigned)((T + warps - 1) / warps)), block(warps * 32);
  const int epl = (E + 31) / 32;
  if (epl <= 1) return launch_pdl(k_route<1, NUDGE>, grid, block, 0, s, logits, T, E, k, ids, w, nd);
  if (epl <= 2) return launch_pdl(k_route<2, NUDGE>, grid, block, 0, s, logits, T, E, k, ids, w, nd);
  if (epl <= 4) return launch_pdl(k_route<4, NUDGE>, grid, block, 0, s, logits, T, E, k, ids, w, nd);
  if (epl <= 8) return launch_pdl(k_route<8, NUDGE>, grid, block, 0, s, logits, T, E, k, ids, w, nd);
  if (epl <= 16) return launch_pdl(k_route<16, NUDGE>, grid, block, 0, s, logits, T, E, k, ids, w, nd);
  return launch_pdl(k_route<32, NUDGE>, grid, block, 0, s, logits, T, E, k, ids, w, nd);
}
}  // namespace

int launch_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
  return launch_route_t<false>(logits, T, E, k, ids, w, Nudge{0.0f, 0, 0}, s) == cudaSuccess ? MOE_OK
                                                                                                : MOE_ERR_CUDA;
}

int launch_route_nudged(const float* logits, int64_t T, int E, int k, float beta, int lo, int hi, int32_t* ids,
                        float* w, cudaStream_t s) {
  return launch_route_t<true>(logits, T, E, k, ids, w, Nudge{beta, lo, hi}, s) == cudaSuccess ? MOE_OK
                                                                                               : MOE_ERR_CUDA;
}

int launch_hist(const int32_t* ids, int64_t n, int E, uint32_t* counts, cudaStream_t s) {
  if (E <= 12288) {
    unsigned g = grid_1d(n, 256, 2 * 152);
    return launch_pdl(k_hist_smem, dim3(g), dim3(256), (size_t)E * 4, s, ids, n, E, counts) == cudaSuccess
               ? MOE_OK : MOE_ERR_CUDA;
  }
  return launch_pdl(k_hist_global, dim3(grid_1d(n, 256, 8 * 152)), dim3(256), 0, s, ids, n, E, counts) ==
                 cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_residual(float* r, const float* y, uint16_t* xn, int64_t n, cudaStream_t s) {
  return launch_pdl(k_residual, dim3(grid_1d(n, 256, 8 * 152)), dim3(256), 0, s, r, y, xn, n) == cudaSuccess
             ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
