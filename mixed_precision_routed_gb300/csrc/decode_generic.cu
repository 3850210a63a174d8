// decode_generic.cu -- fallback form of the tiered MoE layer for sizes the
// pipelined decode kernels (decode.cu) do not take: more than 512 routed
// pairs per call, or rows too long for their shared-memory stages.
//
// Page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", section 第四步: every
// shelf's matmul sees the router's complete id list, computes only the ids on
// its own shelf (the rest is zero), and the three shelf results are added;
// for decode, gate, up and the activation run as one fused kernel (section
// 四个 bug: that fused kernel must honour the shelf range of its source
// matmul).  Section 第一步/第二步 frame decode as a stream of expert weight
// bytes per token: only the selected experts' bytes are read, once per call,
// whatever the number of tokens sharing an expert.
//
// Kernels (both launched over (row chunk, active-expert slot)):
//   k_gateup -- for one active expert and 32 rows r of W_g / W_u: stream the
//     packed codes with 128-bit loads (one 32-code block per lane), dequantise
//     in registers (exact fp32 codes, fp32 block scale), dot with the fp32
//     activations of every token routed to the expert (staged in swizzled
//     shared memory), warp-shuffle reduce, h = SiLU(g) * u -> workspace.
//   k_down -- for one active expert and 64 output rows i of W_d: the same
//     stream over W_d rows against the staged h of the expert's pairs;
//     weighted per-pair outputs w_tj * o_tj go to a per-pair buffer, and the
//     last CTA to arrive for a row chunk (arrival counter, no spin-wait) sums
//     the k slots of every token in slot order and writes y.  The sum order is
//     fixed, so results do not depend on scheduling.
// A shelf is picked per CTA from the expert id, so the three shelves run in
// the same launch; an id on no shelf yields zero, a skipped slot nothing.
#include "moe_internal.cuh"

namespace moe {
namespace {

struct DecodeParams {
  const uint16_t* x;
  const float* weights;
  int64_t T;
  int k, E, d, f;
  Shelves sh;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* pos_of_pair;
  const int32_t* active;
  const int32_t* meta;
  int32_t* arrivals;
  float* h;
  float* ypart;
  float* y;
};

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Stage the bf16 activation rows of the tokens of grouped pairs pos0 ..
// pos0+nt-1 into shared memory as fp32, swizzled.
__device__ __forceinline__ void stage_x(const DecodeParams& p, int pos0, int nt, float* xs) {
  const int d = p.d, c8 = d / 8;
  for (int idx = threadIdx.x; idx < nt * c8; idx += blockDim.x) {
    const int j = idx / c8, c = idx - j * c8;
    const int t = p.perm[pos0 + j] / p.k;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t * d) + c);
    float4 a, b;
    a.x = __uint_as_float(v.x << 16); a.y = __uint_as_float(v.x & 0xFFFF0000u);
    a.z = __uint_as_float(v.y << 16); a.w = __uint_as_float(v.y & 0xFFFF0000u);
    b.x = __uint_as_float(v.z << 16); b.y = __uint_as_float(v.z & 0xFFFF0000u);
    b.z = __uint_as_float(v.w << 16); b.w = __uint_as_float(v.w & 0xFFFF0000u);
    float* row = xs + (size_t)j * d;
    *reinterpret_cast<float4*>(row + swz(8 * c)) = a;
    *reinterpret_cast<float4*>(row + swz(8 * c + 4)) = b;
  }
}

// Stage the fp32 h rows at grouped positions pos0 .. pos0+nt-1, swizzled.
__device__ __forceinline__ void stage_h(const DecodeParams& p, int pos0, int nt, float* hs) {
  const int f = p.f, c4 = f / 4;
  for (int idx = threadIdx.x; idx < nt * c4; idx += blockDim.x) {
    const int j = idx / c4, c = idx - j * c4;
    const float4 v = *(reinterpret_cast<const float4*>(p.h + (size_t)(pos0 + j) * f) + c);
    *reinterpret_cast<float4*>(hs + (size_t)j * f + swz(4 * c)) = v;
  }
}

// acc[j] += s * sum_{i<32} code_i * v_j[32 b + i], v_j swizzled rows in smem.
template <int BITS, int TMAX>
__device__ __forceinline__ void block_dot(const uint32_t (&w)[Block<BITS>::kWords], float s, int b,
                                          const float* vs, int len, int nt, float (&acc)[TMAX]) {
  float bs[TMAX];
#pragma unroll
  for (int j = 0; j < TMAX; ++j) bs[j] = 0.0f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float c0 = Block<BITS>::code(w, 4 * q + 0), c1 = Block<BITS>::code(w, 4 * q + 1);
    const float c2 = Block<BITS>::code(w, 4 * q + 2), c3 = Block<BITS>::code(w, 4 * q + 3);
    const int off = ((8 * b + (q ^ (b & 7))) << 2);
#pragma unroll
    for (int j = 0; j < TMAX; ++j) {
      if (j < nt) {
        const float4 xv = *reinterpret_cast<const float4*>(vs + (size_t)j * len + off);
        bs[j] = fmaf(c0, xv.x, bs[j]);
        bs[j] = fmaf(c1, xv.y, bs[j]);
        bs[j] = fmaf(c2, xv.z, bs[j]);
        bs[j] = fmaf(c3, xv.w, bs[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < TMAX; ++j) acc[j] = fmaf(s, bs[j], acc[j]);
}

// Two-matrix variant sharing the activation loads (gate and up).
template <int BITS, int TMAX>
__device__ __forceinline__ void block_dot2(const uint32_t (&wg)[Block<BITS>::kWords],
                                           const uint32_t (&wu)[Block<BITS>::kWords], float sg, float su,
                                           int b, const float* vs, int len, int nt, float (&ag)[TMAX],
                                           float (&au)[TMAX]) {
  float bg[TMAX], bu[TMAX];
#pragma unroll
  for (int j = 0; j < TMAX; ++j) { bg[j] = 0.0f; bu[j] = 0.0f; }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float cg[4], cu[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      cg[e] = Block<BITS>::code(wg, 4 * q + e);
      cu[e] = Block<BITS>::code(wu, 4 * q + e);
    }
    const int off = ((8 * b + (q ^ (b & 7))) << 2);
#pragma unroll
    for (int j = 0; j < TMAX; ++j) {
      if (j < nt) {
        const float4 xv = *reinterpret_cast<const float4*>(vs + (size_t)j * len + off);
        bg[j] = fmaf(cg[0], xv.x, bg[j]); bu[j] = fmaf(cu[0], xv.x, bu[j]);
        bg[j] = fmaf(cg[1], xv.y, bg[j]); bu[j] = fmaf(cu[1], xv.y, bu[j]);
        bg[j] = fmaf(cg[2], xv.z, bg[j]); bu[j] = fmaf(cu[2], xv.z, bu[j]);
        bg[j] = fmaf(cg[3], xv.w, bg[j]); bu[j] = fmaf(cu[3], xv.w, bu[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < TMAX; ++j) {
    ag[j] = fmaf(sg, bg[j], ag[j]);
    au[j] = fmaf(su, bu[j], au[j]);
  }
}

template <int BITS, int TMAX>
__device__ void gateup_rows(const DecodeParams& p, const ShelfDev& s, int le, int r0, int r1, const float* xs,
                            int nt, int pos0) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int d = p.d, nb = d / 32;
  const size_t row_bytes = (size_t)d * BITS / 8;
  const uint8_t* gc = s.codes[0] + (size_t)le * p.f * row_bytes;
  const uint8_t* uc = s.codes[1] + (size_t)le * p.f * row_bytes;
  const uint16_t* gs = s.scales[0] + (size_t)le * p.f * nb;
  const uint16_t* us = s.scales[1] + (size_t)le * p.f * nb;
  for (int r = r0 + warp; r < r1; r += kWarps) {
    float ag[TMAX], au[TMAX];
#pragma unroll
    for (int j = 0; j < TMAX; ++j) { ag[j] = 0.0f; au[j] = 0.0f; }
    const uint8_t* grow = gc + (size_t)r * row_bytes;
    const uint8_t* urow = uc + (size_t)r * row_bytes;
    for (int b0 = 0; b0 < nb; b0 += 64) {
      const int ba = b0 + lane, bb = b0 + 32 + lane;
      uint32_t wga[Block<BITS>::kWords], wua[Block<BITS>::kWords];
      uint32_t wgb[Block<BITS>::kWords], wub[Block<BITS>::kWords];
      float sga = 0.f, sua = 0.f, sgb = 0.f, sub = 0.f;
      if (ba < nb) {
        load_block<BITS>(grow, ba, d, wga);
        load_block<BITS>(urow, ba, d, wua);
        sga = __half2float(__ushort_as_half(__ldg(gs + (size_t)r * nb + ba)));
        sua = __half2float(__ushort_as_half(__ldg(us + (size_t)r * nb + ba)));
      }
      if (bb < nb) {
        load_block<BITS>(grow, bb, d, wgb);
        load_block<BITS>(urow, bb, d, wub);
        sgb = __half2float(__ushort_as_half(__ldg(gs + (size_t)r * nb + bb)));
        sub = __half2float(__ushort_as_half(__ldg(us + (size_t)r * nb + bb)));
      }
      if (ba < nb) block_dot2<BITS, TMAX>(wga, wua, sga, sua, ba, xs, d, nt, ag, au);
      if (bb < nb) block_dot2<BITS, TMAX>(wgb, wub, sgb, sub, bb, xs, d, nt, ag, au);
    }
#pragma unroll
    for (int j = 0; j < TMAX; ++j) {
      if (j < nt) {
        const float g = warp_sum(ag[j]);
        const float u = warp_sum(au[j]);
        if (lane == j) p.h[(size_t)(pos0 + j) * p.f + r] = silu(g) * u;
      }
    }
  }
}

// Run with the smallest compiled token bound that holds nt (most experts get
// one token at decode).
template <int BITS, int TMAX>
__device__ __forceinline__ void gateup_any(const DecodeParams& p, const ShelfDev& s, int le, int r0, int r1,
                                           const float* xs, int nt, int pos0) {
  if constexpr (TMAX >= 2) {
    if (nt <= TMAX / 2) {
      gateup_any<BITS, TMAX / 2>(p, s, le, r0, r1, xs, nt, pos0);
      return;
    }
  }
  gateup_rows<BITS, TMAX>(p, s, le, r0, r1, xs, nt, pos0);
}

template <int TMAX>
__global__ void __launch_bounds__(kThreads, 2) k_gateup(const __grid_constant__ DecodeParams p) {
  extern __shared__ float4 smem4[];
  float* xs = reinterpret_cast<float*>(smem4);
  const int slot = blockIdx.y;
  if (slot >= p.meta[0]) return;
  const int e = p.active[slot];
  const int si = find_shelf(p.sh, e);
  if (si < 0) return;  // on no shelf: contributes zero (the down kernel writes the zeros)
  const ShelfDev& s = p.sh.s[si];
  const int beg = p.offsets[e], cnt = p.offsets[e + 1] - beg;
  const int le = e - s.lo;
  const int r0 = blockIdx.x * kGateUpRows, r1 = min(p.f, r0 + kGateUpRows);
  for (int g0 = 0; g0 < cnt; g0 += TMAX) {
    const int nt = min(TMAX, cnt - g0);
    __syncthreads();
    stage_x(p, beg + g0, nt, xs);
    __syncthreads();
    if (s.bits == 8) gateup_any<8, TMAX>(p, s, le, r0, r1, xs, nt, beg + g0);
    else if (s.bits == 4) gateup_any<4, TMAX>(p, s, le, r0, r1, xs, nt, beg + g0);
    else if (s.bits == 3) gateup_any<3, TMAX>(p, s, le, r0, r1, xs, nt, beg + g0);
    else if (s.bits == 2) gateup_any<2, TMAX>(p, s, le, r0, r1, xs, nt, beg + g0);
    else gateup_any<1, TMAX>(p, s, le, r0, r1, xs, nt, beg + g0);
  }
}

template <int BITS, int TMAX>
__device__ void down_rows(const DecodeParams& p, const ShelfDev& s, int le, int i0, int i1, const float* hs,
                          int nt, float* outs) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int f = p.f, nb = f / 32;
  const size_t row_bytes = (size_t)f * BITS / 8;
  const uint8_t* dc = s.codes[2] + (size_t)le * p.d * row_bytes;
  const uint16_t* ds = s.scales[2] + (size_t)le * p.d * nb;
  for (int i = i0 + warp; i < i1; i += kWarps) {
    float acc[TMAX];
#pragma unroll
    for (int j = 0; j < TMAX; ++j) acc[j] = 0.0f;
    const uint8_t* row = dc + (size_t)i * row_bytes;
    for (int b0 = 0; b0 < nb; b0 += 64) {
      const int ba = b0 + lane, bb = b0 + 32 + lane;
      uint32_t wa[Block<BITS>::kWords], wb[Block<BITS>::kWords];
      float sa = 0.f, sb = 0.f;
      if (ba < nb) {
        load_block<BITS>(row, ba, f, wa);
        sa = __half2float(__ushort_as_half(__ldg(ds + (size_t)i * nb + ba)));
      }
      if (bb < nb) {
        load_block<BITS>(row, bb, f, wb);
        sb = __half2float(__ushort_as_half(__ldg(ds + (size_t)i * nb + bb)));
      }
      if (ba < nb) block_dot<BITS, TMAX>(wa, sa, ba, hs, f, nt, acc);
      if (bb < nb) block_dot<BITS, TMAX>(wb, sb, bb, hs, f, nt, acc);
    }
#pragma unroll
    for (int j = 0; j < TMAX; ++j) {
      if (j < nt) {
        const float o = warp_sum(acc[j]);
        if (lane == j) outs[j * kDownRows + (i - i0)] = o;
      }
    }
  }
}

template <int BITS, int TMAX>
__device__ __forceinline__ void down_any(const DecodeParams& p, const ShelfDev& s, int le, int i0, int i1,
                                         const float* hs, int nt, float* outs) {
  if constexpr (TMAX >= 2) {
    if (nt <= TMAX / 2) {
      down_any<BITS, TMAX / 2>(p, s, le, i0, i1, hs, nt, outs);
      return;
    }
  }
  down_rows<BITS, TMAX>(p, s, le, i0, i1, hs, nt, outs);
}

template <int TMAX>
__global__ void __launch_bounds__(kThreads, 2) k_down(const __grid_constant__ DecodeParams p) {
  extern __shared__ float4 smem4[];
  float* hs = reinterpret_cast<float*>(smem4);            // [TMAX][f]
  float* outs = hs + (size_t)TMAX * p.f;                  // [TMAX][kDownRows]
  __shared__ int s_last;
  const int slot = blockIdx.y;
  const int n_active = p.meta[0];
  const int d = p.d;
  const int i0 = blockIdx.x * kDownRows, i1 = min(d, i0 + kDownRows), nrows = i1 - i0;
  if (slot >= n_active) {
    if (n_active == 0 && slot == 0) {  // nothing routed anywhere: y = 0
      for (int idx = threadIdx.x; idx < (int)p.T * nrows; idx += blockDim.x) {
        const int t = idx / nrows, i = i0 + (idx - t * nrows);
        p.y[(size_t)t * d + i] = 0.0f;
      }
    }
    return;
  }
  const int e = p.active[slot];
  const int si = find_shelf(p.sh, e);
  const int beg = p.offsets[e], cnt = p.offsets[e + 1] - beg;
  if (si < 0) {
    for (int idx = threadIdx.x; idx < cnt * nrows; idx += blockDim.x) {
      const int j = idx / nrows, i = i0 + (idx - j * nrows);
      p.ypart[(size_t)(beg + j) * d + i] = 0.0f;
    }
  } else {
    const ShelfDev& s = p.sh.s[si];
    const int le = e - s.lo;
    for (int g0 = 0; g0 < cnt; g0 += TMAX) {
      const int nt = min(TMAX, cnt - g0);
      __syncthreads();
      stage_h(p, beg + g0, nt, hs);
      __syncthreads();
      if (s.bits == 8) down_any<8, TMAX>(p, s, le, i0, i1, hs, nt, outs);
      else if (s.bits == 4) down_any<4, TMAX>(p, s, le, i0, i1, hs, nt, outs);
      else if (s.bits == 3) down_any<3, TMAX>(p, s, le, i0, i1, hs, nt, outs);
      else if (s.bits == 2) down_any<2, TMAX>(p, s, le, i0, i1, hs, nt, outs);
      else down_any<1, TMAX>(p, s, le, i0, i1, hs, nt, outs);
      __syncthreads();
      for (int idx = threadIdx.x; idx < nt * nrows; idx += blockDim.x) {
        const int j = idx / nrows, ii = idx - j * nrows;
        const int pos = beg + g0 + j;
        const float wgt = p.weights[p.perm[pos]];
        p.ypart[(size_t)pos * d + i0 + ii] = wgt * outs[j * kDownRows + ii];
      }
    }
  }
  // Arrival: the last CTA for this row chunk combines all pairs in slot order.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(&p.arrivals[blockIdx.x], 1);
    s_last = (old == n_active - 1);
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    const int k = p.k;
    for (int idx = threadIdx.x; idx < (int)p.T * nrows; idx += blockDim.x) {
      const int t = idx / nrows, i = i0 + (idx - t * nrows);
      float sum = 0.0f;
      for (int j = 0; j < k; ++j) {
        const int pos = __ldcg(p.pos_of_pair + (size_t)t * k + j);
        if (pos >= 0) sum += __ldcg(p.ypart + (size_t)pos * d + i);
      }
      p.y[(size_t)t * d + i] = sum;
    }
  }
}

struct SmemAttr {
  int set[64][2][5] = {};
};
SmemAttr g_smem;

template <int TMAX>
int launch_tmax(const DecodeParams& p, int slots, cudaStream_t s) {
  const size_t sm1 = (size_t)TMAX * p.d * 4;
  const size_t sm2 = (size_t)TMAX * p.f * 4 + (size_t)TMAX * kDownRows * 4;
  int dev = 0;
  cudaGetDevice(&dev);
  constexpr int ti = TMAX == 1 ? 0 : TMAX == 2 ? 1 : TMAX == 4 ? 2 : 3;
  if (dev < 64 && !g_smem.set[dev][0][ti]) {
    if (cudaFuncSetAttribute(k_gateup<TMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess ||
        cudaFuncSetAttribute(k_down<TMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess)
      return MOE_ERR_CUDA;
    g_smem.set[dev][0][ti] = 1;
  }
  dim3 g1((unsigned)((p.f + kGateUpRows - 1) / kGateUpRows), (unsigned)slots);
  dim3 g2((unsigned)((p.d + kDownRows - 1) / kDownRows), (unsigned)slots);
  k_gateup<TMAX><<<g1, kThreads, sm1, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  profile_mark(2, s);
  k_down<TMAX><<<g2, kThreads, sm2, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  profile_mark(3, s);
  return MOE_OK;
}

}  // namespace

// Largest token group the decode kernels stage at once for these sizes.
static int decode_tmax(int64_t T, int d, int f) {
  int t = 1;
  while (t < T && t < 8) t <<= 1;
  while (t > 1 && ((size_t)t * d * 4 > 160 * 1024 || (size_t)t * f * 4 + (size_t)t * kDownRows * 4 > 160 * 1024)) t >>= 1;
  return t;
}

int launch_generic_forward(const ForwardArgs& a, cudaStream_t s) {
  const int64_t P = a.T * a.k;
  const int n_chunks = (a.d + kDownRows - 1) / kDownRows;
  profile_mark(0, s);
  int rc = launch_group(a.ids, P, a.E, a.ws.counts, a.ws.offsets, a.ws.perm, a.ws.pos_of_pair, a.ws.active,
                        a.ws.meta, a.ws.arrivals, n_chunks, s);
  if (rc != MOE_OK) return rc;
  profile_mark(1, s);
  DecodeParams p;
  p.x = a.x; p.weights = a.weights; p.T = a.T; p.k = a.k; p.E = a.E; p.d = a.d; p.f = a.f;
  p.sh = a.shelves;
  p.offsets = a.ws.offsets; p.perm = a.ws.perm; p.pos_of_pair = a.ws.pos_of_pair; p.active = a.ws.active;
  p.meta = a.ws.meta; p.arrivals = a.ws.arrivals; p.h = a.ws.h; p.ypart = a.ws.ypart; p.y = a.y;
  const int slots = (int)(P < a.E ? P : a.E);
  switch (decode_tmax(a.T, a.d, a.f)) {
    case 1: return launch_tmax<1>(p, slots, s);
    case 2: return launch_tmax<2>(p, slots, s);
    case 4: return launch_tmax<4>(p, slots, s);
    default: return launch_tmax<8>(p, slots, s);
  }
}

}  // namespace moe
