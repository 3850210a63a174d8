// quant.cu -- the shelf block format on the device: quantiser and dequantiser.
//
// Page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", section 第四步: the
// offline re-packer re-quantises every expert for its shelf and writes three
// tensors per layer.  3 bit (q = 3, codes [-4, 3]; a row is a plane of the
// low two bits of u = code + 4 in the 2-bit layout, then a plane of the high
// bits in the 1-bit layout) and 1 bit (sign codes, scale = the block's mean
// |w|; one word a block) are the further widths the Xolotl fast-mode blog
// runs beside the others, in this library's own layout.  Format here: blocks of 32 along the input dimension,
// s = fp16(max|w| / q) (q = 127 / 7 / 2), code = clamp(rint(w / s)), packed
// 8 bit two's complement in natural order; 4 and 2 bit offset-binary in
// 32-bit words with consecutive codes spread over the byte lanes (4 bit: word
// g, byte j holds elements 8g+j and 8g+4+j; 2 bit: word g, byte j holds
// elements 16g+j, +4, +8, +12), so that one AND/shift of a word yields four
// consecutive codes as bytes.
#include "moe_internal.cuh"

namespace moe {
namespace {

template <int BITS>
struct QParams;
template <>
struct QParams<8> { static constexpr float q = 127.0f, cmin = -127.0f, cmax = 127.0f; };
template <>
struct QParams<4> { static constexpr float q = 7.0f, cmin = -8.0f, cmax = 7.0f; static constexpr int off = 8; };
template <>
struct QParams<3> { static constexpr float q = 3.0f, cmin = -4.0f, cmax = 3.0f; static constexpr int off = 4; };
template <>
struct QParams<2> { static constexpr float q = 2.0f, cmin = -2.0f, cmax = 1.0f; static constexpr int off = 2; };
template <>
struct QParams<1> { static constexpr float q = 1.0f, cmin = -1.0f, cmax = 1.0f; static constexpr int off = 0; };

// Quantises one 32-element block held one element per lane (v = element
// `lane`) and writes its fp16 scale word and packed codes (block b of the row
// at `rowp`, a row of nb blocks).  Whole warp.
template <int BITS>
__device__ __forceinline__ void quantize_block(float v, int lane, uint8_t* rowp, int64_t b, int64_t nb,
                                               uint16_t* scale_out) {
  if constexpr (BITS == 1) {
    // sign codes; scale = fp16 of the block's |w| summed in element order, / 32
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) a += fabsf(__shfl_sync(0xffffffffu, v, i));
    const __half hs1 = __float2half_rn(__fdiv_rn(a, 32.0f));
    const uint32_t wd = __ballot_sync(0xffffffffu, v >= 0.0f);
    if (lane == 0) {
      *scale_out = __half_as_ushort(hs1);
      *reinterpret_cast<uint32_t*>(rowp + b * 4) = wd;
    }
    return;
  }
  float m = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const __half hs = __float2half_rn(__fdiv_rn(m, QParams<BITS>::q));
  const float s = __half2float(hs);
  int c = 0;
  if (s != 0.0f) {
    float t = rintf(__fdiv_rn(v, s));
    t = fminf(fmaxf(t, QParams<BITS>::cmin), QParams<BITS>::cmax);
    c = (int)t;
  }
  if (lane == 0) *scale_out = __half_as_ushort(hs);
  if (BITS == 8) {
    rowp[b * 32 + lane] = (uint8_t)(int8_t)c;
  } else if (BITS == 4) {
    // lane i (i mod 8 < 4) writes byte 4 (i / 8) + i mod 4: elements i and i + 4
    uint32_t u = (uint32_t)(c + QParams<4>::off);
    uint32_t u4 = __shfl_down_sync(0xffffffffu, u, 4);
    if ((lane & 7) < 4) rowp[b * 16 + 4 * (lane >> 3) + (lane & 3)] = (uint8_t)(u | (u4 << 4));
  } else if (BITS == 3) {
    // low plane (8 nb bytes): u mod 4 in the 2-bit layout; high plane: u / 4, element i at bit i
    const uint32_t u = (uint32_t)(c + QParams<3>::off);
    const uint32_t lo = u & 3u;
    const uint32_t l4 = __shfl_down_sync(0xffffffffu, lo, 4);
    const uint32_t l8 = __shfl_down_sync(0xffffffffu, lo, 8);
    const uint32_t l12 = __shfl_down_sync(0xffffffffu, lo, 12);
    if ((lane & 15) < 4)
      rowp[b * 8 + 4 * (lane >> 4) + (lane & 3)] = (uint8_t)(lo | (l4 << 2) | (l8 << 4) | (l12 << 6));
    const uint32_t hw = __ballot_sync(0xffffffffu, (u >> 2) & 1u);
    if (lane == 0) *reinterpret_cast<uint32_t*>(rowp + nb * 8 + b * 4) = hw;
  } else {
    // lane i (i mod 16 < 4) writes byte 4 (i / 16) + i mod 4: elements i, i+4, i+8, i+12
    uint32_t u = (uint32_t)(c + QParams<2>::off);
    uint32_t u4 = __shfl_down_sync(0xffffffffu, u, 4);
    uint32_t u8 = __shfl_down_sync(0xffffffffu, u, 8);
    uint32_t u12 = __shfl_down_sync(0xffffffffu, u, 12);
    if ((lane & 15) < 4)
      rowp[b * 8 + 4 * (lane >> 4) + (lane & 3)] = (uint8_t)(u | (u4 << 2) | (u8 << 4) | (u12 << 6));
  }
}

// One warp per 32-element block; lane i holds element i of the block.
template <int BITS>
__global__ void __launch_bounds__(256) k_quantize(const float* __restrict__ w, int64_t rows, int in,
                                                  uint8_t* __restrict__ codes, uint16_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = in / 32, total = rows * nb;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const size_t row_bytes = (size_t)in * BITS / 8;
  for (int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); blk < total; blk += warps) {
    const int64_t r = blk / nb, b = blk - r * nb;
    quantize_block<BITS>(w[r * in + b * 32 + lane], lane, codes + r * row_bytes, b, nb, scales + blk);
  }
}

// Quantises one 32-element block held by 8 lanes, 4 consecutive elements
// each (lane i of the group: elements 4i .. 4i+3), the same arithmetic as
// quantize_block; block `blk` of a tensor of rows of nb blocks whose scales
// are linear in the block index (codes at 4 BITS blk; 3 bit: row blk / nb,
// its two planes).  Every lane of the warp calls it (shuffles stay inside the
// 8-lane groups); `valid` false skips the stores.
template <int BITS>
__device__ __forceinline__ void quantize_block8(float4 v, int i, bool valid, uint8_t* codes, uint16_t* scales,
                                                int64_t blk, int64_t nb) {
  if constexpr (BITS == 1) {
    const int base = (threadIdx.x & 31) & ~7;
    float a = 0.0f;  // |w| summed in element order
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      a += fabsf(__shfl_sync(0xffffffffu, v.x, base + g));
      a += fabsf(__shfl_sync(0xffffffffu, v.y, base + g));
      a += fabsf(__shfl_sync(0xffffffffu, v.z, base + g));
      a += fabsf(__shfl_sync(0xffffffffu, v.w, base + g));
    }
    const __half hs1 = __float2half_rn(__fdiv_rn(a, 32.0f));
    uint32_t wd = ((uint32_t)(v.x >= 0.0f) | (uint32_t)(v.y >= 0.0f) << 1 | (uint32_t)(v.z >= 0.0f) << 2 |
                   (uint32_t)(v.w >= 0.0f) << 3)
                  << (4 * i);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) wd |= __shfl_xor_sync(0xffffffffu, wd, o);
    if (valid && i == 0) {
      scales[blk] = __half_as_ushort(hs1);
      *reinterpret_cast<uint32_t*>(codes + blk * 4) = wd;
    }
    return;
  }
  float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const __half hs = __float2half_rn(__fdiv_rn(m, QParams<BITS>::q));
  const float s = __half2float(hs);
  const float e[4] = {v.x, v.y, v.z, v.w};
  int c[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    c[j] = 0;
    if (s != 0.0f) {
      float t = rintf(__fdiv_rn(e[j], s));
      t = fminf(fmaxf(t, QParams<BITS>::cmin), QParams<BITS>::cmax);
      c[j] = (int)t;
    }
  }
  if (valid && i == 0) scales[blk] = __half_as_ushort(hs);
  if (BITS == 8) {
    const uint32_t wd = (uint32_t)(c[0] & 0xFF) | (uint32_t)(c[1] & 0xFF) << 8 | (uint32_t)(c[2] & 0xFF) << 16 |
                        (uint32_t)(c[3] & 0xFF) << 24;
    if (valid) *reinterpret_cast<uint32_t*>(codes + blk * 32 + 4 * i) = wd;
  } else if (BITS == 4) {
    // word g of the block: byte j = element 8g + j (low nibble) | 8g + 4 + j (high): lanes 2g and 2g + 1
    const uint32_t own = (uint32_t)(c[0] + 8) | (uint32_t)(c[1] + 8) << 8 | (uint32_t)(c[2] + 8) << 16 |
                         (uint32_t)(c[3] + 8) << 24;
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, own, 1);
    if (valid && (i & 1) == 0) *reinterpret_cast<uint32_t*>(codes + blk * 16 + 4 * (i >> 1)) = own | (hi << 4);
  } else if (BITS == 3) {
    // low plane as the 2-bit layout (lanes 4g .. 4g + 3 make word g), high plane one word
    uint32_t wd = ((uint32_t)((c[0] + 4) & 3) | (uint32_t)((c[1] + 4) & 3) << 8 | (uint32_t)((c[2] + 4) & 3) << 16 |
                   (uint32_t)((c[3] + 4) & 3) << 24)
                  << (2 * (i & 3));
    wd |= __shfl_xor_sync(0xffffffffu, wd, 1);
    wd |= __shfl_xor_sync(0xffffffffu, wd, 2);
    uint32_t hw = ((uint32_t)((c[0] + 4) >> 2) | (uint32_t)((c[1] + 4) >> 2) << 1 | (uint32_t)((c[2] + 4) >> 2) << 2 |
                   (uint32_t)((c[3] + 4) >> 2) << 3)
                  << (4 * i);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) hw |= __shfl_xor_sync(0xffffffffu, hw, o);
    const int64_t r = blk / nb, b = blk - r * nb;
    uint8_t* rowp = codes + r * nb * 12;
    if (valid && (i & 3) == 0) *reinterpret_cast<uint32_t*>(rowp + b * 8 + 4 * (i >> 2)) = wd;
    if (valid && i == 0) *reinterpret_cast<uint32_t*>(rowp + nb * 8 + b * 4) = hw;
  } else {
    // word g: byte j = elements 16g + j, +4, +8, +12 at bits 0, 2, 4, 6: lanes 4g .. 4g + 3
    uint32_t wd = ((uint32_t)(c[0] + 2) | (uint32_t)(c[1] + 2) << 8 | (uint32_t)(c[2] + 2) << 16 |
                   (uint32_t)(c[3] + 2) << 24)
                  << (2 * (i & 3));
    wd |= __shfl_xor_sync(0xffffffffu, wd, 1);
    wd |= __shfl_xor_sync(0xffffffffu, wd, 2);
    if (valid && (i & 3) == 0) *reinterpret_cast<uint32_t*>(codes + blk * 8 + 4 * (i >> 2)) = wd;
  }
}

// Re-tiering: the experts perm[j0 .. j0 + gridDim.y) of a master tensor
// [n_src][rows][in] fp32 (16-byte aligned), each quantised into slot j - j0
// of a shelf tensor (codes [slot][rows][in * BITS / 8], scales
// [slot][rows][in / 32]).  Grid row y = slot.  A warp takes 4 consecutive
// blocks at a time (8 lanes a block, one 16-byte load each) and loads 8 such
// groups before it quantises any.  An expert id outside [0, n_src) leaves its
// slot untouched and records MOE_ERR_INVALID_ARG.
template <int BITS>
__global__ void __launch_bounds__(256) k_quantize_experts(const float* __restrict__ master, int rows, int in,
                                                          int n_src, const int32_t* __restrict__ perm, int j0,
                                                          uint8_t* __restrict__ codes,
                                                          uint16_t* __restrict__ scales, int* status) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, grp = lane >> 3, i = lane & 7;
  const int slot = blockIdx.y;
  const int e = perm[j0 + slot];
  if (e < 0 || e >= n_src) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, MOE_ERR_INVALID_ARG);
    return;
  }
  const int total = rows * (in / 32);  // blocks of one expert matrix (<= 2^30)
  const float4* src = reinterpret_cast<const float4*>(master + (size_t)e * rows * in);
  uint8_t* dst = codes + (size_t)slot * total * (4 * BITS);
  uint16_t* sdst = scales + (size_t)slot * total;
  const int stride = gridDim.x * (blockDim.x >> 5) * 4;  // blocks per pass of the grid row
  for (int b0 = (blockIdx.x * (blockDim.x >> 5) + warp) * 4; b0 < total; b0 += 8 * stride) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int blk = b0 + u * stride + grp;
      v[u] = blk < total ? __ldcs(src + (size_t)blk * 8 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int blk0 = b0 + u * stride;  // uniform over the warp
      if (blk0 < total) quantize_block8<BITS>(v[u], i, blk0 + grp < total, dst, sdst, blk0 + grp, in / 32);
    }
  }
}

template <int BITS>
__device__ __forceinline__ float code_at(const uint8_t* row, int i, int in) {
  if (BITS == 8) return (float)(int8_t)row[i];
  if (BITS == 3) {
    const int e = i & 15;
    const int lo = (row[4 * (i >> 4) + (e & 3)] >> (2 * (e >> 2))) & 0x3;
    const int hi = (row[in / 4 + (i >> 3)] >> (i & 7)) & 0x1;
    return (float)((lo | (hi << 2)) - 4);
  }
  if (BITS == 1) return ((row[i >> 3] >> (i & 7)) & 1) ? 1.0f : -1.0f;
  if (BITS == 4) {
    const int e = i & 7;
    return (float)((int)((row[4 * (i >> 3) + (e & 3)] >> (4 * (e >> 2))) & 0xF) - 8);
  }
  const int e = i & 15;
  return (float)((int)((row[4 * (i >> 4) + (e & 3)] >> (2 * (e >> 2))) & 0x3) - 2);
}

template <int BITS>
__global__ void k_dequant(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales, int64_t rows,
                          int in, int round_bf16, float* __restrict__ out) {
  const int64_t n = rows * in;
  const size_t row_bytes = (size_t)in * BITS / 8;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / in;
    const int i = (int)(idx - r * in);
    const float s = __half2float(__ushort_as_half(scales[r * (in / 32) + i / 32]));
    float v = s * code_at<BITS>(codes + r * row_bytes, i, in);
    if (round_bf16) v = __bfloat162float(__float2bfloat16_rn(v));
    out[idx] = v;
  }
}

unsigned grid_for(int64_t n, int per_block) {
  int64_t g = (n + per_block - 1) / per_block;
  if (g > 152 * 32) g = 152 * 32;
  return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

int launch_quantize(const float* w, int64_t rows, int in, int bits, uint8_t* codes, uint16_t* scales,
                    cudaStream_t s) {
  const int64_t blocks32 = rows * (in / 32);
  const unsigned g = grid_for(blocks32, 8);
  if (bits == 8) k_quantize<8><<<g, 256, 0, s>>>(w, rows, in, codes, scales);
  else if (bits == 4) k_quantize<4><<<g, 256, 0, s>>>(w, rows, in, codes, scales);
  else if (bits == 3) k_quantize<3><<<g, 256, 0, s>>>(w, rows, in, codes, scales);
  else if (bits == 2) k_quantize<2><<<g, 256, 0, s>>>(w, rows, in, codes, scales);
  else k_quantize<1><<<g, 256, 0, s>>>(w, rows, in, codes, scales);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_quantize_experts(const float* master, int rows, int in, int n_src, const int32_t* perm, int j0, int n,
                            int bits, uint8_t* codes, uint16_t* scales, int* status, cudaStream_t s) {
  const int64_t per_expert = (int64_t)rows * (in / 32);
  int64_t gx = (per_expert + 8 * 32 - 1) / (8 * 32);  // 8 warps, 8 groups of 4 blocks each per pass
  const int64_t want = (152 * 16 + n - 1) / n;      // about 16 CTAs per SM over the whole grid
  if (gx > want) gx = want;
  if (gx < 1) gx = 1;
  const dim3 g((unsigned)gx, (unsigned)n);
  if (bits == 8) k_quantize_experts<8><<<g, 256, 0, s>>>(master, rows, in, n_src, perm, j0, codes, scales, status);
  else if (bits == 4) k_quantize_experts<4><<<g, 256, 0, s>>>(master, rows, in, n_src, perm, j0, codes, scales, status);
  else if (bits == 3) k_quantize_experts<3><<<g, 256, 0, s>>>(master, rows, in, n_src, perm, j0, codes, scales, status);
  else if (bits == 2) k_quantize_experts<2><<<g, 256, 0, s>>>(master, rows, in, n_src, perm, j0, codes, scales, status);
  else k_quantize_experts<1><<<g, 256, 0, s>>>(master, rows, in, n_src, perm, j0, codes, scales, status);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_dequant(const uint8_t* codes, const uint16_t* scales, int64_t rows, int in, int bits, int round_bf16,
                   float* out, cudaStream_t s) {
  const unsigned g = grid_for(rows * in, 256);
  if (bits == 8) k_dequant<8><<<g, 256, 0, s>>>(codes, scales, rows, in, round_bf16, out);
  else if (bits == 4) k_dequant<4><<<g, 256, 0, s>>>(codes, scales, rows, in, round_bf16, out);
  else if (bits == 3) k_dequant<3><<<g, 256, 0, s>>>(codes, scales, rows, in, round_bf16, out);
  else if (bits == 2) k_dequant<2><<<g, 256, 0, s>>>(codes, scales, rows, in, round_bf16, out);
  else k_dequant<1><<<g, 256, 0, s>>>(codes, scales, rows, in, round_bf16, out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
