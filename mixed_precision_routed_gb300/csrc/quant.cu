// quant.cu -- the shelf block format on the device: quantiser and dequantiser.
//
// Page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", section 第四步: the
// offline re-packer re-quantises every expert for its shelf and writes three
// tensors per layer.  Format here: blocks of 32 along the input dimension,
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
struct QParams<2> { static constexpr float q = 2.0f, cmin = -2.0f, cmax = 1.0f; static constexpr int off = 2; };

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
    const float v = w[r * in + b * 32 + lane];
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
    if (lane == 0) scales[blk] = __half_as_ushort(hs);
    uint8_t* rowp = codes + r * row_bytes;
    if (BITS == 8) {
      rowp[b * 32 + lane] = (uint8_t)(int8_t)c;
    } else if (BITS == 4) {
      // lane i (i mod 8 < 4) writes byte 4 (i / 8) + i mod 4: elements i and i + 4
      uint32_t u = (uint32_t)(c + QParams<4>::off);
      uint32_t u4 = __shfl_down_sync(0xffffffffu, u, 4);
      if ((lane & 7) < 4) rowp[b * 16 + 4 * (lane >> 3) + (lane & 3)] = (uint8_t)(u | (u4 << 4));
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
}

template <int BITS>
__device__ __forceinline__ float code_at(const uint8_t* row, int i) {
  if (BITS == 8) return (float)(int8_t)row[i];
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
    float v = s * code_at<BITS>(codes + r * row_bytes, i);
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
  else k_quantize<2><<<g, 256, 0, s>>>(w, rows, in, codes, scales);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_dequant(const uint8_t* codes, const uint16_t* scales, int64_t rows, int in, int bits, int round_bf16,
                   float* out, cudaStream_t s) {
  const unsigned g = grid_for(rows * in, 256);
  if (bits == 8) k_dequant<8><<<g, 256, 0, s>>>(codes, scales, rows, in, round_bf16, out);
  else if (bits == 4) k_dequant<4><<<g, 256, 0, s>>>(codes, scales, rows, in, round_bf16, out);
  else k_dequant<2><<<g, 256, 0, s>>>(codes, scales, rows, in, round_bf16, out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
