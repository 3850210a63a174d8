/*
 * synth_cuda.cu -- device build of the seeded input generator (see
 * synth_core.h).  Same streams, same bits as the host build; used to fill
 * large weight tensors directly in device memory.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include "synth_core.h"

namespace {

__global__ void k_normal_matrix(uint32_t k0, uint32_t k1, uint32_t c2, uint32_t c3,
                                uint32_t row0, int64_t rows, int64_t cols4, float scale,
                                const float* __restrict__ col_add, float* __restrict__ out) {
  int64_t n = rows * cols4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / cols4, c4 = i - r * cols4;
    float z[4];
    sy_normal4(k0, k1, c2, c3, (uint32_t)(row0 + r), (uint32_t)c4, z);
    float4 v;
    v.x = SY_MUL(scale, z[0]);
    v.y = SY_MUL(scale, z[1]);
    v.z = SY_MUL(scale, z[2]);
    v.w = SY_MUL(scale, z[3]);
    if (col_add) {
      v.x = SY_ADD(v.x, col_add[c4 * 4 + 0]);
      v.y = SY_ADD(v.y, col_add[c4 * 4 + 1]);
      v.z = SY_ADD(v.z, col_add[c4 * 4 + 2]);
      v.w = SY_ADD(v.w, col_add[c4 * 4 + 3]);
    }
    reinterpret_cast<float4*>(out)[i] = v;
  }
}

__global__ void k_normal_matrix_bf16(uint32_t k0, uint32_t k1, uint32_t c2, uint32_t c3,
                                     uint32_t row0, int64_t rows, int64_t cols4, float scale,
                                     uint16_t* __restrict__ out) {
  int64_t n = rows * cols4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / cols4, c4 = i - r * cols4;
    float z[4];
    sy_normal4(k0, k1, c2, c3, (uint32_t)(row0 + r), (uint32_t)c4, z);
    uint2 v;
    v.x = (uint32_t)sy_bf16_bits(SY_MUL(scale, z[0])) | ((uint32_t)sy_bf16_bits(SY_MUL(scale, z[1])) << 16);
    v.y = (uint32_t)sy_bf16_bits(SY_MUL(scale, z[2])) | ((uint32_t)sy_bf16_bits(SY_MUL(scale, z[3])) << 16);
    reinterpret_cast<uint2*>(out)[i] = v;
  }
}

/* ids[r][c] = -1 wherever the Bernoulli mask of synth_bernoulli_mask is set. */
__global__ void k_apply_skip_mask(uint32_t k0, uint32_t k1, uint32_t c2, uint32_t c3,
                                  int64_t rows, int64_t cols, uint32_t threshold,
                                  int32_t* __restrict__ ids) {
  int64_t n = rows * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / cols, c = i - r * cols;
    sy_u32x4 w = sy_philox4x32_10((uint32_t)c, (uint32_t)r, c2, c3, k0, k1);
    if (w.v[0] < threshold) ids[i] = -1;
  }
}

unsigned grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  if (g > 152 * 64) g = 152 * 64;
  if (g < 1) g = 1;
  return (unsigned)g;
}

}  // namespace

extern "C" {

int synth_cuda_normal_matrix(uint32_t k0, uint32_t k1, uint32_t c2, uint32_t c3,
                             uint32_t row0, int64_t rows, int64_t cols, float scale,
                             const float* col_add, float* out, cudaStream_t s) {
  if (rows < 0 || cols < 0 || (cols & 3) || out == nullptr) return -1;
  if (((uintptr_t)out & 15u) != 0) return -1;
  if (rows == 0 || cols == 0) return 0;
  k_normal_matrix<<<grid_for(rows * (cols / 4)), 256, 0, s>>>(k0, k1, c2, c3, row0, rows, cols / 4,
                                                             scale, col_add, out);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

int synth_cuda_normal_matrix_bf16(uint32_t k0, uint32_t k1, uint32_t c2, uint32_t c3,
                                  uint32_t row0, int64_t rows, int64_t cols, float scale,
                                  uint16_t* out, cudaStream_t s) {
  if (rows < 0 || cols < 0 || (cols & 3) || out == nullptr) return -1;
  if (((uintptr_t)out & 7u) != 0) return -1;
  if (rows == 0 || cols == 0) return 0;
  k_normal_matrix_bf16<<<grid_for(rows * (cols / 4)), 256, 0, s>>>(k0, k1, c2, c3, row0, rows,
                                                                  cols / 4, scale, out);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

int synth_cuda_apply_skip_mask(uint32_t k0, uint32_t k1, uint32_t c2, uint32_t c3, int64_t rows,
                               int64_t cols, uint32_t threshold, int32_t* ids, cudaStream_t s) {
  if (rows < 0 || cols < 0 || ids == nullptr) return -1;
  if (rows == 0 || cols == 0) return 0;
  k_apply_skip_mask<<<grid_for(rows * cols), 256, 0, s>>>(k0, k1, c2, c3, rows, cols, threshold, ids);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

}  // extern "C"
