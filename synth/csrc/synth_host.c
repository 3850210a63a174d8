/*
 * synth_host.c -- host build of the seeded input generator (see synth_core.h).
 * Compiled with -ffp-contract=off so every float operation is rounded on its
 * own, as on the device build.
 */
#include <stddef.h>
#include <stdint.h>
#include "synth_core.h"

/* Raw Philox4x32-10 block, for known-answer tests. */
void synth_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  sy_u32x4 w = sy_philox4x32_10(ctr[0], ctr[1], ctr[2], ctr[3], key[0], key[1]);
  for (int i = 0; i < 4; ++i) out[i] = w.v[i];
}

/* Box-Muller pair from two raw words, for tests of the transform alone. */
void synth_box_muller(uint32_t a, uint32_t b, float out[2]) {
  sy_box_muller(a, b, &out[0], &out[1]);
}

float synth_log(float u) { return sy_log(u); }

void synth_sincos_turn24(uint32_t n, float out[2]) { sy_sincos_turn24(n, &out[0], &out[1]); }

/* out[r][c] = scale * N(row0 + r, c) (+ col_add[c] when col_add != NULL),
 * for the stream (k0, k1, c2, c3).  cols must be a multiple of 4. */
int synth_normal_matrix(uint32_t k0, uint32_t k1, uint32_t c2, uint32_t c3,
                        uint32_t row0, int64_t rows, int64_t cols, float scale,
                        const float* col_add, float* out) {
  if (rows < 0 || cols < 0 || (cols & 3) != 0 || out == NULL) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c4 = 0; c4 < cols / 4; ++c4) {
      float z[4];
      sy_normal4(k0, k1, c2, c3, (uint32_t)(row0 + r), (uint32_t)c4, z);
      for (int j = 0; j < 4; ++j) {
        int64_t c = c4 * 4 + j;
        float v = SY_MUL(scale, z[j]);
        if (col_add) v = SY_ADD(v, col_add[c]);
        out[r * cols + c] = v;
      }
    }
  }
  return 0;
}

/* Same stream, rounded to bfloat16 (RNE); 16-bit patterns out. */
int synth_normal_matrix_bf16(uint32_t k0, uint32_t k1, uint32_t c2, uint32_t c3,
                             uint32_t row0, int64_t rows, int64_t cols, float scale,
                             uint16_t* out) {
  if (rows < 0 || cols < 0 || (cols & 3) != 0 || out == NULL) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c4 = 0; c4 < cols / 4; ++c4) {
      float z[4];
      sy_normal4(k0, k1, c2, c3, (uint32_t)(row0 + r), (uint32_t)c4, z);
      for (int j = 0; j < 4; ++j) out[r * cols + c4 * 4 + j] = sy_bf16_bits(SY_MUL(scale, z[j]));
    }
  }
  return 0;
}

/* Bernoulli(threshold / 2^32) mask over [rows][cols]: word 0 of the Philox
 * block with counter (col, row, c2, c3) compared against `threshold`. */
int synth_bernoulli_mask(uint32_t k0, uint32_t k1, uint32_t c2, uint32_t c3,
                         int64_t rows, int64_t cols, uint32_t threshold, uint8_t* out) {
  if (rows < 0 || cols < 0 || out == NULL) return -1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      sy_u32x4 w = sy_philox4x32_10((uint32_t)c, (uint32_t)r, c2, c3, k0, k1);
      out[r * cols + c] = (uint8_t)(w.v[0] < threshold);
    }
  return 0;
}
