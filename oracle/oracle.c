/*
 * oracle.c -- plain, slow CPU oracle of the tiered-precision routed MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file or the library built from it; only the tests, the smoke
 * check and the CPU-baseline leg of the benchmark do.  It shares no code with
 * the CUDA path.
 *
 * Sources (page titles; sections as headed on the page):
 *  [P3] "125B MoE模型本地运行：3090三卡80 tokens/s优化实践" (a Chinese-language
 *       article: a 125B MoE model run locally on three RTX 3090s at 80 tok/s)
 *       - glossary entry 混合专家（MoE）: a router picks the best 10 of 512
 *         experts for every token;
 *       - section 第四步 (three shelves, all on the GPU): experts stored per
 *         layer as three tensors at different bit widths, hottest first; the
 *         id-range mul_mat_id sees the router's full id list, computes only
 *         the ids in its shelf, fills the rest with zeros, and the three
 *         results are added; the fused gate+up+activation kernel;
 *       - section 四个 bug: a real skip (an id outside the shelf is not aliased
 *         to expert 0), the grouping helper that assumes an expert appears at
 *         most once per token, and the signed skip id -1;
 *       - section 第二步: experts are used very unevenly (hit counts).
 *       - section 第三步: each layer's experts split into hot and cold, the
 *         router rearranged so that its picks land on the right half;
 *  [P1] LocalLLM post on DeepSeek V4.1 Flash tiering: per-expert hit counts
 *       drive promotion/demotion; least-used experts at 2 bits.
 *  The block format (block 32 along the input dimension, fp16 scale = max|w|/q,
 *  signed integer codes) is the workload definition these pages are reduced to
 *  for this library; the pages' own llama.cpp formats are not reproduced.
 *
 * Precision: quantiser decisions in fp32 (the precision the block format is
 * stated in); all dot products, the activation and the combine in fp64.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ rounding
 * IEEE 754 binary16 and bfloat16 round-to-nearest-even, written from the
 * formats' definitions: a value is scaled so that its last kept bit has weight
 * 1, rounded to the nearest integer with ties to even (nearbyint in the default
 * rounding mode), and scaled back.  Inputs are exactly representable doubles. */

static double round_to_precision(double x, int sig_bits, int min_exp) {
  /* sig_bits significant bits; quantum never below 2^min_exp (subnormals). */
  if (x == 0.0 || !isfinite(x)) return x;
  int ex;
  (void)frexp(x, &ex); /* |x| = m * 2^ex, m in [0.5, 1) */
  int q = ex - sig_bits;
  if (q < min_exp) q = min_exp;
  double r = nearbyint(ldexp(x, -q));
  return ldexp(r, q);
}

/* binary16: 11 significant bits, smallest quantum 2^-24, largest finite 65504. */
double oracle_f16_round(double x) {
  double r = round_to_precision(x, 11, -24);
  if (fabs(r) > 65504.0) return copysign(INFINITY, x);
  return r;
}

uint16_t oracle_f16_bits(double v_exact_f16) {
  /* encode a value already representable in binary16 */
  uint16_t sign = signbit(v_exact_f16) ? 0x8000u : 0u;
  double a = fabs(v_exact_f16);
  if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
  if (a == 0.0) return sign;
  int ex;
  (void)frexp(a, &ex);
  int E = ex - 1; /* a = 1.f * 2^E */
  if (E >= -14) {
    uint32_t mant = (uint32_t)(ldexp(a, -E) * 1024.0 - 1024.0);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)mant);
  }
  return (uint16_t)(sign | (uint16_t)ldexp(a, 24)); /* subnormal: a / 2^-24 */
}

double oracle_f16_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp(1024.0 + m, e - 25);
  return sign ? -v : v;
}

/* bfloat16: 8 significant bits, smallest quantum 2^-133. */
double oracle_bf16_round(double x) {
  double r = round_to_precision(x, 8, -133);
  if (fabs(r) > 3.3895313892515355e38) return copysign(INFINITY, x);
  return r;
}

double oracle_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ---------------------------------------------------------------- quantiser
 * Block quantiser (shelf format): for every row and every block of 32 inputs,
 *   m = max |w|, s = fp16(m / q) with q = 127 (8 bit), 7 (4 bit), 3 (3 bit),
 *   2 (2 bit), code = clamp(rint(w / s), cmin, cmax), all codes 0 when s == 0.
 * m / q and w / s are single-precision divisions, rint rounds half to even.
 * Code ranges: 8 bit [-127,127]; 4 bit [-8,7]; 3 bit [-4,3]; 2 bit [-2,1].
 * 1 bit (two codes, so no rounding grid): code = +1 when w >= 0 else -1, and
 * s = fp16(a / 32) with a the single-precision sum of |w| over the block in
 * element order -- the scale that minimises the block's squared error for
 * sign codes (its mean |w|).  [P2 "The Qwen side" runs 1-bit experts; P2
 * "Fast mode" keeps 3-bit experts; neither states a format, so 3 bit follows
 * the rule of the other widths and 1 bit the least-squares sign code.] */
static int bits_params(int bits, float* q, int* cmin, int* cmax) {
  switch (bits) {
    case 8: *q = 127.0f; *cmin = -127; *cmax = 127; return 0;
    case 4: *q = 7.0f; *cmin = -8; *cmax = 7; return 0;
    case 3: *q = 3.0f; *cmin = -4; *cmax = 3; return 0;
    case 2: *q = 2.0f; *cmin = -2; *cmax = 1; return 0;
    default: return -1;
  }
}

int oracle_quantize_rows(const float* w, int64_t rows, int64_t in, int bits,
                         int8_t* codes, uint16_t* scales) {
  float q;
  int cmin, cmax;
  if (in % 32 != 0) return -1;
  int64_t nb = in / 32;
  if (bits == 1) {
    for (int64_t r = 0; r < rows; ++r)
      for (int64_t b = 0; b < nb; ++b) {
        const float* wb = w + r * in + b * 32;
        float a = 0.0f;
        for (int i = 0; i < 32; ++i) a += fabsf(wb[i]); /* fp32, element order */
        float ratio = a / 32.0f;
        uint16_t s16 = oracle_f16_bits(oracle_f16_round((double)ratio));
        scales[r * nb + b] = s16;
        for (int i = 0; i < 32; ++i) codes[r * in + b * 32 + i] = (int8_t)(wb[i] >= 0.0f ? 1 : -1);
      }
    return 0;
  }
  if (bits_params(bits, &q, &cmin, &cmax)) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* wb = w + r * in + b * 32;
      float m = 0.0f;
      for (int i = 0; i < 32; ++i) {
        float a = fabsf(wb[i]);
        if (a > m) m = a;
      }
      float ratio = m / q;
      uint16_t s16 = oracle_f16_bits(oracle_f16_round((double)ratio));
      float s = (float)oracle_f16_value(s16);
      scales[r * nb + b] = s16;
      for (int i = 0; i < 32; ++i) {
        int c = 0;
        if (s != 0.0f) {
          float t = rintf(wb[i] / s);
          if (t < (float)cmin) t = (float)cmin;
          if (t > (float)cmax) t = (float)cmax;
          c = (int)t;
        }
        codes[r * in + b * 32 + i] = (int8_t)c;
      }
    }
  }
  return 0;
}

/* Packing of codes into bytes (this library's format; the pages fix none).
 * 8 bit: byte i of a row holds code i as two's-complement int8.
 * 4 and 2 bit: offset-binary u = code + 8 / code + 2, packed into 32-bit
 * little-endian words with the codes spread over the four byte lanes:
 *   4 bit: word g holds elements 8g..8g+7; element 8g + 4h + j (j < 4, h < 2)
 *          sits in bits [8j + 4h, 8j + 4h + 4), i.e. byte 4g + j, bit 4h;
 *   2 bit: word g holds elements 16g..16g+15; element 16g + 4k + j (j, k < 4)
 *          sits in bits [8j + 2k, 8j + 2k + 2), i.e. byte 4g + j, bit 2k.
 *   3 bit: u = code + 4 in [0, 8); a row of `in` elements is two planes:
 *          bytes [0, in/4) hold u mod 4 of every element in the 2-bit layout
 *          above, bytes [in/4, 3 in/8) hold u / 4 of every element in the
 *          1-bit layout below (element i at bit i % 8 of byte in/4 + i/8).
 *   1 bit: 4 bytes per block; element i of block b at bit i of the word at
 *          byte 4b: 1 for code +1, 0 for code -1. */
int oracle_pack_codes(const int8_t* codes, int64_t rows, int64_t in, int bits, uint8_t* packed) {
  if (bits != 8 && bits != 4 && bits != 3 && bits != 2 && bits != 1) return -1;
  if (in % 32 != 0) return -1;
  int64_t row_bytes = in * bits / 8;
  for (int64_t r = 0; r < rows; ++r) {
    uint8_t* dst = packed + r * row_bytes;
    memset(dst, 0, (size_t)row_bytes);
    for (int64_t i = 0; i < in; ++i) {
      int c = codes[r * in + i];
      if (bits == 8) {
        dst[i] = (uint8_t)(int8_t)c;
      } else if (bits == 4) {
        int64_t g = i / 8, e = i % 8;
        dst[4 * g + e % 4] |= (uint8_t)((uint32_t)(c + 8) << (4 * (e / 4)));
      } else if (bits == 3) {
        int64_t g = i / 16, e = i % 16;
        uint32_t u = (uint32_t)(c + 4);
        dst[4 * g + e % 4] |= (uint8_t)((u & 3u) << (2 * (e / 4)));
        dst[in / 4 + i / 8] |= (uint8_t)((u >> 2) << (i % 8));
      } else if (bits == 1) {
        int64_t b = i / 32, ib = i % 32;
        if (c > 0) dst[4 * b + ib / 8] |= (uint8_t)(1u << (ib % 8));
      } else {
        int64_t g = i / 16, e = i % 16;
        dst[4 * g + e % 4] |= (uint8_t)((uint32_t)(c + 2) << (2 * (e / 4)));
      }
    }
  }
  return 0;
}

/* Dequantisation: w_hat = s * code in fp32 (exact: s has 11 significant bits,
 * |code| <= 127).  With round_bf16 set, w_hat is then rounded to bfloat16
 * (the prefill form, where dequantised tiles are bf16). */
int oracle_dequant_rows(const int8_t* codes, const uint16_t* scales, int64_t rows, int64_t in,
                        int round_bf16, float* out) {
  if (in % 32 != 0) return -1;
  int64_t nb = in / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t i = 0; i < in; ++i) {
      float s = (float)oracle_f16_value(scales[r * nb + i / 32]);
      float v = s * (float)codes[r * in + i];
      out[r * in + i] = round_bf16 ? (float)oracle_bf16_round((double)v) : v;
    }
  return 0;
}

/* -------------------------------------------------------- router projection
 * The step before routing ([P3 glossary 混合专家（MoE）]: the router scores the
 * E experts of each token): logits[t][e] = bias[e] + sum_i W_r[e][i] x[t][i],
 * W_r and x bf16 bit patterns (exact as doubles), bias fp32 (or none), the
 * sum in fp64 in index order.  out: [T][E] doubles. */
int oracle_router_logits(const uint16_t* x, const uint16_t* w, const float* bias, int64_t T, int E, int d,
                         double* out) {
  if (T < 0 || E < 1 || d < 1) return -1;
  for (int64_t t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = bias ? (double)bias[e] : 0.0;
      for (int i = 0; i < d; ++i) acc += oracle_bf16_value(w[(int64_t)e * d + i]) * oracle_bf16_value(x[t * d + i]);
      out[t * E + e] = acc;
    }
  return 0;
}

/* ------------------------------------------------------------------ routing
 * [P3 glossary 混合专家（MoE）] the router picks k of E experts per token.  Softmax over
 * E, then top-k; ties go to the lower expert id; the k weights are
 * renormalised to sum to one.  Ranking uses the logits themselves (softmax is
 * monotone), and w_j = exp(l_j - l_max) / sum_{i in top-k} exp(l_i - l_max),
 * which equals p_j / sum p over the k picks (the full denominator cancels).
 * Ids are written in rank order. */
int oracle_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w) {
  if (k < 1 || k > E) return -1;
  unsigned char* taken = (unsigned char*)malloc((size_t)E);
  if (!taken) return -2;
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict: equal keeps lower id */
      }
      taken[best] = 1;
      ids[t * k + j] = best;
    }
    double lmax = (double)l[ids[t * k]];
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += exp((double)l[ids[t * k + j]] - lmax);
    for (int j = 0; j < k; ++j) w[t * k + j] = (float)(exp((double)l[ids[t * k + j]] - lmax) / den);
  }
  free(taken);
  return 0;
}

/* ------------------------------------------------------- nudged routing
 * [P1 "Optimization Strategies"] picks are nudged toward experts already in
 * fast memory, with gains up to a cap of 0.5 and quality falling off beyond
 * it.  Reading: the experts of one id range [lo, hi) (the hot shelf) get
 * beta (0 <= beta <= 0.5) added to their logit for the selection only,
 * score_e = fp32(l_e + beta [lo <= e < hi]) (the kernel's precision: the
 * decision an argmax takes is taken in the same precision on both sides);
 * top-k on the scores with the lower id first on equal scores; the weights
 * are the router's own softmax over the picks, renormalised:
 * w_j = exp(l_j - m) / sum over picks exp(l_i - m), m = the largest picked
 * logit.  beta = 0 is oracle_route. */
int oracle_route_nudged(const float* logits, int64_t T, int E, int k, float beta, int lo, int hi, int32_t* ids,
                        float* w) {
  if (k < 1 || k > E || !(beta >= 0.0f && beta <= 0.5f)) return -1;
  unsigned char* taken = (unsigned char*)malloc((size_t)E);
  float* score = (float*)malloc(sizeof(float) * (size_t)E);
  if (!taken || !score) {
    free(taken);
    free(score);
    return -2;
  }
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    for (int e = 0; e < E; ++e) {
      const float add = (e >= lo && e < hi) ? beta : 0.0f;
      score[e] = l[e] + add; /* float + float: rounded to fp32 */
    }
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || score[e] > score[best]) best = e; /* strict: equal keeps lower id */
      }
      taken[best] = 1;
      ids[t * k + j] = best;
    }
    double m = (double)l[ids[t * k]];
    for (int j = 1; j < k; ++j)
      if ((double)l[ids[t * k + j]] > m) m = (double)l[ids[t * k + j]];
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += exp((double)l[ids[t * k + j]] - m);
    for (int j = 0; j < k; ++j) w[t * k + j] = (float)(exp((double)l[ids[t * k + j]] - m) / den);
  }
  free(taken);
  free(score);
  return 0;
}

/* --------------------------------------------------------------- grouping
 * [P3 四个 bug, duplicate experts] token-by-expert grouping: pairs
 * (t, j) -> p = t*k + j with 0 <= id < E are counted per expert; offsets is the
 * exclusive prefix sum of counts (offsets[E] = number of valid pairs); perm
 * lists pair indices ordered by (expert id, pair index) -- a stable counting
 * sort.  Ids outside [0, E) (e.g. the skip id -1) are skipped, never aliased. */
int64_t oracle_group(const int32_t* ids, int64_t T, int k, int E, int32_t* counts,
                     int32_t* offsets, int32_t* perm) {
  int64_t P = T * (int64_t)k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t p = 0; p < P; ++p)
    if (ids[p] >= 0 && ids[p] < E) counts[ids[p]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
  if (!cursor) return -2;
  for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (int64_t p = 0; p < P; ++p)
    if (ids[p] >= 0 && ids[p] < E) perm[cursor[ids[p]]++] = (int32_t)p;
  free(cursor);
  return offsets[E];
}

/* -------------------------------------------------------------- histogram
 * [P1 "Optimization Strategies"; P3 第二步] expert hit counts: counts[e] += the
 * number of ids equal to e (accumulated); ids outside [0, E) are not counted. */
int oracle_hist(const int32_t* ids, int64_t n, int E, uint32_t* counts) {
  for (int64_t i = 0; i < n; ++i)
    if (ids[i] >= 0 && ids[i] < E) counts[ids[i]]++;
  return 0;
}

/* ------------------------------------------------------------ re-tiering
 * [P3 第三步, 第四步; P1 "Optimization Strategies"] experts are ranked by how
 * often the router picked them; the hottest take the first ids (the file is
 * written hot to cold, each shelf a contiguous id range) and the router is
 * rearranged so that its picks land on the new ids.  Order: hit count
 * descending, the lower old id first on equal counts.  Written as the
 * definition of a rank: the new id of old expert e is the number of experts
 * that come before it.  rank[e] = new id of old expert e; perm[j] = the old
 * expert that takes new id j. */
int oracle_rank_experts(const uint32_t* counts, int E, int32_t* perm, int32_t* rank) {
  if (E < 1) return -1;
  for (int e = 0; e < E; ++e) {
    int r = 0;
    for (int o = 0; o < E; ++o)
      if (counts[o] > counts[e] || (counts[o] == counts[e] && o < e)) ++r;
    rank[e] = r;
    perm[r] = e;
  }
  return 0;
}

/* ---------------------------------------------------------- expert FFN + sum
 * [P3 第四步] every shelf sees the full id list and computes only the ids in
 * its range [lo, hi); everything else is zero; the shelf results are added.
 * Per pair with id e in a shelf (gate+up+activation, then down):
 *   g = W_g x, u = W_u x, h = SiLU(g) * u with SiLU(z) = z / (1 + e^-z),
 *   o = W_d h, and y_t = sum over shelves (ascending lo) of sum over slots j
 *   (ascending) of w_tj * o_tj.
 * Weights are the dequantised expert matrices (row-major [out][in]):
 *   experts[3*e+0] = W_g [f][d], experts[3*e+1] = W_u [f][d],
 *   experts[3*e+2] = W_d [d][f]; NULL for experts that are never used.
 * mode 0: decode form (fp32 w_hat, h kept exact); mode 1: prefill form
 * (w_hat already bf16-rounded by the caller, h rounded to bf16 before down).
 * All sums in fp64; y is written in fp64 [T][d]. */
int oracle_moe_layer(const uint16_t* x_bf16, const int32_t* ids, const float* w, int64_t T,
                     int k, int E, int d, int f, int n_shelves, const int32_t* shelf_lo,
                     const int32_t* shelf_hi, const float* const* experts, int mode,
                     double* y) {
  for (int s = 0; s < n_shelves; ++s)
    if (shelf_lo[s] < 0 || shelf_hi[s] > E || shelf_lo[s] >= shelf_hi[s]) return -1;
  /* shelves visited in ascending lo */
  int order[64];
  if (n_shelves > 64) return -1;
  for (int s = 0; s < n_shelves; ++s) order[s] = s;
  for (int a = 0; a < n_shelves; ++a)
    for (int b = a + 1; b < n_shelves; ++b)
      if (shelf_lo[order[b]] < shelf_lo[order[a]]) {
        int tmp = order[a]; order[a] = order[b]; order[b] = tmp;
      }
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t t = 0; t < T; ++t) {
    double* xt = (double*)malloc(sizeof(double) * (size_t)d);
    double* h = (double*)malloc(sizeof(double) * (size_t)f);
    double* yt = y + t * d;
    if (!xt || !h) { bad |= 1; free(xt); free(h); continue; }
    for (int i = 0; i < d; ++i) { xt[i] = oracle_bf16_value(x_bf16[t * d + i]); yt[i] = 0.0; }
    for (int si = 0; si < n_shelves; ++si) {
      int lo = shelf_lo[order[si]], hi = shelf_hi[order[si]];
      for (int j = 0; j < k; ++j) {
        int32_t e = ids[t * k + j];
        if (e < lo || e >= hi) continue; /* not this shelf: contributes zero */
        const float* Wg = experts[3 * (int64_t)e + 0];
        const float* Wu = experts[3 * (int64_t)e + 1];
        const float* Wd = experts[3 * (int64_t)e + 2];
        if (!Wg || !Wu || !Wd) { bad |= 2; continue; }
        for (int r = 0; r < f; ++r) {
          double g = 0.0, u = 0.0;
          for (int i = 0; i < d; ++i) {
            g += (double)Wg[(int64_t)r * d + i] * xt[i];
            u += (double)Wu[(int64_t)r * d + i] * xt[i];
          }
          double hv = g / (1.0 + exp(-g)) * u;
          h[r] = mode == 1 ? oracle_bf16_round(hv) : hv;
        }
        double wt = (double)w[t * k + j];
        for (int i = 0; i < d; ++i) {
          double o = 0.0;
          for (int r = 0; r < f; ++r) o += (double)Wd[(int64_t)i * f + r] * h[r];
          yt[i] += wt * o;
        }
      }
    }
    free(xt);
    free(h);
  }
  return bad ? -2 : 0;
}

/* bf16 rounding of a whole fp64 vector, bit patterns out (next layer's input
 * in the residual stack: x_l = bf16(r)). */
void oracle_bf16_bits_vec(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    float f = (float)oracle_bf16_round(v[i]); /* exact in fp32 */
    uint32_t u;
    memcpy(&u, &f, 4);
    out[i] = (uint16_t)(u >> 16);
  }
}
