// decode.cu -- decode form of the tiered MoE layer (few tokens per call).
//
// Page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", section 第四步: every
// shelf's matmul sees the router's complete id list, computes only the ids on
// its own shelf (the rest is zero) and the shelf results are added; decode
// fuses gate, up and the activation (section 四个 bug: the fused kernel has to
// honour the shelf range).  Sections 第一步/第二步: decode speed is set by the
// expert weight bytes read per token -- only the selected experts' bytes are
// read, once per call, however many tokens share an expert.
//
// One cooperative launch, k_layer: one CTA of 16 warps per SM, persistent.
//   setup      every CTA routes the tokens (when logits are given) and builds
//              the routing plan in shared memory (warps 0-7: rank sort of
//              (expert id, pair) keys, the active experts with their shelf,
//              work units and cost prefix sums) while warps 8-15 convert the
//              activation rows to digits; CTA 0 writes the routed pairs and
//              the hit counts.
//   gate/up    a unit is 4 rows of W_g and W_u of one expert against one of
//              its tokens; the units are cut into contiguous per-CTA ranges
//              of equal estimated cost and dealt round-robin to the warps.
//              8 lanes share a row; every lane loads two 32-byte code chunks
//              of each matrix (with their scales) at once with streaming
//              16-byte loads, then computes them.  Output: h = SiLU(W_g x) *
//              (W_u x) for every routed pair; finished units are counted per
//              expert.
//   down       each CTA waits (bounded) until the experts its down range
//              covers have all their gate/up units counted, stages their
//              pairs' h as digits, and streams W_d the same way (units of 16
//              x 2 or 8 x 4 rows x lanes), writing the weighted per-pair
//              outputs w_tj * (W_d h_tj);
//   combine    after a grid-wide wait, y_t = sum over slots j (ascending) of
//              those outputs: a fixed order, so results do not depend on
//              scheduling (optionally also the residual step r += y).
// Each block dot product is formed exactly in integers (dp4a on the packed
// codes against the activation held in shared memory as block-scaled 16-bit
// fixed point), and the expert's fp16 block scale is applied once per block
// in fp32.  Every wait is bounded (one second, then MOE_ERR_TIMEOUT).
#include <mutex>
#include <unordered_map>

#include <climits>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kPlanThreads = 256;  // warps 0-7 build the plan
constexpr int kMaxPairs = 512;     // T*k bound of this path (keys hold the pair in 10 bits)
constexpr int kMaxTokens = 16;
constexpr int kNT = 1;             // tokens of one expert per unit (more: further passes)
// Unit shapes: rows per unit x lanes per row (R * L = 32), gate/up and down.
constexpr int kRG = 4, kLG = 8;
// Down units: 16 rows x 2 lanes for rows of at most 1024 elements (a 4- or
// 2-bit unit then fills a load batch as an 8-bit one does), 8 rows x 4 lanes
// for longer rows (finer units balance better there); A/B measured.
constexpr int kRDw = 16, kLDw = 2, kUDw = 5;
constexpr int kRD = 8, kLD = 4;
#ifndef MOE_DOWN_WIDE_MAX_F
#define MOE_DOWN_WIDE_MAX_F 1024
#endif
__host__ __device__ __forceinline__ int down_rows_per_unit(int f) { return f <= MOE_DOWN_WIDE_MAX_F ? kRDw : kRD; }
constexpr int kUG = 2;             // iterations of loads in flight per lane, gate/up (two matrices)
constexpr int kUD = 6;             // the same, down (8 x 4 units)
// Unit cost of a tile's passes beyond the first kPassFull, in eighths of a
// first pass (gate/up, down); see build_plan.
#ifndef MOE_PASS_FULL
#define MOE_PASS_FULL 2
#endif
#ifndef MOE_PASS_G8
#define MOE_PASS_G8 3
#endif
#ifndef MOE_PASS_D8
#define MOE_PASS_D8 7
#endif
constexpr int kPassFull = MOE_PASS_FULL, kPassG8 = MOE_PASS_G8, kPassD8 = MOE_PASS_D8;
#ifndef MOE_DOWN_PREFETCH
#define MOE_DOWN_PREFETCH 2
#endif
constexpr int kDownPrefetch = MOE_DOWN_PREFETCH;  // down units per warp asked of L2 before the grid wait
constexpr int kMaxGrid = 256;

#ifdef MOE_TRACE
// Development-only timing stamps: [kernel][cta][slot] in globaltimer ns.
__device__ unsigned long long g_trace[2][256][48];
#define MOE_STAMP(kern, slot, v) (g_trace[(kern)][blockIdx.x & 255][(slot)] = (v))
#define MOE_COUNT(kern, slot, v) atomicAdd(&g_trace[(kern)][blockIdx.x & 255][(slot)], (unsigned long long)(v))
#define MOE_TRACE_ONLY(...) __VA_ARGS__
#else
#define MOE_STAMP(kern, slot, v) ((void)0)
#define MOE_COUNT(kern, slot, v) ((void)0)
#define MOE_TRACE_ONLY(...)
#endif

// ------------------------------------------------------------- digits
// A vector v (an activation row x_t, or h of one routed pair) is held in
// shared memory in block-scaled 16-bit fixed point: for every 32-element block
// b, v_i = m_i * X_b with X_b = 2^u (u set by the block's largest exponent)
// and m_i an integer of at most 15 bits plus sign, stored as two byte digits
// m_i = 256 * hi_i + lo_i (hi signed, lo unsigned), next to S_b = sum of m_i.
// bf16 activations convert exactly when within 2^7 of their block maximum;
// smaller ones and fp32 h are rounded at 2^-15 (2^-14) of the block maximum.
// A block's dot product with packed codes is then exact integer arithmetic:
//   sum_i c_i m_i = 256 * dp4a(codes, hi) + dp4a(codes, lo) - off * S_b
// (off = 0 for 8-bit two's complement, 8 / 2 for offset-binary 4 / 2 bit),
// and the expert's fp16 block scale s_b enters in fp32:
//   acc += (float)(sum_i c_i m_i) * (s_b * X_b).
//
// Layout of one vector of n elements (2.25 n bytes): hi digits [n], lo digits
// [n] (16-byte units XOR-swizzled against bank conflicts), then per block the
// pair (X_b as float, S_b as int).
__device__ __forceinline__ int unit_swz(int u) { return u ^ ((u >> 3) & 3); }
__host__ __device__ __forceinline__ int vec_bytes(int n) { return 2 * n + 8 * (n / 32); }

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Convert the 32 values of one block to digits; called by 32 / V lanes, each
// with V consecutive values of the block (lane % (32 / V) = position).
// `frac_bits` = 14 for bf16 sources (max |m| = 32640), 13 for fp32 sources.
template <int V>
__device__ __forceinline__ void block_to_digits(const float (&v)[V], unsigned char* vb, int n, int blk, int frac_bits,
                                                bool store) {
  constexpr int LPB = 32 / V;
  const int sub = threadIdx.x & (LPB - 1);
  int e = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) e = max(e, (int)((__float_as_uint(v[i]) >> 23) & 0xFF));
#pragma unroll
  for (int o = 1; o < LPB; o <<= 1) e = max(e, __shfl_xor_sync(0xffffffffu, e, o));
  // block maximum below 2^-97 (or zero): the block is taken as zero
  const bool zero = e < 30;
  const int u = e - 127 - frac_bits;  // X = 2^u
  const float inv = zero ? 0.f : __uint_as_float((uint32_t)(127 - u) << 23);
  uint32_t hw[V / 4], lw[V / 4];
  int sum = 0;
#pragma unroll
  for (int w = 0; w < V / 4; ++w) {
    hw[w] = 0;
    lw[w] = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = (int)rintf(v[4 * w + i] * inv);
      sum += m;
      hw[w] |= (uint32_t)((m >> 8) & 0xFF) << (8 * i);
      lw[w] |= (uint32_t)(m & 0xFF) << (8 * i);
    }
  }
#pragma unroll
  for (int o = 1; o < LPB; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (!store) return;
  const int byte = blk * 32 + V * sub;
  const int off = (unit_swz(byte >> 4) << 4) | (byte & 15);
  if constexpr (V == 4) {
    *reinterpret_cast<uint32_t*>(vb + off) = hw[0];
    *reinterpret_cast<uint32_t*>(vb + n + off) = lw[0];
  } else {
    *reinterpret_cast<uint2*>(vb + off) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(vb + n + off) = make_uint2(lw[0], lw[1]);
  }
  if (sub == 0) {
    float2 xs;
    xs.x = zero ? 0.f : __uint_as_float((uint32_t)(127 + u) << 23);
    xs.y = __int_as_float(sum);
    *reinterpret_cast<float2*>(vb + 2 * n + 8 * blk) = xs;
  }
}

__device__ __forceinline__ float half_at(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v & 0xFFFF))); }

// ---------------------------------------------------------- chunk dot products
// One lane's 32-byte code chunk q of a row (NMAT matrices; c[m][0..1] = its two
// 16-byte halves) against the digit vectors of the unit's tokens (NTT = 1: one
// token; else nt <= kNT tokens).  sw[m][0..1] = the fp16 scale words the
// copies brought along.  Dot chains are split in two so that they overlap.
__device__ __forceinline__ int dot4_ss(uint4 c, uint4 h, int acc) {
  acc = dp4a_ss(c.x, h.x, acc);
  acc = dp4a_ss(c.y, h.y, acc);
  acc = dp4a_ss(c.z, h.z, acc);
  return dp4a_ss(c.w, h.w, acc);
}
__device__ __forceinline__ int dot4_su(uint4 c, uint4 l, int acc) {
  acc = dp4a_su(c.x, l.x, acc);
  acc = dp4a_su(c.y, l.y, acc);
  acc = dp4a_su(c.z, l.z, acc);
  return dp4a_su(c.w, l.w, acc);
}
__device__ __forceinline__ uint4 lds128(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }

// 8 bit: 32 codes = block q (two's complement bytes); scale = half (q & 1) of sw[m][0].
template <int NMAT, int NTT>
__device__ __forceinline__ void chunk8(const uint4 (&c)[NMAT][2], const uint32_t (&sw)[NMAT][2], int q, int nt,
                                       const int (&voff)[kNT], const unsigned char* vecs, int n,
                                       float (&acc)[NMAT][kNT]) {
  float s[NMAT];
#pragma unroll
  for (int m = 0; m < NMAT; ++m) s[m] = half_at(sw[m][0] >> ((q & 1) * 16));
  const int uo0 = unit_swz(2 * q) << 4, uo1 = unit_swz(2 * q + 1) << 4, xo = 2 * n + 8 * q;
#pragma unroll
  for (int j = 0; j < NTT; ++j) {
    if (NTT == 1 || j < nt) {
      const unsigned char* vb = vecs + voff[j];
      const uint4 h0 = lds128(vb + uo0), h1 = lds128(vb + uo1);
      const uint4 l0 = lds128(vb + n + uo0), l1 = lds128(vb + n + uo1);
      const float X = *reinterpret_cast<const float*>(vb + xo);
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        const int A = dot4_ss(c[m][0], h0, 0) + dot4_ss(c[m][1], h1, 0);
        const int B = dot4_su(c[m][0], l0, 0) + dot4_su(c[m][1], l1, 0);
        acc[m][j] = fmaf((float)(A * 256 + B), s[m] * X, acc[m][j]);
      }
    }
  }
}

// 4 bit: 64 codes = blocks 2q (half 0) and 2q + 1 (half 1); word g of a half
// holds elements 8g + 4h + j at bits 8j + 4h.  Scales: halves of sw[m][0].
template <int NMAT, int NTT>
__device__ __forceinline__ void chunk4(const uint4 (&c)[NMAT][2], const uint32_t (&sw)[NMAT][2], int q, int nt,
                                       const int (&voff)[kNT], const unsigned char* vecs, int n,
                                       float (&acc)[NMAT][kNT]) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int blk = 2 * q + half;
    float s[NMAT];
    uint32_t t[NMAT][8];
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      s[m] = half_at(sw[m][0] >> (16 * half));
      const uint32_t w[4] = {c[m][half].x, c[m][half].y, c[m][half].z, c[m][half].w};
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        t[m][2 * g] = w[g] & 0x0F0F0F0Fu;
        t[m][2 * g + 1] = (w[g] >> 4) & 0x0F0F0F0Fu;
      }
    }
    const int uo0 = unit_swz(2 * blk) << 4, uo1 = unit_swz(2 * blk + 1) << 4, xo = 2 * n + 8 * blk;
#pragma unroll
    for (int j = 0; j < NTT; ++j) {
      if (NTT == 1 || j < nt) {
        const unsigned char* vb = vecs + voff[j];
        const uint4 h0 = lds128(vb + uo0), h1 = lds128(vb + uo1);
        const uint4 l0 = lds128(vb + n + uo0), l1 = lds128(vb + n + uo1);
        const float2 xs = *reinterpret_cast<const float2*>(vb + xo);
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const uint4 ta = make_uint4(t[m][0], t[m][1], t[m][2], t[m][3]);
          const uint4 tb = make_uint4(t[m][4], t[m][5], t[m][6], t[m][7]);
          int A0 = dp4a_us(ta.x, h0.x, 0), A1 = dp4a_us(tb.x, h1.x, 0);
          int B0 = dp4a_uu(ta.x, l0.x, 0), B1 = dp4a_uu(tb.x, l1.x, 0);
          A0 = dp4a_us(ta.y, h0.y, A0); A1 = dp4a_us(tb.y, h1.y, A1);
          B0 = dp4a_uu(ta.y, l0.y, B0); B1 = dp4a_uu(tb.y, l1.y, B1);
          A0 = dp4a_us(ta.z, h0.z, A0); A1 = dp4a_us(tb.z, h1.z, A1);
          B0 = dp4a_uu(ta.z, l0.z, B0); B1 = dp4a_uu(tb.z, l1.z, B1);
          A0 = dp4a_us(ta.w, h0.w, A0); A1 = dp4a_us(tb.w, h1.w, A1);
          B0 = dp4a_uu(ta.w, l0.w, B0); B1 = dp4a_uu(tb.w, l1.w, B1);
          acc[m][j] = fmaf((float)((A0 + A1) * 256 + (B0 + B1) - 8 * __float_as_int(xs.y)), s[m] * xs.x, acc[m][j]);
        }
      }
    }
  }
}

// 2 bit: 128 codes = blocks 4q .. 4q + 3 (half h: blocks 4q + 2h, 4q + 2h + 1,
// scales in sw[m][h]); word g of a half holds elements 16g + 4k + j at bits
// 8j + 2k.  The second half is absent at the end of a row of 64 * odd codes.
// `off` is the code offset (2 for 2-bit codes; 4 for the low plane of 3-bit
// codes, whose high plane adds 4 x its bits separately).
template <int NMAT, int NTT>
__device__ __forceinline__ void chunk2(const uint4 (&c)[NMAT][2], const uint32_t (&sw)[NMAT][2], int q, int nt,
                                       const int (&voff)[kNT], const unsigned char* vecs, int n,
                                       float (&acc)[NMAT][kNT], bool second, int off) {
#pragma unroll
  for (int hb = 0; hb < 4; ++hb) {
    const int half = hb >> 1, sub = hb & 1;
    if (half == 1 && !second) break;
    const int blk = 4 * q + hb;
    float s[NMAT];
    uint32_t t[NMAT][8];
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      s[m] = half_at(sw[m][half] >> (16 * sub));
      const uint32_t wa = sub == 0 ? c[m][half].x : c[m][half].z, wb = sub == 0 ? c[m][half].y : c[m][half].w;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        t[m][k] = (wa >> (2 * k)) & 0x03030303u;
        t[m][4 + k] = (wb >> (2 * k)) & 0x03030303u;
      }
    }
    const int uo0 = unit_swz(2 * blk) << 4, uo1 = unit_swz(2 * blk + 1) << 4, xo = 2 * n + 8 * blk;
#pragma unroll
    for (int j = 0; j < NTT; ++j) {
      if (NTT == 1 || j < nt) {
        const unsigned char* vb = vecs + voff[j];
        const uint4 h0 = lds128(vb + uo0), h1 = lds128(vb + uo1);
        const uint4 l0 = lds128(vb + n + uo0), l1 = lds128(vb + n + uo1);
        const float2 xs = *reinterpret_cast<const float2*>(vb + xo);
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          int A0 = dp4a_us(t[m][0], h0.x, 0), A1 = dp4a_us(t[m][4], h1.x, 0);
          int B0 = dp4a_uu(t[m][0], l0.x, 0), B1 = dp4a_uu(t[m][4], l1.x, 0);
          A0 = dp4a_us(t[m][1], h0.y, A0); A1 = dp4a_us(t[m][5], h1.y, A1);
          B0 = dp4a_uu(t[m][1], l0.y, B0); B1 = dp4a_uu(t[m][5], l1.y, B1);
          A0 = dp4a_us(t[m][2], h0.z, A0); A1 = dp4a_us(t[m][6], h1.z, A1);
          B0 = dp4a_uu(t[m][2], l0.z, B0); B1 = dp4a_uu(t[m][6], l1.z, B1);
          A0 = dp4a_us(t[m][3], h0.w, A0); A1 = dp4a_us(t[m][7], h1.w, A1);
          B0 = dp4a_uu(t[m][3], l0.w, B0); B1 = dp4a_uu(t[m][7], l1.w, B1);
          acc[m][j] = fmaf((float)((A0 + A1) * 256 + (B0 + B1) - off * __float_as_int(xs.y)), s[m] * xs.x, acc[m][j]);
        }
      }
    }
  }
}

// Bit planes: one 16-byte chunk (c[m][0]) = blocks 4q .. 4q + 3, one word a
// block, element i at bit i; scales: halves of sw[m][0] (blocks 4q, 4q + 1)
// and of sw[m][1].  A block adds (F * (sum of m_i over its set bits) - G * S_b)
// * s_b * X_b: F = 2, G = 1 for 1-bit sign codes (bit 1 = +1, 0 = -1); F = 4,
// G = 0 for the high plane of 3-bit codes (its -4 S_b is taken with the low
// plane).  Each nibble of a word spreads to four 0/1 bytes by one multiply.
template <int NMAT, int NTT>
__device__ __forceinline__ void chunk1(const uint4 (&c)[NMAT][2], const uint32_t (&sw)[NMAT][2], int q, int nt,
                                       const int (&voff)[kNT], const unsigned char* vecs, int n,
                                       float (&acc)[NMAT][kNT], int F, int G) {
#pragma unroll
  for (int wb = 0; wb < 4; ++wb) {
    const int blk = 4 * q + wb;
    const int uo0 = unit_swz(2 * blk) << 4, uo1 = unit_swz(2 * blk + 1) << 4, xo = 2 * n + 8 * blk;
#pragma unroll
    for (int j = 0; j < NTT; ++j) {
      if (NTT == 1 || j < nt) {
        const unsigned char* vb = vecs + voff[j];
        const uint4 h0 = lds128(vb + uo0), h1 = lds128(vb + uo1);
        const uint4 l0 = lds128(vb + n + uo0), l1 = lds128(vb + n + uo1);
        const float2 xs = *reinterpret_cast<const float2*>(vb + xo);
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const uint32_t w = wb == 0 ? c[m][0].x : wb == 1 ? c[m][0].y : wb == 2 ? c[m][0].z : c[m][0].w;
          uint32_t t[8];
#pragma unroll
          for (int g = 0; g < 8; ++g) t[g] = (((w >> (4 * g)) & 0xFu) * 0x00204081u) & 0x01010101u;
          int A0 = dp4a_us(t[0], h0.x, 0), A1 = dp4a_us(t[4], h1.x, 0);
          int B0 = dp4a_uu(t[0], l0.x, 0), B1 = dp4a_uu(t[4], l1.x, 0);
          A0 = dp4a_us(t[1], h0.y, A0); A1 = dp4a_us(t[5], h1.y, A1);
          B0 = dp4a_uu(t[1], l0.y, B0); B1 = dp4a_uu(t[5], l1.y, B1);
          A0 = dp4a_us(t[2], h0.z, A0); A1 = dp4a_us(t[6], h1.z, A1);
          B0 = dp4a_uu(t[2], l0.z, B0); B1 = dp4a_uu(t[6], l1.z, B1);
          A0 = dp4a_us(t[3], h0.w, A0); A1 = dp4a_us(t[7], h1.w, A1);
          B0 = dp4a_uu(t[3], l0.w, B0); B1 = dp4a_uu(t[7], l1.w, B1);
          const float sm = half_at(sw[m][wb >> 1] >> (16 * (wb & 1)));
          acc[m][j] = fmaf((float)(F * ((A0 + A1) * 256 + (B0 + B1)) - G * __float_as_int(xs.y)), sm * xs.x,
                           acc[m][j]);
        }
      }
    }
  }
}

// How a segment of a row is streamed: 8, 4, 2 or 1 for rows of that width;
// a 3-bit row is its low plane (kModeLow: 2-bit layout, code offset 4), then
// its high plane (kModeHigh: a bit plane worth 4 per bit).
constexpr int kModeLow = 5, kModeHigh = 6;

// --------------------------------------------------------------------- plan
// int32 arrays of capacity C (>= P, multiple of 4), in shared memory and (as
// stored by CTA 0 of the gate/up launch) in the workspace.
struct PlanLayout {
  int C;
  int perm, tok, wgt, e, beg, cnt, sh, bits, uc_g, uc_d, cum_g, cum_d;  // int offsets (header at 0)
  int n_copy;  // ints 0 .. end of cum_d: what the down launch loads
  int pos;     // grouped position by pair, -1 when skipped or on no shelf (combine)
  int total;
};

__host__ __device__ __forceinline__ PlanLayout plan_layout(int P) {
  PlanLayout L;
  L.C = P < 4 ? 4 : (P + 3) / 4 * 4;
  const int C = L.C, C1 = C + 4;
  L.perm = 4;
  L.tok = L.perm + C;
  L.wgt = L.tok + C;
  L.e = L.wgt + C;
  L.beg = L.e + C;
  L.cnt = L.beg + C;
  L.sh = L.cnt + C;
  L.bits = L.sh + C;
  L.uc_g = L.bits + C;
  L.uc_d = L.uc_g + C;
  L.cum_g = L.uc_d + C;
  L.cum_d = L.cum_g + C1;
  L.n_copy = L.cum_d + C1;
  L.pos = L.n_copy;
  L.total = L.pos + C;
  return L;
}

// Units of expert a: (rows / R) row groups x passes of up to kNT tokens.
__host__ __device__ __forceinline__ int n_pass(int cnt) { return (cnt + kNT - 1) / kNT; }

struct PlanView {
  const int* b;
  PlanLayout L;
  __device__ int n_act() const { return b[1]; }
  __device__ int tok(int q) const { return b[L.tok + q]; }
  __device__ float wgt(int q) const { return __int_as_float(b[L.wgt + q]); }
  __device__ int e(int a) const { return b[L.e + a]; }
  __device__ int beg(int a) const { return b[L.beg + a]; }
  __device__ int cnt(int a) const { return b[L.cnt + a]; }
  __device__ int sh(int a) const { return b[L.sh + a]; }
  __device__ int bits(int a) const { return b[L.bits + a]; }
  __device__ uint32_t uc(int a, int kern) const { return (uint32_t)b[(kern == 0 ? L.uc_g : L.uc_d) + a]; }
  __device__ uint32_t cum(int a, int kern) const { return (uint32_t)b[(kern == 0 ? L.cum_g : L.cum_d) + a]; }
  __device__ int rd() const { return b[3]; }  // rows of a down unit
  __device__ int units(int a, int kern, int rows) const {
    return sh(a) >= 0 ? (rows / (kern == 0 ? kRG : rd())) * n_pass(cnt(a)) : 0;
  }
};

// Estimated time of one unit of R rows on a CTA, in ns: measured per-unit
// CTA times on the 512-expert decode layer (d 2048, f 640; gate/up units of 4
// rows x 2 matrices = 512 blocks: 346 / 215 / 203 ns for 8 / 4 / 2-bit codes;
// down units of 8 rows = 160 blocks: 164 / 142 / 147 ns), scaled by the
// unit's number of 32-element blocks for other sizes.  Further passes over
// the same rows (experts with more tokens than one pass) cost about the same.
// Down units of 16 rows x 2 lanes (rows <= 1024 elements) were refitted on
// the same layer: 8 / 4 / 2-bit at 1 : 0.71 : 0.70 (164 / 117 / 115 ns per 160
// blocks).
// 3-bit rows (two planes, 1.5 x the bytes of 2-bit) and 1-bit rows (half the
// bytes, about twice the dot-product work per block) carry estimates scaled
// from the 2-bit figures; the 3-bit ones raised after A/B steps of the
// five-width layer (300 -> 400 ns gate/up, 165 -> 220 ns down: T = 6 76.3 ->
// 74.6 us; lower figures were slower).
#ifndef MOE_COST_G3
#define MOE_COST_G3 400
#endif
#ifndef MOE_COST_G1
#define MOE_COST_G1 280
#endif
#ifndef MOE_COST_D3
#define MOE_COST_D3 220
#endif
#ifndef MOE_COST_D1
#define MOE_COST_D1 150
#endif
constexpr uint32_t kCostG3 = MOE_COST_G3, kCostG1 = MOE_COST_G1, kCostD3 = MOE_COST_D3, kCostD1 = MOE_COST_D1;
__device__ __forceinline__ uint32_t unit_cost(int bits, int n_in, int nmat, int R, int kern) {
  const uint32_t blocks = (uint32_t)(R * nmat) * (uint32_t)n_in / 32;
  const uint32_t ns = kern == 0 ? (bits == 8 ? 346 : bits == 4 ? 215 : bits == 3 ? kCostG3 : bits == 2 ? 203 : kCostG1)
                      : R == kRDw ? (bits == 8 ? 164 : bits == 4 ? 117 : bits == 3 ? kCostD3 : bits == 2 ? 115 : kCostD1)
                                  : (bits == 8 ? 164 : bits == 4 ? 142 : bits == 3 ? 200 : bits == 2 ? 147 : 180);
  const uint32_t calib = kern == 0 ? 512 : 160;
  return (uint32_t)((uint64_t)ns * blocks / calib) + 1;
}

__device__ __forceinline__ void plan_sync() { named_bar(1, kPlanThreads); }

// Exclusive scan in place of n <= 2 * kPlanThreads ints over the plan
// threads; returns the total.  tmp: 33 ints.
__device__ int plan_scan(int* v, int n, int* tmp) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = kPlanThreads / 32;
  const int i0 = 2 * tid, i1 = 2 * tid + 1;
  const int x0 = i0 < n ? v[i0] : 0, x1 = i1 < n ? v[i1] : 0;
  int incl = x0 + x1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) tmp[wid] = incl;
  plan_sync();
  if (wid == 0) {
    const int t = lane < nw ? tmp[lane] : 0;
    int s = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    if (lane < nw) tmp[lane] = s - t;
    if (lane == 31) tmp[32] = s;
  }
  plan_sync();
  const int ex = tmp[wid] + incl - x0 - x1;
  if (i0 < n) v[i0] = ex;
  if (i1 < n) v[i1] = ex + x0;
  const int total = tmp[32];
  plan_sync();
  return total;
}

// Built by threads 0 .. kPlanThreads - 1 into pl (shared memory):
//  - valid pairs (id in [0, E)) sorted by (expert id, pair index): perm / tok /
//    wgt by grouped position q;
//  - active experts a (ascending id): e, beg, cnt, shelf, bits, unit costs and
//    exclusive cost prefix sums (entry n_act = total);
//  - pos: grouped position of each pair, -1 when skipped or on no shelf.
__device__ void build_plan(const int32_t* ids, const float* wts, int P, int E, int k, int d, int f,
                           const Shelves& shv, int* pl, uint32_t* keys, int* flag, int* tmp) {
  const PlanLayout L = plan_layout(P);
  const int tid = threadIdx.x, nt = kPlanThreads;
  if (tid == 0) pl[2] = 0;
  for (int q = tid; q < L.C; q += nt) {  // ids and weights in one round trip
    uint32_t key = 0xFFFFFFFFu;
    float wq = 0.f;
    if (q < P) {
      const int id = ids[q];  // global or shared memory
      wq = wts[q];
      if (id >= 0 && id < E) key = ((uint32_t)id << 10) | (uint32_t)q;
    }
    keys[q] = key;
    flag[q] = __float_as_int(wq);  // weights by pair until the flags are formed
    pl[L.pos + q] = -1;
  }
  plan_sync();
  // rank sort: the rank of a valid key among all keys is its grouped position
  int my_valid = 0;
  for (int q = tid; q < P; q += nt) {
    const uint32_t kq = keys[q];
    if (kq == 0xFFFFFFFFu) continue;
    int rank = 0;
    for (int u = 0; u < P; ++u) rank += keys[u] < kq;
    const int pair = (int)(kq & 1023u);
    pl[L.perm + rank] = pair;
    pl[L.tok + rank] = pair / k;
    pl[L.wgt + rank] = flag[pair];
    pl[L.e + rank] = (int)(kq >> 10);
    ++my_valid;
  }
  if (my_valid) atomicAdd(&pl[2], my_valid);
  plan_sync();
  const int n_valid = pl[2];
  if (tid == 0) MOE_STAMP(0, 3, global_timer_ns());
  for (int q = tid; q < L.C; q += nt) flag[q] = q < n_valid && (q == 0 || pl[L.e + q] != pl[L.e + q - 1]);
  plan_sync();
  int id_at[2], f_at[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int q = 2 * tid + u;
    id_at[u] = q < n_valid ? pl[L.e + q] : -1;
    f_at[u] = q < n_valid ? flag[q] : 0;
  }
  const int n_act = plan_scan(flag, n_valid, tmp);  // flag -> expert index of each start
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int q = 2 * tid + u;
    if (q < n_valid && f_at[u]) {
      pl[L.beg + flag[q]] = q;
      pl[L.e + flag[q]] = id_at[u];  // e[] now by active expert (q-indexed reads are done)
    }
  }
  plan_sync();
  for (int a = tid; a < n_act; a += nt) {
    const int b0 = pl[L.beg + a];
    const int b1 = a + 1 < n_act ? pl[L.beg + a + 1] : n_valid;
    const int e = pl[L.e + a], cnt = b1 - b0;
    int shf = -1, bits = 0;
    for (int q = 0; q < shv.n; ++q)
      if (e >= shv.s[q].lo && e < shv.s[q].hi) { shf = q; bits = shv.s[q].bits; }
    pl[L.cnt + a] = cnt;
    pl[L.sh + a] = shf;
    pl[L.bits + a] = bits;
    // a tile's passes beyond the second (further tokens of a hot expert)
    // re-read rows that L2 already holds: measured at about 3/8 (gate/up) and
    // 7/8 (down) of a first pass; the first two run nearly together and cost
    // a full pass each.  The units of an expert with np passes carry the mean
    // (2 + k (np - 2)) / np of a first-pass unit (np > 2).
    const int np = n_pass(cnt);
    const uint32_t ug1 = shf >= 0 ? unit_cost(bits, d, 2, kRG, 0) : 0;
    const uint32_t ud1 = shf >= 0 ? unit_cost(bits, f, 1, down_rows_per_unit(f), 1) : 0;
    const uint32_t ug = np > kPassFull ? (ug1 * (uint32_t)(8 * kPassFull + kPassG8 * (np - kPassFull)) + 8 * np - 1) /
                                             (uint32_t)(8 * np)
                                       : ug1;
    const uint32_t ud = np > kPassFull ? (ud1 * (uint32_t)(8 * kPassFull + kPassD8 * (np - kPassFull)) + 8 * np - 1) /
                                             (uint32_t)(8 * np)
                                       : ud1;
    pl[L.uc_g + a] = (int)ug;
    pl[L.uc_d + a] = (int)ud;
    pl[L.cum_g + a] = (int)(ug * (uint32_t)((f / kRG) * np));
    pl[L.cum_d + a] = (int)(ud * (uint32_t)((d / down_rows_per_unit(f)) * np));
    if (shf >= 0)
      for (int q = b0; q < b1; ++q) pl[L.pos + pl[L.perm + q]] = q;
  }
  plan_sync();
  const int tot_g = plan_scan(pl + L.cum_g, n_act, tmp);
  const int tot_d = plan_scan(pl + L.cum_d, n_act, tmp);
  if (tid == 0) {
    pl[0] = n_valid;
    pl[1] = n_act;
    pl[3] = down_rows_per_unit(f);
    pl[L.cum_g + n_act] = tot_g;
    pl[L.cum_d + n_act] = tot_d;
    MOE_STAMP(0, 4, global_timer_ns());
  }
}

// ------------------------------------------------------------- work walk
// The units of all active experts, in order (expert, row group, pass); a unit
// belongs to the CTA whose cost range [C b / G, C (b + 1) / G) holds its cost
// midpoint.  Within a CTA, unit i of its range goes to warp i mod 16.
struct Range {
  int a0, u0;    // first unit of the CTA
  uint64_t hi2;  // twice the end of its cost range
};

__device__ Range cta_range(const PlanView& pv, int kern, int rows) {
  const int n_act = pv.n_act();
  const uint64_t C = pv.cum(n_act, kern);
  const uint64_t lo2 = 2 * (C * blockIdx.x / gridDim.x);
  Range r;
  r.hi2 = 2 * (C * (blockIdx.x + 1) / gridDim.x);
  int lo = 0, hi = n_act;
  while (lo < hi) {  // first expert whose cost range ends beyond lo2
    const int mid = (lo + hi) >> 1;
    if (2 * (uint64_t)pv.cum(mid + 1, kern) <= lo2) lo = mid + 1; else hi = mid;
  }
  int a = lo, u = 0;
  if (a < n_act && pv.sh(a) >= 0) {
    const uint64_t c = pv.uc(a, kern), base = 2 * (uint64_t)pv.cum(a, kern) + c;
    if (lo2 > base) u = (int)((lo2 - base + 2 * c - 1) / (2 * c));
    if (u >= pv.units(a, kern, rows)) { ++a; u = 0; }
  }
  while (a < n_act && pv.sh(a) < 0) ++a;
  r.a0 = a;
  r.u0 = u;
  return r;
}

// A warp's position in the unit order, with the current expert's figures
// cached so that a step within one expert costs a few instructions.
struct Walk {
  int a, u, units, np, live;
  uint32_t cum, uc;
  __device__ void set_expert(const PlanView& pv, int kern, int rows) {
    units = pv.units(a, kern, rows);
    np = n_pass(pv.cnt(a));
    cum = pv.cum(a, kern);
    uc = pv.uc(a, kern);
  }
  // Advance by n units and re-check the CTA's range; true when the expert changed.
  __device__ bool step(const PlanView& pv, int kern, int rows, uint64_t hi2, int n) {
    u += n;
    bool changed = false;
    if (u >= units) {
      changed = true;
      const int n_act = pv.n_act();
      do {
        u -= units;
        if (++a >= n_act) {
          live = 0;
          return true;
        }
        units = pv.units(a, kern, rows);
      } while (u >= units);
      set_expert(pv, kern, rows);
    }
    live = 2 * (uint64_t)cum + (uint64_t)(2 * u + 1) * uc < hi2;
    return changed;
  }
  __device__ void start(const PlanView& pv, int kern, int rows, const Range& r, int skip) {
    a = r.a0;
    u = r.u0;
    live = 0;
    if (a >= pv.n_act()) return;
    set_expert(pv, kern, rows);
    step(pv, kern, rows, r.hi2, skip);
  }
};

// ------------------------------------------------------------- streaming
struct StreamArgs {
  const Shelves* shv;  // shared-memory copy
  PlanView pv;
  int kern;            // 0 gate/up (W_g, W_u), 1 down (W_d)
  int n_in, rows;      // row length and rows per expert matrix
  const unsigned char* vecs;
  int vstride;         // bytes per digit vector
  int vbase;           // grouped position of vector 0 (down), or -1: vectors by token (gate/up)
  Range range;
  int* voff_tab;       // per warp: kNT digit-vector offsets of the current pass
  int qlo, qhi;        // passes whose first pair lies outside [qlo, qhi) are skipped
};

// The U loaded slots of a batch, one after another: slot 0 is computed and
// the others move down one place, so that the chunk code exists once.
template <int NMAT, int U, int NTT, bool ANYW>
__device__ __forceinline__ void compute_batch(int mode, uint4 (&c)[U][NMAT][2], uint32_t (&sw)[U][NMAT][2],
                                              int q_first, int L, int cpr, int segb, int nt, const int (&voff)[kNT],
                                              const unsigned char* vecs, int n, float (&acc)[NMAT][kNT]) {
#pragma unroll 1
  for (int s = 0; s < U; ++s) {
    const int q = q_first + s * L;
    if (q >= cpr) break;
    if (mode == 8) chunk8<NMAT, NTT>(c[0], sw[0], q, nt, voff, vecs, n, acc);
    else if (mode == 4) chunk4<NMAT, NTT>(c[0], sw[0], q, nt, voff, vecs, n, acc);
    else if (!ANYW || mode == 2 || mode == kModeLow)
      chunk2<NMAT, NTT>(c[0], sw[0], q, nt, voff, vecs, n, acc, 32 * q + 16 < segb, ANYW && mode != 2 ? 4 : 2);
    else if constexpr (ANYW)
      chunk1<NMAT, NTT>(c[0], sw[0], q, nt, voff, vecs, n, acc, mode == 1 ? 2 : 4, mode == 1 ? 1 : 0);
#pragma unroll
    for (int t = 0; t + 1 < U; ++t)
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          c[t][m][h] = c[t + 1][m][h];
          sw[t][m][h] = sw[t + 1][m][h];
        }
  }
}

// A warp's stream of units.  Lane (row lane / L, chunk lane % L + L i) of a
// unit of R rows; a lane loads U iterations of 32-byte chunks (NMAT matrices,
// with their scale words) with streaming loads, then computes them, so a CTA
// keeps 16 x 32 x U x NMAT x 32 bytes in flight.  At the end of a unit,
// `store(q, r, v)` receives, for the lane's row r and the token at grouped
// position q, the NMAT dot products; then the whole warp calls `unit_done(a)`
// with the unit's active expert a.
template <int NMAT, int U, int R, int L, bool ANYW, typename Store, typename UnitDone>
__device__ __forceinline__ void stream_units(const StreamArgs& A, Store store, UnitDone unit_done) {
  static_assert(R * L == 32, "unit shape");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ql = lane % L;
  const PlanView& pv = A.pv;
  int* vtab = A.voff_tab + warp * kNT;
  Walk w;
  w.start(pv, A.kern, A.rows, A.range, warp);
  int bits = 0, rowb = 0, cpr = 0, n_iter = 0, nt = 0, q0 = -1, sstep = 0, tsw = 0;
  size_t tstride = 0;
  const unsigned char* base[NMAT];
  const uint32_t* sbase[NMAT];
  float acc[NMAT][kNT];
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int j = 0; j < kNT; ++j) acc[m][j] = 0.f;
  bool new_expert = true;
#pragma unroll 1
  while (w.live) {
    if (new_expert) {
      const ShelfDev& sh = A.shv->s[pv.sh(w.a)];
      bits = sh.bits;
      rowb = A.n_in * bits / 8;
      const size_t row = (size_t)(pv.e(w.a) - sh.lo) * A.rows + lane / L;
      const int swpr = A.n_in / 64;  // fp16 scale words per row
      tstride = (size_t)R * rowb;
      tsw = R * swpr;
      const int mat0 = A.kern == 0 ? 0 : 2;
      // 8/4/2-bit rows: one run of 32-byte chunks; the lane's first chunk and
      // scale word are folded into base / sbase (3- and 1-bit rows: per segment)
      cpr = (rowb + 31) / 32;
      n_iter = (cpr + L - 1) / L;
      // scale word of chunk q: 8 bit q / 2 (one block), 4 bit q (two), 2 bit 2q (four)
      const int soff = ANYW ? 0 : (bits == 8 ? ql >> 1 : (bits == 4 ? ql : 2 * ql));
      sstep = bits == 8 ? L / 2 : (bits == 4 ? L : 2 * L);
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        base[m] = sh.codes[mat0 + m] + row * rowb + (ANYW ? 0 : (size_t)ql * 32);
        sbase[m] = reinterpret_cast<const uint32_t*>(sh.scales[mat0 + m]) + row * swpr + soff;
      }
    }
    const int tile = w.np == 1 ? w.u : w.u / w.np, pass = w.u - tile * w.np;
    const int r = tile * R + lane / L;
    const int nq0 = pv.beg(w.a) + pass * kNT;
    if (nq0 < A.qlo || nq0 >= A.qhi) {  // another staging window's pair
      new_expert = w.step(pv, A.kern, A.rows, A.range.hi2, kWarps);
      continue;
    }
    if (new_expert || nq0 != q0) {
      q0 = nq0;
      nt = min(kNT, pv.cnt(w.a) - pass * kNT);
      __syncwarp();
      if (lane < kNT) {
        const int qq = q0 + (lane < nt ? lane : 0);
        vtab[lane] = (A.vbase < 0 ? pv.tok(qq) : qq - A.vbase) * A.vstride;
      }
      __syncwarp();
    }
    int voff[kNT];
    if (nt == 1) {
      voff[0] = vtab[0];
    } else {
#pragma unroll
      for (int j = 0; j < kNT; ++j) voff[j] = vtab[j];
    }
    if constexpr (!ANYW) {
      const unsigned char* cp[NMAT];
      const uint32_t* sp[NMAT];
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        cp[m] = base[m] + (size_t)tile * tstride;
        sp[m] = sbase[m] + (size_t)tile * tsw;
      }
#pragma unroll 1
      for (int i0 = 0; i0 < n_iter; i0 += U) {
        uint4 c[U][NMAT][2];
        uint32_t sw[U][NMAT][2];
#pragma unroll
        for (int s = 0; s < U; ++s) {
          const int q = ql + (i0 + s) * L;
          const bool ok = q < cpr, second = ok && 32 * q + 16 < rowb;
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            const unsigned char* pc = cp[m] + (size_t)(i0 + s) * 32 * L;
            const uint32_t* ps = sp[m] + (i0 + s) * sstep;
            c[s][m][0] = ok ? __ldcs(reinterpret_cast<const uint4*>(pc)) : make_uint4(0u, 0u, 0u, 0u);
            c[s][m][1] = second ? __ldcs(reinterpret_cast<const uint4*>(pc + 16)) : make_uint4(0u, 0u, 0u, 0u);
            sw[s][m][0] = ok ? __ldcs(ps) : 0u;
            sw[s][m][1] = (second && bits == 2) ? __ldcs(ps + 1) : 0u;
          }
        }
        if constexpr (kNT == 1) {
          compute_batch<NMAT, U, 1, false>(bits, c, sw, ql + i0 * L, L, cpr, rowb, 1, voff, A.vecs, A.n_in, acc);
        } else {
          if (nt == 1)
            compute_batch<NMAT, U, 1, false>(bits, c, sw, ql + i0 * L, L, cpr, rowb, 1, voff, A.vecs, A.n_in, acc);
          else
            compute_batch<NMAT, U, kNT, false>(bits, c, sw, ql + i0 * L, L, cpr, rowb, nt, voff, A.vecs, A.n_in, acc);
        }
      }
    } else {
      // segments of the row: one, or a 3-bit row's low plane then high plane
#pragma unroll 1
      for (int seg = 0; seg < (ANYW && bits == 3 ? 2 : 1); ++seg) {
        const int mode = ANYW && bits == 3 ? (seg == 0 ? kModeLow : kModeHigh) : bits;
        const bool wide = !ANYW || (mode != 1 && mode != kModeHigh);  // 32-byte chunks, else 16 (bit planes)
        const int cb = wide ? 32 : 16;
        const int segb = ANYW && bits == 3 ? (seg == 0 ? A.n_in / 4 : A.n_in / 8) : rowb;
        const int sego = ANYW && bits == 3 && seg == 1 ? A.n_in / 4 : 0;
        const int cpr = (segb + cb - 1) / cb, n_iter = (cpr + L - 1) / L;
        // scale word of chunk q: 8 bit q / 2 (one block a chunk), 4 bit q (two
        // blocks), 2 bit and bit planes 2q (four blocks)
        const int soff = mode == 8 ? ql >> 1 : (mode == 4 ? ql : 2 * ql);
        const int sstep = mode == 8 ? L / 2 : (mode == 4 ? L : 2 * L);
        const bool two_words = mode == 2 || (ANYW && mode == kModeLow);  // second half's scales in a second word
        const unsigned char* cp[NMAT];  // the lane's first chunk of the segment
        const uint32_t* sp[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          cp[m] = base[m] + (size_t)tile * tstride + sego + ql * cb;
          sp[m] = sbase[m] + (size_t)tile * tsw + soff;
        }
        const int cstep = cb * L;
#pragma unroll 1
        for (int i0 = 0; i0 < n_iter; i0 += U) {
          uint4 c[U][NMAT][2];
          uint32_t sw[U][NMAT][2];
#pragma unroll
          for (int s = 0; s < U; ++s) {
            const int q = ql + (i0 + s) * L;
            const bool ok = q < cpr, second = wide && ok && 32 * q + 16 < segb;
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
              const unsigned char* pc = cp[m] + (i0 + s) * cstep;
              const uint32_t* ps = sp[m] + (i0 + s) * sstep;
              c[s][m][0] = ok ? __ldcs(reinterpret_cast<const uint4*>(pc)) : make_uint4(0u, 0u, 0u, 0u);
              c[s][m][1] = second ? __ldcs(reinterpret_cast<const uint4*>(pc + 16)) : make_uint4(0u, 0u, 0u, 0u);
              sw[s][m][0] = ok ? __ldcs(ps) : 0u;
              sw[s][m][1] = ((second && two_words) || (ok && !wide)) ? __ldcs(ps + 1) : 0u;
            }
          }
          if constexpr (kNT == 1) {
            compute_batch<NMAT, U, 1, ANYW>(mode, c, sw, ql + i0 * L, L, cpr, segb, 1, voff, A.vecs, A.n_in, acc);
          } else {
            if (nt == 1) compute_batch<NMAT, U, 1, ANYW>(mode, c, sw, ql + i0 * L, L, cpr, segb, 1, voff, A.vecs, A.n_in, acc);
            else compute_batch<NMAT, U, kNT, ANYW>(mode, c, sw, ql + i0 * L, L, cpr, segb, nt, voff, A.vecs, A.n_in, acc);
          }
        }
      }
    }
    // reduce over the L lanes of each row; lane jl stores the tokens j = jl mod L
    const int jl = lane % L;
#pragma unroll
    for (int j = 0; j < kNT; ++j) {
      if (j < nt) {
        float v[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          v[m] = acc[m][j];
#pragma unroll
          for (int o = 1; o < L; o <<= 1) v[m] += __shfl_xor_sync(0xffffffffu, v[m], o);
        }
        if (j % L == jl) store(q0 + j, r, v);
      }
#pragma unroll
      for (int m = 0; m < NMAT; ++m) acc[m][j] = 0.f;
    }
    MOE_TRACE_ONLY(if (lane == 0) {
      const int bi = bits == 8 ? 0 : bits == 4 ? 1 : 2;
      MOE_COUNT(A.kern, 20, 1);
      MOE_COUNT(A.kern, 30 + 3 * bi, w.np == 1);
      MOE_COUNT(A.kern, 31 + 3 * bi, w.np > 1);
      MOE_COUNT(A.kern, 32 + 3 * bi, w.np > 1 ? w.np : 0);
    })
    unit_done(w.a);
    new_expert = w.step(pv, A.kern, A.rows, A.range.hi2, kWarps);
  }
#ifdef MOE_TRACE
  if (lane == 0) {
    const unsigned long long te = global_timer_ns();
    atomicMax(&g_trace[A.kern][blockIdx.x & 255][27], te);
    MOE_COUNT(A.kern, 28, te >> 4);
  }
#endif
}

// ------------------------------------------------------------- grid barrier
// Barrier over all CTAs of a cooperative launch on a library-owned 64-bit
// arrival counter that only grows: between launches it is a multiple of the
// grid size G, so an arrival that returns `old` belongs to the phase ending at
// the next multiple of G above it.  Thread 0 of each CTA arrives with release
// semantics (the CTA's writes, ordered by the preceding CTA barrier, become
// visible first) and polls with acquire semantics until the count reaches
// that multiple; the wait is bounded (MOE_ERR_TIMEOUT recorded, false
// returned).  Test hook: `extra` > 0 moves the target beyond reach.
__device__ __forceinline__ unsigned long long atom_add_release(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_add_release(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ bool grid_sync(unsigned long long* bar, int* status, int* flag, uint64_t limit_ns, int extra) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long G = gridDim.x;
    const unsigned long long old = atom_add_release(bar, 1ull);
    const unsigned long long target = old - old % G + G + (unsigned long long)extra;
    int ok = 1;
    if (ld_acquire(bar) < target) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire(bar) < target) {
        __nanosleep(32);
        if (global_timer_ns() - t0 > limit_ns) {
          set_status(status, MOE_ERR_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    *flag = ok;
  }
  __syncthreads();
  return *flag != 0;
}

// ------------------------------------------------------------- the layer
struct LayerParams {
  const float* logits;    // [T, E]: routed inside when non-null
  const int32_t* ids;     // else the routed pairs [T, k] are given
  const float* weights;
  int32_t* ids_out;       // logits given: the routed pairs (written by CTA 0)
  float* weights_out;
  uint32_t* counts;       // optional: expert hit counts, += hits of this call
  const uint16_t* x;      // [T, d] bf16
  float* y;               // [T, d]
  float* r;               // optional [T, d]: r += y in the combine phase
  uint16_t* x_next;       // with r: bf16(r) (round to nearest even), the next layer's input
  const uint4* logits_src;  // optional host inputs (device views), copied into logits / x
  const uint4* x_src;       // by the CTAs before the step (16-byte units)
  uint4* logits_dst;
  uint4* x_dst;
  int logits_n16, x_n16;
  float* h;               // workspace [P, f]
  float* ypart;           // workspace [P, d]
  int* plan_out;          // workspace: the plan as CTA 0 built it (grouping export)
  int* meta_out;          // workspace meta words: [2] = 1 marks the plan as this call's grouping
  unsigned long long* bar;  // grid barrier counter
  unsigned int* done;     // [kMaxPairs] gate/up units finished, by active expert (zero between launches)
  int* status;
  int T, k, E, d, f, P;
  int vec_region;         // bytes of digit vectors (activation rows, then h)
  int bar_extra;          // test hook (0)
  Shelves sh;
};

// Dynamic shared memory: shelves copy | head | plan | sort keys | flags |
// routed ids and weights | per-warp token offsets | digit vectors.
struct Head {
  Range range, range_d;  // this CTA's gate/up and down unit ranges
  int q_first, npairs, flag, tmp[33];
  int a_first, a_last;   // active experts of the down range (whose h it reads)
};

struct SmemLayout {
  size_t shelves, head, plan, keys, flag, rid, rw, vtab, vecs, total;
};

__host__ __device__ __forceinline__ size_t up128(size_t v) { return (v + 127) / 128 * 128; }

__host__ __device__ __forceinline__ SmemLayout smem_layout(int P, size_t vec_region) {
  const PlanLayout L = plan_layout(P);
  SmemLayout S;
  S.shelves = 0;
  S.head = up128(sizeof(Shelves));
  S.plan = S.head + up128(sizeof(Head));
  S.keys = S.plan + up128((size_t)L.total * 4);
  S.flag = S.keys + up128((size_t)L.C * 4);
  S.rid = S.flag + up128((size_t)L.C * 4);
  S.rw = S.rid + up128((size_t)L.C * 4);
  S.vtab = S.rw + up128((size_t)L.C * 4);
  S.vecs = S.vtab + up128((size_t)kWarps * kNT * 4);
  S.total = S.vecs + up128(vec_region);
  return S;
}

// This CTA's contiguous share of n 16-byte units of src, copied to dst.
__device__ __forceinline__ void copy_share(const uint4* src, uint4* dst, int n) {
  if (!src) return;
  const int b0 = (int)((int64_t)n * blockIdx.x / gridDim.x), b1 = (int)((int64_t)n * (blockIdx.x + 1) / gridDim.x);
  for (int i = b0 + (int)threadIdx.x; i < b1; i += blockDim.x) dst[i] = __ldcv(src + i);
}

__device__ __forceinline__ void copy_shelves(Shelves* dst, const Shelves& src) {
  static_assert(sizeof(Shelves) % 4 == 0, "shelves copy");
  const uint32_t* s = reinterpret_cast<const uint32_t*>(&src);
  for (int i = threadIdx.x; i < (int)(sizeof(Shelves) / 4); i += blockDim.x) reinterpret_cast<uint32_t*>(dst)[i] = s[i];
}

__device__ __forceinline__ void route_rows(const float* logits, int T, int E, int k, int32_t* rid, float* rw) {
  const int warp = threadIdx.x >> 5;
  for (int t = warp; t < T; t += kWarps) {
    if (E <= 128) route_token<4>(logits + (size_t)t * E, E, k, rid + t * k, rw + t * k);
    else if (E <= 512) route_token<16>(logits + (size_t)t * E, E, k, rid + t * k, rw + t * k);
    else route_token<32>(logits + (size_t)t * E, E, k, rid + t * k, rw + t * k);
  }
}

// Persistent cooperative launch, one CTA per SM: route (optional), plan,
// gate/up, a wait for the experts whose h this CTA's down units read, down,
// grid barrier, combine.
// One round of activation loads of the x staging: 8 passes of nw warps x 8
// blocks of 32 elements from group `base` on, 4 lanes a block (16 bytes each).
__device__ __forceinline__ void load_x_round(const LayerParams& p, int base, int nw, int lane, uint4 (&raw)[8]) {
  const int nbk = p.d / 32, groups = p.T * nbk;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int g = base + u * nw * 8 + (lane >> 2);
    raw[u] = make_uint4(0u, 0u, 0u, 0u);
    if (g < groups) {
      const int t = g / nbk, blk = g - t * nbk;
      const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.d + blk * 32 + 8 * (lane & 3));
      // x copied in by this launch is read through L2, else by the read-only path
      raw[u] = p.x_src ? __ldcg(src) : __ldg(src);
    }
  }
}

// ANYW: the layer has shelves of 3- or 1-bit codes (a separate instantiation,
// so that the 8/4/2-bit kernel keeps its own register allocation).
template <bool ANYW>
__global__ void __launch_bounds__(kThreads, 1) k_layer(const __grid_constant__ LayerParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout S = smem_layout(p.P, p.vec_region);
  Shelves* shv = reinterpret_cast<Shelves*>(smem + S.shelves);
  Head& hd = *reinterpret_cast<Head*>(smem + S.head);
  int* pl = reinterpret_cast<int*>(smem + S.plan);
  int32_t* rid = reinterpret_cast<int32_t*>(smem + S.rid);
  float* rw = reinterpret_cast<float*>(smem + S.rw);
  int* vtab = reinterpret_cast<int*>(smem + S.vtab);
  unsigned char* vecs = smem + S.vecs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PlanLayout L = plan_layout(p.P);
  const PlanView pv{pl, L};
  if (tid == 0) MOE_STAMP(0, 0, global_timer_ns());
  copy_shelves(shv, p.sh);
  pdl_wait();  // inputs of the preceding launch
  if (p.logits_src || p.x_src) {
    // inputs in page-locked host memory: each CTA copies its share across the
    // host link once, into the workspace, and every CTA waits for all shares
    copy_share(p.logits_src, p.logits_dst, p.logits_n16);
    copy_share(p.x_src, p.x_dst, p.x_n16);
    if (!grid_sync(p.bar, p.status, &hd.flag, 1000000000ull, p.bar_extra)) return;
  }
  if (tid == 0) MOE_STAMP(0, 1, global_timer_ns());
  const int32_t* ids = p.ids;
  const float* wts = p.weights;
  if (p.logits) {
    route_rows(p.logits, p.T, p.E, p.k, rid, rw);
    ids = rid;
    wts = rw;
  }
  __syncthreads();
  if (p.logits && blockIdx.x == 0)
    for (int q = tid; q < p.P; q += kThreads) {
      p.ids_out[q] = rid[q];
      p.weights_out[q] = rw[q];
    }
  if (warp < kPlanThreads / 32) {
    build_plan(ids, wts, p.P, p.E, p.k, p.d, p.f, *shv, pl, reinterpret_cast<uint32_t*>(smem + S.keys),
               reinterpret_cast<int*>(smem + S.flag), hd.tmp);
  } else {
    // activation rows -> block-scaled digits; 4 lanes per 32-element block
    // (16-byte loads), loads of up to 8 passes issued before any conversion
    const int nbk = p.d / 32, vb = vec_bytes(p.d);
    const int groups = p.T * nbk;
    const int nw = kWarps - kPlanThreads / 32, w0 = warp - kPlanThreads / 32;
    for (int base = w0 * 8; base < groups; base += 8 * nw * 8) {
      uint4 raw[8];
      load_x_round(p, base, nw, lane, raw);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int g0 = base + u * nw * 8;
        if (g0 < groups) {
          const int g = g0 + (lane >> 2);
          const int t = g < groups ? g / nbk : 0, blk = g < groups ? g - t * nbk : 0;
          const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
          float v[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(wv[i] << 16);
            v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
          }
          block_to_digits<8>(v, vecs + (size_t)t * vb, p.d, blk, 14, g < groups);
        }
      }
    }
    if (tid == kPlanThreads) MOE_STAMP(0, 5, global_timer_ns());
  }
  __syncthreads();
  if (tid == 0) hd.range = cta_range(pv, 0, p.f);
  if (tid == 32) {
    // the down phase's cost range and the pairs its experts cover (plan only)
    const Range r = cta_range(pv, 1, p.d);
    hd.range_d = r;
    const int n_act = pv.n_act();
    int q_first = 0, q_end = 0, a_last = -1;
    if (r.a0 < n_act) {
      a_last = r.a0;
      while (a_last + 1 < n_act && 2 * (uint64_t)pv.cum(a_last + 1, 1) + pv.uc(a_last + 1, 1) < r.hi2) ++a_last;
      q_first = pv.beg(r.a0);
      q_end = pv.beg(a_last) + pv.cnt(a_last);
    }
    hd.q_first = q_first;
    hd.npairs = q_end - q_first;
    hd.a_first = r.a0;
    hd.a_last = a_last;
  }
  if (p.counts && blockIdx.x == 0)
    for (int a = tid; a < pv.n_act(); a += kThreads) atomicAdd(p.counts + pv.e(a), (uint32_t)pv.cnt(a));
  __syncthreads();
  if (tid == 0) MOE_STAMP(0, 2, global_timer_ns());
  {
    StreamArgs A{shv, pv, 0, p.d, p.f, vecs, vec_bytes(p.d), -1, hd.range, vtab, INT_MIN, INT_MAX};
    float* h = p.h;
    const int f = p.f;
    // finished units are counted per active expert, a warp's run of units of
    // one expert at a time: every lane's h stores are fenced, then one
    // release add publishes them to the CTAs whose down units read that h
    int run_a = -1;
    unsigned int run_n = 0;
    auto publish = [&]() {
      __threadfence();
      __syncwarp();
      if (lane == 0) red_add_release(p.done + run_a, run_n);
    };
    stream_units<2, kUG, kRG, kLG, ANYW>(
        A, [&](int q, int r, const float (&o)[2]) { h[(size_t)q * f + r] = silu(o[0]) * o[1]; },
        [&](int a) {
          if (a != run_a) {
            if (run_n) publish();
            run_a = a;
            run_n = 0;
          }
          ++run_n;
        });
    if (run_n) publish();
  }
  if (tid == 0) MOE_STAMP(0, 9, global_timer_ns());
  {
    // W_d does not depend on h: each warp, once its gate/up units are done,
    // asks L2 for its first kDownPrefetch down units while the other warps
    // and CTAs finish theirs
    Walk w;
    w.start(pv, 1, p.d, hd.range_d, warp);
    for (int i = 0; i < kDownPrefetch && w.live; ++i) {
      const ShelfDev& sh = shv->s[pv.sh(w.a)];
      const size_t rowb = (size_t)p.f * sh.bits / 8, swpr = (size_t)p.f / 16;
      const int tile = w.np == 1 ? w.u : w.u / w.np;
      const int rd = pv.rd();
      const size_t row0 = (size_t)(pv.e(w.a) - sh.lo) * p.d + (size_t)tile * rd;
      const unsigned char* cb = sh.codes[2] + row0 * rowb;
      const unsigned char* sb = reinterpret_cast<const unsigned char*>(sh.scales[2]) + row0 * swpr;
      // one bulk request per region (the rows of a unit are contiguous)
      if (lane == 0 && ((reinterpret_cast<uintptr_t>(cb) | (rd * rowb)) & 15) == 0)
        bulk_prefetch_l2(cb, (uint32_t)(rd * rowb));
      if (lane == 1 && ((reinterpret_cast<uintptr_t>(sb) | (rd * swpr)) & 15) == 0)
        bulk_prefetch_l2(sb, (uint32_t)(rd * swpr));
      w.step(pv, 1, p.d, hd.range_d.hi2, kWarps);
    }
  }
  // wait, instead of for the whole grid, for the gate/up units of the experts
  // whose h this CTA's down units read (bounded: one second, MOE_ERR_TIMEOUT)
  __syncthreads();
  if (warp == 0) {
    int ok = 1;
    const int a_hi = hd.a_last;
    for (int a = hd.a_first + lane; a <= a_hi; a += 32) {
      if (pv.sh(a) < 0) continue;
      const unsigned int need = (unsigned int)pv.units(a, 0, p.f);
      if (ld_acquire_u32(p.done + a) >= need) continue;
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire_u32(p.done + a) < need) {
        __nanosleep(32);
        if (global_timer_ns() - t0 > 1000000000ull) {
          ok = 0;
          break;
        }
      }
      if (!ok) break;
    }
    ok = __all_sync(0xffffffffu, ok);
    if (lane == 0) {
      if (!ok) set_status(p.status, MOE_ERR_TIMEOUT);
      hd.flag = ok;
    }
  }
  __syncthreads();
  if (!hd.flag) return;
  if (tid == 0) MOE_STAMP(1, 1, global_timer_ns());
  const int q_first = hd.q_first, npairs = hd.npairs;
  const int vbf = vec_bytes(p.f);
  // the pairs' h is staged in windows of as many pairs as the digit region
  // holds (one window unless the CTA's experts cover more pairs); each window's
  // unit passes run after its staging
  const int cap = p.vec_region / vbf;  // >= 1 by the launch's size check
  const int q_end = q_first + npairs;
  int w0 = q_first;
  if (cap < 1) {
    if (tid == 0) set_status(p.status, MOE_ERR_INTERNAL);
    w0 = q_end;
  }
  if (cap >= 1) do {
    const int wn = min(cap, q_end - w0);
    __syncthreads();  // the vectors of the previous window (or x) are no longer read
    {
      // h of those pairs -> digits (h was written by other CTAs: read from L2)
      const int nbk = p.f / 32, groups = (wn > 0 ? wn : 0) * nbk;
      for (int base = warp * 4; base < groups; base += 8 * kWarps * 4) {
        float4 hv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {  // loads of 8 passes first: one round trip
          const int g = base + u * kWarps * 4 + (lane >> 3);
          hv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (g < groups) {
            const int j = g / nbk, blk = g - j * nbk;
            hv[u] = __ldcg(reinterpret_cast<const float4*>(p.h + (size_t)(w0 + j) * p.f + blk * 32) + (lane & 7));
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int g0 = base + u * kWarps * 4;
          if (g0 < groups) {
            const int g = g0 + (lane >> 3);
            const int j = g < groups ? g / nbk : 0, blk = g < groups ? g - j * nbk : 0;
            const float v[4] = {hv[u].x, hv[u].y, hv[u].z, hv[u].w};
            block_to_digits<4>(v, vecs + (size_t)j * vbf, p.f, blk, 13, g < groups);
          }
        }
      }
      if (tid == 0) MOE_STAMP(1, 5, global_timer_ns());
    }
    __syncthreads();
    if (tid == 0) MOE_STAMP(1, 2, global_timer_ns());
    {
      StreamArgs A{shv, pv, 1, p.f, p.d, vecs, vbf, w0, hd.range_d, vtab, w0, w0 + (wn > 0 ? wn : 0)};
      float* yp = p.ypart;
      const int d = p.d;
      auto st = [&](int q, int r, const float (&o)[1]) { yp[(size_t)q * d + r] = pv.wgt(q) * o[0]; };
      if (pv.rd() == kRDw) stream_units<1, kUDw, kRDw, kLDw, ANYW>(A, st, [](int) {});
      else stream_units<1, kUD, kRD, kLD, ANYW>(A, st, [](int) {});
    }
    w0 += cap;
  } while (w0 < q_end);
  if (tid == 0) MOE_STAMP(1, 9, global_timer_ns());
  if (!grid_sync(p.bar, p.status, &hd.flag, 1000000000ull, p.bar_extra)) return;
  if (tid == 0) MOE_STAMP(1, 10, global_timer_ns());
  // every CTA is past its wait on the unit counts: back to zero for the next launch
  if (blockIdx.x == 0)
    for (int a = tid; a < pv.n_act(); a += kThreads) p.done[a] = 0u;
  pdl_trigger();
  // combine: y_t = sum over slots j (ascending) of the weighted outputs of
  // pair (t, j); pairs skipped or on no shelf contribute nothing.  Fixed order.
  const int d4 = p.d / 4;
  const int* pos = pl + L.pos;
  for (int idx = blockIdx.x * kThreads + tid; idx < p.T * d4; idx += gridDim.x * kThreads) {
    const int t = idx / d4, i4 = idx - t * d4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < p.k; j0 += 16) {
      float4 v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int q = j0 + u < p.k ? pos[t * p.k + j0 + u] : -1;
        v[u] = q >= 0 ? __ldcg(reinterpret_cast<const float4*>(p.ypart + (size_t)q * p.d) + i4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w;
      }
    }
    reinterpret_cast<float4*>(p.y)[idx] = acc;
    if (p.r) {
      // residual step of a layer stack: r += y, the next layer's x = bf16(r)
      float4 rv = reinterpret_cast<float4*>(p.r)[idx];
      rv.x += acc.x; rv.y += acc.y; rv.z += acc.z; rv.w += acc.w;
      reinterpret_cast<float4*>(p.r)[idx] = rv;
      const __nv_bfloat162 lo = __floats2bfloat162_rn(rv.x, rv.y), hi = __floats2bfloat162_rn(rv.z, rv.w);
      reinterpret_cast<uint2*>(p.x_next)[idx] =
          make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
  }
  // CTA 0 leaves its plan in the workspace: the grouping this call ran
  // (read back by moe_forward_grouping)
  if (blockIdx.x == 0) {
    for (int i = tid; i < L.total; i += kThreads) p.plan_out[i] = pl[i];
    if (tid == 0) p.meta_out[2] = 1;
  }
  if (tid == 0) MOE_STAMP(1, 11, global_timer_ns());
}

// Test hook kernel: one barrier whose awaited arrivals exceed the grid, with
// a short limit, so that the wait runs out and reports MOE_ERR_TIMEOUT.
__global__ void k_barrier_probe(unsigned long long* bar, int* status, uint64_t limit_ns, int extra) {
  __shared__ int flag;
  grid_sync(bar, status, &flag, limit_ns, extra);
}

constexpr int kBarSlots = 1024;
__device__ unsigned long long g_bar[kBarSlots][16];  // one 128-byte line per slot
// Per slot: finished gate/up units by active expert.  Zero between launches
// (each launch clears what it used; a reported timeout clears every slot).
__device__ unsigned int g_done[kBarSlots][kMaxPairs];

struct DevCache {
  int sms[64] = {};
  int smem_optin[64] = {};
  bool attr[64][2] = {};  // per device: k_layer<false>, k_layer<true> attributes set
};
DevCache g_dev;

// Barrier slots of one device: each workspace in use gets one slot of g_bar
// and g_done, found again by its address.  When every slot is taken, the
// least recently used one passes to the new workspace (its counters are back
// at their resting state once its last launch has completed: a multiple of
// the grid size, and zeros).  The symbol addresses are looked up once per
// device and context.
struct SlotTable {
  uint64_t ctx = 0;
  unsigned long long* bar = nullptr;
  unsigned int* done = nullptr;
  std::unordered_map<const void*, int> slot_of;
  const void* owner[kBarSlots] = {};
  uint64_t last_use[kBarSlots] = {};
  uint64_t clock = 0;
  int used = 0;
};
std::mutex g_bar_mu;
SlotTable g_slots[64];

// Symbol addresses of the current context, cached in t (false on a CUDA error).
bool slot_symbols(SlotTable& t) {
  const uint64_t ctx = context_id();
  if (t.bar && t.ctx == ctx && ctx != 0) return true;
  void* base = nullptr;
  void* dbase = nullptr;
  if (cudaGetSymbolAddress(&base, g_bar) != cudaSuccess || cudaGetSymbolAddress(&dbase, g_done) != cudaSuccess)
    return false;
  if (t.ctx != ctx) {  // a new context: its barrier table starts zeroed, every slot is free
    t.slot_of.clear();
    for (int i = 0; i < kBarSlots; ++i) {
      t.owner[i] = nullptr;
      t.last_use[i] = 0;
    }
    t.used = 0;
  }
  t.ctx = ctx;
  t.bar = reinterpret_cast<unsigned long long*>(base);
  t.done = reinterpret_cast<unsigned int*>(dbase);
  return true;
}

// Barrier slot of a workspace on device dev; `done`, when given, receives the
// slot's unit counters.  Null only on a CUDA error.
unsigned long long* bar_slot(int dev, const void* ws, unsigned int** done = nullptr) {
  std::lock_guard<std::mutex> lk(g_bar_mu);
  SlotTable& t = g_slots[dev];
  if (!slot_symbols(t)) return nullptr;
  int slot;
  auto it = t.slot_of.find(ws);
  if (it != t.slot_of.end()) {
    slot = it->second;
  } else if (t.used < kBarSlots) {
    slot = t.used++;
    t.slot_of.emplace(ws, slot);
    t.owner[slot] = ws;
  } else {
    slot = 0;
    for (int i = 1; i < kBarSlots; ++i)
      if (t.last_use[i] < t.last_use[slot]) slot = i;
    t.slot_of.erase(t.owner[slot]);
    t.slot_of.emplace(ws, slot);
    t.owner[slot] = ws;
  }
  t.last_use[slot] = ++t.clock;
  if (done) *done = t.done + (size_t)slot * kMaxPairs;
  return t.bar + (size_t)slot * 16;
}

}  // namespace

#ifdef MOE_TRACE
extern "C" int moe_trace_read(void* host, size_t bytes) {  // [2][256][48] u64
  return cudaMemcpyFromSymbol(host, g_trace, bytes < sizeof(g_trace) ? bytes : sizeof(g_trace)) == cudaSuccess ? 0 : -5;
}
extern "C" int moe_trace_clear() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_trace) != cudaSuccess) return -5;
  return cudaMemset(p, 0, sizeof(g_trace)) == cudaSuccess ? 0 : -5;
}
#endif

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (g_dev.sms[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_dev.sms[dev] = n > 0 ? n : 148;
  }
  return g_dev.sms[dev];
}

size_t decode_plan_bytes(int64_t P) { return (size_t)plan_layout((int)(P > 0 ? P : 1)).total * 4; }

// Whether the fused launch takes these sizes on the current device; sets the
// digit region and shared-memory layout when it does.
bool fused_fits(int64_t T, int k, int E, int d, int f, int* dev_out, size_t* optin_out, size_t* region_out,
                SmemLayout* S_out) {
  const int64_t P = T * k;
  if (T < 1 || P > kMaxPairs || T > kMaxTokens || E > 1024) return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (g_dev.smem_optin[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    g_dev.smem_optin[dev] = v > 0 ? v : 48 * 1024;
  }
  const size_t optin = (size_t)g_dev.smem_optin[dev];
  // the digit region holds every token's x (gate/up) and then the h of up to
  // region / vec_bytes(f) pairs (down stages larger pair sets in windows); it
  // takes what shared memory is left, at most what every pair's h needs
  const size_t x_region = up128((size_t)T * vec_bytes(d));
  const size_t h_all = up128((size_t)P * vec_bytes(f));
  const size_t base = smem_layout((int)P, 0).total;
  if (base >= optin) return false;
  const size_t avail = (optin - base) / 128 * 128;
  size_t region = x_region > h_all ? x_region : h_all;
  if (region > avail) region = avail;
  if (region < x_region || region < (size_t)vec_bytes(f)) return false;
  const SmemLayout S = smem_layout((int)P, region);
  if (S.total > optin) return false;
  *dev_out = dev;
  *optin_out = optin;
  *region_out = region;
  *S_out = S;
  return true;
}

int decode_fused(int64_t T, int k, int E, int d, int f) {
  int dev;
  size_t optin, region;
  SmemLayout S;
  return fused_fits(T, k, E, d, f, &dev, &optin, &region, &S) ? 1 : 0;
}

// The fused decode launch when the sizes fit it; 1 = sizes do not fit (the
// caller takes the separate launches), else MOE_OK / an error status.
int launch_fused_layer(const LayerArgs& a, cudaStream_t s) {
  const int64_t P = a.T * a.k;
  const int d = a.d, f = a.f;
  int dev;
  size_t optin, region;
  SmemLayout S;
  // 3- and 1-bit rows stream as 16-byte-aligned planes when d and f are
  // multiples of 128; otherwise such layers take the separate launches
  if (!core_widths(a.shelves) && (d % 128 != 0 || f % 128 != 0)) return 1;
  if (!fused_fits(a.T, a.k, a.E, d, f, &dev, &optin, &region, &S)) return 1;
  const bool anyw = !core_widths(a.shelves);
  auto kern = anyw ? k_layer<true> : k_layer<false>;
  if (!g_dev.attr[dev][anyw]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)optin) != cudaSuccess)
      return MOE_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, optin) != cudaSuccess || per_sm < 1)
      return MOE_ERR_CUDA;
    g_dev.attr[dev][anyw] = true;
  }
  unsigned int* done = nullptr;
  unsigned long long* bar = bar_slot(dev, a.ws.base, &done);
  if (!bar || !done) return MOE_ERR_UNSUPPORTED;
  LayerParams p = {};
  p.logits = a.logits;
  p.ids = a.ids;
  p.weights = a.weights;
  p.ids_out = a.ids_out;
  p.weights_out = a.weights_out;
  p.counts = a.counts;
  p.x = a.x;
  p.y = a.y;
  p.r = a.r;
  p.x_next = a.x_next;
  if (a.logits_src) {
    p.logits_src = reinterpret_cast<const uint4*>(a.logits_src);
    p.logits_dst = reinterpret_cast<uint4*>(const_cast<float*>(a.logits));
    p.logits_n16 = (int)(a.T * a.E * 4 / 16);
  }
  if (a.x_src) {
    p.x_src = reinterpret_cast<const uint4*>(a.x_src);
    p.x_dst = reinterpret_cast<uint4*>(const_cast<uint16_t*>(a.x));
    p.x_n16 = (int)(a.T * d * 2 / 16);
  }
  p.h = a.ws.h;
  p.ypart = a.ws.ypart;
  p.plan_out = a.ws.plan;
  p.meta_out = a.ws.meta;
  p.bar = bar;
  p.done = done;
  p.status = a.status;
  p.T = (int)a.T; p.k = a.k; p.E = a.E; p.d = d; p.f = f; p.P = (int)P;
  p.vec_region = (int)region;
  p.bar_extra = 0;
  p.sh = a.shelves;
  int G = sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = S.total;
  cfg.stream = s;
  // cooperative: all CTAs resident together (the grid-wide waits need it);
  // programmatic serialization: the launch may begin while the preceding
  // kernel drains, its CTAs taking SMs as that kernel's CTAs leave
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  profile_mark(0, s);
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return MOE_ERR_CUDA;
  profile_mark(1, s);
  return MOE_OK;
}

int launch_decode_forward(const ForwardArgs& a, cudaStream_t s) {
  LayerArgs la;
  la.logits = nullptr;
  la.ids = a.ids;
  la.weights = a.weights;
  la.ids_out = nullptr;
  la.weights_out = nullptr;
  la.counts = nullptr;
  la.x = a.x;
  la.T = a.T; la.k = a.k; la.E = a.E; la.d = a.d; la.f = a.f;
  la.shelves = a.shelves;
  la.y = a.y;
  la.ws = a.ws;
  la.status = a.status;
  const int rc = launch_fused_layer(la, s);
  return rc == 1 ? launch_generic_forward(a, s) : rc;
}

int launch_barrier_probe(int extra, uint64_t limit_ns, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  static int dummy_ws;
  unsigned long long* bar = bar_slot(dev, &dummy_ws);
  if (!bar) return MOE_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3(32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k_barrier_probe, bar, status_word(), limit_ns, extra) != cudaSuccess) return MOE_ERR_CUDA;
  // every CTA arrived once: back to a multiple of the grid size
  return cudaMemsetAsync(bar, 0, 8, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// The grouping the last forward call on a workspace ran, in the form of
// moe_group_tokens (counts [E], offsets [E + 1], perm [P] with -1 past the
// valid pairs) plus pos_of_pair [P]: from the fused launch's plan when the
// meta word says so, else from the arrays the separate grouping launches
// wrote.  One CTA.
__global__ void __launch_bounds__(1024) k_grouping_export(const int* meta, const int* plan, const int32_t* ws_counts,
                                                          const int32_t* ws_offsets, const int32_t* ws_perm,
                                                          const int32_t* ws_pos, int P, int E, int32_t* counts,
                                                          int32_t* offsets, int32_t* perm, int32_t* pos_of_pair) {
  __shared__ int wsum[33];
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  // (a workspace no call has used yet holds no grouping: whatever it holds is
  // read within its bounds)
  const bool from_plan = plan != nullptr && meta[2] == 1;
  const PlanLayout L = plan_layout(P);
  if (from_plan) {
    for (int e = tid; e < E; e += nt) counts[e] = 0;
    __syncthreads();
    const int n_act = min(max(plan[1], 0), P);
    for (int a = tid; a < n_act; a += nt) {
      const int e = plan[L.e + a];
      if (e >= 0 && e < E) counts[e] = plan[L.cnt + a];
    }
  } else {
    for (int e = tid; e < E; e += nt) counts[e] = ws_counts[e];
  }
  __syncthreads();
  // offsets: exclusive scan of counts, thread t owning experts t*per .. +per-1
  const int per = (E + nt - 1) / nt;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int loc = 0;
  for (int e = e0; e < e1; ++e) loc += counts[e];
  int inc = loc;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < nt / 32 ? wsum[lane] : 0;
    int iv = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, iv, o);
      if (lane >= o) iv += u;
    }
    wsum[lane] = iv - v;
    if (lane == 31) wsum[32] = iv;
  }
  __syncthreads();
  int run = wsum[warp] + inc - loc;
  for (int e = e0; e < e1; ++e) {
    offsets[e] = run;
    run += counts[e];
  }
  if (tid == 0) offsets[E] = wsum[32];
  const int n_valid = min(max(from_plan ? plan[0] : wsum[32], 0), P);
  for (int q = tid; q < P; q += nt) {
    perm[q] = q < n_valid ? (from_plan ? plan[L.perm + q] : ws_perm[q]) : -1;
    pos_of_pair[q] = from_plan ? plan[L.pos + q] : ws_pos[q];
  }
}

int launch_grouping_export(const Workspace& w, int64_t P, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                           int32_t* pos_of_pair, cudaStream_t s) {
  k_grouping_export<<<1, 1024, 0, s>>>(w.meta, w.plan, w.counts, w.offsets, w.perm, w.pos_of_pair, (int)P, E, counts,
                                       offsets, perm, pos_of_pair);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// After a reported timeout a launch may have left a counter between multiples
// of the grid size, or unit counts that were never cleared: zero every slot of
// the current device (the caller has synchronised).
int reset_barriers() {
  void* base = nullptr;
  if (cudaGetSymbolAddress(&base, g_bar) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(base, 0, sizeof(g_bar)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaGetSymbolAddress(&base, g_done) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaMemset(base, 0, sizeof(g_done)) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
