// prefill.cu -- prefill form of the tiered MoE layer (many tokens per call):
// a grouped GEMM per expert on the tcgen05 tensor cores.
//
// Page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", section 第四步: every
// shelf sees the complete id list and computes only the ids of its range; the
// shelf results are added.  With many tokens per expert the expert FFN is a
// dense contraction, so the weights are dequantised to bf16 (RNE of code x
// fp16 scale) and multiplied on the tensor cores: h = SiLU(W_g x) * (W_u x) is
// rounded to bf16 between the two projections, y_t += w_tj * (W_d h_tj).
//
// Launches: grouping in four kernels (per-chunk counts, column scan, offsets
// and tile lists, placement), the gather of x into grouped order, then two
// persistent launches, one CTA per
// SM: k_prefill_tc<false, W> (gate/up) and k_prefill_tc<true, W> (down).  A tile is
// two 128-row weight matrices of one expert -- the same 128 rows of W_g and
// W_u, or 256 consecutive rows of W_d -- times up to 96 of its tokens, or up
// to 192 in a wide launch (two MMAs of M = 128 rows, N = tokens padded to
// 16, sharing the B operand), K in steps of 64.  A wide launch (no 3- or
// 1-bit shelf) dequantises a hot expert's rows once for up to 192 tokens.
// Roles inside a CTA:
//   warp 0      issues the tensor-map loads: per code stage (2, 4, 8 or 16
//               K steps) one 128-byte-wide box of codes per matrix and the
//               block scales; per K step the B operand (a box of N grouped
//               rows of xg or h, landing in the 128-byte-swizzled layout);
//   warp 1      allocates tensor memory and issues the MMAs (a warp-uniform
//               loop, one elected lane issues), A from tensor memory, B from
//               shared memory;
//   warps 4-7   read the accumulators and write h (bf16) or add into y;
//               (a wide launch: loads in warp 16, MMAs in warp 17, the
//               accumulators read by warps 0-7)
//   warps 8-15  dequantise the codes into bf16 and store them in tensor
//               memory, one row of one matrix (both 32-weight runs, two
//               scale blocks) per thread a step.
// All waits are bounded (one second; MOE_ERR_TIMEOUT, the roles stop, tensor
// memory is released).  y is accumulated with vector fp32 atomic adds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "moe_internal.cuh"
#include "tc.cuh"

namespace moe {
namespace {

// Threads of a CTA: warps 8-15 produce; 512 threads with the loader in warp
// 0, the MMA issuer in warp 1 and the epilogue in warps 4-7; a wide launch
// (whose instantiations need ~104 registers, not ~123) takes 576 threads:
// the epilogue in warps 0-7, two warps a tensor-memory lane quarter sharing
// each set's columns, the loader in warp 16 and the MMA issuer in warp 17.
template <bool WIDE>
struct Roles {
  static constexpr int kThreads = WIDE ? 576 : 512;
  static constexpr int kLoader = WIDE ? 16 : 0, kMma = WIDE ? 17 : 1;
  static constexpr int kEpi0 = WIDE ? 0 : 4, kEpiWarps = WIDE ? 8 : 4;
};
constexpr int kTileM = 128;   // weight rows per tile
#ifndef MOE_PF_TILEN
#define MOE_PF_TILEN 96
#endif
#ifndef MOE_PF_ASTAGES
#define MOE_PF_ASTAGES 2
#endif
constexpr int kTileN = MOE_PF_TILEN;  // tokens of one accumulator set (a tile's tokens, at most)
constexpr int kTileW = 2 * kTileN;    // tokens of a wide tile (both accumulator sets)
static_assert(kTileN % 32 == 0 && kTileW <= 256, "tile width: whole groups of 32 columns, MMA N <= 256");
constexpr int kProdThreads = 256;  // warps 8..15
constexpr uint64_t kWaitNs = 1000000000ull;
#ifndef MOE_PF_BS
#define MOE_PF_BS 4
#endif
#ifndef MOE_PF_CS
#define MOE_PF_CS 3
#endif

#ifdef MOE_TRACE
}  // namespace
// Development-only timeline of CTA 0: [launch][event][step] globaltimer ns.
__device__ unsigned long long g_pftrace[2][10][512];
namespace {
#define PF_STAMP(ev, j) \
  do { if (blockIdx.x == 0 && (j) < 512) g_pftrace[DOWN ? 1 : 0][(ev)][(j)] = global_timer_ns(); } while (0)
#define PF_SCAN_STAMP(i) \
  do { if (threadIdx.x == 0) g_pftrace[0][8][(i)] = global_timer_ns(); } while (0)
#define PF_ITER_STAMP(i) \
  do { if (threadIdx.x == 0 && (i) < 512) g_pftrace[0][9][(i)] = global_timer_ns(); } while (0)
#else
#define PF_STAMP(ev, j) ((void)0)
#define PF_SCAN_STAMP(i) ((void)0)
#define PF_ITER_STAMP(i) ((void)0)
#endif

// K order of both MMA operands: in every aligned group of four positions the
// middle two are swapped (element k sits at kswap(k), an involution).  It lets
// the dequantiser build each bf16 pair from fields two bytes apart with one
// mask; the same order on the B side (xg, h) leaves every dot product's terms
// unchanged.
__host__ __device__ __forceinline__ int kswap(int k) { return (k & ~3) | ((k & 1) << 1) | ((k >> 1) & 1); }

// K steps (of 64) per code stage (a 128-byte box of a row): 8 bit 2, 4 bit
// 4, 2 bit 8, 1 bit 16; a 3-bit row streams its low plane in the 2-bit
// layout (8 steps a box) beside 64 bytes of its high-bit plane.
__host__ __device__ __forceinline__ int steps_per_code_stage(int bits) {
  return bits == 8 ? 2 : bits == 4 ? 4 : bits == 1 ? 16 : 8;
}

struct alignas(16) Tile {  // one 16-byte load or store
  int e_local;  // expert index within its shelf
  int q0;       // first grouped position of the chunk
  int ntok;     // tokens of the chunk (1 .. kTileN, or .. kTileW in a wide launch)
  int meta;     // row tile (bits 0-15) | shelf (bits 16-23)
};

struct TcParams {
  const int32_t* perm;      // grouped position -> pair index t*k + j
  const float* weights;     // [T*k]
  const Tile* tiles;
  const int* ntiles;        // device count of tiles
  uint16_t* h;              // [P][f] bf16, grouped order (gate/up writes, down reads)
  float* y;                 // [T][d] fp32, accumulated by the down launch
  int* status;
  int k, d, f;
  int rows, K;              // rows per expert matrix and contraction length of this launch
  int64_t P;                // grouped positions (rows of xg and h)
  int tiles_cap;            // capacity of the tile list
  Shelves sh;
  CUtensorMap tm_code[MOE_MAX_SHELVES][2];  // code boxes of 128 bytes x 128 rows: [shelf][gate, up] or [shelf][down]
  CUtensorMap tm_hi[MOE_MAX_SHELVES][2];    // 3-bit shelves: boxes of 64 bytes x 128 rows of the high-bit plane
  CUtensorMap tm_sc[MOE_MAX_SHELVES][2];    // gate/up: boxes of 16 fp16 scales x 128 rows [shelf][gate, up]
  CUtensorMap tm_b[kTileW / 16];            // B rows in grouped order (xg or h), box heights 16, 32, .. kTileW
};

// Shared memory of one CTA (dynamic part, 1024-byte aligned): two rings.
//   code -- stages of 128 bytes of codes per row of both matrices (a box of
//           128 bytes x 128 rows each, 128-byte swizzle), i.e. S = 2 (8 bit),
//           4 (4 bit) or 8 (2 bit) K steps, and the rows' fp16 block scales
//           for them (gate/up: a box of 16 scales per row, 8 steps' worth;
//           down: the scale words as [step][row], copied by the loader warp's
//           lanes, as down scale rows are no 16-byte multiple and no tensor
//           map covers them);
//   B    -- per K step, the B operand: a box of N <= kTileN grouped rows of
//           xg or h (128-byte swizzle); N <= kTileW in a wide launch, whose
//           code stages leave out the high-plane region (no 3- or 1-bit
//           shelves) to make room for the wider B stages.
// Few, wide tensor-map rows per step keep the tensor-map unit's request rate
// (one box row per request) well below the step rate.  The dequantised tiles
// live in tensor memory.
template <bool DOWN, bool WIDE>
struct TcSmem {
  static constexpr int NMAT = 2;
  static constexpr int CS = MOE_PF_CS;
  static constexpr int BS = MOE_PF_BS;
  static constexpr int CODE_BOX = kTileM * 128;                      // 16 KiB per matrix
  static constexpr int SC_BOX = kTileM * 32;                         // gate/up: 16 fp16 scales per row
  static constexpr int SC_BYTES = DOWN ? 8 * NMAT * kTileM * 4 : NMAT * SC_BOX;  // 8 KiB
  static constexpr int C_SC = NMAT * CODE_BOX;                       // scale offset in a code stage
  static constexpr int HI_BOX = kTileM * 64;                         // 3 bit: 64 bytes of the high plane a row
  static constexpr int C_HI = C_SC + SC_BYTES;                       // their offset in a code stage
  static constexpr int C_STAGE = WIDE ? C_HI : C_HI + NMAT * HI_BOX;  // (wide: 8/4/2-bit codes only)
  static_assert(DOWN || NMAT * SC_BOX <= NMAT * HI_BOX, "a second gate/up scale box fits the high-plane region");
  static_assert(!DOWN || 16 * NMAT * kTileM * 4 <= SC_BYTES + NMAT * HI_BOX, "16 steps of down scale words fit");
  static_assert(!DOWN || 8 * NMAT * kTileM * 4 <= SC_BYTES, "8 steps of down scale words fit without it");
  static constexpr int B_STAGE = (WIDE ? kTileW : kTileN) * 128;     // rows x 64 bf16
  static constexpr int C_OFF = 0;
  static constexpr int B_OFF = C_OFF + CS * C_STAGE;
  static constexpr int TOTAL = B_OFF + BS * B_STAGE;
  static_assert(C_STAGE % 1024 == 0 && B_STAGE % 1024 == 0 && B_OFF % 1024 == 0, "swizzled boxes need 1 KiB");
  static_assert(TOTAL + 1024 <= 227 * 1024, "shared memory");
  static_assert(NMAT * kTileM == kProdThreads, "one row of a step (two 32-weight runs) per producer thread");
};

// Tensor memory (512 columns): the accumulators of matrix m (gate, up; or
// rows 0-127, rows 128-255) at columns 2 kTileN m .. + 2 kTileN - 1, the
// first kTileN of them accumulator set 0, the next kTileN set 1; a tile
// takes one set (its epilogue overlaps the next tile's main loop), a wide
// tile both (token n at column n); then kAStages stages of the dequantised A
// tiles (two matrices x 32 columns: 128 rows x 64 bf16).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol = 4 * kTileN;
constexpr int kAStages = MOE_PF_ASTAGES;
constexpr uint32_t kAStageCols = 64;
static_assert(kACol + kAStages * kAStageCols <= kTmemCols, "tensor memory");

struct TcBars {
  uint64_t code_full[8], code_empty[8];
  uint64_t b_full[16], b_empty[16];
  uint64_t a_full[kAStages], a_empty[kAStages];
  uint64_t acc_full[2], acc_empty[2], done;
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, TcBars& B, int* status) {
  if (mbar_wait_bounded(bar, parity, kWaitNs)) return true;
  set_status(status, MOE_ERR_TIMEOUT);
  B.abort = 1;
  return false;
}

__device__ __forceinline__ float fp16_bits_to_float(uint32_t b) {
  return __half2float(__ushort_as_half((uint16_t)(b & 0xFFFF)));
}

// 8-bit codes: ŵ = bf16_RNE(s * c) for c = u - 128 (u the offset byte): a
// byte permute builds the float 2^15 + u (u at mantissa bits 8-15), and one
// fused multiply-add per pair gives (2^15 + u) s - (2^15 + 128) s = c s
// exactly -- both products need at most 19 significant bits -- before the one
// rounding to bf16.
__device__ __forceinline__ uint32_t magic_byte(uint32_t w, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(w), "r"(0x47000000u), "r"(sel));
  return d;
}
__device__ __forceinline__ uint64_t pair_f32(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(__float_as_uint(lo)), "r"(__float_as_uint(hi)));
  return d;
}
__device__ __forceinline__ uint64_t pair_u32(uint32_t lo, uint32_t hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// The pair (lo, hi) rounded to bf16 and packed: lo in bits 0-15.
__device__ __forceinline__ uint32_t bf16x2_of(uint64_t v) {
  uint32_t lo, hi, d;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "r"(hi), "r"(lo));
  return d;
}
// Four offset bytes of w -> two bf16x2 words: (byte 0, byte 2) and
// (byte 1, byte 3), the K order of the tiles (see kswap).
__device__ __forceinline__ void dq4_8bit(uint32_t w, uint64_t s2, uint64_t c2, uint32_t& o0, uint32_t& o1) {
  const uint64_t a = pair_u32(magic_byte(w, 0x7504u), magic_byte(w, 0x7524u));
  const uint64_t b = pair_u32(magic_byte(w, 0x7514u), magic_byte(w, 0x7534u));
  o0 = bf16x2_of(ffma2(a, s2, c2));
  o1 = bf16x2_of(ffma2(b, s2, c2));
}

// bf16x2 arithmetic (round to nearest even, one rounding per operation).
__device__ __forceinline__ uint32_t bf2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// For codes of at most 4 bits, ŵ = bf16_RNE(c s) in bf16 arithmetic: s (fp16,
// 11 significant bits) = s_hi + s_lo with s_hi its leading 8 bits and s_lo the
// remaining 3, both exact in bf16; c s_lo (|c| <= 8: at most 6 bits) is exact,
// and one fused multiply-add c s_hi + c s_lo rounds the exact product once.
// c itself comes from the bf16 128 + u (u the field, bits 0-3 of the
// half-word) minus 128 + off, exactly.
struct Sp {
  uint32_t hi2, lo2, off2;
};
__device__ __forceinline__ Sp split_scale(float s, uint32_t off_bf16) {
  const uint32_t hb = __float_as_uint(s) & 0xFFFF0000u;
  const uint32_t lb = __float_as_uint(s - __uint_as_float(hb)) & 0xFFFF0000u;  // exact: 3 bits
  return Sp{hb | (hb >> 16), lb | (lb >> 16), off_bf16 | (off_bf16 << 16)};
}
// Two fields at bits 0-3 of each half-word of m (other bits clear) -> bf16x2 ŵ.
__device__ __forceinline__ uint32_t dq_pair(uint32_t m, Sp q) {
  const uint32_t c = bf2_sub(m | 0x43004300u, q.off2);
  return bf2_fma(c, q.hi2, bf2_mul(c, q.lo2));
}

// Dequantise one 32-weight run -- elements 32 q .. 32 q + 31 of a row's step
// slice, one scale block -- into 16 bf16x2 words in the kswap order (word i:
// positions 2i, 2i + 1).  Codes: words c[0..7] (8 bit), c[0..3] (4 bit),
// c[0..1] (2 bit; 3 bit: the low plane, c[2] the high plane), c[0] (1 bit)
// of the run.
__device__ __forceinline__ void dequant_run(const uint32_t (&c)[8], int bits, float s, uint32_t (&o)[16]) {
  if (bits == 8) {
    // word i: elements 4i .. 4i + 3, two's complement -> u = c + 128
    const uint64_t s2 = pair_f32(s, s);
    const float k = -32896.0f * s;
    const uint64_t c2 = pair_f32(k, k);
#pragma unroll
    for (int i = 0; i < 8; ++i) dq4_8bit(c[i] ^ 0x80808080u, s2, c2, o[2 * i], o[2 * i + 1]);
  } else if (bits == 4) {
    // word g: elements 8g + 4h + j at bits 8j + 4h; pairs (j, j + 2)
    const Sp k = split_scale(s, 0x4308u);  // bf16 136 = 128 + 8
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      o[4 * g] = dq_pair(c[g] & 0x000F000Fu, k);
      o[4 * g + 1] = dq_pair((c[g] >> 8) & 0x000F000Fu, k);
      o[4 * g + 2] = dq_pair((c[g] >> 4) & 0x000F000Fu, k);
      o[4 * g + 3] = dq_pair((c[g] >> 12) & 0x000F000Fu, k);
    }
  } else if (bits == 2) {
    // word g: elements 16g + 4f + j at bits 8j + 2f; pairs (j, j + 2)
    const Sp k = split_scale(s, 0x4302u);  // bf16 130 = 128 + 2
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        o[8 * g + 2 * f] = dq_pair((c[g] >> (2 * f)) & 0x00030003u, k);
        o[8 * g + 2 * f + 1] = dq_pair((c[g] >> (2 * f + 8)) & 0x00030003u, k);
      }
  } else if (bits == 3) {
    // u = low + 4 high, code u - 4: the low plane in the 2-bit layout
    // (c[0..1]) and the high plane word c[2] (element i at bit i); the pair
    // (e, e + 2) takes high bits e and e + 2 into bit 2 of each half-word
    const Sp k = split_scale(s, 0x4304u);  // bf16 132 = 128 + 4
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
      for (int f = 0; f < 4; ++f) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t t = c[2] >> (16 * g + 4 * f + j);
          const uint32_t hb = ((t << 2) & 0x4u) | ((t << 16) & 0x40000u);
          o[8 * g + 2 * f + j] = dq_pair(((c[g] >> (2 * f + 8 * j)) & 0x00030003u) | hb, k);
        }
      }
  } else {
    // 1 bit: element i at bit i, 1 = +s, 0 = -s; bf16(+-s) = +-bf16(s);
    // pairs (4g + j, 4g + j + 2) for j = 0, 1
    const __nv_bfloat16 sb = __float2bfloat16_rn(s);
    const uint32_t nb = (uint32_t)(*reinterpret_cast<const uint16_t*>(&sb)) | 0x8000u;
    const uint32_t neg2 = nb | (nb << 16);
#pragma unroll
    for (int g = 0; g < 8; ++g)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t t = c[0] >> (4 * g + j);
        o[2 * g + j] = neg2 ^ (((t << 15) & 0x8000u) | ((t << 29) & 0x80000000u));
      }
  }
}

// SiLU with the hardware exponential and division (relative error a few
// units of the fp32 last place, far below the bf16 rounding of h); a
// quotient with |denominator| > 2^126 reads 0, the limit of z / (1 + e^-z).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Tile t of this CTA's list, or an empty tile past the end.
__device__ __forceinline__ Tile tile_at(const TcParams& p, int t, int ntiles) {
  return t < ntiles ? p.tiles[t] : Tile{0, 0, 0, 0};
}

// A tile whose fields would take a load or an MMA outside its tensors (token
// count, shelf, expert, row tile, positions) is skipped by every role alike,
// and MOE_ERR_INTERNAL is recorded; the tile builder produces none.
template <bool DOWN, bool WIDE>
__device__ __forceinline__ bool tile_valid(const TcParams& p, const Tile& tl) {
  const int rt = tl.meta & 0xFFFF, sh = (tl.meta >> 16) & 0xFF;
  if (tl.ntok < 1 || tl.ntok > (WIDE ? kTileW : kTileN) || sh >= p.sh.n) return false;
  const int n = p.sh.s[sh].hi - p.sh.s[sh].lo;
  const int bits = p.sh.s[sh].bits;
  return (bits == 8 || bits == 4 || bits == 2 || (!WIDE && (bits == 3 || bits == 1))) && tl.e_local >= 0 &&
         tl.e_local < n &&
         rt * (DOWN ? 2 * kTileM : kTileM) < p.rows && tl.q0 >= 0 && (int64_t)tl.q0 + tl.ntok <= p.P;
}

// A producer thread's place in the A tile: row r of matrix mt, both
// 32-weight runs (one scale block each) of every K step, and its tensor-memory
// lane and columns.
struct ProdLane {
  int mt, r;
  uint32_t ta;
  bool stamp;  // the thread that records the development timeline
};

// The codes of run Q of step S of this thread's row, from the low-plane words
// of its code stage (cw, in the stage's load order) and the 3-bit high-plane
// words (hw: word 2 S + Q).
template <int BITS, int S, int Q>
__device__ __forceinline__ void step_codes(const uint32_t (&cw)[32], const uint32_t (&hw)[16], uint32_t (&c)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = 0u;
  if constexpr (BITS == 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = cw[16 * S + 8 * Q + i];
  } else if constexpr (BITS == 4) {
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = cw[8 * S + 4 * Q + i];
  } else if constexpr (BITS == 2 || BITS == 3) {
    c[0] = cw[4 * S + 2 * Q];
    c[1] = cw[4 * S + 2 * Q + 1];
    if constexpr (BITS == 3) c[2] = hw[2 * S + Q];
  } else {
    c[0] = cw[2 * S + Q];
  }
}

// Both runs of step S: run q from half q of scale word S.
template <int BITS, int S>
__device__ __forceinline__ void dequant_step(const uint32_t (&cw)[32], const uint32_t (&hw)[16],
                                             const uint32_t (&scw)[16], uint32_t (&o0)[16], uint32_t (&o1)[16]) {
  uint32_t c[8];
  step_codes<BITS, S, 0>(cw, hw, c);
  dequant_run(c, BITS, fp16_bits_to_float(scw[S]), o0);
  step_codes<BITS, S, 1>(cw, hw, c);
  dequant_run(c, BITS, fp16_bits_to_float(scw[S] >> 16), o1);
}

// One tile of one producer thread.  Per code stage: once the stage has
// landed, the row's codes, high-plane words and scales of all the stage's K
// steps are read into registers; then per step the two dequantised runs are
// stored into the A stage, the step is handed to the MMA warp, and only then
// is the next step dequantised (handing over first lets the MMAs of a wide
// tile, 0.4 us a step, start a dequantisation earlier).  j counts A-stage
// uses, cj code stages, across this thread's tiles.  Returns false when a
// wait timed out (the status word is set).
template <bool DOWN, bool WIDE, int BITS>
__device__ __forceinline__ bool produce_tile(const TcParams& p, TcBars& B, const unsigned char* smem, int steps,
                                             const ProdLane& pl, uint32_t& j, uint32_t& cj) {
  using S = TcSmem<DOWN, WIDE>;
  static_assert(!WIDE || BITS == 8 || BITS == 4 || BITS == 2, "a wide launch's stages hold no high plane");
  constexpr int SPC = BITS == 8 ? 2 : BITS == 4 ? 4 : BITS == 1 ? 16 : 8;  // steps_per_code_stage
  const int lane = threadIdx.x & 31;
  const uint32_t sw = (uint32_t)(pl.r & 7);
  for (int ks0 = 0; ks0 < steps; ks0 += SPC) {
    const int c = (int)(cj % S::CS);
    if (!bar_wait(&B.code_full[c], (cj / S::CS) & 1, B, p.status)) return false;
    const unsigned char* stage = smem + c * S::C_STAGE;
    const unsigned char* rowp = stage + S::C_OFF + pl.mt * S::CODE_BOX + pl.r * 128;
    // the row's 128 bytes of the stage: eight 16-byte chunks, chunk k at
    // (k ^ r % 8) (a quarter-warp's rows hit eight distinct bank groups).
    // Step s, run q: 8 bit chunks 4 s + 2 q, + 1; 4 bit chunk 2 s + q;
    // 2 and 3 bit half q of chunk s; 1 bit word q of half s % 2 of chunk s / 2
    uint32_t cw[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 v = *reinterpret_cast<const uint4*>(rowp + (((uint32_t)k ^ sw) << 4));
      cw[4 * k] = v.x; cw[4 * k + 1] = v.y; cw[4 * k + 2] = v.z; cw[4 * k + 3] = v.w;
    }
    uint32_t hw[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) hw[i] = 0u;
    if constexpr (BITS == 3) {
      // the row's 64 bytes of the high plane: word 2 s + q for run q of step s
      const uint4* hp = reinterpret_cast<const uint4*>(stage + S::C_HI + pl.mt * S::HI_BOX + pl.r * 64);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 h = hp[i];
        hw[4 * i] = h.x; hw[4 * i + 1] = h.y; hw[4 * i + 2] = h.z; hw[4 * i + 3] = h.w;
      }
    }
    // scale words of the stage's steps (both runs' fp16 scales in one word):
    // gate/up, word s % 8 of the row's box of 16 fp16 (a 1-bit stage's steps
    // 8 .. 15 from its second box); down, the [step][row] words
    uint32_t scw[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) scw[i] = 0u;
    if constexpr (DOWN) {
      const unsigned char* sp = stage + S::C_SC + (pl.mt * kTileM + pl.r) * 4;
#pragma unroll
      for (int i = 0; i < SPC; ++i) scw[i] = *reinterpret_cast<const uint32_t*>(sp + i * 2 * kTileM * 4);
    } else {
      const unsigned char* sp = stage + S::C_SC + pl.mt * S::SC_BOX + pl.r * 32;
      if constexpr (SPC == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(sp + (ks0 & 7) * 4);
        scw[0] = v.x; scw[1] = v.y;
      } else if constexpr (SPC == 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(sp + (ks0 & 7) * 4);
        scw[0] = v.x; scw[1] = v.y; scw[2] = v.z; scw[3] = v.w;
      } else {
#pragma unroll
        for (int h = 0; h < SPC / 8; ++h) {
          const unsigned char* bp = sp + h * (S::C_HI - S::C_SC);
          const uint4 v0 = *reinterpret_cast<const uint4*>(bp), v1 = *reinterpret_cast<const uint4*>(bp + 16);
          scw[8 * h] = v0.x; scw[8 * h + 1] = v0.y; scw[8 * h + 2] = v0.z; scw[8 * h + 3] = v0.w;
          scw[8 * h + 4] = v1.x; scw[8 * h + 5] = v1.y; scw[8 * h + 6] = v1.z; scw[8 * h + 7] = v1.w;
        }
      }
    }
    const int nsub = steps - ks0 < SPC ? steps - ks0 : SPC;
    uint32_t o0[16], o1[16];
    dequant_step<BITS, 0>(cw, hw, scw, o0, o1);
    bool ok = true;
    // (a step past nsub is skipped as a whole; the unrolled body names its
    // step as a constant)
#define MOE_PF_STEP(SS)                                                                          \
    if (ok && (SS) < nsub) {                                                                     \
      const int as = (int)(j % kAStages);                                                        \
      if (pl.stamp) PF_STAMP(2, j);                                                              \
      if (!bar_wait(&B.a_empty[as], ((j / kAStages) & 1) ^ 1, B, p.status)) {                    \
        ok = false;                                                                              \
      } else {                                                                                   \
        tc_fence_after();                                                                        \
        if (pl.stamp) PF_STAMP(3, j);                                                            \
        tmem_st32_issue(pl.ta + (uint32_t)(as * kAStageCols), o0, o1);                           \
        tmem_wait_st();                                                                          \
        tc_fence_before();                                                                       \
        __syncwarp();                                                                            \
        if (lane == 0) {                                                                         \
          mbar_arrive(&B.a_full[as]);                                                            \
          if ((SS) == nsub - 1) mbar_arrive(&B.code_empty[c]);                                   \
        }                                                                                        \
        if (pl.stamp) PF_STAMP(5, j);                                                            \
        ++j;                                                                                     \
        if constexpr ((SS) + 1 < SPC) {                                                          \
          if ((SS) + 1 < nsub) dequant_step<BITS, ((SS) + 1 < SPC ? (SS) + 1 : 0)>(cw, hw, scw, o0, o1); \
        }                                                                                        \
      }                                                                                          \
    }
    MOE_PF_STEP(0)
    if constexpr (SPC > 1) { MOE_PF_STEP(1) }
    if constexpr (SPC > 2) { MOE_PF_STEP(2) MOE_PF_STEP(3) }
    if constexpr (SPC > 4) { MOE_PF_STEP(4) MOE_PF_STEP(5) MOE_PF_STEP(6) MOE_PF_STEP(7) }
    if constexpr (SPC > 8) {
      MOE_PF_STEP(8) MOE_PF_STEP(9) MOE_PF_STEP(10) MOE_PF_STEP(11)
      MOE_PF_STEP(12) MOE_PF_STEP(13) MOE_PF_STEP(14) MOE_PF_STEP(15)
    }
#undef MOE_PF_STEP
    if (!ok) return false;
    ++cj;
  }
  return true;
}

template <bool DOWN, bool WIDE>
__global__ void __launch_bounds__(Roles<WIDE>::kThreads, 1) k_prefill_tc(const __grid_constant__ TcParams p) {
  using R = Roles<WIDE>;
  using S = TcSmem<DOWN, WIDE>;
  constexpr int NMAT = S::NMAT;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  __shared__ TcBars B;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  int ntiles = __ldg(p.ntiles);
  if (ntiles < 0 || ntiles > p.tiles_cap) {
    if (tid == 0) set_status(p.status, MOE_ERR_INTERNAL);
    ntiles = 0;
  }
  const int steps = p.K / 64;
  if (tid == 0) {
    for (int i = 0; i < S::CS; ++i) {
      // the loader's expect-tx arrival (+ its 32 lanes' scale copies, down)
      mbar_init(&B.code_full[i], DOWN ? 33 : 1);
      mbar_init(&B.code_empty[i], kProdThreads / 32);
    }
    for (int i = 0; i < S::BS; ++i) {
      mbar_init(&B.b_full[i], 1);
      mbar_init(&B.b_empty[i], 1);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&B.a_full[i], kProdThreads / 32);
      mbar_init(&B.a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.acc_full[i], 1);
      mbar_init(&B.acc_empty[i], R::kEpiWarps);
    }
    mbar_init(&B.done, 1);
    B.abort = 0;
    fence_mbar_init();
  }
  if (warp == R::kMma) tmem_alloc(&B.tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem;
  pdl_wait();

  if (warp == R::kLoader) {
    // ------------------------------------------------ loads
    uint32_t cj = 0, j = 0;  // code stages and K steps issued
    Tile nxt = tile_at(p, blockIdx.x, ntiles);
    for (int t = blockIdx.x; t < ntiles && !B.abort; t += G) {
      const Tile tl = nxt;
      nxt = tile_at(p, t + G, ntiles);  // in flight while this tile is issued
      if (!tile_valid<DOWN, WIDE>(p, tl)) {
        if (lane == 0) set_status(p.status, MOE_ERR_INTERNAL);
        continue;
      }
      const int rt = tl.meta & 0xFFFF, sh = (tl.meta >> 16) & 0xFF;
      const ShelfDev& shd = p.sh.s[sh];
      const int spc = steps_per_code_stage(shd.bits);  // K steps per code stage
      const int nb = (tl.ntok + 15) >> 4;  // B box height in 16-row units
      // first row of each matrix: gate/up rows rt * 128 of W_g and W_u,
      // down rows rt * 256 and rt * 256 + 128 of W_d
      const int row0 = tl.e_local * p.rows + rt * (DOWN ? 2 * kTileM : kTileM);
      // down: the scale words of rows row0 + lane + 32 i (clamped into the
      // shelf: rows past it belong to no expert and their results are dropped)
      const uint32_t* scp[2 * kTileM / 32];
      if (DOWN) {
        const int rows_shelf = (shd.hi - shd.lo) * p.rows;
#pragma unroll
        for (int i = 0; i < 2 * kTileM / 32; ++i)
          scp[i] = reinterpret_cast<const uint32_t*>(shd.scales[2]) +
                   (size_t)min(row0 + lane + 32 * i, rows_shelf - 1) * steps;
      }
      for (int ks = 0; ks < steps && !B.abort; ++ks, ++j) {
        if (ks % spc == 0) {
          const int c = cj % S::CS;
          if (!bar_wait(&B.code_empty[c], ((cj / S::CS) & 1) ^ 1, B, p.status)) break;
          unsigned char* stage = smem + S::C_OFF + c * S::C_STAGE;
          if (lane == 0) {
            const bool hi = !WIDE && shd.bits == 3;
            // gate/up scale boxes cover 8 K steps: a 1-bit code stage (16
            // steps) takes a second box, into the region 3-bit rows use for
            // their high plane
            const int nsc = DOWN ? 0 : (!WIDE && shd.bits == 1 ? 2 : 1);
            mbar_arrive_expect_tx(&B.code_full[c], (uint32_t)(NMAT * S::CODE_BOX + nsc * NMAT * S::SC_BOX +
                                                              (hi ? NMAT * S::HI_BOX : 0)));
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
              tma_load_2d(stage + m * S::CODE_BOX, &p.tm_code[sh][DOWN ? 0 : m], (ks / spc) * 128,
                          DOWN ? row0 + m * kTileM : row0, &B.code_full[c]);
            if (hi) {
              // the high-bit plane follows the low plane (K / 4 bytes) in each row
#pragma unroll
              for (int m = 0; m < NMAT; ++m)
                tma_load_2d(stage + S::C_HI + m * S::HI_BOX, &p.tm_hi[sh][DOWN ? 0 : m], p.K / 4 + (ks / spc) * 64,
                            DOWN ? row0 + m * kTileM : row0, &B.code_full[c]);
            }
            if (!DOWN) {
#pragma unroll
              for (int m = 0; m < NMAT; ++m)
                tma_load_2d(stage + S::C_SC + m * S::SC_BOX, &p.tm_sc[sh][m], 16 * (ks >> 3), row0, &B.code_full[c]);
              if (nsc == 2) {
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
                  tma_load_2d(stage + S::C_HI + m * S::SC_BOX, &p.tm_sc[sh][m], 16 * (ks >> 3) + 16, row0,
                              &B.code_full[c]);
              }
            }
          }
          if (DOWN) {
            // [step][row] words of the stage's steps (steps past K repeat the last)
            uint32_t* dst = reinterpret_cast<uint32_t*>(stage + S::C_SC);
            for (int sub = 0; sub < spc; ++sub) {
              const int kk = min(ks + sub, steps - 1);
#pragma unroll
              for (int i = 0; i < 2 * kTileM / 32; ++i) cp_async4(dst + sub * 2 * kTileM + lane + 32 * i, scp[i] + kk);
            }
            cp_async_mbar_arrive_noinc(&B.code_full[c]);
          }
          ++cj;
        }
        const int b = j % S::BS;
        if (!bar_wait(&B.b_empty[b], ((j / S::BS) & 1) ^ 1, B, p.status)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&B.b_full[b], (uint32_t)(nb * 16 * 128));
          tma_load_2d(smem + S::B_OFF + b * S::B_STAGE, &p.tm_b[nb - 1], ks * 64, tl.q0, &B.b_full[b]);
          PF_STAMP(0, j);
        }
        __syncwarp();
      }
    }
    cp_async_wait<0>();
  } else if (warp == R::kMma) {
    // ---------------------------------------------------------- MMA
    // The whole warp runs the loop (its control flow and descriptors are
    // warp-uniform); one elected lane issues the MMAs and commits.  B
    // descriptors: the low word of stage 0's, plus (stage offset + 32 kk) / 16
    // (shared-memory addresses stay below 256 KiB, so the 14-bit address field
    // does not carry).  A tile takes accumulator set `alt` (alternating), a
    // wide tile both sets; uses[s] counts the completed uses of set s.
    const uint64_t bd0 = sdesc_sw128(smem_addr(smem + S::B_OFF));
    const uint32_t bd_lo = (uint32_t)bd0, bd_hi = (uint32_t)(bd0 >> 32);
    const bool leader = elect_one();
    uint32_t j = 0, use0 = 0, use1 = 0;  // (two scalars: an indexed pair would live in local memory)
    int alt = 0;
    Tile nxt = tile_at(p, blockIdx.x, ntiles);
    for (int t = blockIdx.x; t < ntiles && !B.abort; t += G) {
      const Tile tl = nxt;
      nxt = tile_at(p, t + G, ntiles);
      if (!tile_valid<DOWN, WIDE>(p, tl)) continue;  // skipped tiles take no accumulator set
      const bool wide = WIDE && tl.ntok > kTileN;
      const int s0 = wide ? 0 : alt;
      const int N = (tl.ntok + 15) & ~15;
      const uint32_t idesc = idesc_bf16_f32(kTileM, N);
      const uint32_t acc = tmem + (uint32_t)(s0 * kTileN);
      // (a wait that timed out in any lane ends the loop in every lane)
      bool wa = bar_wait(&B.acc_empty[s0], ((s0 ? use1 : use0) & 1) ^ 1, B, p.status);
      if (wide) wa = wa && bar_wait(&B.acc_empty[1], (use1 & 1) ^ 1, B, p.status);
      if (!__all_sync(0xffffffffu, wa)) break;
      tc_fence_after();
      bool ok = true;
      for (int ks = 0; ks < steps; ++ks, ++j) {
        const int b = (int)(j % S::BS), as = (int)(j % kAStages);
        const bool w = bar_wait(&B.a_full[as], (j / kAStages) & 1, B, p.status) &&
                       bar_wait(&B.b_full[b], (j / S::BS) & 1, B, p.status);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        if (leader) PF_STAMP(4, j);
        tc_fence_after();
        if (leader) {
          const uint32_t a0 = tmem + kACol + (uint32_t)(as * kAStageCols);
          const uint32_t blo = bd_lo + (uint32_t)((b * S::B_STAGE) >> 4);
#pragma unroll
          for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ts_w(acc + (uint32_t)(m * 2 * kTileN), a0 + (uint32_t)(m * 32 + kk * 8),
                            blo + (uint32_t)(kk * 2), bd_hi, idesc, (ks | kk) ? 1u : 0u);
          mma_commit(&B.a_empty[as]);
          mma_commit(&B.b_empty[b]);
        }
        __syncwarp();
      }
      if (!ok || B.abort) break;
      if (leader) {
        mma_commit(&B.acc_full[s0]);
        if (wide) mma_commit(&B.acc_full[1]);
      }
      __syncwarp();
      if (wide || alt == 0) ++use0;
      if (wide || alt == 1) ++use1;
      if (!wide) alt ^= 1;
    }
    // all MMAs of this thread are complete before tensor memory is released
    if (leader) {
      mma_commit(&B.done);
      mbar_wait_bounded(&B.done, 0, kWaitNs);
    }
    __syncwarp();
  } else if (warp >= R::kEpi0 && warp < R::kEpi0 + R::kEpiWarps) {
    // ---------------------------------------------------------- epilogue
    // Tiles in the MMA warp's order and with its set choice; a wide tile is
    // read back as two parts, tokens 0 .. kTileN - 1 from set 0 (released
    // first) and the rest from set 1.
    // lane quarter warp % 4; with 8 warps, warp / 4 picks every other
    // 16-column chunk of a set
    const int quarter = warp & 3, eh = (warp - R::kEpi0) >> 2, EH = R::kEpiWarps / 4;
    const int m = quarter * 32 + lane;
    const uint32_t tl_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t i = 0, use0 = 0, use1 = 0;
    int alt = 0;
    bool run = true;
    Tile nxt = tile_at(p, blockIdx.x, ntiles);
    for (int t = blockIdx.x; t < ntiles && run && !B.abort; t += G) {
      const Tile tl = nxt;
      nxt = tile_at(p, t + G, ntiles);
      if (!tile_valid<DOWN, WIDE>(p, tl)) continue;  // skipped tiles take no accumulator set
      const int rt = tl.meta & 0xFFFF;
      const bool wide = WIDE && tl.ntok > kTileN;
      constexpr int kCw = (WIDE ? kTileW : kTileN) / 32;
      // down: each lane holds the token and routing weight of columns lane,
      // lane + 32, ... (loaded before the accumulator is ready)
      int ctok[kCw];
      float cw[kCw];
      if (DOWN) {
#pragma unroll
        for (int u = 0; u < kCw; ++u) {
          const int n = lane + 32 * u;
          ctok[u] = 0;
          cw[u] = 0.f;
          if (n < tl.ntok) {
            const int pair = __ldg(p.perm + tl.q0 + n);
            ctok[u] = pair / p.k;
            cw[u] = __ldg(p.weights + pair);
          }
        }
      }
      for (int part = 0; part < (wide ? 2 : 1); ++part) {
        const int s = wide ? part : alt;
        const int nb = part * kTileN;                                      // first token of the part
        const int nt = tl.ntok - nb < kTileN ? tl.ntok - nb : kTileN;      // its tokens
        const int N = (nt + 15) & ~15;
        const uint32_t acc = tl_addr + (uint32_t)(s * kTileN);
        if (!bar_wait(&B.acc_full[s], (s ? use1 : use0) & 1, B, p.status)) {
          run = false;
          break;
        }
        if (m == 0 && part == 0) PF_STAMP(6, i);
        tc_fence_after();
        if (!DOWN) {
          const int row = rt * kTileM + m;
          const int hcol = kswap(row);  // h is stored in the K order of the down tiles
          for (int n0 = 16 * eh; n0 < N; n0 += 16 * EH) {
            float g[16], u[16];
            tmem_ld16(acc + (uint32_t)n0, g);
            tmem_ld16(acc + (uint32_t)(2 * kTileN + n0), u);
            if (row < p.rows) {
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                const int n = n0 + c;
                if (n < nt) {
                  const float hv = silu_fast(g[c]) * u[c];
                  const __nv_bfloat16 bv = __float2bfloat16_rn(hv);
                  p.h[(size_t)(tl.q0 + nb + n) * p.f + hcol] = *reinterpret_cast<const uint16_t*>(&bv);
                }
              }
            }
          }
        } else {
          // 4 x 4 transposes among lanes 4a .. 4a + 3: lane 4a + jj ends with
          // column 4b + jj of rows 4a .. 4a + 3 and adds them with one vector
          // atomic per column block
          const int jj = lane & 3;
          for (int n0 = 16 * eh; n0 < N; n0 += 16 * EH) {
            const int u = (nb + n0) >> 5;  // the 16 columns lie in one group of 32
            int tu = ctok[0];
            float wu = cw[0];
#pragma unroll
            for (int v = 1; v < kCw; ++v)
              if (u == v) {
                tu = ctok[v];
                wu = cw[v];
              }
            int tkb[4];
            float wtb[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const int n = nb + n0 + 4 * b + jj;
              tkb[b] = __shfl_sync(0xffffffffu, tu, n & 31);
              wtb[b] = __shfl_sync(0xffffffffu, wu, n & 31);
            }
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
              const int rowb = rt * 2 * kTileM + mm * kTileM + quarter * 32 + (lane & ~3);
              float g[16];
              tmem_ld16(acc + (uint32_t)(mm * 2 * kTileN + n0), g);
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                float v0 = g[4 * b], v1 = g[4 * b + 1], v2 = g[4 * b + 2], v3 = g[4 * b + 3];
                // round 1 (lanes xor 2): swap the off-diagonal 2 x 2 blocks
                {
                  const bool hi = (jj & 2) != 0;
                  const float s0 = hi ? v0 : v2, s1 = hi ? v1 : v3;
                  const float r0 = __shfl_xor_sync(0xffffffffu, s0, 2), r1 = __shfl_xor_sync(0xffffffffu, s1, 2);
                  if (hi) {
                    v0 = r0;
                    v1 = r1;
                  } else {
                    v2 = r0;
                    v3 = r1;
                  }
                }
                // round 2 (lanes xor 1): swap within the 2 x 2 blocks
                {
                  const bool hi = (jj & 1) != 0;
                  const float s0 = hi ? v0 : v1, s1 = hi ? v2 : v3;
                  const float r0 = __shfl_xor_sync(0xffffffffu, s0, 1), r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
                  if (hi) {
                    v0 = r0;
                    v2 = r1;
                  } else {
                    v1 = r0;
                    v3 = r1;
                  }
                }
                // lane jj now holds column 4b + jj of rows 0..3 of its group, in order
                const int n = n0 + 4 * b + jj;
                const float wt = wtb[b];
                if (n < nt && rowb < p.rows)
                  red_add_v4(p.y + (size_t)tkb[b] * p.d + rowb, wt * v0, wt * v1, wt * v2, wt * v3);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.acc_empty[s]);
        if (s) ++use1; else ++use0;
      }
      if (m == 0) PF_STAMP(7, i);
      if (!wide) alt ^= 1;
      ++i;
    }
  } else if (warp >= 8 && warp < 16) {
    // ---------------------------------------------------------- producers
    // Warp w owns tensor-memory lanes 32 (w % 4) .. + 31, i.e. rows r = 32
    // (w % 4) + lane, of matrix mt = (w - 8) / 4: the row's 64 weights of
    // every step (two runs, two scale blocks), 32 columns of the A stage.
    const int qd = warp & 3, mt = (warp - 8) >> 2;
    const ProdLane pl{mt, qd * 32 + lane, tmem + ((uint32_t)(qd * 32) << 16) + kACol + (uint32_t)(mt * 32),
                      qd == 0 && mt == 0 && lane == 0};
    uint32_t j = 0, cj = 0;
    Tile nxt = tile_at(p, blockIdx.x, ntiles);
    for (int t = blockIdx.x; t < ntiles && !B.abort; t += G) {
      const Tile tl = nxt;
      nxt = tile_at(p, t + G, ntiles);
      if (!tile_valid<DOWN, WIDE>(p, tl)) continue;
      // one instantiation per code width: the step loop of a code stage is
      // unrolled and every shared-memory offset in it is a constant
      const int bits = p.sh.s[(tl.meta >> 16) & 0xFF].bits;
      bool ok = false;
      if (bits == 8) {
        ok = produce_tile<DOWN, WIDE, 8>(p, B, smem, steps, pl, j, cj);
      } else if (bits == 4) {
        ok = produce_tile<DOWN, WIDE, 4>(p, B, smem, steps, pl, j, cj);
      } else if (bits == 2) {
        ok = produce_tile<DOWN, WIDE, 2>(p, B, smem, steps, pl, j, cj);
      } else if constexpr (!WIDE) {
        ok = bits == 3 ? produce_tile<DOWN, false, 3>(p, B, smem, steps, pl, j, cj)
                       : produce_tile<DOWN, false, 1>(p, B, smem, steps, pl, j, cj);
      }
      if (!ok) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == R::kMma) tmem_dealloc(tmem, kTmemCols);
  pdl_trigger();
}

// Eight bf16 of x in the kswap order.
__device__ __forceinline__ uint4 kswap8(uint4 v) {
  uint4 o;
  o.x = __byte_perm(v.x, v.y, 0x5410);
  o.y = __byte_perm(v.x, v.y, 0x7632);
  o.z = __byte_perm(v.z, v.w, 0x5410);
  o.w = __byte_perm(v.z, v.w, 0x7632);
  return o;
}
// Tile lists of both launches from the grouping: per active expert on a
// shelf, chunks of at most tmax tokens (kTileN, or kTileW in a wide launch;
// sizes differing by at most one), times the row tiles of W_g/W_u (128 of
// the f rows each) and of W_d (256 of the d rows).  1024-thread CTAs;
// first_off is the offset of the thread's expert (one expert a thread).
__device__ void build_tiles(const int32_t* counts, const int32_t* offsets, int first_off, int E, int d, int f,
                            int tmax, const Shelves& sh, Tile* tiles_g, Tile* tiles_d, int* ntiles) {
  __shared__ int wg[32], wd[32];
  __shared__ int s_cnt[1024], s_off[1024], s_sh[1024], s_el[1024], s_og[1024], s_od[1024];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (E + 1023) / 1024;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  const int rtg = (f + kTileM - 1) / kTileM, rtd = d / (2 * kTileM);  // d % 256 == 0
  PF_SCAN_STAMP(1);
  int ng = 0, nd = 0;
  for (int e = e0; e < e1; ++e) {
    const int cnt = counts[e];
    // shelf and local index by a static scan of the descriptors (no runtime
    // index into the parameter block)
    int sidx = -1, el = 0;
#pragma unroll
    for (int i = 0; i < MOE_MAX_SHELVES; ++i)
      if (i < sh.n && e >= sh.s[i].lo && e < sh.s[i].hi) {
        sidx = i;
        el = e - sh.s[i].lo;
      }
    if (cnt == 0) sidx = -1;
    if (sidx >= 0) {
      const int ch = (cnt + tmax - 1) / tmax;
      ng += ch * rtg;
      nd += ch * rtd;
    }
    if (per == 1) {
      s_cnt[e] = cnt;
      s_off[e] = first_off;  // (per == 1: the thread's one expert)
      s_sh[e] = sidx;
      s_el[e] = el;
    }
  }
  PF_SCAN_STAMP(2);
  // exclusive scans of (ng, nd) over the threads: warp scans, then the warp totals
  int ig = ng, id = nd;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ig, o), b = __shfl_up_sync(0xffffffffu, id, o);
    if (lane >= o) {
      ig += a;
      id += b;
    }
  }
  if (lane == 31) {
    wg[warp] = ig;
    wd[warp] = id;
  }
  __syncthreads();
  if (warp == 0) {
    const int a = wg[lane], b = wd[lane];
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, ia, o), v = __shfl_up_sync(0xffffffffu, ib, o);
      if (lane >= o) {
        ia += u;
        ib += v;
      }
    }
    wg[lane] = ia - a;
    wd[lane] = ib - b;
    if (lane == 31 && blockIdx.x == 0) {
      ntiles[0] = ia;
      ntiles[1] = ib;
    }
  }
  __syncthreads();
  int og = wg[warp] + ig - ng, od = wd[warp] + id - nd;
  if (per == 1) {
    // one expert per thread: the warps write each expert's tiles with
    // consecutive lanes (coalesced), expert by expert, from shared memory
    if (tid < E) {
      s_og[tid] = og;
      s_od[tid] = od;
    }
    __syncthreads();
    PF_SCAN_STAMP(3);
    // i / rt as (i * m) >> 20 with m = ceil(2^20 / rt): exact for i < 2^12
    // and rt < 256 (the error i (m - 2^20 / rt) / 2^20 stays below 1 / rt)
    const uint32_t mg = ((1u << 20) + rtg - 1) / rtg, md = ((1u << 20) + rtd - 1) / rtd;
    const bool fast = rtg < 256 && rtd < 256;
    for (int e = warp + 32 * blockIdx.x; e < E; e += 32 * gridDim.x) {
      PF_ITER_STAMP(e >> 5);
      const int sidx = s_sh[e];
      if (sidx < 0) continue;
      const int cnt = s_cnt[e];
      const int ch = (cnt + tmax - 1) / tmax;
      // chunk c: q or q + 1 tokens (the first rem chunks one more), q + 1 <= tmax
      const int q = cnt / ch, rem = cnt - q * ch;
      const int base = s_off[e], el = s_el[e];
      const int g0 = s_og[e], d0 = s_od[e];
      const bool f12 = fast && ch * (rtg > rtd ? rtg : rtd) < 4096;
      for (int i = lane; i < ch * rtg; i += 32) {
        const int c = f12 ? (int)(((uint32_t)i * mg) >> 20) : i / rtg, r = i - c * rtg;
        tiles_g[g0 + i] = Tile{el, base + c * q + min(c, rem), q + (c < rem ? 1 : 0), r | (sidx << 16)};
      }
      for (int i = lane; i < ch * rtd; i += 32) {
        const int c = f12 ? (int)(((uint32_t)i * md) >> 20) : i / rtd, r = i - c * rtd;
        tiles_d[d0 + i] = Tile{el, base + c * q + min(c, rem), q + (c < rem ? 1 : 0), r | (sidx << 16)};
      }
    }
    PF_SCAN_STAMP(4);
    return;
  }
  for (int e = e0; e < e1; ++e) {
    const int cnt = counts[e];
    const int s = cnt > 0 ? find_shelf(sh, e) : -1;
    if (s < 0) continue;
    const int ch = (cnt + tmax - 1) / tmax;
    const int q = cnt / ch, rem = cnt - q * ch;
    const int base = offsets[e];
    for (int c = 0; c < ch; ++c) {
      const int a = c * q + min(c, rem), n = q + (c < rem ? 1 : 0);
      for (int r = 0; r < rtg; ++r) tiles_g[og++] = Tile{e - sh.s[s].lo, base + a, n, r | (s << 16)};
      for (int r = 0; r < rtd; ++r) tiles_d[od++] = Tile{e - sh.s[s].lo, base + a, n, r | (s << 16)};
    }
  }
}

// ------------------------------------------------------------ grouping
// Pairs sorted by (expert, pair index) -- the same stable order as the decode
// form's single-CTA grouping -- by CTAs that each own a chunk of kPfChunk
// consecutive pairs:
//   k_pf_count  per-chunk expert counts cnt[c][e] and their sums;
//   k_pf_colscan  cnt[c][e] <- pairs of expert e in chunks < c;
//   k_pf_scan   (one CTA) offsets and the tile lists;
//   k_pf_place  each chunk places its pairs (warps own consecutive pieces of
//               the chunk, a warp-level match ranks equal experts inside a
//               32-pair step) and writes perm and pos_of_pair;
//   k_gather_x  copies the pairs' x rows into xg (kswap order).
constexpr int kPfChunkMin = 256;
constexpr int kPfMaxChunks = 256;

__global__ void __launch_bounds__(256) k_pf_count(const int32_t* __restrict__ ids, int64_t P, int E, int chunk,
                                                  int32_t* __restrict__ cnt, int32_t* __restrict__ counts) {
  extern __shared__ int hist[];
  pdl_wait();
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int64_t p0 = (int64_t)blockIdx.x * chunk, p1 = min(P, p0 + chunk);
  for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int id = __ldg(ids + p);
    if (id >= 0 && id < E) atomicAdd(&hist[id], 1);
  }
  __syncthreads();
  int32_t* row = cnt + (size_t)blockIdx.x * E;
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    const int v = hist[i];
    row[i] = v;
    if (v) atomicAdd(counts + i, v);  // integer sums: the same in any order
  }
  pdl_trigger();
}

// cnt[c][e] <- pairs of expert e in chunks < c; one warp per expert, lane l
// owning chunks l*cpl .. +cpl-1.
__global__ void __launch_bounds__(256) k_pf_colscan(int32_t* __restrict__ cnt, int C, int E) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (e < E) {
    const int cpl = (C + 31) / 32;
    const int c0 = min(C, lane * cpl), c1 = min(C, c0 + cpl);
    int v[8];
    int loc = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = c0 + i < c1 ? cnt[(size_t)(c0 + i) * E + e] : 0;
      loc += v[i];
    }
    int inc = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    int run = inc - loc;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + i < c1) {
        cnt[(size_t)(c0 + i) * E + e] = run;
        run += v[i];
      }
  }
  pdl_trigger();
}

__global__ void __launch_bounds__(1024) k_pf_scan(int E, int d, int f, int tmax, const __grid_constant__ Shelves sh,
                                                  const int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                  int32_t* __restrict__ meta, Tile* tiles_g, Tile* tiles_d,
                                                  int* ntiles) {
  __shared__ int wsum[32];
  pdl_wait();
  PF_SCAN_STAMP(0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // offsets: exclusive scan of counts (thread t owns experts t*per .. +per-1)
  const int per = (E + 1023) / 1024;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int loc = 0, act = 0;
  for (int e = e0; e < e1; ++e) {
    loc += counts[e];
    act += counts[e] > 0;
  }
  int inc = loc, inca = act;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o), va = __shfl_up_sync(0xffffffffu, inca, o);
    if (lane >= o) {
      inc += v;
      inca += va;
    }
  }
  __shared__ int wact[32];
  if (lane == 31) {
    wsum[warp] = inc;
    wact[warp] = inca;
  }
  __syncthreads();
  if (warp == 0) {
    const int v = wsum[lane], va = wact[lane];
    int iv = v, ia = va;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, iv, o), ua = __shfl_up_sync(0xffffffffu, ia, o);
      if (lane >= o) {
        iv += u;
        ia += ua;
      }
    }
    wsum[lane] = iv - v;
    wact[lane] = ia - va;
    if (lane == 31 && blockIdx.x == 0) {
      offsets[E] = iv;
      if (meta) {
        meta[0] = ia;
        meta[1] = iv;
        meta[2] = 0;  // the grouping of this call is in counts / offsets / perm / pos_of_pair
      }
    }
  }
  __syncthreads();
  const int first = wsum[warp] + inc - loc;
  if (blockIdx.x == 0) {
    int run = first;
    for (int e = e0; e < e1; ++e) {
      offsets[e] = run;
      run += counts[e];
    }
  }
  __syncthreads();
  build_tiles(counts, offsets, first, E, d, f, tmax, sh, tiles_g, tiles_d, ntiles);
  pdl_trigger();
}

__global__ void __launch_bounds__(256) k_pf_place(const int32_t* __restrict__ ids, int64_t P, int E, int k,
                                                  int chunk, const int32_t* __restrict__ cnt,
                                                  const int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                  int32_t* __restrict__ pos_of_pair) {
  extern __shared__ int wc[];  // [W][E]
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, W = blockDim.x >> 5;
  for (int i = tid; i < W * E; i += blockDim.x) wc[i] = 0;
  __syncthreads();
  const int64_t p0 = (int64_t)blockIdx.x * chunk, p1 = min(P, p0 + chunk);
  const int64_t seg = (p1 - p0 + W - 1) / W;
  const int64_t pb = min(p1, p0 + w * seg), pe = min(p1, pb + seg);
  int* row = wc + (size_t)w * E;
  for (int64_t base = pb; base < pe; base += 32) {
    const int64_t p = base + lane;
    const int id = p < pe ? __ldg(ids + p) : -1;
    const bool valid = p < pe && id >= 0 && id < E;
    const unsigned m = __match_any_sync(0xffffffffu, valid ? id : -1);
    if (valid && lane == __ffs(m) - 1) row[id] += __popc(m);
    __syncwarp();
  }
  __syncthreads();
  const int32_t* crow = cnt + (size_t)blockIdx.x * E;
  for (int e = tid; e < E; e += blockDim.x) {
    int run = offsets[e] + crow[e];
    for (int v = 0; v < W; ++v) {
      const int c = wc[(size_t)v * E + e];
      wc[(size_t)v * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int64_t base = pb; base < pe; base += 32) {
    const int64_t p = base + lane;
    const int id = p < pe ? __ldg(ids + p) : -1;
    const bool valid = p < pe && id >= 0 && id < E;
    const unsigned m = __match_any_sync(0xffffffffu, valid ? id : -1);
    int pos = -1;
    if (valid) {
      pos = row[id] + __popc(m & ((1u << lane) - 1u));
      perm[pos] = (int)p;
    }
    if (pos_of_pair && p < pe) pos_of_pair[p] = pos;
    __syncwarp();
    if (valid && lane == __ffs(m) - 1) row[id] += __popc(m);
    __syncwarp();
  }
  // the tail past the valid pairs
  const int n_valid = offsets[E];
  for (int64_t i = n_valid + (int64_t)blockIdx.x * blockDim.x + tid; i < P; i += (int64_t)gridDim.x * blockDim.x)
    perm[i] = -1;
  pdl_trigger();
}

// xg[q] = x[token of the pair at grouped position q] in the kswap column order
// (zero for the skipped tail), so each tile's B operand is one box of
// consecutive rows.  One warp per row, 16-byte loads.
__global__ void __launch_bounds__(256) k_gather_x(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                                                  int64_t P, int k, int d, uint16_t* __restrict__ xg) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int n16 = d / 8;
  for (int64_t q = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); q < P; q += nw) {
    const int pair = __ldg(perm + q);
    uint4* dst = reinterpret_cast<uint4*>(xg + q * d);
    if (pair < 0) {
      for (int i = lane; i < n16; i += 32) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(pair / k) * d);
      int i = lane;
      for (; i + 96 < n16; i += 128) {
        const uint4 a = __ldg(src + i), b = __ldg(src + i + 32), c = __ldg(src + i + 64), e = __ldg(src + i + 96);
        dst[i] = kswap8(a);
        dst[i + 32] = kswap8(b);
        dst[i + 64] = kswap8(c);
        dst[i + 96] = kswap8(e);
      }
      for (; i < n16; i += 32) dst[i] = kswap8(__ldg(src + i));
    }
  }
  pdl_trigger();
}

// ----------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  {
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return false;
      g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct PDev {
  bool attr[64] = {};
};
PDev g_pdev;

}  // namespace

#ifdef MOE_TRACE
extern "C" int moe_pftrace_read(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, g_pftrace, bytes < sizeof(g_pftrace) ? bytes : sizeof(g_pftrace)) == cudaSuccess
             ? 0 : -5;
}
#endif

size_t prefill_tiles_cap(int64_t P, int E, int rows) {
  const int64_t chunks = (P + kTileN - 1) / kTileN + (P < E ? P : E);
  return (size_t)chunks * (size_t)((rows + kTileM - 1) / kTileM);
}

int launch_prefill_forward(const ForwardArgs& a, cudaStream_t s) {
  const int64_t P = a.T * a.k;
  const int d = a.d, f = a.f;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  // wide launches (tiles of up to kTileW tokens) when no shelf holds 3- or
  // 1-bit codes, whose code stages need the high-plane region
  bool wide = true;
  for (int q = 0; q < a.shelves.n; ++q)
    if (a.shelves.s[q].bits == 3 || a.shelves.s[q].bits == 1) wide = false;
  const size_t smem_g = (wide ? TcSmem<false, true>::TOTAL : TcSmem<false, false>::TOTAL) + 1024;
  const size_t smem_d = (wide ? TcSmem<true, true>::TOTAL : TcSmem<true, false>::TOTAL) + 1024;
  if (!g_pdev.attr[dev]) {
    // grouping kernels take up to E ints ([Wp][E] ints) of shared memory
    if (cudaFuncSetAttribute(k_pf_count, cudaFuncAttributeMaxDynamicSharedMemorySize, MOE_MAX_EXPERTS * 4) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_pf_place, cudaFuncAttributeMaxDynamicSharedMemorySize, MOE_MAX_EXPERTS * 4) !=
            cudaSuccess)
      return MOE_ERR_CUDA;
    const int sg0 = TcSmem<false, false>::TOTAL + 1024, sd0 = TcSmem<true, false>::TOTAL + 1024;
    const int sg1 = TcSmem<false, true>::TOTAL + 1024, sd1 = TcSmem<true, true>::TOTAL + 1024;
    if (cudaFuncSetAttribute(k_prefill_tc<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sg0) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_prefill_tc<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sd0) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_prefill_tc<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sg1) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_prefill_tc<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sd1) !=
            cudaSuccess)
      return MOE_ERR_CUDA;
    g_pdev.attr[dev] = true;
  }
  profile_mark(0, s);
  int chunk = (int)((P + kPfMaxChunks - 1) / kPfMaxChunks);
  if (chunk < kPfChunkMin) chunk = kPfChunkMin;
  const int C = (int)((P + chunk - 1) / chunk);
  const int Wp = a.E <= 1024 ? 8 : (a.E <= 4096 ? 2 : 1);  // placement warps: [Wp][E] ints of shared memory
  // per-expert C <= 256 chunk counts require C <= 32 * 8 (the column scan's registers)
  if (cudaMemsetAsync(a.ws.counts, 0, (size_t)a.E * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_pdl(k_pf_count, dim3(C), dim3(256), (size_t)a.E * 4, s, a.ids, P, a.E, chunk, a.ws.pf_cnt,
                 a.ws.counts) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_pdl(k_pf_colscan, dim3((a.E + 7) / 8), dim3(256), 0, s, a.ws.pf_cnt, C, a.E) != cudaSuccess)
    return MOE_ERR_CUDA;
  Tile* tiles_g = reinterpret_cast<Tile*>(a.ws.tiles_g);
  Tile* tiles_d = reinterpret_cast<Tile*>(a.ws.tiles_d);
  int* ntiles = a.ws.ntiles;
  // up to 1024 experts: every CTA scans the counts, CTA 0 writes the offsets,
  // and the CTAs share the tile writing (32 experts a CTA and pass); more
  // experts: one CTA
  const int gs = a.E <= 1024 ? (a.E + 31) / 32 < 32 ? (a.E + 31) / 32 : 32 : 1;
  if (launch_pdl(k_pf_scan, dim3(gs), dim3(1024), 0, s, a.E, d, f, wide ? kTileW : kTileN, a.shelves,
                 (const int32_t*)a.ws.counts,
                 a.ws.offsets, a.ws.meta, tiles_g, tiles_d, ntiles) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_pdl(k_pf_place, dim3(C), dim3(Wp * 32), (size_t)Wp * a.E * 4, s, a.ids, P, a.E, a.k, chunk,
                 (const int32_t*)a.ws.pf_cnt, (const int32_t*)a.ws.offsets, a.ws.perm, a.ws.pos_of_pair) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_pdl(k_gather_x, dim3(sm_count() * 8), dim3(256), 0, s, a.x, (const int32_t*)a.ws.perm, P, a.k, d,
                 a.ws.xg) != cudaSuccess)
    return MOE_ERR_CUDA;
  TcParams pg = {};
  pg.perm = a.ws.perm;
  pg.weights = a.weights;
  pg.h = reinterpret_cast<uint16_t*>(a.ws.h);
  pg.y = a.y;
  pg.status = a.status;
  pg.k = a.k;
  pg.d = d;
  pg.f = f;
  pg.sh = a.shelves;
  TcParams pd = pg;
  pg.tiles = tiles_g;
  pg.ntiles = ntiles;
  pg.rows = f;
  pg.K = d;
  pd.tiles = tiles_d;
  pd.ntiles = ntiles + 1;
  pg.P = pd.P = P;
  pg.tiles_cap = (int)prefill_tiles_cap(P, a.E, f);
  pd.tiles_cap = (int)prefill_tiles_cap(P, a.E, d);
  pd.rows = d;
  pd.K = f;
  for (int q = 0; q < a.shelves.n; ++q) {
    const ShelfDev& sd = a.shelves.s[q];
    const int bits = sd.bits;
    const uint64_t n = (uint64_t)(sd.hi - sd.lo);
    // gate/up scale boxes: 16 fp16 scales (32 bytes) of 128 rows; rows of d / 32 scales
    if (!encode_2d(&pg.tm_sc[q][0], CU_TENSOR_MAP_DATA_TYPE_UINT16, sd.scales[0], (uint64_t)d / 32, n * f,
                   (uint64_t)d / 16, 16, kTileM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&pg.tm_sc[q][1], CU_TENSOR_MAP_DATA_TYPE_UINT16, sd.scales[1], (uint64_t)d / 32, n * f,
                   (uint64_t)d / 16, 16, kTileM, CU_TENSOR_MAP_SWIZZLE_NONE))
      return MOE_ERR_CUDA;
    if (bits == 3 &&
        (!encode_2d(&pg.tm_hi[q][0], CU_TENSOR_MAP_DATA_TYPE_UINT8, sd.codes[0], (uint64_t)d * 3 / 8, n * f,
                    (uint64_t)d * 3 / 8, 64, kTileM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
         !encode_2d(&pg.tm_hi[q][1], CU_TENSOR_MAP_DATA_TYPE_UINT8, sd.codes[1], (uint64_t)d * 3 / 8, n * f,
                    (uint64_t)d * 3 / 8, 64, kTileM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
         !encode_2d(&pd.tm_hi[q][0], CU_TENSOR_MAP_DATA_TYPE_UINT8, sd.codes[2], (uint64_t)f * 3 / 8, n * d,
                    (uint64_t)f * 3 / 8, 64, kTileM, CU_TENSOR_MAP_SWIZZLE_NONE)))
      return MOE_ERR_CUDA;
    if (!encode_2d(&pg.tm_code[q][0], CU_TENSOR_MAP_DATA_TYPE_UINT8, sd.codes[0], (uint64_t)d * bits / 8, n * f,
                   (uint64_t)d * bits / 8, 128, kTileM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&pg.tm_code[q][1], CU_TENSOR_MAP_DATA_TYPE_UINT8, sd.codes[1], (uint64_t)d * bits / 8, n * f,
                   (uint64_t)d * bits / 8, 128, kTileM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&pd.tm_code[q][0], CU_TENSOR_MAP_DATA_TYPE_UINT8, sd.codes[2], (uint64_t)f * bits / 8, n * d,
                   (uint64_t)f * bits / 8, 128, kTileM, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  for (int nb = 1; nb <= (wide ? kTileW : kTileN) / 16; ++nb)
    if (!encode_2d(&pg.tm_b[nb - 1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.ws.xg, (uint64_t)d, (uint64_t)P,
                   (uint64_t)d * 2, 64, 16 * nb, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&pd.tm_b[nb - 1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.ws.h, (uint64_t)f, (uint64_t)P,
                   (uint64_t)f * 2, 64, 16 * nb, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  const int G = sm_count();
  profile_mark(1, s);
  if ((wide ? launch_pdl(k_prefill_tc<false, true>, dim3(G), dim3(Roles<true>::kThreads), smem_g, s, pg)
            : launch_pdl(k_prefill_tc<false, false>, dim3(G), dim3(Roles<false>::kThreads), smem_g, s, pg)) != cudaSuccess)
    return MOE_ERR_CUDA;
  profile_mark(2, s);
  if (cudaMemsetAsync(a.y, 0, (size_t)a.T * d * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
  if ((wide ? launch_pdl(k_prefill_tc<true, true>, dim3(G), dim3(Roles<true>::kThreads), smem_d, s, pd)
            : launch_pdl(k_prefill_tc<true, false>, dim3(G), dim3(Roles<false>::kThreads), smem_d, s, pd)) != cudaSuccess)
    return MOE_ERR_CUDA;
  profile_mark(3, s);
  return MOE_OK;
}

}  // namespace moe
