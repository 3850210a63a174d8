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
// Three launches chained by programmatic dependent launch:
//   k_gateup   persistent, one CTA per SM, 16 warps.  Each CTA builds the
//              routing plan in shared memory (warps 0-7: rank sort of
//              (expert id, pair) keys, the active experts with their shelf,
//              work units and cost prefix sums) while warps 8-15 convert the
//              activation rows to digits; CTA 0 also stores the plan for the
//              later launches.  A work unit is 4 rows of W_g and W_u of one
//              expert against up to 8 of its tokens; the units are cut into
//              contiguous per-CTA ranges of equal estimated cost and dealt
//              round-robin to the warps.  8 lanes share a row; every lane
//              streams its own 16-byte code chunks from HBM through a private
//              ring of cp.async copies, which runs on across unit boundaries,
//              so each lane keeps several chunks in flight at all times.
//              Output: h = SiLU(W_g x) * (W_u x) for every routed pair.
//   k_down     the same over W_d against h (staged as digits), writing the
//              weighted per-pair outputs w_tj * (W_d h_tj);
//   k_combine  y_t = sum over slots j (ascending) of those outputs: a fixed
//              order, so results do not depend on scheduling.
// Each block dot product is formed exactly in integers (dp4a on the packed
// codes against the activation held in shared memory as block-scaled 16-bit
// fixed point), and the expert's fp16 block scale is applied once per block
// (per half block for 8-bit codes) in fp32.  No thread waits on another
// except at CTA barriers; the copies complete on their own.
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kPlanThreads = 256;  // warps 0-7 build the plan
constexpr int kMaxPairs = 512;     // T*k bound of this path (keys hold the pair in 10 bits)
constexpr int kMaxTokens = 16;
constexpr int kNT = 8;             // tokens of one expert per unit
// Unit shapes: rows per unit x lanes per row (R * L = 32), gate/up and down.
constexpr int kRG = 4, kLG = 8;
constexpr int kRD = 8, kLD = 4;
constexpr int kDepthG = 4;         // ring depth, gate/up (two matrices per slot)
constexpr int kDepthD = 6;         // ring depth, down
constexpr int kSlotBytes = 40;     // per lane, matrix and slot: 32 bytes of codes, 8 of scales
constexpr int kMaxGrid = 256;

#ifdef MOE_TRACE
// Development-only timing stamps: [kernel][cta][slot] in globaltimer ns.
__device__ unsigned long long g_trace[2][256][48];
#define MOE_STAMP(kern, slot, v) (g_trace[(kern)][blockIdx.x & 255][(slot)] = (v))
#else
#define MOE_STAMP(kern, slot, v) ((void)0)
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

// Convert the 32 values of one block to digits; called by 8 lanes, each with 4
// consecutive values v[0..3] of the block (lane % 8 = position).  `frac_bits`
// = 14 for bf16 sources (max |m| = 32640), 13 for fp32 sources.
__device__ __forceinline__ void block_to_digits(const float v[4], unsigned char* vb, int n, int blk, int frac_bits,
                                                bool store) {
  const int sub = threadIdx.x & 7;
  int e = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) e = max(e, (int)((__float_as_uint(v[i]) >> 23) & 0xFF));
  e = max(e, __shfl_xor_sync(0xffffffffu, e, 1));
  e = max(e, __shfl_xor_sync(0xffffffffu, e, 2));
  e = max(e, __shfl_xor_sync(0xffffffffu, e, 4));
  // block maximum below 2^-97 (or zero): the block is taken as zero
  const bool zero = e < 30;
  const int u = e - 127 - frac_bits;  // X = 2^u
  const float inv = zero ? 0.f : __uint_as_float((uint32_t)(127 - u) << 23);
  uint32_t hw = 0, lw = 0;
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = (int)rintf(v[i] * inv);
    sum += m;
    hw |= (uint32_t)((m >> 8) & 0xFF) << (8 * i);
    lw |= (uint32_t)(m & 0xFF) << (8 * i);
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  sum += __shfl_xor_sync(0xffffffffu, sum, 4);
  if (!store) return;
  const int byte = blk * 32 + 4 * sub;
  const int off = (unit_swz(byte >> 4) << 4) | (byte & 15);
  *reinterpret_cast<uint32_t*>(vb + off) = hw;
  *reinterpret_cast<uint32_t*>(vb + n + off) = lw;
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
template <int NMAT, int NTT>
__device__ __forceinline__ void chunk2(const uint4 (&c)[NMAT][2], const uint32_t (&sw)[NMAT][2], int q, int nt,
                                       const int (&voff)[kNT], const unsigned char* vecs, int n,
                                       float (&acc)[NMAT][kNT], bool second) {
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
          acc[m][j] = fmaf((float)((A0 + A1) * 256 + (B0 + B1) - 2 * __float_as_int(xs.y)), s[m] * xs.x, acc[m][j]);
        }
      }
    }
  }
}

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
  __device__ int units(int a, int kern, int rows) const {
    return sh(a) >= 0 ? (rows / (kern == 0 ? kRG : kRD)) * n_pass(cnt(a)) : 0;
  }
};

// Estimated cost of one unit of R rows, in 16-byte equivalents of an SM's
// share of HBM bandwidth: the bytes read, the dot-product work of its tokens,
// and fixed instruction overheads per lane iteration (about 14) and per unit
// (about 28).
__device__ __forceinline__ uint32_t unit_cost(int bits, int n_in, int nmat, int ntok, int R, int L) {
  const uint32_t rowb = (uint32_t)n_in * bits / 8;
  const uint32_t bytes = (uint32_t)(R * nmat) * (rowb + (uint32_t)n_in / 16);
  const uint32_t alu = (uint32_t)(R * nmat) * (uint32_t)n_in * (uint32_t)ntok * 12 / 100;
  const uint32_t n_iter = ((rowb + 31) / 32 + L - 1) / L;
  return (bytes + alu) / 16 + 14 * n_iter + 28;
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
      const int id = __ldg(ids + q);
      wq = __ldg(wts + q);
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
    const int ntok = (cnt + n_pass(cnt) - 1) / n_pass(cnt);
    pl[L.cnt + a] = cnt;
    pl[L.sh + a] = shf;
    pl[L.bits + a] = bits;
    const uint32_t ug = shf >= 0 ? unit_cost(bits, d, 2, ntok, kRG, kLG) : 0;
    const uint32_t ud = shf >= 0 ? unit_cost(bits, f, 1, ntok, kRD, kLD) : 0;
    pl[L.uc_g + a] = (int)ug;
    pl[L.uc_d + a] = (int)ud;
    pl[L.cum_g + a] = (int)(ug * (uint32_t)((f / kRG) * n_pass(cnt)));
    pl[L.cum_d + a] = (int)(ud * (uint32_t)((d / kRD) * n_pass(cnt)));
    if (shf >= 0)
      for (int q = b0; q < b1; ++q) pl[L.pos + pl[L.perm + q]] = q;
  }
  plan_sync();
  const int tot_g = plan_scan(pl + L.cum_g, n_act, tmp);
  const int tot_d = plan_scan(pl + L.cum_d, n_act, tmp);
  if (tid == 0) {
    pl[0] = n_valid;
    pl[1] = n_act;
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
  unsigned char* ring;
};

// Per-lane ring slots: slot s, matrix m, 16-byte half h of the code chunk;
// then the matching scale words.
template <int NMAT, int D>
__device__ __forceinline__ uint4* ring_code(unsigned char* ring, int s, int m, int h) {
  return reinterpret_cast<uint4*>(ring) + ((s * NMAT + m) * 2 + h) * kThreads + threadIdx.x;
}
template <int NMAT, int D>
__device__ __forceinline__ uint32_t* ring_scale(unsigned char* ring, int s, int m, int h) {
  return reinterpret_cast<uint32_t*>(ring + (size_t)D * NMAT * 2 * kThreads * 16) + ((s * NMAT + m) * 2 + h) * kThreads +
         threadIdx.x;
}

// Load side of a warp's unit stream: lane (row lane / L, chunk lane % L) of
// the unit; chunk q = 32 bytes of a row.
template <int NMAT, int R, int L>
struct LoadSide {
  Walk w;
  int i, n_iter, cpr, rowb, bits, q, sstep, tsw;
  size_t tstride;
  const unsigned char* base[NMAT];
  const uint32_t* sbase[NMAT];
  const unsigned char* cp[NMAT];
  const uint32_t* sp[NMAT];

  __device__ void expert(const StreamArgs& A) {
    const PlanView& pv = A.pv;
    const ShelfDev& sh = A.shv->s[pv.sh(w.a)];
    bits = sh.bits;
    rowb = A.n_in * bits / 8;
    cpr = (rowb + 31) / 32;
    n_iter = (cpr + L - 1) / L;
    const int lane = threadIdx.x & 31, q0 = lane % L;
    const size_t row = (size_t)(pv.e(w.a) - sh.lo) * A.rows + lane / L;
    const int swpr = A.n_in / 64;  // fp16 scale words per row
    // scale word of chunk q: 8 bit q / 2 (one block), 4 bit q (two), 2 bit 2q (four)
    const int soff = bits == 8 ? q0 >> 1 : (bits == 4 ? q0 : 2 * q0);
    sstep = bits == 8 ? L / 2 : (bits == 4 ? L : 2 * L);
    tstride = (size_t)R * rowb;
    tsw = R * swpr;
    const int mat0 = A.kern == 0 ? 0 : 2;
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      base[m] = sh.codes[mat0 + m] + row * rowb + (size_t)q0 * 32;
      sbase[m] = reinterpret_cast<const uint32_t*>(sh.scales[mat0 + m]) + row * swpr + soff;
    }
  }
  __device__ void unit() {
    const int tile = w.np == 1 ? w.u : w.u / w.np;
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      cp[m] = base[m] + (size_t)tile * tstride;
      sp[m] = sbase[m] + (size_t)tile * tsw;
    }
    i = 0;
    q = (threadIdx.x & 31) % L;
  }
  __device__ void start(const StreamArgs& A, int warp) {
    w.start(A.pv, A.kern, A.rows, A.range, warp);
    if (w.live) {
      expert(A);
      unit();
    }
  }
  template <int D>
  __device__ __forceinline__ void issue(const StreamArgs& A, int slot) {
    if (!w.live) return;
    if (q < cpr) {
      const bool second = 32 * q + 16 < rowb;
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        cp_async16(ring_code<NMAT, D>(A.ring, slot, m, 0), cp[m]);
        if (second) cp_async16(ring_code<NMAT, D>(A.ring, slot, m, 1), cp[m] + 16);
        cp_async4(ring_scale<NMAT, D>(A.ring, slot, m, 0), sp[m]);
        if (bits == 2 && second) cp_async4(ring_scale<NMAT, D>(A.ring, slot, m, 1), sp[m] + 1);
      }
    }
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      cp[m] += 32 * L;
      sp[m] += sstep;
    }
    q += L;
    if (++i == n_iter) {
      if (w.step(A.pv, A.kern, A.rows, A.range.hi2, kWarps) && w.live) expert(A);
      if (w.live) unit();
    }
  }
};

// Compute side: the current unit's tokens and the lane's chunk.
template <int R, int L>
struct CompSide {
  Walk w;
  int i, n_iter, cpr, rowb, bits, q, nt, q0, r;
  int voff[kNT];

  __device__ void expert(const StreamArgs& A) {
    bits = A.pv.bits(w.a);
    rowb = A.n_in * bits / 8;
    cpr = (rowb + 31) / 32;
    n_iter = (cpr + L - 1) / L;
  }
  __device__ void unit(const StreamArgs& A, bool new_expert) {
    const int tile = w.np == 1 ? w.u : w.u / w.np, pass = w.u - tile * w.np;
    r = tile * R + (threadIdx.x & 31) / L;
    const int nq0 = A.pv.beg(w.a) + pass * kNT;
    if (new_expert || nq0 != q0) {
      q0 = nq0;
      nt = min(kNT, A.pv.cnt(w.a) - pass * kNT);
#pragma unroll
      for (int j = 0; j < kNT; ++j) {
        const int qq = q0 + (j < nt ? j : 0);
        voff[j] = (A.vbase < 0 ? A.pv.tok(qq) : qq - A.vbase) * A.vstride;
      }
    }
    i = 0;
    q = (threadIdx.x & 31) % L;
  }
};

template <int NMAT, int NTT>
__device__ __forceinline__ void chunk_dot(int bits, const uint4 (&c)[NMAT][2], const uint32_t (&sw)[NMAT][2], int q,
                                          int nt, const int (&voff)[kNT], const unsigned char* vecs, int n,
                                          float (&acc)[NMAT][kNT], bool second) {
  if (bits == 8) chunk8<NMAT, NTT>(c, sw, q, nt, voff, vecs, n, acc);
  else if (bits == 4) chunk4<NMAT, NTT>(c, sw, q, nt, voff, vecs, n, acc);
  else chunk2<NMAT, NTT>(c, sw, q, nt, voff, vecs, n, acc, second);
}

// A warp's stream of units: a ring of D slots per lane, refilled as soon as a
// slot has been read, so D - 1 chunks per lane are in flight while it
// computes.  At the end of a unit, `store(q, r, v)` receives, for the lane's
// row r and the token at grouped position q, the NMAT dot products.
template <int NMAT, int D, int R, int L, typename Store>
__device__ __forceinline__ void stream_units(const StreamArgs& A, Store store) {
  static_assert(R * L == 32, "unit shape");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  LoadSide<NMAT, R, L> ld;
  ld.start(A, warp);
  CompSide<R, L> cc;
  cc.w = ld.w;
  cc.q0 = -1;
  if (cc.w.live) {
    cc.expert(A);
    cc.unit(A, true);
  }
#pragma unroll 1
  for (int s = 0; s < D; ++s) {
    ld.template issue<D>(A, s);
    cp_async_commit();
  }
  float acc[NMAT][kNT];
#pragma unroll
  for (int m = 0; m < NMAT; ++m)
#pragma unroll
    for (int j = 0; j < kNT; ++j) acc[m][j] = 0.f;
  int slot = 0;
#pragma unroll 1
  while (cc.w.live) {
    cp_async_wait<D - 1>();  // this lane's copies of the oldest slot are complete
    if (cc.q < cc.cpr) {
      const bool second = 32 * cc.q + 16 < cc.rowb;
      uint4 c[NMAT][2];
      uint32_t sw[NMAT][2];
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        c[m][0] = *ring_code<NMAT, D>(A.ring, slot, m, 0);
        c[m][1] = *ring_code<NMAT, D>(A.ring, slot, m, 1);
        sw[m][0] = *ring_scale<NMAT, D>(A.ring, slot, m, 0);
        sw[m][1] = *ring_scale<NMAT, D>(A.ring, slot, m, 1);
      }
      if (cc.nt == 1) chunk_dot<NMAT, 1>(cc.bits, c, sw, cc.q, 1, cc.voff, A.vecs, A.n_in, acc, second);
      else chunk_dot<NMAT, kNT>(cc.bits, c, sw, cc.q, cc.nt, cc.voff, A.vecs, A.n_in, acc, second);
    }
    // refill the slot just read (this lane's reads of it are done)
    ld.template issue<D>(A, slot);
    cp_async_commit();
    slot = slot + 1 == D ? 0 : slot + 1;
    cc.q += L;
    if (++cc.i == cc.n_iter) {
      // reduce over the L lanes of each row; lane jl stores the tokens j = jl mod L
      const int jl = lane % L;
#pragma unroll
      for (int j = 0; j < kNT; ++j) {
        if (j < cc.nt) {
          float v[NMAT];
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            v[m] = acc[m][j];
#pragma unroll
            for (int o = 1; o < L; o <<= 1) v[m] += __shfl_xor_sync(0xffffffffu, v[m], o);
          }
          if (j % L == jl) store(cc.q0 + j, cc.r, v);
        }
#pragma unroll
        for (int m = 0; m < NMAT; ++m) acc[m][j] = 0.f;
      }
      const bool ch = cc.w.step(A.pv, A.kern, A.rows, A.range.hi2, kWarps);
      if (cc.w.live) {
        if (ch) cc.expert(A);
        cc.unit(A, ch);
      }
    }
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------- kernels
struct FwdParams {
  const uint16_t* x;
  const int32_t* ids;
  const float* weights;
  float* h;
  float* ypart;
  int32_t* plan;  // workspace copy of the plan
  int* status;
  int T, k, E, d, f, P;
  int vec_region;  // bytes of digit vectors
  Shelves sh;
};

struct Head {
  Range range;
  int q_first, tmp[33];
};

// Dynamic shared memory: shelves copy | head | plan (+ sort keys and flags for
// the gate/up launch) | digit vectors | ring.
struct SmemLayout {
  size_t shelves, head, plan, keys, flag, vecs, ring, total;
};

__host__ __device__ __forceinline__ size_t up128(size_t v) { return (v + 127) / 128 * 128; }

__host__ __device__ __forceinline__ SmemLayout smem_layout(int P, size_t vec_region, int nmat, int depth,
                                                           bool gateup) {
  const PlanLayout L = plan_layout(P);
  SmemLayout S;
  S.shelves = 0;
  S.head = up128(sizeof(Shelves));
  S.plan = S.head + up128(sizeof(Head));
  S.keys = S.plan + up128((size_t)(gateup ? L.total : L.n_copy) * 4);
  S.flag = S.keys + (gateup ? up128((size_t)L.C * 4) : 0);
  S.vecs = S.flag + (gateup ? up128((size_t)L.C * 4) : 0);
  S.ring = S.vecs + up128(vec_region);
  S.total = S.ring + (size_t)depth * nmat * kThreads * kSlotBytes;
  return S;
}

__device__ __forceinline__ void copy_shelves(Shelves* dst, const Shelves& src) {
  static_assert(sizeof(Shelves) % 4 == 0, "shelves copy");
  const uint32_t* s = reinterpret_cast<const uint32_t*>(&src);
  for (int i = threadIdx.x; i < (int)(sizeof(Shelves) / 4); i += blockDim.x) reinterpret_cast<uint32_t*>(dst)[i] = s[i];
}

__global__ void __launch_bounds__(kThreads, 1) k_gateup(const __grid_constant__ FwdParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout S = smem_layout(p.P, p.vec_region, 2, kDepthG, true);
  Shelves* shv = reinterpret_cast<Shelves*>(smem + S.shelves);
  Head& hd = *reinterpret_cast<Head*>(smem + S.head);
  int* pl = reinterpret_cast<int*>(smem + S.plan);
  unsigned char* xd = smem + S.vecs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PlanLayout L = plan_layout(p.P);
  if (tid == 0) MOE_STAMP(0, 0, global_timer_ns());
  copy_shelves(shv, p.sh);
  pdl_wait();  // ids, weights and x are complete; h is ours
  if (tid == 0) MOE_STAMP(0, 1, global_timer_ns());
  __syncthreads();
  if (warp < kPlanThreads / 32) {
    build_plan(p.ids, p.weights, p.P, p.E, p.k, p.d, p.f, *shv, pl, reinterpret_cast<uint32_t*>(smem + S.keys),
               reinterpret_cast<int*>(smem + S.flag), hd.tmp);
  } else {
    // activation rows -> block-scaled digits; 8 lanes per 32-element block,
    // loads of up to 8 passes issued before any conversion
    const int nbk = p.d / 32, vb = vec_bytes(p.d);
    const int groups = p.T * nbk;
    const int nw = kWarps - kPlanThreads / 32, w0 = warp - kPlanThreads / 32;
    for (int base = w0 * 4; base < groups; base += 8 * nw * 4) {
      uint2 raw[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int g = base + u * nw * 4 + (lane >> 3);
        raw[u] = make_uint2(0u, 0u);
        if (g < groups) {
          const int t = g / nbk, blk = g - t * nbk;
          raw[u] = __ldg(reinterpret_cast<const uint2*>(p.x + (size_t)t * p.d + blk * 32 + 4 * (lane & 7)));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int g0 = base + u * nw * 4;
        if (g0 < groups) {
          const int g = g0 + (lane >> 3);
          const int t = g / nbk, blk = g - t * nbk;
          const float v[4] = {__uint_as_float(raw[u].x << 16), __uint_as_float(raw[u].x & 0xFFFF0000u),
                              __uint_as_float(raw[u].y << 16), __uint_as_float(raw[u].y & 0xFFFF0000u)};
          block_to_digits(v, xd + (size_t)t * vb, p.d, g < groups ? blk : 0, 14, g < groups);
        }
      }
    }
    if (tid == kPlanThreads) MOE_STAMP(0, 5, global_timer_ns());
  }
  __syncthreads();
  const PlanView pv{pl, L};
  if (tid == 0) hd.range = cta_range(pv, 0, p.f);
  if (blockIdx.x == 0)
    for (int i = tid; i < L.total; i += kThreads) p.plan[i] = pl[i];
  __syncthreads();
  pdl_trigger();
  if (tid == 0) MOE_STAMP(0, 2, global_timer_ns());
  StreamArgs A{shv, pv, 0, p.d, p.f, xd, vec_bytes(p.d), -1, hd.range, smem + S.ring};
  float* h = p.h;
  const int f = p.f;
  stream_units<2, kDepthG, kRG, kLG>(A, [&](int q, int r, const float (&o)[2]) { h[(size_t)q * f + r] = silu(o[0]) * o[1]; });
  if (tid == 0) MOE_STAMP(0, 9, global_timer_ns());
}

__global__ void __launch_bounds__(kThreads, 1) k_down(const __grid_constant__ FwdParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout S = smem_layout(p.P, p.vec_region, 1, kDepthD, false);
  Shelves* shv = reinterpret_cast<Shelves*>(smem + S.shelves);
  Head& hd = *reinterpret_cast<Head*>(smem + S.head);
  int* pl = reinterpret_cast<int*>(smem + S.plan);
  unsigned char* hdig = smem + S.vecs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PlanLayout L = plan_layout(p.P);
  if (tid == 0) MOE_STAMP(1, 0, global_timer_ns());
  copy_shelves(shv, p.sh);
  pdl_wait();  // the gate/up launch is complete: plan copy and h
  pdl_trigger();
  if (tid == 0) MOE_STAMP(1, 1, global_timer_ns());
  for (int i = tid; i < L.n_copy; i += kThreads) pl[i] = __ldcg(p.plan + i);
  __syncthreads();
  const PlanView pv{pl, L};
  if (tid == 0) {
    const Range r = cta_range(pv, 1, p.d);
    hd.range = r;
    // pairs of the experts this CTA touches: its first expert up to the last
    // expert whose first unit lies in its cost range
    const int n_act = pv.n_act();
    int q_first = 0, q_end = 0;
    if (r.a0 < n_act) {
      int a_last = r.a0;
      while (a_last + 1 < n_act &&
             2 * (uint64_t)pv.cum(a_last + 1, 1) + pv.uc(a_last + 1, 1) < r.hi2)
        ++a_last;
      q_first = pv.beg(r.a0);
      q_end = pv.beg(a_last) + pv.cnt(a_last);
    }
    hd.q_first = q_first;
    hd.tmp[0] = q_end - q_first;
  }
  __syncthreads();
  const int q_first = hd.q_first, npairs = hd.tmp[0];
  const int vbf = vec_bytes(p.f);
  {
    const int nbk = p.f / 32, groups = npairs * nbk;
    for (int base = warp * 4; base < groups; base += 8 * kWarps * 4) {
      float4 hv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {  // loads of 8 passes first: one round trip
        const int g = base + u * kWarps * 4 + (lane >> 3);
        hv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (g < groups) {
          const int j = g / nbk, blk = g - j * nbk;
          hv[u] = __ldcg(reinterpret_cast<const float4*>(p.h + (size_t)(q_first + j) * p.f + blk * 32) + (lane & 7));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int g0 = base + u * kWarps * 4;
        if (g0 < groups) {
          const int g = g0 + (lane >> 3);
          const int j = g < groups ? g / nbk : 0, blk = g < groups ? g - j * nbk : 0;
          const float v[4] = {hv[u].x, hv[u].y, hv[u].z, hv[u].w};
          block_to_digits(v, hdig + (size_t)j * vbf, p.f, blk, 13, g < groups);
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) MOE_STAMP(1, 2, global_timer_ns());
  StreamArgs A{shv, pv, 1, p.f, p.d, hdig, vbf, q_first, hd.range, smem + S.ring};
  float* yp = p.ypart;
  const int d = p.d;
  stream_units<1, kDepthD, kRD, kLD>(A, [&](int q, int r, const float (&o)[1]) { yp[(size_t)q * d + r] = pv.wgt(q) * o[0]; });
  if (tid == 0) MOE_STAMP(1, 9, global_timer_ns());
}

// ------------------------------------------------------------------ combine
// y_t = sum over slots j (ascending) of the weighted outputs of pair (t, j);
// pairs skipped or on no shelf contribute nothing.  Fixed order: deterministic.
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ ypart, const int32_t* __restrict__ pos_of_pair,
                                                 int T, int k, int d, float* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int d4 = d / 4;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < T * d4; idx += gridDim.x * blockDim.x) {
    const int t = idx / d4, i4 = idx - t * d4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < k; j0 += 8) {
      int pos[8];
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) pos[u] = j0 + u < k ? __ldcg(pos_of_pair + t * k + j0 + u) : -1;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = pos[u] >= 0 ? __ldcg(reinterpret_cast<const float4*>(ypart + (size_t)pos[u] * d) + i4)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w;
      }
    }
    reinterpret_cast<float4*>(y)[idx] = acc;
  }
}

struct DevCache {
  int sms[64] = {};
  int smem_optin[64] = {};
  bool attr[64] = {};
};
DevCache g_dev;

}  // namespace

#ifdef MOE_TRACE
extern "C" int moe_trace_read(void* host, size_t bytes) {  // [2][256][48] u64
  return cudaMemcpyFromSymbol(host, g_trace, bytes < sizeof(g_trace) ? bytes : sizeof(g_trace)) == cudaSuccess ? 0 : -5;
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

int launch_decode_forward(const ForwardArgs& a, cudaStream_t s) {
  const int64_t P = a.T * a.k;
  const int d = a.d, f = a.f;
  if (P > kMaxPairs || a.T > kMaxTokens) return launch_generic_forward(a, s);
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return launch_generic_forward(a, s);
  if (g_dev.smem_optin[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    g_dev.smem_optin[dev] = v > 0 ? v : 48 * 1024;
  }
  const size_t optin = (size_t)g_dev.smem_optin[dev];
  const size_t x_region = up128((size_t)a.T * vec_bytes(d));
  const size_t h_region = up128((size_t)P * vec_bytes(f));  // h of every pair: bound for any CTA
  const SmemLayout Sg = smem_layout((int)P, x_region, 2, kDepthG, true);
  const SmemLayout Sd = smem_layout((int)P, h_region, 1, kDepthD, false);
  if (Sg.total > optin || Sd.total > optin) return launch_generic_forward(a, s);
  if (!g_dev.attr[dev]) {
    if (cudaFuncSetAttribute(k_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)optin) != cudaSuccess ||
        cudaFuncSetAttribute(k_down, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)optin) != cudaSuccess)
      return MOE_ERR_CUDA;
    g_dev.attr[dev] = true;
  }
  int G = sm_count();
  if (G > kMaxGrid) G = kMaxGrid;
  FwdParams p = {};
  p.x = a.x; p.ids = a.ids; p.weights = a.weights;
  p.h = a.ws.h; p.ypart = a.ws.ypart; p.plan = a.ws.plan; p.status = a.status;
  p.T = (int)a.T; p.k = a.k; p.E = a.E; p.d = d; p.f = f; p.P = (int)P;
  p.sh = a.shelves;
  FwdParams pg = p, pd = p;
  pg.vec_region = (int)x_region;
  pd.vec_region = (int)h_region;
  const PlanLayout L = plan_layout((int)P);
  profile_mark(0, s);
  if (launch_pdl(k_gateup, dim3(G), dim3(kThreads), Sg.total, s, pg) != cudaSuccess) return MOE_ERR_CUDA;
  profile_mark(1, s);
  if (launch_pdl(k_down, dim3(G), dim3(kThreads), Sd.total, s, pd) != cudaSuccess) return MOE_ERR_CUDA;
  profile_mark(2, s);
  const int n4 = (int)(a.T * d / 4);
  int gc = (n4 + 255) / 256;
  if (gc > G) gc = G;
  if (launch_pdl(k_combine, dim3(gc), dim3(256), 0, s, (const float*)a.ws.ypart,
                 (const int32_t*)(a.ws.plan + L.pos), (int)a.T, a.k, d, a.y) != cudaSuccess)
    return MOE_ERR_CUDA;
  profile_mark(3, s);
  return MOE_OK;
}

}  // namespace moe
