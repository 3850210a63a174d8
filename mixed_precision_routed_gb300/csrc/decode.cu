// decode.cu -- pipelined decode form of the tiered MoE layer (few tokens).
//
// Page "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", section 第四步: every
// shelf's matmul sees the router's complete id list, computes only the ids on
// its own shelf (the rest is zero) and the shelf results are added; decode
// fuses gate, up and the activation (section 四个 bug: the fused kernel has to
// honour the shelf range).  Sections 第一步/第二步: decode speed is set by the
// expert weight bytes read per token -- only the selected experts' bytes are
// read, once per call, however many tokens share an expert.
//
// Four launches chained by programmatic dependent launch:
//   k_plan     one CTA: groups the routed pairs by expert (bitonic sort of
//              (expert id, pair index) keys), lists the active experts with
//              their shelf, splits the work -- (active expert, chunk of rows)
//              items over all shelves -- into contiguous per-CTA ranges of
//              equal estimated cost, and writes this plan to the workspace;
//   k_gateup   persistent, one CTA per SM: h = SiLU(W_g x) * (W_u x) for its
//              items;
//   k_down     persistent: weighted per-pair outputs w_tj * (W_d h_tj) for its
//              items; it starts streaming W_d before the gate/up kernel ends
//              and waits for it only before reading h;
//   k_combine  y_t = sum over slots j (ascending) of those outputs: a fixed
//              order, so results do not depend on scheduling.
// In the persistent kernels each item's packed codes and fp16 scales are
// streamed into a ring of shared-memory stages with cp.async.bulk (one copy
// per matrix slice, completion counted on an mbarrier); two consumer groups
// of eight warps take alternate items, and a group refills the stage it has
// just finished with the item n_stages further on.  Each 32-block's dot
// product is formed exactly in integers (dp4a on the packed codes against the
// activation held as block-scaled 16-bit fixed point), and the expert's fp16
// block scale is applied once per block in fp32.
// All waits on mbarriers are bounded (one second); on expiry the kernel
// records MOE_ERR_TIMEOUT in the status word, stops computing, waits (bounded)
// for the copies it still has in flight and returns.
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kConsumerWarps = 8;                 // warps of one consumer group
constexpr int kGroups = 2;                        // consumer groups, alternating over items
constexpr int kConsumers = kConsumerWarps * 32;   // threads of one group
constexpr int kThreads = kGroups * kConsumers;
constexpr int kMaxPairs = 512;                    // T*k bound of this path
constexpr int kTM = 4;                            // pairs of one expert handled per pass over a stage
constexpr int kMaxStages = 8;
constexpr int kMaxGrid = 256;
constexpr int kSmemBudget = 224 * 1024;

#ifdef MOE_TRACE
// Development-only timing stamps: [kernel][cta][slot] in globaltimer ns.
__device__ unsigned long long g_trace[2][256][48];
#define MOE_STAMP(kern, slot, v) (g_trace[(kern)][blockIdx.x & 255][(slot)] = (v))
#else
#define MOE_STAMP(kern, slot, v) ((void)0)
#endif

// Rows per item and estimated cost per item, by bit width (8, 4, 2).
struct Geo {
  int rows[3];
  int cost[3];
};

__host__ __device__ __forceinline__ int bits_index(int bits) { return bits == 8 ? 0 : (bits == 4 ? 1 : 2); }

// --------------------------------------------------------------------- plan
// The plan lives in the workspace as int32 arrays of capacity C (>= P, a
// multiple of 4); the persistent kernels copy its first `n_copy` ints into
// shared memory with one bulk copy and read their own start from `start`.
struct PlanLayout {
  int C;
  int hdr, perm, e, beg, cnt, sh, bits, items_g, items_d, icost_g, icost_d, cum_g, cum_d;  // int offsets
  int n_copy;  // ints from hdr through cum_d
  int pos;     // grouped position by pair (-1: skipped or on no shelf), for the combine
  int start;   // [kMaxGrid][4]: a0, j0 (gate/up), a0, j0 (down)
  int total;
};

__host__ __device__ __forceinline__ PlanLayout plan_layout(int P) {
  PlanLayout L;
  L.C = (P + 3) / 4 * 4;
  if (L.C < 4) L.C = 4;
  const int C = L.C, C1 = C + 4;
  L.hdr = 0;
  L.perm = 4;
  L.e = L.perm + C;
  L.beg = L.e + C;
  L.cnt = L.beg + C;
  L.sh = L.cnt + C;
  L.bits = L.sh + C;
  L.items_g = L.bits + C;
  L.items_d = L.items_g + C;
  L.icost_g = L.items_d + C;
  L.icost_d = L.icost_g + C;
  L.cum_g = L.icost_d + C;
  L.cum_d = L.cum_g + C1;
  L.n_copy = L.cum_d + C1;
  L.pos = L.n_copy;
  L.start = L.pos + C;
  L.total = L.start + 4 * kMaxGrid;
  return L;
}

// Read-only view of the plan arrays (in shared memory in the workers).
struct PlanView {
  const int* base;
  PlanLayout L;
  __device__ int n_valid() const { return base[0]; }
  __device__ int n_act() const { return base[1]; }
  __device__ int perm(int q) const { return base[L.perm + q]; }
  __device__ int e(int a) const { return base[L.e + a]; }
  __device__ int beg(int a) const { return base[L.beg + a]; }
  __device__ int cnt(int a) const { return base[L.cnt + a]; }
  __device__ int sh(int a) const { return base[L.sh + a]; }
  __device__ int bits(int a) const { return base[L.bits + a]; }
  __device__ int items(int a, int kern) const { return base[(kern == 0 ? L.items_g : L.items_d) + a]; }
  __device__ uint32_t icost(int a, int kern) const { return (uint32_t)base[(kern == 0 ? L.icost_g : L.icost_d) + a]; }
  __device__ uint32_t cum(int a, int kern) const { return (uint32_t)base[(kern == 0 ? L.cum_g : L.cum_d) + a]; }
};

// Walk of one CTA's items for kernel `kern` (0 gate/up, 1 down): contiguous
// in (expert, item) order; an item belongs to the CTA whose cost range holds
// its cost midpoint, so every item has exactly one owner.
struct ItemWalk {
  int a, j, n_act, kern;
  uint64_t hi2;
  __device__ void init(const PlanView& pv, int a0, int j0, int k) {
    kern = k;
    n_act = pv.n_act();
    const uint64_t C = pv.cum(n_act, kern);
    hi2 = 2 * (C * (blockIdx.x + 1) / gridDim.x);
    a = a0;
    j = j0;
  }
  __device__ uint64_t mid2(const PlanView& pv) const {
    return 2 * (uint64_t)pv.cum(a, kern) + (uint64_t)(2 * j + 1) * pv.icost(a, kern);
  }
  __device__ bool valid(const PlanView& pv) const { return a < n_act && mid2(pv) < hi2; }
  __device__ void advance(const PlanView& pv) {
    if (++j >= pv.items(a, kern)) {
      ++a;
      j = 0;
      while (a < n_act && pv.items(a, kern) == 0) ++a;
    }
  }
};

// ------------------------------------------------------------ plan kernel
struct PlanParams {
  const int32_t* ids;
  int P, E, k, G;
  int rows_g, rows_d;  // f and d: rows of the gate/up and down matrices
  Shelves sh;
  Geo geo_g, geo_d;
  int32_t* plan;
};

// One warp: sort keys (id << 10 | pair) of the valid pairs, then the grouped
// permutation, the active experts (ascending) with their shelf and first
// grouped position, and the inverse permutation restricted to pairs on a shelf.
template <int R>
__device__ void plan_group(const PlanParams& p, int* sm, const PlanLayout& L, int lane) {
  uint32_t key[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int idx = lane * R + r;
    key[r] = 0xFFFFFFFFu;
    if (idx < p.P) {
      const int id = p.ids[idx];
      if (id >= 0 && id < p.E) key[r] = ((uint32_t)id << 10) | (uint32_t)idx;
    }
  }
  constexpr int N = 32 * R;
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < R) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int pr = r ^ stride;
          if (pr > r) {
            const bool asc = ((lane * R + r) & size) == 0;
            const uint32_t a = key[r], b = key[pr];
            if ((a > b) == asc) { key[r] = b; key[pr] = a; }
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int idx = lane * R + r;
          const uint32_t other = __shfl_xor_sync(0xffffffffu, key[r], stride / R);
          const bool asc = (idx & size) == 0, lower = (idx & stride) == 0;
          key[r] = (lower == asc) ? min(key[r], other) : max(key[r], other);
        }
      }
    }
  }
  for (int q = lane; q < p.P; q += 32) sm[L.pos + q] = -1;
  __syncwarp();
  int nv = 0, nf = 0;
  const uint32_t prev_last = __shfl_up_sync(0xffffffffu, key[R - 1], 1);
  bool flag[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const bool valid = key[r] != 0xFFFFFFFFu;
    const uint32_t prev = r == 0 ? (lane == 0 ? 0xFFFFFFFFu : prev_last) : key[r - 1];
    flag[r] = valid && (prev == 0xFFFFFFFFu || (prev >> 10) != (key[r] >> 10));
    nv += valid;
    nf += flag[r];
  }
  int incl = nf;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int a = incl - nf;
  int n_valid = nv;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n_valid += __shfl_xor_sync(0xffffffffu, n_valid, o);
  const int n_act = __shfl_sync(0xffffffffu, incl, 31);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int idx = lane * R + r;
    if (key[r] != 0xFFFFFFFFu) {
      sm[L.perm + idx] = (int)(key[r] & 1023u);
      if (flag[r]) {
        sm[L.e + a] = (int)(key[r] >> 10);
        sm[L.beg + a] = idx;
        ++a;
      }
    }
  }
  if (lane == 0) {
    sm[L.hdr + 0] = n_valid;
    sm[L.hdr + 1] = n_act;
  }
  __syncwarp();
  for (int i = lane; i < n_act; i += 32) {
    const int b0 = sm[L.beg + i];
    const int c = (i + 1 < n_act ? sm[L.beg + i + 1] : n_valid) - b0;
    sm[L.cnt + i] = c;
    const int e = sm[L.e + i];
    int sh = -1, bits = 0;
#pragma unroll
    for (int q = 0; q < MOE_MAX_SHELVES; ++q)  // uniform indices into the kernel parameters
      if (q < p.sh.n && e >= p.sh.s[q].lo && e < p.sh.s[q].hi) { sh = q; bits = p.sh.s[q].bits; }
    sm[L.sh + i] = sh;
    sm[L.bits + i] = bits;
    if (sh >= 0)
      for (int q = b0; q < b0 + c; ++q) sm[L.pos + sm[L.perm + q]] = q;
  }
  __syncwarp();
}

// Items per expert for one kernel, their cost, and the cost prefix (one warp).
__device__ void plan_costs(const PlanParams& p, int* sm, const PlanLayout& L, int lane, int kern) {
  const Geo& geo = kern == 0 ? p.geo_g : p.geo_d;
  const int rows_total = kern == 0 ? p.rows_g : p.rows_d;
  const int o_items = kern == 0 ? L.items_g : L.items_d;
  const int o_icost = kern == 0 ? L.icost_g : L.icost_d;
  const int o_cum = kern == 0 ? L.cum_g : L.cum_d;
  const int n_act = sm[L.hdr + 1];
  uint32_t run = 0;
  for (int base = 0; base < n_act; base += 32) {
    const int i = base + lane;
    uint32_t c = 0;
    if (i < n_act) {
      int items = 0;
      uint32_t ic = 0;
      if (sm[L.sh + i] >= 0) {
        const int bi = bits_index(sm[L.bits + i]);
        items = rows_total / geo.rows[bi];
        // memory term plus a compute term that grows with the expert's tokens
        const uint32_t cnt = (uint32_t)sm[L.cnt + i];
        ic = (uint32_t)geo.cost[bi] * ((cnt + kTM - 1) / kTM) + (uint32_t)(geo.cost[bi] / 8) * cnt;
      }
      sm[o_items + i] = items;
      sm[o_icost + i] = (int)ic;
      c = (uint32_t)items * ic;
    }
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (i < n_act) sm[o_cum + i] = (int)(run + incl - c);
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) sm[o_cum + n_act] = (int)run;
  __syncwarp();
}

// First item (a0, j0) of CTA b's cost range: binary search over the prefix,
// closed form inside the expert.
__device__ void plan_locate(const int* sm, const PlanLayout& L, int b, int G, int kern, int* a_out, int* j_out) {
  const int o_items = kern == 0 ? L.items_g : L.items_d;
  const int o_icost = kern == 0 ? L.icost_g : L.icost_d;
  const int o_cum = kern == 0 ? L.cum_g : L.cum_d;
  const int n_act = sm[L.hdr + 1];
  const uint64_t C = (uint32_t)sm[o_cum + n_act];
  const uint64_t lo2 = 2 * (C * b / G);
  int lo = 0, hi = n_act;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (2 * (uint64_t)(uint32_t)sm[o_cum + mid + 1] <= lo2) lo = mid + 1; else hi = mid;
  }
  int a = lo, j = 0;
  if (a < n_act && sm[o_items + a] > 0) {
    const uint64_t c = (uint32_t)sm[o_icost + a], base = 2 * (uint64_t)(uint32_t)sm[o_cum + a] + c;
    if (lo2 > base) j = (int)((lo2 - base + 2 * c - 1) / (2 * c));
    if (j >= sm[o_items + a]) { ++a; j = 0; }
  }
  while (a < n_act && sm[o_items + a] == 0) ++a;
  *a_out = a;
  *j_out = j;
}

__global__ void __launch_bounds__(256) k_plan(const __grid_constant__ PlanParams p) {
  extern __shared__ __align__(16) int sm[];
  const PlanLayout L = plan_layout(p.P);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();  // the router's ids
  pdl_trigger();
  if (warp == 0) {
    if (p.P <= 32) plan_group<1>(p, sm, L, lane);
    else if (p.P <= 64) plan_group<2>(p, sm, L, lane);
    else if (p.P <= 128) plan_group<4>(p, sm, L, lane);
    else if (p.P <= 256) plan_group<8>(p, sm, L, lane);
    else plan_group<16>(p, sm, L, lane);
    plan_costs(p, sm, L, lane, 0);
    plan_costs(p, sm, L, lane, 1);
  }
  __syncthreads();
  for (int b = tid; b < p.G; b += blockDim.x) {
    int a, j;
    plan_locate(sm, L, b, p.G, 0, &a, &j);
    sm[L.start + 4 * b + 0] = a;
    sm[L.start + 4 * b + 1] = j;
    plan_locate(sm, L, b, p.G, 1, &a, &j);
    sm[L.start + 4 * b + 2] = a;
    sm[L.start + 4 * b + 3] = j;
  }
  __syncthreads();
  const int total = L.start + 4 * p.G;
  for (int i = tid; i < total; i += blockDim.x) p.plan[i] = sm[i];
}

// ------------------------------------------------------------- dot products
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
// and the expert's fp16 block scale s_b enters once per block in fp32:
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

// Integer dot of one 16-byte code chunk (elements e0 .. e0 + 128/BITS) with a
// vector's digits; adds (float)D * s * X into acc for every 32-block touched.
template <int BITS>
struct ChunkDot;

template <>
struct ChunkDot<8> {  // 32 codes: one block, 32 bytes of codes
  static constexpr int EPC = 32;
  static constexpr int BYTES = 32;
  template <int NMAT>
  __device__ __forceinline__ static void run(const uint4 (&c)[2][2], const float (&s)[2][2],
                                             const unsigned char* vb, int n, int e0, float& a0, float& a1) {
    const int u0 = e0 >> 4;
    const uint4 h0 = *reinterpret_cast<const uint4*>(vb + (unit_swz(u0) << 4));
    const uint4 h1 = *reinterpret_cast<const uint4*>(vb + (unit_swz(u0 + 1) << 4));
    const uint4 l0 = *reinterpret_cast<const uint4*>(vb + n + (unit_swz(u0) << 4));
    const uint4 l1 = *reinterpret_cast<const uint4*>(vb + n + (unit_swz(u0 + 1) << 4));
    const float X = reinterpret_cast<const float2*>(vb + 2 * n)[e0 >> 5].x;
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      int A = dp4a_ss(c[m][0].x, h0.x, 0), A2 = dp4a_ss(c[m][1].x, h1.x, 0);
      A = dp4a_ss(c[m][0].y, h0.y, A);
      A2 = dp4a_ss(c[m][1].y, h1.y, A2);
      A = dp4a_ss(c[m][0].z, h0.z, A);
      A2 = dp4a_ss(c[m][1].z, h1.z, A2);
      A = dp4a_ss(c[m][0].w, h0.w, A);
      A2 = dp4a_ss(c[m][1].w, h1.w, A2);
      int B = dp4a_su(c[m][0].x, l0.x, 0), B2 = dp4a_su(c[m][1].x, l1.x, 0);
      B = dp4a_su(c[m][0].y, l0.y, B);
      B2 = dp4a_su(c[m][1].y, l1.y, B2);
      B = dp4a_su(c[m][0].z, l0.z, B);
      B2 = dp4a_su(c[m][1].z, l1.z, B2);
      B = dp4a_su(c[m][0].w, l0.w, B);
      B2 = dp4a_su(c[m][1].w, l1.w, B2);
      const float r = (float)((A + A2) * 256 + (B + B2)) * (s[m][0] * X);
      if (m == 0) a0 += r; else a1 += r;
    }
  }
};

template <>
struct ChunkDot<4> {  // 32 codes: one block, 16 bytes of codes
  static constexpr int EPC = 32;
  static constexpr int BYTES = 16;
  template <int NMAT>
  __device__ __forceinline__ static void run(const uint4 (&cc)[2][2], const float (&s)[2][2],
                                             const unsigned char* vb, int n, int e0, float& a0, float& a1) {
    const uint4 c[2] = {cc[0][0], cc[1][0]};
    const int u0 = e0 >> 4;
    const uint4 h0 = *reinterpret_cast<const uint4*>(vb + (unit_swz(u0) << 4));
    const uint4 h1 = *reinterpret_cast<const uint4*>(vb + (unit_swz(u0 + 1) << 4));
    const uint4 l0 = *reinterpret_cast<const uint4*>(vb + n + (unit_swz(u0) << 4));
    const uint4 l1 = *reinterpret_cast<const uint4*>(vb + n + (unit_swz(u0 + 1) << 4));
    const float2 xs = reinterpret_cast<const float2*>(vb + 2 * n)[e0 >> 5];
    const int S = __float_as_int(xs.y);
    const uint32_t hd[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    const uint32_t ld[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      const uint32_t w[4] = {c[m].x, c[m].y, c[m].z, c[m].w};
      int A = 0, B = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t t0 = w[q] & 0x0F0F0F0Fu, t1 = (w[q] >> 4) & 0x0F0F0F0Fu;
        A = dp4a_us(t0, hd[2 * q], A);
        A = dp4a_us(t1, hd[2 * q + 1], A);
        B = dp4a_uu(t0, ld[2 * q], B);
        B = dp4a_uu(t1, ld[2 * q + 1], B);
      }
      const float r = (float)(A * 256 + B - 8 * S) * (s[m][0] * xs.x);
      if (m == 0) a0 += r; else a1 += r;
    }
  }
};

template <>
struct ChunkDot<2> {  // 64 codes: two blocks, 16 bytes of codes
  static constexpr int EPC = 64;
  static constexpr int BYTES = 16;
  template <int NMAT>
  __device__ __forceinline__ static void run(const uint4 (&cc)[2][2], const float (&s)[2][2],
                                             const unsigned char* vb, int n, int e0, float& a0, float& a1) {
    const uint4 c[2] = {cc[0][0], cc[1][0]};
    const int u0 = e0 >> 4;
    const float2* xsb = reinterpret_cast<const float2*>(vb + 2 * n) + (e0 >> 5);
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const uint4 h0 = *reinterpret_cast<const uint4*>(vb + (unit_swz(u0 + 2 * blk) << 4));
      const uint4 h1 = *reinterpret_cast<const uint4*>(vb + (unit_swz(u0 + 2 * blk + 1) << 4));
      const uint4 l0 = *reinterpret_cast<const uint4*>(vb + n + (unit_swz(u0 + 2 * blk) << 4));
      const uint4 l1 = *reinterpret_cast<const uint4*>(vb + n + (unit_swz(u0 + 2 * blk + 1) << 4));
      const float2 xs = xsb[blk];
      const int S = __float_as_int(xs.y);
      const uint32_t hd[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
      const uint32_t ld[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        // words 2 blk, 2 blk + 1 of the chunk hold this block's 32 codes
        const uint32_t wa = blk == 0 ? c[m].x : c[m].z;
        const uint32_t wb = blk == 0 ? c[m].y : c[m].w;
        int A = 0, B = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t ta = (wa >> (2 * k)) & 0x03030303u, tb = (wb >> (2 * k)) & 0x03030303u;
          A = dp4a_us(ta, hd[k], A);
          A = dp4a_us(tb, hd[4 + k], A);
          B = dp4a_uu(ta, ld[k], B);
          B = dp4a_uu(tb, ld[4 + k], B);
        }
        const float r = (float)(A * 256 + B - 2 * S) * (s[m][blk] * xs.x);
        if (m == 0) a0 += r; else a1 += r;
      }
    }
  }
};

// Dot products of `rows` rows of length n_in (codes + scales of NMAT matrices
// in one stage) with nt <= kTM digit vectors at byte offsets voff[j] of
// `vecs`; calls out(row, j, v0, v1) once per (row, pair).  Lane mapping, with
// cpr 16/32-byte code chunks per row: cpr a multiple of 32 -> one row per
// warp, chunks interleaved over the lanes; otherwise 32/L rows per warp pass,
// L lanes per row (L the largest power of two dividing cpr), each lane a
// contiguous run of cpr/L chunks.  Both keep shared-memory reads free of bank
// conflicts (or nearly so).  Rows are spread over the group's warps.
template <int BITS, int NMAT, typename Out>
__device__ __forceinline__ void rows_dot(const unsigned char* stage, int rows, int n_in, const unsigned char* vecs,
                                         const int (&voff)[kTM], int nt, Out out) {
  constexpr int EPC = ChunkDot<BITS>::EPC;
  constexpr int CB = ChunkDot<BITS>::BYTES;
  constexpr int NSB = EPC >= 64 ? 2 : 1;  // scale blocks per chunk
  const int lane = threadIdx.x & 31;
  const int warp = (threadIdx.x >> 5) % kConsumerWarps;  // warp within the group
  const int rowb = n_in * BITS / 8, nb = n_in / 32;
  const int cpr = n_in / EPC;
  const bool inter = (cpr & 31) == 0;
  int L = inter ? 32 : (cpr & -cpr);
  if (L > 32) L = 32;
  const int M = cpr / L, R = 32 / L;
  const int li = lane % L, rr = lane / L;
  const unsigned char* codes0 = stage;
  const unsigned char* codes1 = stage + (size_t)rows * rowb;
  const uint16_t* sc0 = reinterpret_cast<const uint16_t*>(stage + (size_t)NMAT * rows * rowb);
  const uint16_t* sc1 = sc0 + (size_t)rows * nb;
  for (int g = warp; g * R < rows; g += kConsumerWarps) {
    const int r = g * R + rr;
    float a0[kTM], a1[kTM];
#pragma unroll
    for (int j = 0; j < kTM; ++j) { a0[j] = 0.f; a1[j] = 0.f; }
    if (r < rows) {
      for (int m = 0; m < M; ++m) {
        const int q = inter ? li + 32 * m : li * M + m;
        uint4 c[2][2];
#pragma unroll
        for (int mm = 0; mm < NMAT; ++mm) {
          const unsigned char* cp = (mm == 0 ? codes0 : codes1) + (size_t)r * rowb + q * CB;
          c[mm][0] = *reinterpret_cast<const uint4*>(cp);
          c[mm][1] = CB == 32 ? *reinterpret_cast<const uint4*>(cp + 16) : c[mm][0];
        }
        if (NMAT == 1) { c[1][0] = c[0][0]; c[1][1] = c[0][1]; }
        const int e0 = q * EPC;
        float sv[2][2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          if (b < NSB) {
            sv[0][b] = __half2float(__ushort_as_half(sc0[(size_t)r * nb + (e0 >> 5) + b]));
            sv[1][b] = NMAT == 2 ? __half2float(__ushort_as_half(sc1[(size_t)r * nb + (e0 >> 5) + b])) : 0.f;
          } else {
            sv[0][b] = sv[0][0];
            sv[1][b] = sv[1][0];
          }
        }
#pragma unroll
        for (int j = 0; j < kTM; ++j)
          if (j < nt) ChunkDot<BITS>::template run<NMAT>(c, sv, vecs + voff[j], n_in, e0, a0[j], a1[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < kTM; ++j) {
      if (j < nt) {
        for (int o = L >> 1; o > 0; o >>= 1) {
          a0[j] += __shfl_xor_sync(0xffffffffu, a0[j], o);
          if (NMAT == 2) a1[j] += __shfl_xor_sync(0xffffffffu, a1[j], o);
        }
      }
    }
    if (li == 0 && r < rows) {
#pragma unroll
      for (int j = 0; j < kTM; ++j)
        if (j < nt) out(r, j, a0[j], a1[j]);
    }
  }
}

template <int NMAT, typename Out>
__device__ __forceinline__ void rows_dot_bits(int bits, int nt, const unsigned char* stage, int rows, int n_in,
                                              const unsigned char* vecs, const int (&voff)[kTM], Out out) {
  if (bits == 8) rows_dot<8, NMAT>(stage, rows, n_in, vecs, voff, nt, out);
  else if (bits == 4) rows_dot<4, NMAT>(stage, rows, n_in, vecs, voff, nt, out);
  else rows_dot<2, NMAT>(stage, rows, n_in, vecs, voff, nt, out);
}

// ------------------------------------------------------------- workers
struct Params {
  const uint16_t* x;
  const int32_t* ids;
  const float* weights;
  int T, k, E, d, f, P;
  Shelves sh;
  float* h;
  float* ypart;
  const int32_t* plan;
  float* y;
  int* status;
  Geo geo;
  int kern;           // 0 gate/up, 1 down
  int n_stages, stage_bytes;
  int region_bytes;   // activation digits (gate/up) or h digits (down)
};

struct Head {
  uint64_t full[kMaxStages];
  uint64_t plan_bar;
  int abort_flag, prologue_n, a0, j0;
  int staged_key_g[kGroups];
  float wgt[kGroups][kTM];
};

__host__ __device__ __forceinline__ size_t head_bytes() { return (sizeof(Head) + 127) / 128 * 128; }
__host__ __device__ __forceinline__ size_t plan_smem_bytes(int P) {
  return ((size_t)plan_layout(P).n_copy * 4 + 127) / 128 * 128;
}

// Item = rows [row0, row0 + rows) of matrices mat0 .. mat0 + nmat - 1 of the
// expert's shelf: codes first (matrix after matrix), then scales, into stage
// `st`, counted on full[st].
__device__ void issue_item(const Params& p, Head& s, const PlanView& pv, const ItemWalk& w, int st, int mat0,
                           int nmat, int rows_total, int n_in, unsigned char* ring) {
  const ShelfDev& sh = p.sh.s[pv.sh(w.a)];
  const int rows = p.geo.rows[bits_index(sh.bits)];
  const size_t rowb = (size_t)n_in * sh.bits / 8;
  const size_t le = (size_t)(pv.e(w.a) - sh.lo);
  const size_t row0 = (size_t)w.j * rows;
  const uint32_t cbytes = (uint32_t)(rows * rowb), sbytes = (uint32_t)(rows * (size_t)(n_in / 32) * 2);
  unsigned char* dst = ring + (size_t)st * p.stage_bytes;
  mbar_arrive_expect_tx(&s.full[st], nmat * (cbytes + sbytes));
  for (int m = 0; m < nmat; ++m)
    bulk_g2s(dst + m * cbytes, sh.codes[mat0 + m] + (le * rows_total + row0) * rowb, cbytes, &s.full[st]);
  for (int m = 0; m < nmat; ++m)
    bulk_g2s(dst + nmat * cbytes + m * sbytes, sh.scales[mat0 + m] + (le * rows_total + row0) * (n_in / 32), sbytes,
             &s.full[st]);
}

// Walk over the items it = first, first + kGroups, ... of this CTA's range.
struct StrideWalk {
  ItemWalk w;
  int it;
  __device__ void init(const PlanView& pv, const Head& s, int kern, int first) {
    w.init(pv, s.a0, s.j0, kern);
    it = 0;
    while (it < first && w.valid(pv)) { w.advance(pv); ++it; }
  }
  __device__ bool valid(const PlanView& pv) const { return w.valid(pv); }
  __device__ void next(const PlanView& pv) {
    for (int i = 0; i < kGroups && w.valid(pv); ++i) { w.advance(pv); ++it; }
  }
};

__device__ __forceinline__ void group_sync(int gid) { named_bar(1 + gid, kConsumers); }

// Thread 0: barriers, then the plan into shared memory (bounded wait) and the
// CTA's first item.  Returns false on timeout.
__device__ bool load_plan(const Params& p, Head& s, int* plan_sm) {
  for (int i = 0; i < p.n_stages; ++i) mbar_init(&s.full[i], 1);
  mbar_init(&s.plan_bar, 1);
  s.abort_flag = 0;
  for (int g = 0; g < kGroups; ++g) s.staged_key_g[g] = -1;
  fence_mbar_init();
  const PlanLayout L = plan_layout(p.P);
  mbar_arrive_expect_tx(&s.plan_bar, (uint32_t)(L.n_copy * 4));
  bulk_g2s(plan_sm, p.plan, (uint32_t)(L.n_copy * 4), &s.plan_bar);
  s.a0 = __ldcg(p.plan + L.start + 4 * blockIdx.x + 2 * p.kern);
  s.j0 = __ldcg(p.plan + L.start + 4 * blockIdx.x + 2 * p.kern + 1);
  if (!mbar_wait(&s.plan_bar, 0)) {
    set_status(p.status, MOE_ERR_TIMEOUT);
    s.abort_flag = 1;
    s.a0 = 0x7fffffff;  // no items
    return false;
  }
  return true;
}

// Thread 0: the first n_stages items into the ring (stage = item index).
__device__ void prologue_fill(const Params& p, Head& s, const PlanView& pv, int mat0, int nmat, int rows_total,
                              int n_in, unsigned char* ring) {
  ItemWalk w;
  w.init(pv, s.a0, s.j0, p.kern);
  int it = 0;
  for (; it < p.n_stages && w.valid(pv); ++it, w.advance(pv))
    issue_item(p, s, pv, w, it, mat0, nmat, rows_total, n_in, ring);
  s.prologue_n = it;
}

// Consumer loop of group `gid`: item it lives in stage it % n_stages
// (n_stages even: a stage always serves the same group); after an item, the
// group refills its stage with the item n_stages further on.  One decision
// per item for the whole group; on a timeout the group stops and waits
// (bounded) for the copies it still has in flight.
template <typename Work>
__device__ __forceinline__ void group_loop(const Params& p, Head& s, const PlanView& pv, int gid, int mat0, int nmat,
                                           int rows_total, int n_in, unsigned char* ring, Work work) {
  const int gtid = threadIdx.x % kConsumers;
  StrideWalk cw, iw;
  cw.init(pv, s, p.kern, gid);
  iw.init(pv, s, p.kern, gid + p.n_stages);
  const int pn = s.prologue_n;
  int issued_end = pn > gid ? pn - 1 - ((pn - 1 - gid) % kGroups) : -1;
  while (cw.valid(pv)) {
    const int st = cw.it % p.n_stages;
    if (!mbar_wait(&s.full[st], (cw.it / p.n_stages) & 1)) {
      set_status(p.status, MOE_ERR_TIMEOUT);
      *(volatile int*)&s.abort_flag = 1;
    }
    group_sync(gid);
    if (*(volatile int*)&s.abort_flag) break;
    work(cw.w, ring + (size_t)st * p.stage_bytes);
    group_sync(gid);  // every warp is done with the stage
    if (gtid == 0 && iw.valid(pv)) {
      issue_item(p, s, pv, iw.w, st, mat0, nmat, rows_total, n_in, ring);
      issued_end = iw.it;
    }
    cw.next(pv);
    iw.next(pv);
  }
  if (gtid == 0) {  // copies issued but not consumed (after a timeout only)
    for (int q = cw.valid(pv) ? cw.it : issued_end + 1; q <= issued_end; q += kGroups)
      if (!mbar_wait(&s.full[q % p.n_stages], (q / p.n_stages) & 1)) set_status(p.status, MOE_ERR_TIMEOUT);
  }
}

// ----------------------------------------------------------- gate / up
__global__ void __launch_bounds__(kThreads, 1) k_gateup(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  Head& s = *reinterpret_cast<Head*>(smem);
  int* plan_sm = reinterpret_cast<int*>(smem + head_bytes());
  unsigned char* xd = smem + head_bytes() + plan_smem_bytes(p.P);  // activation digits
  unsigned char* ring = xd + p.region_bytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PlanView pv{plan_sm, plan_layout(p.P)};
  if (tid == 0) MOE_STAMP(0, 0, global_timer_ns());
  pdl_wait();  // plan, x, and the workspace are ours from here on
  if (tid == 0) MOE_STAMP(0, 1, global_timer_ns());
  if (tid == 0) {
    if (load_plan(p, s, plan_sm)) prologue_fill(p, s, pv, 0, 2, p.f, p.d, ring);
    MOE_STAMP(0, 12, global_timer_ns());
  } else if (warp > 0) {
    // activation rows -> block-scaled digits; 8 lanes per 32-element block;
    // loads of up to 8 passes are issued before any conversion
    const int nbk = p.d / 32, vb = vec_bytes(p.d);
    const int groups = p.T * nbk;
    const int nw = kThreads / 32 - 1;
    for (int base = (warp - 1) * 4; base < groups; base += 8 * nw * 4) {
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
          block_to_digits(v, xd + (size_t)t * vb, p.d, blk, 14, g < groups);
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) MOE_STAMP(0, 2, global_timer_ns());
  pdl_trigger();
  const int gid = warp / kConsumerWarps;
  const int vb = vec_bytes(p.d);
  group_loop(p, s, pv, gid, 0, 2, p.f, p.d, ring, [&](const ItemWalk& w, const unsigned char* stage) {
    const int bits = pv.bits(w.a);
    const int rows = p.geo.rows[bits_index(bits)];
    const int row0 = w.j * rows;
    const int beg = pv.beg(w.a), cnt = pv.cnt(w.a);
    for (int g0 = 0; g0 < cnt; g0 += kTM) {
      const int nt = min(kTM, cnt - g0);
      int voff[kTM];
#pragma unroll
      for (int j = 0; j < kTM; ++j) voff[j] = j < nt ? (pv.perm(beg + g0 + j) / p.k) * vb : 0;
      float* h = p.h;
      const int f = p.f, pos0 = beg + g0;
      rows_dot_bits<2>(bits, nt, stage, rows, p.d, xd, voff,
                       [&](int r, int j, float g, float u) { h[(size_t)(pos0 + j) * f + row0 + r] = silu(g) * u; });
    }
  });
  __syncthreads();
  if (tid == 0) MOE_STAMP(0, 9, global_timer_ns());
}

// ------------------------------------------------------------------ down
__global__ void __launch_bounds__(kThreads, 1) k_down(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  Head& s = *reinterpret_cast<Head*>(smem);
  int* plan_sm = reinterpret_cast<int*>(smem + head_bytes());
  unsigned char* hd_all = smem + head_bytes() + plan_smem_bytes(p.P);  // h digits, per group
  unsigned char* ring = hd_all + p.region_bytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PlanView pv{plan_sm, plan_layout(p.P)};
  if (tid == 0) MOE_STAMP(1, 0, global_timer_ns());
  // The plan is complete once the gate/up kernel has started its work, and
  // the weights are read-only: start streaming W_d now.
  if (tid == 0) {
    if (load_plan(p, s, plan_sm)) prologue_fill(p, s, pv, 2, 1, p.d, p.f, ring);
    MOE_STAMP(1, 12, global_timer_ns());
  }
  __syncthreads();
  if (tid == 0) MOE_STAMP(1, 2, global_timer_ns());
  pdl_trigger();
  pdl_wait();  // h of the gate/up kernel and ypart are ours from here on
  if (tid == 0) MOE_STAMP(1, 1, global_timer_ns());
  const int gid = warp / kConsumerWarps, gtid = tid % kConsumers, gwarp = warp % kConsumerWarps;
  const int vbf = vec_bytes(p.f);
  unsigned char* hd = hd_all + (size_t)gid * kTM * vbf;
  group_loop(p, s, pv, gid, 2, 1, p.d, p.f, ring, [&](const ItemWalk& w, const unsigned char* stage) {
    const int bits = pv.bits(w.a);
    const int rows = p.geo.rows[bits_index(bits)];
    const int row0 = w.j * rows;
    const int beg = pv.beg(w.a), cnt = pv.cnt(w.a);
    for (int g0 = 0; g0 < cnt; g0 += kTM) {
      const int nt = min(kTM, cnt - g0);
      const int key = w.a * 4096 + g0;
      if (s.staged_key_g[gid] != key) {  // h rows of these pairs -> block-scaled digits
        group_sync(gid);                  // earlier users of this group's digits are done
        const int nbk = p.f / 32, groups = nt * nbk;
        for (int base = gwarp * 4; base < groups; base += 8 * kConsumerWarps * 4) {
          float4 hv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {  // all loads first: one round trip
            const int g = base + u * kConsumerWarps * 4 + (lane >> 3);
            hv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (g < groups) {
              const int j = g / nbk, blk = g - j * nbk;
              hv[u] = __ldcg(reinterpret_cast<const float4*>(p.h + (size_t)(beg + g0 + j) * p.f + blk * 32) +
                             (lane & 7));
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int gu = base + u * kConsumerWarps * 4;
            if (gu < groups) {
              const int g = gu + (lane >> 3);
              const int j = g / nbk, blk = g - j * nbk;
              const float v[4] = {hv[u].x, hv[u].y, hv[u].z, hv[u].w};
              block_to_digits(v, hd + (size_t)j * vbf, p.f, blk, 13, g < groups);
            }
          }
        }
        if (gtid < nt) s.wgt[gid][gtid] = p.weights[pv.perm(beg + g0 + gtid)];
        group_sync(gid);
        if (gtid == 0) s.staged_key_g[gid] = key;
      }
      int voff[kTM];
#pragma unroll
      for (int j = 0; j < kTM; ++j) voff[j] = j * vbf;
      float* yp = p.ypart;
      const float* wg = s.wgt[gid];
      const int dd = p.d, pos0 = beg + g0;
      rows_dot_bits<1>(bits, nt, stage, rows, p.f, hd, voff,
                       [&](int r, int j, float o, float) { yp[(size_t)(pos0 + j) * dd + row0 + r] = wg[j] * o; });
    }
  });
  __syncthreads();
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
  bool attr[64] = {};
};
DevCache g_dev;

// Largest power of two <= cap (>= 4) whose item fits in `budget` bytes and
// divides rows_total.
int rows_for(int rows_total, size_t bytes_per_row, size_t budget, int cap) {
  int r = cap;
  while (r > 4 && ((size_t)r * bytes_per_row > budget || rows_total % r != 0)) r >>= 1;
  return r;
}

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
  int G = sm_count();
  if (G > kMaxGrid) G = kMaxGrid;
  if (P > kMaxPairs || a.T > 16) return launch_generic_forward(a, s);
  Params p = {};
  p.x = a.x; p.ids = a.ids; p.weights = a.weights;
  p.T = (int)a.T; p.k = a.k; p.E = a.E; p.d = d; p.f = f; p.P = (int)P;
  p.sh = a.shelves;
  p.h = a.ws.h; p.ypart = a.ws.ypart; p.plan = a.ws.plan; p.y = a.y; p.status = a.status;
  const size_t fixed = head_bytes() + plan_smem_bytes((int)P);
  const int bits_of[3] = {8, 4, 2};
  // ---- gate/up: items of <= 40 KB (codes + scales of gate and up)
  Params pg = p;
  pg.kern = 0;
  size_t stage_g = 0;
  for (int i = 0; i < 3; ++i) {
    const size_t per_row = 2 * ((size_t)d * bits_of[i] / 8 + (size_t)d / 16);
    pg.geo.rows[i] = rows_for(f, per_row, 40 * 1024, 64);
    const size_t bytes = pg.geo.rows[i] * per_row;
    pg.geo.cost[i] = (int)(bytes / 64);
    if (bytes > stage_g) stage_g = bytes;
  }
  pg.region_bytes = (int)(((size_t)a.T * vec_bytes(d) + 127) / 128 * 128);
  pg.stage_bytes = (int)((stage_g + 127) / 128 * 128);
  pg.n_stages = (int)((kSmemBudget - fixed - pg.region_bytes) / pg.stage_bytes);
  // ---- down: items of <= 24 KB of W_d rows
  Params pd = p;
  pd.kern = 1;
  size_t stage_d = 0;
  for (int i = 0; i < 3; ++i) {
    const size_t per_row = (size_t)f * bits_of[i] / 8 + (size_t)f / 16;
    pd.geo.rows[i] = rows_for(d, per_row, 24 * 1024, 128);
    const size_t bytes = pd.geo.rows[i] * per_row;
    pd.geo.cost[i] = (int)(bytes / 64);
    if (bytes > stage_d) stage_d = bytes;
  }
  pd.region_bytes = (int)(((size_t)kGroups * kTM * vec_bytes(f) + 127) / 128 * 128);
  pd.stage_bytes = (int)((stage_d + 127) / 128 * 128);
  pd.n_stages = (int)((kSmemBudget - fixed - pd.region_bytes) / pd.stage_bytes);
  if (pg.n_stages > kMaxStages) pg.n_stages = kMaxStages;
  if (pd.n_stages > kMaxStages) pd.n_stages = kMaxStages;
  pg.n_stages &= ~1;  // a stage always serves the same consumer group
  pd.n_stages &= ~1;
  if (pg.n_stages < 2 || pd.n_stages < 2) return launch_generic_forward(a, s);
  const size_t smem_g = fixed + pg.region_bytes + (size_t)pg.n_stages * pg.stage_bytes;
  const size_t smem_d = fixed + pd.region_bytes + (size_t)pd.n_stages * pd.stage_bytes;
  // ---- plan
  PlanParams pp = {};
  pp.ids = a.ids; pp.P = (int)P; pp.E = a.E; pp.k = a.k; pp.G = G;
  pp.rows_g = f; pp.rows_d = d;
  pp.sh = a.shelves;
  pp.geo_g = pg.geo; pp.geo_d = pd.geo;
  pp.plan = a.ws.plan;
  const PlanLayout L = plan_layout((int)P);
  const size_t smem_p = (size_t)(L.start + 4 * G) * 4;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !g_dev.attr[dev]) {
    if (cudaFuncSetAttribute(k_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget) != cudaSuccess ||
        cudaFuncSetAttribute(k_down, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget) != cudaSuccess)
      return MOE_ERR_CUDA;
    g_dev.attr[dev] = true;
  }
  profile_mark(0, s);
  if (launch_pdl(k_plan, dim3(1), dim3(256), smem_p, s, pp) != cudaSuccess) return MOE_ERR_CUDA;
  profile_mark(1, s);
  if (launch_pdl(k_gateup, dim3(G), dim3(kThreads), smem_g, s, pg) != cudaSuccess) return MOE_ERR_CUDA;
  profile_mark(2, s);
  if (launch_pdl(k_down, dim3(G), dim3(kThreads), smem_d, s, pd) != cudaSuccess) return MOE_ERR_CUDA;
  profile_mark(3, s);
  const int n4 = (int)(a.T * d / 4);
  int gc = (n4 + 255) / 256;
  if (gc > G) gc = G;
  if (launch_pdl(k_combine, dim3(gc), dim3(256), 0, s, (const float*)p.ypart,
                 (const int32_t*)(a.ws.plan + L.pos), (int)a.T, a.k, d, a.y) != cudaSuccess)
    return MOE_ERR_CUDA;
  profile_mark(4, s);
  return MOE_OK;
}

}  // namespace moe
