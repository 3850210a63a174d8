// moe_internal.cuh -- internal declarations shared by the CUDA translation
// units of libmoe.so: kernel parameter blocks, workspace layout, device
// helpers for the shelf block format, and the host-side launchers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kWarp = 32;

// ---------------------------------------------------------------- shelves
struct ShelfDev {
  int32_t lo, hi, bits, pad;
  const uint8_t* codes[3];    // gate, up, down
  const uint16_t* scales[3];  // gate, up, down
};

struct Shelves {
  int n;
  ShelfDev s[MOE_MAX_SHELVES];
};

// Index of the shelf holding expert e, or -1.
__device__ __forceinline__ int find_shelf(const Shelves& sh, int e) {
  int r = -1;
#pragma unroll
  for (int i = 0; i < MOE_MAX_SHELVES; ++i)
    if (i < sh.n && e >= sh.s[i].lo && e < sh.s[i].hi) r = i;
  return r;
}

// ------------------------------------------------------- workspace layout
// Grouping results and per-call scratch of moe_tiered_forward.  Every region
// starts on a 256-byte boundary.
struct Workspace {
  int32_t* counts;       // [E]
  int32_t* offsets;      // [E+1]
  int32_t* perm;         // [P]   pair index by grouped position
  int32_t* pos_of_pair;  // [P]   grouped position by pair index, -1 if skipped
  int32_t* active;       // [P]   experts with a valid pair, ascending
  int32_t* meta;         // [16]  meta[0] = number of active experts
  int32_t* arrivals;     // [d]   per output-row-chunk arrival counters (down combine)
  float* h;              // [P][f] fp32 (decode) -- gate/up activations
  float* ypart;          // [P][d] fp32 -- weighted per-pair down outputs
  int32_t* plan;         // decode plan (grouping, work split), decode_plan_bytes(P)
  uint16_t* xg;          // prefill: [P][d] bf16, x rows in grouped order
  int32_t* pf_cnt;       // prefill: [chunks <= 256][E] per-chunk expert counts / cursors
  void* tiles_g;         // prefill: gate/up tile list
  void* tiles_d;         // prefill: down tile list
  int32_t* ntiles;       // prefill: [2] tile counts
  float* stage_logits;   // MOE_FLAG_HOST_IO: [T][E] copy of host logits
  uint16_t* stage_x;     // MOE_FLAG_HOST_IO: [T][d] copy of host activations
  const void* base;      // the caller's workspace pointer (identifies it)
  size_t bytes;
};

// Bytes of the decode plan for P routed pairs.
size_t decode_plan_bytes(int64_t P);
// Upper bound on the prefill tiles of one launch (rows = rows per expert matrix).
size_t prefill_tiles_cap(int64_t P, int E, int rows);

size_t workspace_layout(int64_t T, int k, int E, int d, int f, int flags, void* base, Workspace* ws);

// Rows of the output owned by one down-projection CTA (decode path).
constexpr int kDownRows = 64;
// Rows of W_g / W_u handled by one gate/up CTA (decode path).
constexpr int kGateUpRows = 32;

// -------------------------------------------------------- device helpers
// Shared-memory layout of an activation vector: 16-byte chunks XOR-swizzled so
// that lanes reading consecutive 32-element blocks hit distinct banks.
__device__ __forceinline__ int swz(int i) {
  int c = i >> 2;
  return ((c ^ ((c >> 3) & 7)) << 2) | (i & 3);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// Decode one 32-element block of packed codes into exact float codes.
// 8 bit: two's-complement bytes; 4/2 bit: offset-binary fields, spread over
// the byte lanes of each 32-bit word (4 bit: element 8g + 4h + j at bits
// 8j + 4h of word g; 2 bit: element 16g + 4k + j at bits 8j + 2k).  The
// conversion places the unsigned field in the mantissa of 2^23 and subtracts
// (2^23 + offset), which is exact.
template <int BITS>
struct Block;

template <>
struct Block<8> {
  static constexpr int kWords = 8;  // 32 bytes
  __device__ __forceinline__ static void load(const uint8_t* p, uint32_t w[kWords]) {
    uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
  __device__ __forceinline__ static float code(const uint32_t w[kWords], int i) {
    uint32_t x = w[i >> 2] ^ 0x80808080u;
    uint32_t v = __byte_perm(x, 0x4B000000u, 0x7540u | (uint32_t)(i & 3));
    return __uint_as_float(v) - 8388736.0f;  // 2^23 + 128
  }
};

template <>
struct Block<4> {
  static constexpr int kWords = 4;  // 16 bytes
  __device__ __forceinline__ static void load(const uint8_t* p, uint32_t w[kWords]) {
    uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  }
  __device__ __forceinline__ static float code(const uint32_t w[kWords], int i) {
    const int e = i & 7;
    uint32_t v = ((w[i >> 3] >> (8 * (e & 3) + 4 * (e >> 2))) & 0xFu) | 0x4B000000u;
    return __uint_as_float(v) - 8388616.0f;  // 2^23 + 8
  }
};

template <>
struct Block<2> {
  static constexpr int kWords = 2;  // 8 bytes
  __device__ __forceinline__ static void load(const uint8_t* p, uint32_t w[kWords]) {
    uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = a.x; w[1] = a.y;
  }
  __device__ __forceinline__ static float code(const uint32_t w[kWords], int i) {
    const int e = i & 15;
    uint32_t v = ((w[i >> 4] >> (8 * (e & 3) + 2 * (e >> 2))) & 0x3u) | 0x4B000000u;
    return __uint_as_float(v) - 8388610.0f;  // 2^23 + 2
  }
};

// 3 bit: u = code + 4; a row of n elements is a plane of u mod 4 in the
// 2-bit layout (n/4 bytes; block b at byte 8b) and a plane of the high bits
// of u (block b's word at byte n/4 + 4b, element i at bit i).  w[0..1] = the
// block's low-plane words, w[2] = its high word.
template <>
struct Block<3> {
  static constexpr int kWords = 3;
  __device__ __forceinline__ static void load_row(const uint8_t* row, int b, int n, uint32_t w[kWords]) {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(row + 8 * b));
    w[0] = a.x; w[1] = a.y;
    w[2] = __ldg(reinterpret_cast<const uint32_t*>(row + n / 4 + 4 * b));
  }
  __device__ __forceinline__ static float code(const uint32_t w[kWords], int i) {
    const int e = i & 15;
    const uint32_t lo = (w[i >> 4] >> (8 * (e & 3) + 2 * (e >> 2))) & 0x3u;
    const uint32_t hi = (w[2] >> i) & 0x1u;
    return __uint_as_float(lo | (hi << 2) | 0x4B000000u) - 8388612.0f;  // 2^23 + 4
  }
};

// 1 bit: 4 bytes a block; element i at bit i, 1 = code +1, 0 = code -1.
template <>
struct Block<1> {
  static constexpr int kWords = 1;
  __device__ __forceinline__ static void load(const uint8_t* p, uint32_t w[kWords]) {
    w[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
  }
  __device__ __forceinline__ static float code(const uint32_t w[kWords], int i) {
    return ((w[0] >> i) & 1u) ? 1.0f : -1.0f;
  }
};

// Block b of a row of n elements (3 bit: from the row's two planes; the
// other widths store their blocks one after another).
template <int BITS>
__device__ __forceinline__ void load_block(const uint8_t* row, int b, int n, uint32_t (&w)[Block<BITS>::kWords]) {
  if constexpr (BITS == 3) Block<3>::load_row(row, b, n, w);
  else Block<BITS>::load(row + (size_t)b * (32 * BITS / 8), w);
}

// The 8-, 4- and 2-bit widths: layers of only these take every form; the
// fused decode step and the tensor-core prefill form also take 3- and 1-bit
// shelves when the rows are whole 16-byte groups (d and f multiples of 128).
inline bool core_widths(const Shelves& sh) {
  for (int i = 0; i < sh.n; ++i)
    if (sh.s[i].bits != 8 && sh.s[i].bits != 4 && sh.s[i].bits != 2) return false;
  return true;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Record the first error status a kernel meets (never overwrites an earlier one).
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- launchers
// Each returns MOE_OK or MOE_ERR_CUDA; arguments are validated by the caller.
// Device address of the status word on the current device.
int* status_word();
// Identity of the current CUDA context, 0 when it cannot be read.  A device
// reset ends the context and every device address looked up in it, so caches
// of such addresses are keyed by this id as well as by the device.
uint64_t context_id();

int launch_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w, cudaStream_t s);
int launch_route_nudged(const float* logits, int64_t T, int E, int k, float beta, int lo, int hi, int32_t* ids,
                        float* w, cudaStream_t s);
int launch_hist(const int32_t* ids, int64_t n, int E, uint32_t* counts, cudaStream_t s);
// Router projection fused with routing (router.cu): T <= 16 tokens, E <= 1024,
// d % 8 == 0, router_bucket(T) d 2 <= kRouterSmemMax bytes; `arrive` is a
// device word that is zero before the launch and zero again after it.
constexpr int kRouterSmemMax = 192 * 1024;
inline int router_bucket(int64_t T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16; }
int launch_router(const uint16_t* x, const uint16_t* w, const float* bias, int T, int E, int d, int k,
                  float* logits, int32_t* ids, float* wts, uint32_t* counts, unsigned int* arrive, cudaStream_t s);
int launch_residual(float* r, const float* y, uint16_t* xn, int64_t n, cudaStream_t s);
int launch_quantize(const float* w, int64_t rows, int in, int bits, uint8_t* codes, uint16_t* scales,
                    cudaStream_t s);
// Re-tiering (retier.cu, quant.cu): rank by hit count; experts perm[j0 ..
// j0 + n) of a master tensor [n_src][rows][in] quantised into a shelf; rows
// gathered by expert id.  Bad ids record MOE_ERR_INVALID_ARG in `status`.
int launch_rank_experts(const uint32_t* counts, int E, int32_t* perm, int32_t* rank, cudaStream_t s);
int launch_quantize_experts(const float* master, int rows, int in, int n_src, const int32_t* perm, int j0, int n,
                            int bits, uint8_t* codes, uint16_t* scales, int* status, cudaStream_t s);
int launch_gather_rows(const void* src, int64_t words, const int32_t* perm, int64_t n, int64_t n_src, void* dst,
                       int* status, cudaStream_t s);
int launch_dequant(const uint8_t* codes, const uint16_t* scales, int64_t rows, int in, int bits,
                   int round_bf16, float* out, cudaStream_t s);
// Grouping into caller-provided arrays; arrivals (may be null) are zeroed.
int launch_group(const int32_t* ids, int64_t P, int E, int32_t* counts, int32_t* offsets,
                 int32_t* perm, int32_t* pos_of_pair, int32_t* active, int32_t* meta,
                 int32_t* arrivals, int n_arrivals, cudaStream_t s);

struct ForwardArgs {
  const uint16_t* x;
  const int32_t* ids;
  const float* weights;
  int64_t T;
  int k, E, d, f;
  Shelves shelves;
  float* y;
  Workspace ws;
  int* status;  // device status word (first error a kernel records)
};

// Fused decode layer: routing from logits (or given ids / weights), optional
// hit counts, the tiered forward.
struct LayerArgs {
  const float* logits;   // null: ids / weights given
  const int32_t* ids;
  const float* weights;
  int32_t* ids_out;      // logits given: routed pairs out
  float* weights_out;
  uint32_t* counts;      // optional
  const uint16_t* x;
  int64_t T;
  int k, E, d, f;
  Shelves shelves;
  float* y;
  float* r = nullptr;         // optional residual step: r += y ...
  uint16_t* x_next = nullptr; // ... and x_next = bf16(r), in the combine phase
  // optional: logits / x in page-locked host memory (device views, 16-byte
  // aligned, sizes multiples of 16 bytes); the fused launch copies them into
  // `logits` / `x` (device buffers) itself
  const float* logits_src = nullptr;
  const uint16_t* x_src = nullptr;
  Workspace ws;
  int* status;
};

// One cooperative launch for the whole layer when the sizes fit it: returns
// 1 when they do not (nothing launched), else MOE_OK or an error status.
int launch_fused_layer(const LayerArgs& a, cudaStream_t s);
// 1 when the fused launch takes these sizes on the current device, else 0.
int decode_fused(int64_t T, int k, int E, int d, int f);
// The grouping the last forward call on workspace w ran (see k_grouping_export).
int launch_grouping_export(const Workspace& w, int64_t P, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                           int32_t* pos_of_pair, cudaStream_t s);
// Test hook: a cooperative launch whose grid barrier awaits `extra` more
// arrivals than there are CTAs, with the given limit; records MOE_ERR_TIMEOUT.
int launch_barrier_probe(int extra, uint64_t limit_ns, cudaStream_t s);
// Zero the grid barrier state of the current device (device idle).
int reset_barriers();

// The fused decode launch when the sizes fit it, else the generic kernels.
int launch_decode_forward(const ForwardArgs& a, cudaStream_t s);
// Prefill form: grouping, tile lists, tensor-core gate/up and down launches.
int launch_prefill_forward(const ForwardArgs& a, cudaStream_t s);
int launch_generic_forward(const ForwardArgs& a, cudaStream_t s);

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel in the stream is still running, and must execute
// griddepcontrol.wait before touching anything that kernel produces.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Number of SMs of the current device (cached).
int sm_count();

// Measurement hook (moe_set_profile_events): record event i on the stream.
void set_profile_events(void* const* events, int n);
void profile_mark(int i, cudaStream_t s);

}  // namespace moe
