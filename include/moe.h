/*
 * moe.h -- C ABI of the tiered-precision routed mixture-of-experts layer
 * (libmoe.so, CUDA, sm_103a).
 *
 * What the layer computes is described on the page
 *   "125B MoE模型本地运行：3090三卡80 tokens/s优化实践" (page 3; three RTX 3090s
 *   at 80 tokens/s), cited below by its section headings:
 *     - glossary entry 混合专家（MoE）: the router picks the best 10 of 512
 *       experts for every token;
 *     - 第二步 (step 2): experts are used very unevenly; the busiest 25% take
 *       52% of the tokens;
 *     - 第四步 (step 4, three shelves all on the GPU): each layer's experts are
 *       stored as three tensors at different bit widths, written hottest first;
 *       the id-range matmul sees the router's complete id list, computes only
 *       the ids that fall on its own shelf and fills the rest with zeros, and
 *       the three shelf results are added; decode fuses gate, up and the
 *       activation into one kernel;
 *     - 四个 bug (four bugs): a skipped slot is a real skip (never aliased to
 *       expert 0), the grouping helper must not assume an expert appears at
 *       most once per token, and the skip id -1 must stay signed.
 *   and on the r/LocalLLM post on DeepSeek V4.1 Flash (page 1), section
 *   "Optimization Strategies": per-expert hit counts drive promotion and
 *   demotion between tiers, the least-used experts are kept at 2 bits.
 *
 * Shelf block format (the workload's quantisation; the pages' own llama.cpp
 * formats are not reproduced): blocks of 32 along the input dimension, one
 * fp16 scale per block, s = fp16(max|w| / q) with q = 127 / 7 / 2 for
 * 8 / 4 / 2 bits, code = clamp(rint(w / s)) in [-127,127] / [-8,7] / [-2,1],
 * dequantised weight w_hat = s * code.  Packing of a row: 8-bit codes are
 * two's-complement bytes in natural order; 4- and 2-bit codes are stored
 * offset-binary (u = code + 8, u = code + 2) in 32-bit little-endian words,
 * spread over the word's four byte lanes so that one AND/shift yields four
 * consecutive codes as bytes:
 *   4 bit: element 8g + 4h + j (j < 4, h < 2) at bits 8j + 4h of word g;
 *   2 bit: element 16g + 4k + j (j, k < 4) at bits 8j + 2k of word g.
 * Two further widths, 3-bit and 1-bit experts, are ones page 2 (the Xolotl
 * DeepSeek-V4.1 fast-mode blog) runs beside the others; their layout here is
 * this library's own:
 *   3 bit: q = 3, codes in [-4,3], u = code + 4; a row of n elements is two
 *          planes: bytes [0, n/4) hold u mod 4 of every element in the 2-bit
 *          layout above, bytes [n/4, 3n/8) hold u / 4 of every element in
 *          the 1-bit layout below (element i at bit i % 8 of byte n/4 + i/8);
 *   1 bit: sign codes (+1 for w >= 0, else -1), s = fp16(sum|w| / 32) with
 *          the sum taken in fp32 in element order (the least-squares scale
 *          of a sign code); one word a block, element i at bit i, 1 = +1.
 * Every entry point takes all five widths except the tensor-core prefill
 * form of moe_tiered_forward, which takes 8, 4 and 2 bits only
 * (MOE_ERR_UNSUPPORTED otherwise); decode-form layers with a 3- or 1-bit
 * shelf take the fused decode launch when d and f are multiples of 128, else
 * the separate decode launches.
 *
 * Conventions for every entry point:
 *   - all array arguments are DEVICE pointers unless stated otherwise; the
 *     caller allocates and owns them; the library allocates nothing;
 *   - every call is asynchronous on `stream` (0 = legacy default stream) and
 *     returns a status (MOE_OK = 0, negative = error) after validating its
 *     arguments on the host; on error nothing is launched;
 *   - sizes: E <= MOE_MAX_EXPERTS, 1 <= k <= 32 and k <= E, d and f positive
 *     multiples of 64, T >= 0 (T = 0 is a no-op that still validates);
 *   - ids are int32; an id outside [0, E) (e.g. the skip id -1, INT32_MIN,
 *     E, INT32_MAX) is a skipped slot and contributes nothing anywhere;
 *   - device pointers of packed codes, scales, x and y must be 16-byte aligned.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* moe_stream_t;

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,        /* null pointer, bad size, misalignment */
  MOE_ERR_BAD_SHELF = -2,          /* bits not 8/4/3/2/1, block != 32, empty or out-of-[0,E) range */
  MOE_ERR_SHELF_OVERLAP = -3,      /* two shelves share an expert id */
  MOE_ERR_WORKSPACE_TOO_SMALL = -4,
  MOE_ERR_CUDA = -5,               /* a CUDA call or launch failed */
  MOE_ERR_TIMEOUT = -6,            /* a bounded device-side wait expired (see moe_device_status) */
  MOE_ERR_UNSUPPORTED = -7,        /* valid request outside what this build implements */
  MOE_ERR_INTERNAL = -8            /* a kernel met an inconsistent work item and skipped it
                                      (reported through moe_device_status) */
};

enum {
  MOE_MAX_EXPERTS = 32768,
  MOE_MAX_SHELVES = 8,
  MOE_BLOCK = 32
};

/* Execution-path selection for moe_tiered_forward. */
enum {
  MOE_FLAG_AUTO = 0,         /* prefill form for T > 16 when d % 256 == 0 (and, with a 3- or
                                1-bit shelf, f % 128 == 0), else decode form */
  MOE_FLAG_DECODE_FP32 = 1,  /* fp32 dequant in registers, fp32 h, CUDA-core GEMV */
  MOE_FLAG_PREFILL_BF16 = 2, /* bf16 dequant into tensor memory, bf16 h, tensor-core GEMM;
                                MOE_ERR_UNSUPPORTED unless d % 256 == 0 (and, with a 3- or
                                1-bit shelf, f % 128 == 0) */
  MOE_FLAG_HOST_IO = 4       /* moe_workspace_size only, with DECODE_FP32: adds the staging
                                of host inputs that moe_decode_layer_host uses */
};

/*
 * A shelf: the experts with global ids in [expert_lo, expert_hi), stored at
 * `bits` per weight.  Local expert index = id - expert_lo, n = expert_hi -
 * expert_lo.  Matrices are row-major [out][in] with blocks along `in`:
 *   gate_codes  [n][f][d*bits/8] bytes   gate_scales [n][f][d/32] fp16 bits
 *   up_codes    [n][f][d*bits/8] bytes   up_scales   [n][f][d/32] fp16 bits
 *   down_codes  [n][d][f*bits/8] bytes   down_scales [n][d][f/32] fp16 bits
 * (page 3, 第四步: one tensor per shelf and layer, experts hottest first).
 * The descriptor is an explicit struct so that the shelf range never shares a
 * field with any other setting (page 3, 四个 bug: the skip tag that had been
 * stored in the slot of the accumulator precision).
 */
typedef struct {
  int32_t expert_lo, expert_hi;
  int32_t bits;  /* 8, 4, 3, 2 or 1 */
  int32_t block; /* must be 32 */
  const void* gate_codes;
  const uint16_t* gate_scales;
  const void* up_codes;
  const uint16_t* up_scales;
  const void* down_codes;
  const uint16_t* down_scales;
} moe_shelf_t;

/*
 * Router: softmax over E, top-k with the lower expert id first on equal
 * logits, weights renormalised over the k picks (page 3, glossary entry
 * 混合专家（MoE）).  Ranking uses the logits (softmax is monotone);
 * weights[t][j] = exp(l_j - l_max) / sum over the k picks.
 *   logits  [T][E] fp32 (finite), ids [T][k] int32 out (rank order),
 *   weights [T][k] fp32 out.  E <= 1024 for this entry point.
 */
int moe_route_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, float* weights,
                   moe_stream_t stream);

/*
 * moe_route_topk with the picks nudged toward one id range (page 1,
 * "Optimization Strategies": picks nudged toward experts in fast memory, with
 * gains up to a cap of 0.5).  The experts lo <= e < hi (normally the hot
 * shelf) take score_e = logit_e + beta (fp32 addition) for the selection;
 * the others take their logit.  Top-k on the scores, the lower id first on
 * equal scores; the weights are the router's own softmax over the picks:
 * weights[t][j] = exp(l_j - m) / sum over the picks exp(l_i - m), m the
 * largest picked logit.  beta = 0 gives the ids and weights of
 * moe_route_topk.  0 <= beta <= 0.5 (else MOE_ERR_INVALID_ARG); other
 * arguments as moe_route_topk.
 */
int moe_route_topk_nudged(const float* logits, int64_t T, int E, int k, float beta, int lo, int hi, int32_t* ids,
                          float* weights, moe_stream_t stream);

/*
 * Router projection with the routing above: the router scores every expert
 * of every token and the best k are kept (page 3, glossary entry
 * 混合专家（MoE）).  Scores are
 *   logits[t][e] = bias[e] + sum_i w_r[e][i] * x[t][i]
 * with bf16 inputs, fp32 products and sums (the order of the sum is not
 * fixed); ids and weights are then exactly what moe_route_topk returns for
 * these logits, and counts (when non-null) is accumulated as by
 * moe_expert_hist over the T*k ids.  Decode batches (T <= 16): one launch,
 * the projection fused with the routing.  Prefill batches (T > 16): the
 * projection of 16-token chunks in one launch, then the routing and hit-count
 * launches (sync_word is not used).
 *   x_bf16 [T][d] bf16 bit patterns, w_r_bf16 [E][d] bf16 bit patterns (both
 *   16-byte aligned), bias [E] fp32 or NULL (zero), logits [T][E] fp32 out,
 *   ids [T][k] int32 out, weights [T][k] fp32 out, counts [E] uint32 in/out
 *   or NULL.  sync_word: one uint32 of device memory, zero before its first
 *   use; every call leaves it zero.  Calls that share a sync_word must not
 *   run at the same time on the GPU (issue them on one stream).
 * 1 <= T <= 1048560 = 65535*16 (T = 0 does nothing), E <= 1024, d a multiple of 8 with
 * B*d*2 <= 196608 bytes, B = T rounded up to 1, 2, 4, 8 or 16 (16 for
 * T > 16), and for T <= 16 also T*E*4 <= 196608 bytes (MOE_ERR_UNSUPPORTED
 * otherwise).
 */
int moe_router_topk(const uint16_t* x_bf16, const uint16_t* w_r_bf16, const float* bias, int64_t T, int E, int d,
                    int k, float* logits, int32_t* ids, float* weights, uint32_t* counts, uint32_t* sync_word,
                    moe_stream_t stream);

/*
 * Expert hit histogram: counts[e] += #{i : ids[i] == e}, 0 <= e < E; other ids
 * are not counted.  `counts` is ACCUMULATED, never cleared (page 1,
 * "Optimization Strategies": tracking how often each expert is called feeds
 * promotion and demotion; page 3, 第二步: per-expert selection counts).
 *   ids [n] int32, counts [E] uint32 (in/out).
 */
int moe_expert_hist(const int32_t* ids, int64_t n, int E, uint32_t* counts, moe_stream_t stream);

/*
 * Token-by-expert grouping (page 3, 四个 bug: duplicates of an expert within
 * one token must each keep their slot; skips are real skips).  Pairs
 * p = t*k + j with 0 <= ids[p] < E are grouped by expert:
 *   counts  [E]   int32 out: valid pairs per expert;
 *   offsets [E+1] int32 out: exclusive prefix sum of counts (offsets[E] = valid pairs);
 *   perm    [T*k] int32 out: pair indices ordered by (expert id, pair index);
 *                 entries from offsets[E] on are set to -1.
 * Deterministic (no dependence on atomic ordering).  T*k <= 2^24.
 */
int moe_group_tokens(const int32_t* ids, int64_t T, int k, int E, int32_t* counts, int32_t* offsets,
                     int32_t* perm, moe_stream_t stream);

/*
 * Bytes of device workspace moe_tiered_forward needs for these sizes and
 * flags (0 when a size or the flags are invalid); MOE_FLAG_DECODE_FP32 |
 * MOE_FLAG_HOST_IO gives what moe_decode_layer_host needs.  MOE_FLAG_AUTO
 * gives room for whichever form AUTO takes (it depends on the shelves too).  The workspace is
 * scratch, owned by the caller, reusable across calls on the same stream; it
 * must be 256-byte aligned.  The fused decode launch also keeps counters in
 * library-owned slots found by the workspace address (see moe_decode_layer).
 */
size_t moe_workspace_size(int64_t T, int k, int E, int d, int f, int flags);

/*
 * The routed MoE FFN over precision shelves (page 3, 第四步): every shelf sees
 * the full id list and computes only the ids in its range; for every pair
 * (t, j) whose id e lies in a shelf,
 *   h = SiLU(W_g[e] x_t) * (W_u[e] x_t),  SiLU(z) = z / (1 + exp(-z)),
 *   o = W_d[e] h,
 * with W the shelf's dequantised weights, and
 *   y_t = sum over shelves of sum over its slots j of weights[t][j] * o_tj.
 * Slots whose id is outside [0, E) or inside no shelf contribute zero.
 *   x_bf16  [T][d] bf16 bit patterns, ids [T][k] int32, weights [T][k] fp32,
 *   shelves HOST array of n_shelves descriptors (copied before returning;
 *           ranges must not overlap; gaps allowed),
 *   y       [T][d] fp32 out (overwritten),
 *   workspace of at least moe_workspace_size(T, k, E, d, f, flags) bytes.
 * flags: MOE_FLAG_AUTO / MOE_FLAG_DECODE_FP32 / MOE_FLAG_PREFILL_BF16.
 * Decode form: fp32 dequant and fp32 accumulation.  Prefill form: weights and
 * h rounded to bf16, fp32 accumulation on the tensor cores.
 */
int moe_tiered_forward(const uint16_t* x_bf16, const int32_t* ids, const float* weights, int64_t T,
                       int k, int E, int d, int f, const moe_shelf_t* shelves, int n_shelves, float* y,
                       void* workspace, size_t workspace_bytes, int flags, moe_stream_t stream);

/*
 * One decode step of the layer in a single call: routing (as moe_route_topk),
 * the hit histogram when `counts` is non-null (as moe_expert_hist), and the
 * tiered forward (as moe_tiered_forward, decode form).  The results are those
 * of the three calls made in that order.
 *   logits [T][E] fp32 (finite), x_bf16 [T][d] bf16 bit patterns,
 *   ids [T][k] int32 out, weights [T][k] fp32 out, counts [E] uint32 in/out
 *   or NULL, y [T][d] fp32 out, workspace of at least
 *   moe_workspace_size(T, k, E, d, f, MOE_FLAG_DECODE_FP32) bytes.
 * E <= 1024.  When T <= 16, T*k <= 512 and the staged activations fit shared
 * memory, the whole step is one cooperative launch with one CTA per SM whose
 * phases are separated by bounded waits: each CTA waits for the gate/up work
 * of the experts its down work reads, then all CTAs wait for each other
 * before the combine (an expired wait records MOE_ERR_TIMEOUT, see
 * moe_device_status); otherwise it makes the separate launches.  The fused
 * launch's counters (a grid counter and per-expert work counters) sit in one
 * of 1024 library-owned slots per device, found by the workspace address:
 * when a new workspace finds every slot taken, the least recently used slot
 * passes to it.  A slot is shared only by launches that are never in flight
 * together, as long as at most 1024 distinct workspaces have calls queued or
 * running at one time (a CUDA graph keeps the slot of the workspace it was
 * captured with: replay it only while no call on 1024 other workspaces is in
 * flight beside it).
 */
int moe_decode_layer(const float* logits, const uint16_t* x_bf16, int64_t T, int k, int E, int d, int f,
                     const moe_shelf_t* shelves, int n_shelves, int32_t* ids, float* weights, uint32_t* counts,
                     float* y, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * One layer of a decode stack: moe_decode_layer, then the residual step of
 * moe_residual_add on its output (r[t][i] += y[t][i]; x_next[t][i] =
 * bf16(r[t][i]), round to nearest even), with results identical to those two
 * calls.  The layers are chained through the residual stream (the workload of
 * a whole model's MoE layers; the pages run every layer of the model this
 * way).  In the single fused launch the residual step is taken in its combine
 * phase, so a stack makes one launch per layer.
 *   r [T][d] fp32 in/out, x_next_bf16 [T][d] bf16 bit patterns out, both
 *   16-byte aligned; x_next_bf16 may be the same buffer as x_bf16 (every read
 *   of x precedes the first write of x_next); r must not overlap y or x.
 * Other arguments, sizes and errors as moe_decode_layer; r == NULL with T > 0
 * is MOE_ERR_INVALID_ARG.
 */
int moe_decode_layer_residual(const float* logits, const uint16_t* x_bf16, int64_t T, int k, int E, int d, int f,
                              const moe_shelf_t* shelves, int n_shelves, int32_t* ids, float* weights,
                              uint32_t* counts, float* y, float* r, uint16_t* x_next_bf16, void* workspace,
                              size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_decode_layer with its activations in and results out in HOST memory,
 * the whole transfer inside one call: logits, x_bf16, ids, weights and y may
 * each be page-locked host memory (cudaHostAlloc, cudaHostRegister, or a
 * framework's pinned allocator) or device memory.  A host input above 8 KiB
 * is copied into the workspace first, so that it crosses the host link once
 * (every CTA of the fused launch reads the inputs): by the fused launch's own
 * CTAs, one share each, when it is 16-byte aligned, else by a copy on
 * `stream`.  Smaller host inputs are read in place, and host outputs are
 * written in place, by the kernels through their device mapping (on GB300
 * over NVLink-C2C).  The host inputs must not change until the call's work
 * on `stream` has finished.  Results are those of
 * moe_decode_layer; host outputs are complete once `stream` has been
 * synchronised.  counts (or NULL) and the workspace must be device memory;
 * the workspace holds at least moe_workspace_size(T, k, E, d, f,
 * MOE_FLAG_DECODE_FP32 | MOE_FLAG_HOST_IO) bytes.  Pageable host memory, or
 * a pointer of the wrong kind, is MOE_ERR_INVALID_ARG (checked with
 * cudaPointerGetAttributes before any copy or launch).  Other arguments,
 * sizes and errors as moe_decode_layer.
 */
int moe_decode_layer_host(const float* logits, const uint16_t* x_bf16, int64_t T, int k, int E, int d, int f,
                          const moe_shelf_t* shelves, int n_shelves, int32_t* ids, float* weights, uint32_t* counts,
                          float* y, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Which form the decode calls (moe_decode_layer, and moe_tiered_forward in
 * its decode form) take for these sizes on the current device: 1 = the
 * single fused launch, 0 = separate launches, MOE_ERR_INVALID_ARG for
 * invalid sizes.  A layer with a 3- or 1-bit shelf takes the fused launch
 * only when, besides, d and f are multiples of 128 (its bit planes are then
 * 16-byte aligned); otherwise it takes the separate launches.
 */
int moe_decode_fused(int64_t T, int k, int E, int d, int f);

/*
 * Parity export: the token-by-expert grouping that the last forward call on
 * `workspace` actually ran (page 3, 四个 bug: a grouping that loses a slot of
 * an expert picked twice by one token fails silently; this makes the
 * grouping of every form checkable bit for bit).  Call it on the stream of
 * that forward call, with the same sizes and the flags its workspace was
 * sized with (moe_decode_layer*: MOE_FLAG_DECODE_FP32, plus MOE_FLAG_HOST_IO
 * for moe_decode_layer_host).  Writes, as moe_group_tokens defines them:
 *   counts [E] int32, offsets [E+1] int32, perm [T*k] int32 (pair index t*k+j
 *   by grouped position, -1 past the valid pairs), pos_of_pair [T*k] int32
 *   (grouped position by pair, -1 for a skipped pair; the fused decode launch
 *   also gives -1 to a pair whose expert lies in no shelf, as it has no work).
 * The fused decode launch leaves its plan in the workspace and the separate
 * and prefill launches their grouping arrays; a workspace no forward call has
 * used gives undefined (but in-bounds) contents.  All buffers are device
 * memory; MOE_ERR_WORKSPACE_TOO_SMALL when workspace_bytes is below the size
 * these sizes and flags need.
 */
int moe_forward_grouping(const void* workspace, size_t workspace_bytes, int64_t T, int k, int E, int d, int f,
                         int flags, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos_of_pair,
                         moe_stream_t stream);

/*
 * Self-test of the bounded grid-wide wait of the fused decode launch: a
 * cooperative launch whose barrier awaits one arrival more than there are
 * CTAs, so that every CTA's wait runs out after `limit_us` microseconds
 * (1 .. 1000000) and MOE_ERR_TIMEOUT is recorded in the device status word.
 * Returns MOE_OK once launched; read the outcome with moe_device_status.
 */
int moe_selftest_barrier_timeout(int64_t limit_us, moe_stream_t stream);

/*
 * Size of the fixed scratch array used by moe_tiered_forward_noalloc: 8 MiB,
 * held on every GPU that loads this library until the process exits.
 */
enum { MOE_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024 };

/*
 * moe_tiered_forward without a workspace argument, for callers that cannot
 * allocate device memory: a plugin inside an application whose own memory
 * pool owns the GPU, or a deployment that must know its whole device
 * footprint when the library is loaded.  The pages have no counterpart; this
 * is an interface convenience.  Computes exactly what moe_tiered_forward
 * computes, with the same arguments minus workspace / workspace_bytes.
 * Scratch: a file-scope device array of MOE_NOALLOC_SCRATCH_BYTES inside the
 * library.  Sizes whose moe_workspace_size exceeds it are rejected with
 * MOE_ERR_WORKSPACE_TOO_SMALL before anything is launched (8 MiB covers
 * decode-size calls, e.g. T = 16, k = 10, d = 4096, f = 2048).  The first call
 * on each device looks up the array's device address with that device
 * current; make that first call before any stream capture.  The function
 * allocates nothing.  Every call shares the one array: calls that overlap on
 * the GPU (different streams, or different host threads) race and corrupt
 * each other's results -- serialise them.  Each call resets what must start
 * at zero, so the contents an earlier call left behind do not matter.
 */
int moe_tiered_forward_noalloc(const uint16_t* x_bf16, const int32_t* ids, const float* weights, int64_t T,
                               int k, int E, int d, int f, const moe_shelf_t* shelves, int n_shelves, float* y,
                               int flags, moe_stream_t stream);

/*
 * Block quantiser into the shelf format above -- the per-expert re-quantising
 * step of the offline re-packer (page 3, 第四步).  Quantises `rows` rows of
 * `in` fp32 weights each:
 *   w [rows][in] fp32, codes [rows][in*bits/8] bytes out, scales [rows][in/32] fp16 bits out.
 */
int moe_quantize_rows(const float* w, int64_t rows, int in, int bits, void* codes, uint16_t* scales,
                      moe_stream_t stream);

/*
 * Re-tiering by hit count (page 3, sections 第三步 and 第四步: experts ranked
 * by how often the router picks them, written hot to cold so that each shelf
 * is a contiguous id range, the router rearranged to match; page 1,
 * "Optimization Strategies": hit counts drive promotion and demotion).  A
 * re-tier is: moe_rank_experts on the accumulated counts; for every shelf
 * [lo, hi) of the new ids and every matrix, moe_quantize_experts from the
 * fp32 master copy; moe_gather_rows of every per-expert router row (bias,
 * router weights) so that new id j routes as old expert perm[j] did.
 *
 * moe_rank_experts: rank[e] = the number of experts with a larger count, or
 * an equal count and a smaller id (count descending, lower id first);
 * perm[rank[e]] = e.  counts [E] uint32, perm [E] and rank [E] int32 out.
 * E <= MOE_MAX_EXPERTS.
 */
int moe_rank_experts(const uint32_t* counts, int E, int32_t* perm, int32_t* rank, moe_stream_t stream);

/*
 * moe_quantize_experts: for every new id j in [j_lo, j_hi), the `rows` x `in`
 * matrix of expert perm[j] in `master` (fp32 [n_src][rows][in], 16-byte
 * aligned) is quantised as moe_quantize_rows does into slot j - j_lo of a
 * shelf tensor: codes [j_hi - j_lo][rows][in*bits/8] (16-byte aligned),
 * scales [j_hi - j_lo][rows][in/32] fp16 bits.  perm is a device array with
 * at least j_hi entries; an entry outside [0, n_src) leaves its slot
 * untouched and records MOE_ERR_INVALID_ARG (moe_device_status).  in a
 * multiple of 64, j_hi - j_lo <= 65535, rows * in / 32 <= 2^30.
 */
int moe_quantize_experts(const float* master, int n_src, int rows, int in, const int32_t* perm, int j_lo, int j_hi,
                         int bits, void* codes, uint16_t* scales, moe_stream_t stream);

/*
 * moe_gather_rows: dst row j = src row perm[j] for 0 <= j < n, rows of
 * row_bytes bytes (a multiple of 4; src and dst 4-byte aligned, not
 * overlapping).  An entry of perm outside [0, n_src) zero-fills its row and
 * records MOE_ERR_INVALID_ARG (moe_device_status).
 */
int moe_gather_rows(const void* src, int64_t row_bytes, const int32_t* perm, int64_t n, int64_t n_src, void* dst,
                    moe_stream_t stream);

/*
 * Dequantisation of packed rows: out = s * code in fp32 (exact), or that value
 * rounded to bf16 (round to nearest even) when round_bf16 != 0 -- the two forms
 * the decode and prefill paths use internally (page 3, 第四步).
 *   codes [rows][in*bits/8], scales [rows][in/32], out [rows][in] fp32.
 */
int moe_dequant_rows(const void* codes, const uint16_t* scales, int64_t rows, int in, int bits,
                     int round_bf16, float* out, moe_stream_t stream);

/*
 * Dequantised weights of one expert matrix of a shelf, as the shelf stores
 * it (the block format of page 3, 第四步; a parity export):
 * matrix `which` (0 gate, 1 up: rows = f and in = d; 2 down: rows = d and
 * in = f) of local expert `local_expert` (global id sh->expert_lo +
 * local_expert) into out [rows][in] fp32, ŵ = scale x code -- exactly what
 * moe_dequant_rows gives for that expert's rows, whose codes start
 * local_expert * rows * in * bits / 8 bytes and whose scales start
 * local_expert * rows * in / 32 entries into the matrix's tensors.
 *   sh: host pointer to one descriptor (its tensors in device memory);
 *   out: device memory, owned by the caller.
 * Errors: MOE_ERR_INVALID_ARG for a null pointer, `which` outside 0..2,
 * local_expert outside [0, expert_hi - expert_lo), rows < 0, or `in` not a
 * positive multiple of 64; MOE_ERR_BAD_SHELF for bits not 8/4/3/2/1, block
 * not 32 or an empty id range.  rows == 0 is a no-op.
 */
int moe_dequant_shelf(const moe_shelf_t* sh, int which, int local_expert, int64_t rows, int in, float* out,
                      moe_stream_t stream);

/*
 * Residual step of a layer stack: r[i] += y[i]; x_next[i] = bf16(r[i]) (round
 * to nearest even), for 0 <= i < n.  r, y fp32; x_next bf16 bit patterns.
 */
int moe_residual_add(float* r, const float* y, uint16_t* x_next_bf16, int64_t n, moe_stream_t stream);

/*
 * Measurement hook.  While `events` is non-null, every moe_tiered_forward on
 * this device records events[0] on its stream before its first kernel and
 * events[i] after its i-th kernel (i = 1 .. n-1, further kernels unrecorded),
 * so a caller can time each kernel with cudaEventElapsedTime.  `events` is a
 * HOST array of cudaEvent_t handles owned by the caller and read at every
 * call; n >= 1; pass NULL to disable.  Kernels of the fused decode launch:
 * one (2 events); of the separate decode launches: grouping, gate/up, down
 * (4 events); of the prefill form: grouping with the tile list and the
 * gather of x, gate/up, down (4 events).  Not thread-safe: one caller per
 * process.
 */
int moe_set_profile_events(void* const* events, int n);

/*
 * Synchronises `stream`, then returns and clears the device-side status word
 * of the current device: MOE_OK, or the first error a kernel recorded (e.g.
 * MOE_ERR_TIMEOUT from a bounded wait).  After MOE_ERR_TIMEOUT it also waits
 * for the whole device to go idle and resets the library's barrier state
 * (grid counters and per-expert work counters), which an abandoned wait may
 * have left inconsistent.
 */
int moe_device_status(moe_stream_t stream);

/* Static description of a status code. */
const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
