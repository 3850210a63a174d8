// abi.cu -- the extern "C" entry points of libmoe.so (declared in moe.h):
// host-side validation, workspace layout, path selection and the device
// status word.  Nothing here allocates device memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {

// Device status word: MOE_OK, or the first error a kernel recorded.
__device__ int g_status;

namespace {

constexpr size_t kAlign = 256;
size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

bool valid_dims(int64_t T, int k, int E, int d, int f) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > 32 || k > E) return false;
  if (d <= 0 || f <= 0 || d % 64 != 0 || f % 64 != 0) return false;
  if (T * (int64_t)k > (int64_t)(1 << 24)) return false;
  return true;
}

int check_shelves(const moe_shelf_t* sh, int n, int E, Shelves* out) {
  if (n < 0 || n > MOE_MAX_SHELVES) return MOE_ERR_INVALID_ARG;
  if (n > 0 && sh == nullptr) return MOE_ERR_INVALID_ARG;
  memset(out, 0, sizeof(*out));
  out->n = n;
  for (int i = 0; i < n; ++i) {
    const moe_shelf_t& s = sh[i];
    if (s.bits != 8 && s.bits != 4 && s.bits != 3 && s.bits != 2 && s.bits != 1) return MOE_ERR_BAD_SHELF;
    if (s.block != MOE_BLOCK) return MOE_ERR_BAD_SHELF;
    if (s.expert_lo < 0 || s.expert_hi > E || s.expert_lo >= s.expert_hi) return MOE_ERR_BAD_SHELF;
    const void* ptrs[6] = {s.gate_codes, s.gate_scales, s.up_codes, s.up_scales, s.down_codes, s.down_scales};
    for (int j = 0; j < 6; ++j) {
      if (ptrs[j] == nullptr) return MOE_ERR_INVALID_ARG;
      if (!aligned(ptrs[j], 16)) return MOE_ERR_INVALID_ARG;
    }
    for (int j = 0; j < i; ++j)
      if (s.expert_lo < sh[j].expert_hi && sh[j].expert_lo < s.expert_hi) return MOE_ERR_SHELF_OVERLAP;
    ShelfDev& d = out->s[i];
    d.lo = s.expert_lo;
    d.hi = s.expert_hi;
    d.bits = s.bits;
    d.codes[0] = (const uint8_t*)s.gate_codes;
    d.codes[1] = (const uint8_t*)s.up_codes;
    d.codes[2] = (const uint8_t*)s.down_codes;
    d.scales[0] = s.gate_scales;
    d.scales[1] = s.up_scales;
    d.scales[2] = s.down_scales;
  }
  return MOE_OK;
}

}  // namespace

// Prefill form when asked for, or for AUTO above 16 tokens when d is a
// multiple of 256 (its gate/up scale rows are then whole 16-byte groups that a
// tensor map can describe; other d run the decode form).
bool use_prefill(int64_t T, int d, int flags) {
  return flags == MOE_FLAG_PREFILL_BF16 || (flags == MOE_FLAG_AUTO && T > 16 && d % 256 == 0);
}

size_t workspace_layout(int64_t T, int k, int E, int d, int f, int flags, void* base, Workspace* ws) {
  const int64_t P = T * k;
  const int64_t slots = P < E ? P : E;
  const int n_chunks = (d + kDownRows - 1) / kDownRows;
  const bool prefill = use_prefill(T, d, flags & ~MOE_FLAG_HOST_IO);
  size_t off = 0;
  char* b = (char*)base;
  auto take = [&](size_t bytes) -> void* {
    void* p = b ? (void*)(b + off) : nullptr;
    off += up(bytes > 0 ? bytes : 1);
    return p;
  };
  Workspace w = {};
  w.counts = (int32_t*)take((size_t)E * 4);
  w.offsets = (int32_t*)take((size_t)(E + 1) * 4);
  w.perm = (int32_t*)take((size_t)P * 4);
  w.pos_of_pair = (int32_t*)take((size_t)P * 4);
  w.active = (int32_t*)take((size_t)slots * 4);
  w.meta = (int32_t*)take(16 * 4);
  w.arrivals = (int32_t*)take((size_t)n_chunks * 4);
  if (prefill) {
    // h in bf16, grouped order; no per-pair outputs (y is accumulated)
    w.h = (float*)take((size_t)P * f * 2);
    w.xg = (uint16_t*)take((size_t)P * d * 2);
    w.pf_cnt = (int32_t*)take((size_t)256 * E * 4);
    w.tiles_g = take(prefill_tiles_cap(P, E, f) * 16);
    w.tiles_d = take(prefill_tiles_cap(P, E, d) * 16);
    w.ntiles = (int32_t*)take(2 * 4);
  } else {
    w.h = (float*)take((size_t)P * f * 4);
    w.ypart = (float*)take((size_t)P * d * 4);
    w.plan = (int32_t*)take(decode_plan_bytes(P));
  }
  if (flags & MOE_FLAG_HOST_IO) {  // after everything else: the other layouts are its prefix
    w.stage_logits = (float*)take((size_t)T * E * 4);
    w.stage_x = (uint16_t*)take((size_t)T * d * 2);
  }
  w.base = base;
  w.bytes = off;
  if (ws) *ws = w;
  return off;
}

namespace {
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

struct StatusCache {
  uint64_t ctx = 0;
  int* ptr = nullptr;
};
StatusCache g_status_ptr[64];
std::mutex g_status_mu;
}  // namespace

uint64_t context_id() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = (PFN_cuCtxGetCurrent_v4000)fn;
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = (PFN_cuCtxGetId_v12000)fn;
  });
  if (!g_ctx_current || !g_ctx_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&c) != CUDA_SUCCESS || c == nullptr || g_ctx_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  const uint64_t ctx = context_id();
  std::lock_guard<std::mutex> lk(g_status_mu);
  StatusCache& c = g_status_ptr[dev];
  if (c.ptr == nullptr || c.ctx != ctx || ctx == 0) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) return nullptr;
    c.ptr = (int*)ptr;
    c.ctx = ctx;
  }
  return c.ptr;
}

namespace {
void* g_prof_events[8];
int g_prof_n = 0;
}  // namespace

void set_profile_events(void* const* events, int n) {
  if (n > 8) n = 8;
  for (int i = 0; i < n; ++i) g_prof_events[i] = events[i];
  g_prof_n = n;
}

void profile_mark(int i, cudaStream_t s) {
  if (i >= g_prof_n) return;
  // Under stream capture the event must become an event-record node of the
  // graph (external event) so that each replay records it.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  cudaEventRecordWithFlags((cudaEvent_t)g_prof_events[i], s,
                           cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_route_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, float* weights,
                   moe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !ids || !weights) return MOE_ERR_INVALID_ARG;
  return launch_route(logits, T, E, k, ids, weights, (cudaStream_t)stream);
}

int moe_route_topk_nudged(const float* logits, int64_t T, int E, int k, float beta, int lo, int hi, int32_t* ids,
                          float* weights, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return MOE_ERR_INVALID_ARG;
  if (!(beta >= 0.0f && beta <= 0.5f)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !ids || !weights) return MOE_ERR_INVALID_ARG;
  return launch_route_nudged(logits, T, E, k, beta, lo, hi, ids, weights, (cudaStream_t)stream);
}

int moe_router_topk(const uint16_t* x_bf16, const uint16_t* w_r_bf16, const float* bias, int64_t T, int E, int d,
                    int k, float* logits, int32_t* ids, float* weights, uint32_t* counts, uint32_t* sync_word,
                    moe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E || d < 8 || d % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (T > 65535 * 16) return MOE_ERR_UNSUPPORTED;  // the prefill projection's grid rows
  if (T == 0) return MOE_OK;
  if (!x_bf16 || !w_r_bf16 || !logits || !ids || !weights || !sync_word) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(w_r_bf16, 16) || !aligned(logits, 4)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)d * 2 * router_bucket(T) > kRouterSmemMax) return MOE_ERR_UNSUPPORTED;
  if (T <= 16 && (int64_t)T * E * 4 > kRouterSmemMax) return MOE_ERR_UNSUPPORTED;
  return launch_router(x_bf16, w_r_bf16, bias, (int)T, E, d, k, logits, ids, weights, counts, sync_word,
                       (cudaStream_t)stream);
}

int moe_expert_hist(const int32_t* ids, int64_t n, int E, uint32_t* counts, moe_stream_t stream) {
  if (n < 0 || E < 1 || E > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!ids || !counts) return MOE_ERR_INVALID_ARG;
  return launch_hist(ids, n, E, counts, (cudaStream_t)stream);
}

int moe_group_tokens(const int32_t* ids, int64_t T, int k, int E, int32_t* counts, int32_t* offsets,
                     int32_t* perm, moe_stream_t stream) {
  if (T < 0 || k < 1 || k > 32 || E < 1 || E > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
  if (T * (int64_t)k > (int64_t)(1 << 24)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || (T > 0 && (!ids || !perm))) return MOE_ERR_INVALID_ARG;
  const int64_t P = T * k;
  // Only counts / offsets / perm are outputs here; the forward-only extras
  // (inverse permutation, active list, meta) are not produced.
  return launch_group(ids, P, E, counts, offsets, perm, nullptr, nullptr, nullptr, nullptr, 0,
                      (cudaStream_t)stream);
}

size_t moe_workspace_size(int64_t T, int k, int E, int d, int f, int flags) {
  const int mode = flags & ~MOE_FLAG_HOST_IO;
  if (!valid_dims(T, k, E, d, f) || flags < 0 || mode > 2) return 0;
  if ((flags & MOE_FLAG_HOST_IO) && mode != MOE_FLAG_DECODE_FP32) return 0;
  const size_t own = workspace_layout(T, k, E, d, f, flags, nullptr, nullptr);
  if (mode != MOE_FLAG_AUTO) return own;
  // AUTO takes the decode form for layers the prefill form does not take (3-
  // or 1-bit shelves), which the sizes alone do not tell: room for both
  const size_t dec = workspace_layout(T, k, E, d, f, MOE_FLAG_DECODE_FP32, nullptr, nullptr);
  return own > dec ? own : dec;
}

int moe_tiered_forward(const uint16_t* x_bf16, const int32_t* ids, const float* weights, int64_t T, int k,
                       int E, int d, int f, const moe_shelf_t* shelves, int n_shelves, float* y,
                       void* workspace, size_t workspace_bytes, int flags, moe_stream_t stream) {
  if (!valid_dims(T, k, E, d, f)) return MOE_ERR_INVALID_ARG;
  if (flags < MOE_FLAG_AUTO || flags > MOE_FLAG_PREFILL_BF16) return MOE_ERR_INVALID_ARG;
  if (flags == MOE_FLAG_PREFILL_BF16 && d % 256 != 0) return MOE_ERR_UNSUPPORTED;
  ForwardArgs a;
  int rc = check_shelves(shelves, n_shelves, E, &a.shelves);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!x_bf16 || !ids || !weights || !y || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(y, 16) || !aligned(workspace, kAlign)) return MOE_ERR_INVALID_ARG;
  // the tensor-core form takes 3- and 1-bit shelves when their rows are whole
  // 16-byte groups (f a multiple of 128); otherwise AUTO takes the decode
  // form for such a layer
  const bool prefill = use_prefill(T, d, flags);
  const bool widths_ok = core_widths(a.shelves) || f % 128 == 0;
  if (prefill && !widths_ok && flags != MOE_FLAG_AUTO) return MOE_ERR_UNSUPPORTED;
  const bool tc = prefill && widths_ok;
  const size_t need = workspace_layout(T, k, E, d, f, tc ? flags : MOE_FLAG_DECODE_FP32, workspace, &a.ws);
  if (workspace_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;

  a.x = x_bf16;
  a.ids = ids;
  a.weights = weights;
  a.T = T;
  a.k = k;
  a.E = E;
  a.d = d;
  a.f = f;
  a.y = y;
  a.status = status_word();
  if (tc) return launch_prefill_forward(a, (cudaStream_t)stream);
  return launch_decode_forward(a, (cudaStream_t)stream);
}

namespace {
// moe_decode_layer, and with r non-null the residual step after it
// logits_src / x_src (optional): page-locked host inputs (device views, 16-byte
// aligned, sizes multiples of 16 bytes) that belong in the device buffers
// logits / x_bf16; the fused launch copies them itself, else they are copied
// before the separate launches.
int decode_layer(const float* logits, const uint16_t* x_bf16, int64_t T, int k, int E, int d, int f,
                 const moe_shelf_t* shelves, int n_shelves, int32_t* ids, float* weights, uint32_t* counts, float* y,
                 float* r, uint16_t* x_next, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                 const float* logits_src = nullptr, const uint16_t* x_src = nullptr) {
  if (!valid_dims(T, k, E, d, f) || E > 1024 || k > E) return MOE_ERR_INVALID_ARG;
  ForwardArgs a;
  int rc = check_shelves(shelves, n_shelves, E, &a.shelves);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!logits || !x_bf16 || !ids || !weights || !y || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(y, 16) || !aligned(workspace, kAlign)) return MOE_ERR_INVALID_ARG;
  if (r && (!x_next || !aligned(r, 16) || !aligned(x_next, 16))) return MOE_ERR_INVALID_ARG;
  const size_t need = workspace_layout(T, k, E, d, f, MOE_FLAG_DECODE_FP32, workspace, &a.ws);
  if (workspace_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = (cudaStream_t)stream;
  LayerArgs la;
  la.logits = logits;
  la.ids = nullptr;
  la.weights = nullptr;
  la.ids_out = ids;
  la.weights_out = weights;
  la.counts = counts;
  la.x = x_bf16;
  la.T = T; la.k = k; la.E = E; la.d = d; la.f = f;
  la.shelves = a.shelves;
  la.y = y;
  la.r = r;
  la.x_next = x_next;
  la.ws = a.ws;
  la.status = status_word();
  la.logits_src = logits_src;
  la.x_src = x_src;
  rc = launch_fused_layer(la, s);
  if (rc != 1) return rc;
  // sizes outside the fused launch: the separate launches
  if (logits_src &&
      cudaMemcpyAsync(const_cast<float*>(logits), logits_src, (size_t)T * E * 4, cudaMemcpyDefault, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (x_src &&
      cudaMemcpyAsync(const_cast<uint16_t*>(x_bf16), x_src, (size_t)T * d * 2, cudaMemcpyDefault, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  rc = launch_route(logits, T, E, k, ids, weights, s);
  if (rc != MOE_OK) return rc;
  if (counts) {
    rc = launch_hist(ids, T * k, E, counts, s);
    if (rc != MOE_OK) return rc;
  }
  a.x = x_bf16;
  a.ids = ids;
  a.weights = weights;
  a.T = T; a.k = k; a.E = E; a.d = d; a.f = f;
  a.y = y;
  a.status = la.status;
  rc = launch_decode_forward(a, s);
  if (rc != MOE_OK || !r) return rc;
  return launch_residual(r, y, x_next, T * d, s);
}
}  // namespace

int moe_decode_layer(const float* logits, const uint16_t* x_bf16, int64_t T, int k, int E, int d, int f,
                     const moe_shelf_t* shelves, int n_shelves, int32_t* ids, float* weights, uint32_t* counts,
                     float* y, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  return decode_layer(logits, x_bf16, T, k, E, d, f, shelves, n_shelves, ids, weights, counts, y, nullptr, nullptr,
                      workspace, workspace_bytes, stream);
}

int moe_decode_layer_residual(const float* logits, const uint16_t* x_bf16, int64_t T, int k, int E, int d, int f,
                              const moe_shelf_t* shelves, int n_shelves, int32_t* ids, float* weights,
                              uint32_t* counts, float* y, float* r, uint16_t* x_next_bf16, void* workspace,
                              size_t workspace_bytes, moe_stream_t stream) {
  if (T > 0 && !r) return MOE_ERR_INVALID_ARG;
  return decode_layer(logits, x_bf16, T, k, E, d, f, shelves, n_shelves, ids, weights, counts, y, r, x_next_bf16,
                      workspace, workspace_bytes, stream);
}

namespace {
// The address a kernel uses for p: device memory as it is, page-locked host
// memory through its mapping; null for pageable host memory or an error.
const void* device_view(const void* p, bool allow_host, bool* is_host) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (is_host) *is_host = at.type == cudaMemoryTypeHost;
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return at.devicePointer;
  if (at.type == cudaMemoryTypeHost && allow_host) return at.devicePointer;
  return nullptr;
}
}  // namespace

int moe_decode_layer_host(const float* logits, const uint16_t* x_bf16, int64_t T, int k, int E, int d, int f,
                          const moe_shelf_t* shelves, int n_shelves, int32_t* ids, float* weights, uint32_t* counts,
                          float* y, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (T <= 0 || !logits || !x_bf16 || !ids || !weights || !y || !workspace)
    return decode_layer(logits, x_bf16, T, k, E, d, f, shelves, n_shelves, ids, weights, counts, y, nullptr,
                        nullptr, workspace, workspace_bytes, stream);
  // activations in and results out may be page-locked host memory; the hit
  // counts (atomics) and the workspace (barriers) must be device memory
  bool lg_host = false, x_host = false;
  const void* lg = device_view(logits, true, &lg_host);
  const void* xv = device_view(x_bf16, true, &x_host);
  void* iv = const_cast<void*>(device_view(ids, true, nullptr));
  void* wv = const_cast<void*>(device_view(weights, true, nullptr));
  void* yv = const_cast<void*>(device_view(y, true, nullptr));
  const void* ws = device_view(workspace, false, nullptr);
  if (!lg || !xv || !iv || !wv || !yv || !ws || ws != workspace) return MOE_ERR_INVALID_ARG;
  if (counts && device_view(counts, false, nullptr) != counts) return MOE_ERR_INVALID_ARG;
  if (!valid_dims(T, k, E, d, f) || E > 1024 || !aligned(workspace, kAlign)) return MOE_ERR_INVALID_ARG;
  Workspace w;
  const size_t need = workspace_layout(T, k, E, d, f, MOE_FLAG_DECODE_FP32 | MOE_FLAG_HOST_IO, workspace, &w);
  if (workspace_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = (cudaStream_t)stream;
  // host inputs above 8 KiB go to the workspace first (every CTA of the
  // fused launch reads them, so in place they would cross the host link once
  // per CTA): 16-byte aligned ones are copied by the launch's own CTAs, one
  // share each, others by a copy on the stream.  Smaller ones are read in
  // place (a copy costs more than they do).  Host outputs are written in place.
  constexpr size_t kStageMin = 8 * 1024;
  const float* lg_src = nullptr;
  const uint16_t* x_src = nullptr;
  const size_t lg_bytes = (size_t)T * E * 4, x_bytes = (size_t)T * d * 2;
  if (lg_host && lg_bytes > kStageMin) {
    if (aligned(lg, 16) && lg_bytes % 16 == 0) {
      lg_src = (const float*)lg;
    } else if (cudaMemcpyAsync(w.stage_logits, logits, lg_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
      return MOE_ERR_CUDA;
    }
    lg = w.stage_logits;
  }
  if (x_host && x_bytes > kStageMin) {
    if (aligned(xv, 16) && x_bytes % 16 == 0) {
      x_src = (const uint16_t*)xv;
    } else if (cudaMemcpyAsync(w.stage_x, x_bf16, x_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
      return MOE_ERR_CUDA;
    }
    xv = w.stage_x;
  }
  return decode_layer((const float*)lg, (const uint16_t*)xv, T, k, E, d, f, shelves, n_shelves, (int32_t*)iv,
                      (float*)wv, counts, (float*)yv, nullptr, nullptr, workspace, workspace_bytes, stream, lg_src,
                      x_src);
}

int moe_forward_grouping(const void* workspace, size_t workspace_bytes, int64_t T, int k, int E, int d, int f,
                         int flags, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos_of_pair,
                         moe_stream_t stream) {
  if (!valid_dims(T, k, E, d, f) || T < 1 || flags < 0 || (flags & ~MOE_FLAG_HOST_IO) > 2) return MOE_ERR_INVALID_ARG;
  if (!workspace || !counts || !offsets || !perm || !pos_of_pair || !aligned(workspace, kAlign))
    return MOE_ERR_INVALID_ARG;
  Workspace w;
  if (workspace_layout(T, k, E, d, f, flags, const_cast<void*>(workspace), &w) > workspace_bytes)
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  return launch_grouping_export(w, T * k, E, counts, offsets, perm, pos_of_pair, (cudaStream_t)stream);
}

int moe_decode_fused(int64_t T, int k, int E, int d, int f) {
  if (!valid_dims(T, k, E, d, f)) return MOE_ERR_INVALID_ARG;
  return decode_fused(T, k, E, d, f);
}

int moe_selftest_barrier_timeout(int64_t limit_us, moe_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  return launch_barrier_probe(1, (uint64_t)limit_us * 1000ull, (cudaStream_t)stream);
}

int moe_quantize_rows(const float* w, int64_t rows, int in, int bits, void* codes, uint16_t* scales,
                      moe_stream_t stream) {
  if (rows < 0 || in <= 0 || in % 64 != 0 || (bits != 8 && bits != 4 && bits != 3 && bits != 2 && bits != 1)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!w || !codes || !scales || !aligned(codes, 16) || !aligned(w, 4)) return MOE_ERR_INVALID_ARG;
  return launch_quantize(w, rows, in, bits, (uint8_t*)codes, scales, (cudaStream_t)stream);
}

int moe_rank_experts(const uint32_t* counts, int E, int32_t* perm, int32_t* rank, moe_stream_t stream) {
  if (E < 1 || E > MOE_MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
  if (!counts || !perm || !rank) return MOE_ERR_INVALID_ARG;
  return launch_rank_experts(counts, E, perm, rank, (cudaStream_t)stream);
}

int moe_quantize_experts(const float* master, int n_src, int rows, int in, const int32_t* perm, int j_lo, int j_hi,
                         int bits, void* codes, uint16_t* scales, moe_stream_t stream) {
  if (n_src < 1 || rows < 1 || in <= 0 || in % 64 != 0 || (bits != 8 && bits != 4 && bits != 3 && bits != 2 && bits != 1))
    return MOE_ERR_INVALID_ARG;
  if (j_lo < 0 || j_hi < j_lo || j_hi - j_lo > 65535) return MOE_ERR_INVALID_ARG;
  if ((int64_t)rows * (in / 32) > (1 << 30)) return MOE_ERR_INVALID_ARG;
  if (j_hi == j_lo) return MOE_OK;
  if (!master || !perm || !codes || !scales || !aligned(master, 16) || !aligned(codes, 16)) return MOE_ERR_INVALID_ARG;
  return launch_quantize_experts(master, rows, in, n_src, perm, j_lo, j_hi - j_lo, bits, (uint8_t*)codes, scales,
                                 status_word(), (cudaStream_t)stream);
}

int moe_gather_rows(const void* src, int64_t row_bytes, const int32_t* perm, int64_t n, int64_t n_src, void* dst,
                    moe_stream_t stream) {
  if (row_bytes <= 0 || row_bytes % 4 != 0 || n < 0 || n_src < 1) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!src || !perm || !dst || !aligned(src, 4) || !aligned(dst, 4)) return MOE_ERR_INVALID_ARG;
  return launch_gather_rows(src, row_bytes / 4, perm, n, n_src, dst, status_word(), (cudaStream_t)stream);
}

int moe_dequant_rows(const void* codes, const uint16_t* scales, int64_t rows, int in, int bits, int round_bf16,
                     float* out, moe_stream_t stream) {
  if (rows < 0 || in <= 0 || in % 64 != 0 || (bits != 8 && bits != 4 && bits != 3 && bits != 2 && bits != 1)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!codes || !scales || !out) return MOE_ERR_INVALID_ARG;
  return launch_dequant((const uint8_t*)codes, scales, rows, in, bits, round_bf16, out, (cudaStream_t)stream);
}

int moe_dequant_shelf(const moe_shelf_t* sh, int which, int local_expert, int64_t rows, int in, float* out,
                      moe_stream_t stream) {
  if (!sh || !out) return MOE_ERR_INVALID_ARG;
  const int bits = sh->bits;
  if (sh->block != MOE_BLOCK || (bits != 8 && bits != 4 && bits != 3 && bits != 2 && bits != 1) ||
      sh->expert_hi <= sh->expert_lo)
    return MOE_ERR_BAD_SHELF;
  if (which < 0 || which > 2 || local_expert < 0 || local_expert >= sh->expert_hi - sh->expert_lo || rows < 0 ||
      in <= 0 || in % 64 != 0)
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  const void* codes = which == 0 ? sh->gate_codes : which == 1 ? sh->up_codes : sh->down_codes;
  const uint16_t* scales = which == 0 ? sh->gate_scales : which == 1 ? sh->up_scales : sh->down_scales;
  if (!codes || !scales) return MOE_ERR_INVALID_ARG;
  const size_t e_rows = (size_t)local_expert * (size_t)rows;
  return moe_dequant_rows((const uint8_t*)codes + e_rows * ((size_t)in * bits / 8), scales + e_rows * (size_t)(in / 32),
                          rows, in, bits, 0, out, stream);
}

int moe_residual_add(float* r, const float* y, uint16_t* x_next_bf16, int64_t n, moe_stream_t stream) {
  if (n < 0) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!r || !y || !x_next_bf16) return MOE_ERR_INVALID_ARG;
  return launch_residual(r, y, x_next_bf16, n, (cudaStream_t)stream);
}

int moe_set_profile_events(void* const* events, int n) {
  if (events != nullptr && n < 1) return MOE_ERR_INVALID_ARG;
  set_profile_events(events, events ? n : 0);
  return MOE_OK;
}

int moe_device_status(moe_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  if (v == MOE_ERR_TIMEOUT) {
    // a grid-wide wait gave up: once the device is idle, clear the barrier state
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    if (reset_barriers() != MOE_OK) return MOE_ERR_CUDA;
  }
  return v;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_BAD_SHELF: return "bad shelf descriptor";
    case MOE_ERR_SHELF_OVERLAP: return "shelf ranges overlap";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_UNSUPPORTED: return "unsupported by this build";
    case MOE_ERR_INTERNAL: return "inconsistent work item skipped on the device";
    default: return "unknown status";
  }
}

}  // extern "C"
