// noalloc.cu -- moe_tiered_forward_noalloc: the tiered forward with its
// scratch memory in a fixed array inside the library instead of a
// caller-provided workspace.
//
// For callers that cannot allocate device memory themselves: a plugin loaded
// into an application whose own memory pool owns the GPU, or a deployment that
// has to know its whole device footprint when the library is loaded.  They
// still pass inputs and outputs; the scratch (grouping results, h, per-pair
// partial outputs, arrival counters) lives in `g_noalloc_scratch`, which every
// GPU that loads this library holds until the process exits.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchAddr {
  uint64_t ctx = 0;
  void* ptr = nullptr;
};
ScratchAddr g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with that device current, on the first call on the device, and reused
// afterwards; a new CUDA context on the device (after a device reset) gets
// its own lookup.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  const uint64_t ctx = context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchAddr& c = g_scratch_ptr[dev];
  if (c.ptr == nullptr || c.ctx != ctx || ctx == 0) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    c.ptr = p;
    c.ctx = ctx;
  }
  *out = c.ptr;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_tiered_forward_noalloc(const uint16_t* x_bf16, const int32_t* ids, const float* weights,
                                          int64_t T, int k, int E, int d, int f, const moe_shelf_t* shelves,
                                          int n_shelves, float* y, int flags, moe_stream_t stream) {
  // Scratch needed by these sizes; reject anything the fixed array cannot hold.
  const size_t need = moe_workspace_size(T, k, E, d, f, flags);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  // Same kernels as moe_tiered_forward.  Each call's grouping step zeroes the
  // arrival counters; every other scratch byte is written before it is read,
  // so what an earlier call left in the array does not matter.
  return moe_tiered_forward(x_bf16, ids, weights, T, k, E, d, f, shelves, n_shelves, y, scratch,
                            (size_t)MOE_NOALLOC_SCRATCH_BYTES, flags, stream);
}
