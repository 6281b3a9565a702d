// moe_prepare_inputs_noalloc: the staging + dispatch call for callers that
// cannot allocate device memory.
//
// Some callers have no allocator to hand: a plugin inside another runtime
// that is only given its input and output buffers, code that runs while a
// CUDA graph is being captured in a framework that forbids allocation there,
// or a process with a fixed device-memory budget that must never call
// cudaMalloc (which may also synchronise the device).  The dispatch of
// moe_prepare_inputs needs a small scratch area (a block-completion counter,
// per-block expert histograms and per-route ranks); here that scratch is a
// fixed array in device memory that belongs to this library instead of a
// caller-provided workspace.
//
// The array exists on every GPU that loads the library, for as long as the
// process lives.  Its device address is looked up once per device, on the
// first call made with that device current (so make that first call before
// any stream capture).  All calls on a device share the one array and it
// keeps whatever the previous call left in it: the completion counter is
// cleared by every call (an async memset), the rest is fully rewritten.
// Calls that can overlap on the GPU (different streams without ordering)
// race on the array; serialise them.
#include <mutex>

#include "common.cuh"

// Fixed dispatch scratch: 256-byte counter slot + hist [B, E] + ranks [T*k].
static __device__ __align__(256) uint8_t g_dispatch_scratch[MOE_PREPARE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

moe_status_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return moe_host::set_error(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return moe_host::set_error(MOE_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess || p == nullptr)
      return moe_host::set_error(MOE_ERR_CUDA, "cudaGetSymbolAddress(dispatch scratch): %s",
                                 cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_prepare_inputs_noalloc(const moe_prepare_args_t* args,
                                                   void* stream) {
  if (args == nullptr)
    return moe_host::set_error(MOE_ERR_INVALID_ARGUMENT, "args is NULL");
  moe_prepare_args_t a = *args;
  if (a.x_b != nullptr && a.num_tokens > 0 && a.top_k > 0 && a.num_experts > 0) {
    const size_t need = moe_prepare_workspace_size(a.num_tokens, a.top_k, a.num_experts);
    if (need > (size_t)MOE_PREPARE_NOALLOC_SCRATCH_BYTES)
      return moe_host::set_error(
          MOE_ERR_WORKSPACE,
          "moe_prepare_inputs_noalloc: %lld tokens x top-k %lld over %lld experts need %zu bytes "
          "of dispatch scratch; the fixed scratch holds %zu bytes",
          (long long)a.num_tokens, (long long)a.top_k, (long long)a.num_experts, need,
          (size_t)MOE_PREPARE_NOALLOC_SCRATCH_BYTES);
    void* p = nullptr;
    moe_status_t st = scratch_address(&p);
    if (st != MOE_OK) return st;
    a.workspace = p;
    a.workspace_bytes = (size_t)MOE_PREPARE_NOALLOC_SCRATCH_BYTES;
  }
  return moe_prepare_inputs(&a, stream);
}
