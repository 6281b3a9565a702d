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
// any stream capture), and again if the device's context has changed since
// (after a device reset the module is loaded anew, maybe elsewhere).  All
// calls on a device share the one array and it keeps whatever the previous
// call left in it: the completion counter is cleared by every call (an async
// memset), the rest is fully rewritten.
// Calls that can overlap on the GPU (different streams without ordering)
// race on the array; serialise them.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

// Fixed dispatch scratch: 256-byte counter slot + hist [B, E] + ranks [T*k].
static __device__ __align__(256) uint8_t g_dispatch_scratch[MOE_PREPARE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
struct ScratchEntry {
  unsigned long long ctx_id;  // context the address belongs to (0: not looked up yet)
  void* ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Unique id of the calling thread's current context (0 when none is current
// yet or the driver does not provide the query).  The array's address belongs
// to the context the module was loaded into: after a device reset the
// primary context is a new one, and the address is looked up again.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrent)(CUcontext*);
  typedef CUresult (*GetId)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static bool resolved = false;
  if (!resolved) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<GetCurrent>(f1);
      get_id = reinterpret_cast<GetId>(f2);
    }
    resolved = true;
  }
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

moe_status_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return moe_host::set_error(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return moe_host::set_error(MOE_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mutex);
  unsigned long long ctx = current_context_id();
  ScratchEntry& ent = g_scratch[dev];
  if (ent.ptr == nullptr || ctx == 0 || ent.ctx_id != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess || p == nullptr)
      return moe_host::set_error(MOE_ERR_CUDA, "cudaGetSymbolAddress(dispatch scratch): %s",
                                 cudaGetErrorString(e));
    ent.ptr = p;
    // the lookup makes the primary context current if it was not yet
    ent.ctx_id = ctx != 0 ? ctx : current_context_id();
  }
  *out = ent.ptr;
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
