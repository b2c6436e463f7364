// noalloc.cu -- ring-attention forward for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain a workspace: code that runs under a host
// framework which owns every device allocation (a plugin handed only its
// input and output buffers), or a serving loop where a cudaMalloc would
// synchronise the device or break a fixed memory budget.  ra_fwd_noalloc runs
// the same forward as ra_fwd, with its workspace taken from a file-scope
// device array that is part of this library's module image.  Every GPU that
// loads the library holds that array until the process exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/ring_attn.h"
#include "ring_attn_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

// The scratch.  In host code this name is only a stand-in for the symbol; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
struct Cached {
  unsigned long long ctx_id;  // the context the address belongs to (0: none yet)
  void* addr;
};
Cached g_cache[kMaxDevices] = {};

// Identity of the thread's current context (cuCtxGetCurrent + cuCtxGetId,
// fetched through the runtime's driver entry points; no libcuda link).
// Returns false when there is no current context or the entry points are
// unavailable.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch on the current device.  The set-up (the
// cudaGetSymbolAddress lookup, with the device current) runs on the first
// call on a device and again whenever that device's context has been
// re-created since (after a cudaDeviceReset, for instance: the module, and
// with it the array, is then loaded anew at another address).
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  if (have_id && g_cache[dev].addr && g_cache[dev].ctx_id == id) {
    *out = g_cache[dev].addr;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  // the lookup made the device's context current if none was: record it now
  g_cache[dev].ctx_id = current_context_id(&id) ? id : 0;
  g_cache[dev].addr = g_cache[dev].ctx_id ? p : nullptr;  // no identity: look it up on every call
  *out = p;
  return cudaSuccess;
}

ra_status address_failure(cudaError_t e) {
  char msg[256];
  snprintf(msg, sizeof(msg), "no-allocation forward: cudaGetSymbolAddress of the scratch failed: %s",
           cudaGetErrorString(e));
  return ra::set_last_error(RA_ERR_CUDA, msg);
}

}  // namespace

extern "C" ra_status ra_fwd_noalloc(const ra_plan* plan, const void* q, const void* k, const void* v, void* o,
                                    int32_t o_is_fp32, float* lse, void* stream) {
  if (!plan) return ra::set_last_error(RA_ERR_INVALID_ARG, "plan is NULL");
  size_t need = 0;
  ra_status rs = ra_plan_workspace_bytes(plan, o_is_fp32, 0, &need, nullptr);
  if (rs != RA_OK) return rs;
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "ra_fwd_noalloc: this plan needs %zu bytes of scratch, above the fixed maximum of %zu bytes "
             "(use ra_fwd with a caller-provided workspace)",
             need, kNoAllocScratchBytes);
    return ra::set_last_error(RA_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return address_failure(e);
  // The forward zeroes the status word and rewrites the work lists before
  // its kernel reads them, so the previous call's contents of the scratch
  // never leak into this one.
  return ra_fwd(plan, q, k, v, o, o_is_fp32, lse, scratch, kNoAllocScratchBytes, stream);
}

extern "C" ra_status ra_noalloc_status(void* stream) {
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return address_failure(e);
  return ra_workspace_status(scratch, stream);
}
