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
void* g_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
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
             "(use ra_fwd with a caller-provided workspace, or o_is_fp32 = 1 to drop the fp32 running output)",
             need, kNoAllocScratchBytes);
    return ra::set_last_error(RA_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "ra_fwd_noalloc: cudaGetSymbolAddress of the scratch failed: %s",
             cudaGetErrorString(e));
    return ra::set_last_error(RA_ERR_CUDA, msg);
  }
  // The forward resets the status word and rewrites the work list and the
  // running output before reading them, so the previous call's contents of
  // the scratch never leak into this one.
  return ra_fwd(plan, q, k, v, o, o_is_fp32, lse, scratch, kNoAllocScratchBytes, stream);
}
