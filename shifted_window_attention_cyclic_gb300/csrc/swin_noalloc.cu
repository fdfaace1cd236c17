// swin_noalloc.cu -- swin_attn_bwd_noalloc: the backward pass for callers
// that cannot allocate device memory.
//
// swin_attn_bwd needs a caller-provided workspace for the per-CTA partial
// dBias tables. Some callers have no way to get one: their host code owns no
// device allocator (a C or Fortran model that only receives tensors from its
// host framework), or every byte of device memory belongs to a pool they may
// not touch while stepping. This entry point takes the same tensors as
// swin_attn_bwd but keeps the partial tables in a fixed array that lives in
// this library's device image, so nothing is allocated on any call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/swin_attn.h"

namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kScratchBytes = SWIN_NOALLOC_MAX_WORKSPACE_BYTES;  // partial dBias tables
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

// The host-side name g_bwd_scratch is only a stand-in; its device address
// belongs to one CUDA context. It is looked up with cudaGetSymbolAddress in
// the current context and cached per device together with that context's
// process-unique id, so that a new context on the device (after
// cudaDeviceReset, or a context the caller made current) is looked up anew.
constexpr int kMaxDevices = 64;
struct CachedAddress {
  unsigned long long ctx_id;
  void *addr;
};
std::mutex g_cache_mutex;
CachedAddress g_cache[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Process-unique id of the current context (driver API, reached through the
// runtime's entry-point query so that the library links no libcuda).
int current_context_id(unsigned long long *id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!get_current || !get_id) return SWIN_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return SWIN_ERR_CUDA;
  if (!ctx) {
    // no context bound to this thread yet: bind the device's primary context
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess ||
        get_current(&ctx) != CUDA_SUCCESS || !ctx)
      return SWIN_ERR_CUDA;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? SWIN_OK : SWIN_ERR_CUDA;
}

// Device address of g_bwd_scratch in the current context.
int scratch_in_current_context(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return SWIN_ERR_CUDA;
  if (dev >= kMaxDevices) return SWIN_ERR_UNSUPPORTED;
  unsigned long long id = 0;
  int rc = current_context_id(&id);
  if (rc != SWIN_OK) return rc;
  std::lock_guard<std::mutex> lock(g_cache_mutex);
  CachedAddress &c = g_cache[dev];
  if (!c.addr || c.ctx_id != id) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return SWIN_ERR_CUDA;
    c.addr = p;
    c.ctx_id = id;
  }
  *out = c.addr;
  return SWIN_OK;
}

}  // namespace

extern "C" int swin_attn_bwd_noalloc(swin_attn_plan_t plan, const void *q, const void *k, const void *v,
                                     const void *dout, const float *lse, const float *bias, const uint8_t *land,
                                     void *dq, void *dk, void *dv, float *dbias, swin_stream_t stream) {
  if (!plan) return SWIN_ERR_INVALID_ARG;
  // Without dbias, swin_attn_bwd needs no workspace at all.
  if (!dbias) return swin_attn_bwd(plan, q, k, v, dout, lse, bias, land, dq, dk, dv, nullptr, nullptr, 0, stream);
  if (swin_attn_workspace_bytes(plan) > kScratchBytes) return SWIN_ERR_WORKSPACE;
  void *scratch = nullptr;
  const int rc = scratch_in_current_context(&scratch);
  if (rc != SWIN_OK) return rc;
  // On the success path every partial table the kernel reads is written
  // earlier in the same call, so the array needs no clearing between calls.
  // (A call whose kernel gives up a bounded wait skips writing some tables;
  // its outputs are undefined, as the header states.)
  return swin_attn_bwd(plan, q, k, v, dout, lse, bias, land, dq, dk, dv, dbias, scratch, kScratchBytes, stream);
}
