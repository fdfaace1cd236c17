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
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/swin_attn.h"

namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kScratchBytes = SWIN_NOALLOC_MAX_WORKSPACE_BYTES;  // partial dBias tables
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];

// Device address of g_bwd_scratch on the current device. The host-side name
// is only a stand-in, so the address is looked up once per device (with that
// device current) and cached.
int scratch_on_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return SWIN_ERR_CUDA;
  if (dev >= kMaxDevices) return SWIN_ERR_UNSUPPORTED;
  void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return SWIN_ERR_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return SWIN_OK;
}

}  // namespace

extern "C" int swin_attn_bwd_noalloc(swin_attn_plan_t plan, const void *q, const void *k, const void *v,
                                     const void *dout, const float *lse, const float *bias, const uint8_t *land,
                                     void *dq, void *dk, void *dv, float *dbias, swin_stream_t stream) {
  if (!plan) return SWIN_ERR_INVALID_ARG;
  if (swin_attn_workspace_bytes(plan) > kScratchBytes) return SWIN_ERR_WORKSPACE;
  void *scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != SWIN_OK) return rc;
  // Every partial table the kernel reads is written earlier in the same call,
  // so the array needs no clearing between calls.
  return swin_attn_bwd(plan, q, k, v, dout, lse, bias, land, dq, dk, dv, dbias, scratch, kScratchBytes, stream);
}
