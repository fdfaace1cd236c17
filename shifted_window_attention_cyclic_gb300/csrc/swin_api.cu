// swin_api.cu -- the C ABI (include/swin_attn.h): plan building, argument
// checks, launches, the dBias fold and the device status word.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "swin_common.cuh"
#include "swin_tc.cuh"

using namespace swin;

struct swin_attn_plan_s {
  swin_attn_desc d;
  Geo g;
  int device;
  int num_sms;
  int impl;
  int fwd_ctas, bwd_ctas;
  int64_t items;           // work items of the backward (and of the forward, but for head_dim 128)
  int64_t fwd_items;       // work items of the forward
  int64_t ws_slots;
  int32_t *d_win_src;
  uint8_t *d_region;
  int32_t *d_tok_dst;
  int32_t *d_relidx;
  int *d_status;
  int *d_slot_base;        // [bwd_ctas]
  int *d_head_slot_begin;  // [heads + 1]
  uint64_t wait_limit_ns;  // bound of every in-kernel wait
  int debug_force_timeout;
  bool large;              // head_dim 128: key-tiled kernels for windows of any size
};

namespace {

// ---- routing tables, built on the device with the kernels' own routing ----
__global__ void tables_kernel(Geo g, int32_t *win_src, uint8_t *region, int32_t *tok_dst) {
  const int64_t total = (int64_t)g.nwin * g.n;
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total; x += (int64_t)gridDim.x * blockDim.x) {
    const int omega = (int)(x / g.n), sigma = (int)(x % g.n);
    int wc[3];
    window_coords(g, omega, wc);
    const SlotRoute r = slot_route(g, wc, sigma);
    win_src[x] = r.src;
    region[x] = (uint8_t)r.reg;
    if (r.src >= 0) tok_dst[r.src] = (int32_t)x;
  }
}

__global__ void relidx_kernel(Geo g, int32_t *relidx) {
  const int wc[3] = {0, 0, 0};
  for (int x = blockIdx.x * blockDim.x + threadIdx.x; x < g.n * g.n; x += gridDim.x * blockDim.x) {
    const int i = x / g.n, j = x % g.n;
    relidx[x] = slot_route(g, wc, i).rbase - slot_route(g, wc, j).roff;
  }
}

// dbias[t][h] = sum over the workspace slots of head h, in slot order.
__global__ void fold_kernel(FoldArgs a) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= a.T * a.heads) return;
  const int t = x / a.heads, h = x % a.heads;
  float sum = 0.f;
  for (int s = a.head_slot_begin[h]; s < a.head_slot_begin[h + 1]; ++s) sum += a.ws[(int64_t)s * a.T + t];
  a.dbias[x] = sum;
}

constexpr int64_t kMaxSlots = 65536;       // slots per window
constexpr int64_t kMaxRelidxSlots = 2048;  // the plan keeps the [n][n] bias-row table up to this n

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_desc(const swin_attn_desc *d) {
  if (!d) return SWIN_ERR_INVALID_ARG;
  if (d->ndim != 2 && d->ndim != 3) return SWIN_ERR_INVALID_ARG;
  if (d->batch < 1 || d->heads < 1) return SWIN_ERR_INVALID_ARG;
  if (d->dtype != SWIN_F32 && d->dtype != SWIN_BF16) return SWIN_ERR_UNSUPPORTED;
  if (d->impl < SWIN_IMPL_AUTO || d->impl > SWIN_IMPL_TC) return SWIN_ERR_INVALID_ARG;
  if (d->has_land != 0 && d->has_land != 1) return SWIN_ERR_INVALID_ARG;
  int64_t tokens = 1, n = 1;
  for (int a = 0; a < d->ndim; ++a) {
    if (d->grid[a] < 1 || d->window[a] < 1) return SWIN_ERR_INVALID_ARG;
    if (d->shift[a] < 0 || d->shift[a] >= d->window[a]) return SWIN_ERR_INVALID_ARG;
    if (d->shift[a] > 0 && d->shift[a] >= d->grid[a]) return SWIN_ERR_INVALID_ARG;
    if (d->periodic[a] != 0 && d->periodic[a] != 1) return SWIN_ERR_INVALID_ARG;
    tokens *= d->grid[a];
    n *= d->window[a];
    if (tokens >= (int64_t(1) << 31) || n > kMaxSlots) return SWIN_ERR_UNSUPPORTED;
  }
  if (d->head_dim != 16 && d->head_dim != 32 && d->head_dim != 128) return SWIN_ERR_UNSUPPORTED;
  // windows of more than 128 slots: head_dim 128, bf16 (the key-tiled kernels)
  if ((n > 128 || d->head_dim == 128) && (d->head_dim != 128 || d->dtype != SWIN_BF16 || d->impl == SWIN_IMPL_SIMT))
    return SWIN_ERR_UNSUPPORTED;
  // The kernels keep the batch in an int and address the [B*T, C] row view
  // (TMA coordinates, land bytes) with 32-bit row numbers.
  if (d->batch > INT32_MAX || d->batch * tokens >= (int64_t(1) << 31)) return SWIN_ERR_UNSUPPORTED;
  if (d->batch * tokens * d->heads >= (int64_t(1) << 40)) return SWIN_ERR_UNSUPPORTED;
  return SWIN_OK;
}

// Step of the window order inside an (head, image) block: the integer
// nearest nwin * (sqrt(5) - 1) / 2 that is coprime with nwin (so that
// k -> k * step mod nwin is a permutation whose consecutive windows lie far
// apart on the grid).
int window_step(int nwin) {
  if (nwin <= 2) return 1;
  int st = std::max(1, (int)((double)nwin * 0.6180339887498949 + 0.5));
  auto gcd = [](int a, int b) {
    while (b) {
      const int t = a % b;
      a = b;
      b = t;
    }
    return a;
  };
  while (gcd(st, nwin) != 1) ++st;
  return st;
}

// Windows per work item. The tensor-core kernels put two windows in one
// 128-row tile when both fit with the second starting on a 16-row boundary
// (whole 1 KB swizzle spans and 16-key MMA groups); the mask step's 16
// columns hold the two windows' region codes (8 each).
void set_pack(Geo &g, int pack) {
  g.pack = pack;
  g.offb = pack == 2 ? ((g.n + 15) & ~15) : g.n;
  g.rows = pack == 2 ? g.offb + g.n : g.n;
  g.nitem = (g.nwin + pack - 1) / pack;
  g.istep = (int)(((int64_t)pack * g.wstep) % g.nwin);
}

Geo make_geo(const swin_attn_desc *d) {
  Geo g;
  std::memset(&g, 0, sizeof(g));
  g.lead = 3 - d->ndim;
  for (int a = 0; a < 3; ++a) {
    const int s = a - g.lead;
    g.G[a] = s >= 0 ? d->grid[s] : 1;
    g.w[a] = s >= 0 ? d->window[s] : 1;
    g.s[a] = s >= 0 ? d->shift[s] : 0;
    g.per[a] = s >= 0 ? d->periodic[s] : 0;
    g.nw[a] = (g.G[a] + g.w[a] - 1) / g.w[a];
  }
  g.n = g.w[0] * g.w[1] * g.w[2];
  g.nwin = g.nw[0] * g.nw[1] * g.nw[2];
  g.nqt = (g.n + 127) / 128;
  // a 128-slot tile is a box of the grid when it is made of whole rows of the
  // window's last dim: w2 x tb1 rows (tb1 dividing w1), or w2 x w1 x tb0 (tb0
  // dividing w0)
  g.tb1 = g.tb0 = 0;
  if (128 % g.w[2] == 0) {
    const int r = 128 / g.w[2];
    if (r <= g.w[1] && g.w[1] % r == 0) {
      g.tb1 = r;
      g.tb0 = 1;
    } else if (r % g.w[1] == 0 && r / g.w[1] <= g.w[0] && g.w[0] % (r / g.w[1]) == 0) {
      g.tb1 = g.w[1];
      g.tb0 = r / g.w[1];
    }
  }
  g.wstep = window_step(g.nwin);
  g.tokens = g.G[0] * g.G[1] * g.G[2];
  g.rstride[2] = 1;
  g.rstride[1] = 2 * g.w[2] - 1;
  g.rstride[0] = (2 * g.w[1] - 1) * (2 * g.w[2] - 1);
  g.T = (2 * g.w[0] - 1) * g.rstride[0];
  g.heads = d->heads;
  g.hd = d->head_dim;
  g.C = d->heads * d->head_dim;
  g.batch = (int)d->batch;
  g.has_land = d->has_land;
  set_pack(g, 1);
  return g;
}

void free_plan(swin_attn_plan_s *p) {
  if (!p) return;
  cudaFree(p->d_win_src);
  cudaFree(p->d_region);
  cudaFree(p->d_tok_dst);
  cudaFree(p->d_relidx);
  cudaFree(p->d_status);
  cudaFree(p->d_slot_base);
  cudaFree(p->d_head_slot_begin);
  delete p;
}

// head_dim-128 plans keep delta_i = sum_j P_ij dP_ij of every query ([B][heads][tokens]
// float) at the start of the workspace, ahead of the partial dBias tables.
size_t delta_bytes(const swin_attn_plan_s *p) {
  if (!p->large) return 0;
  const size_t bytes = (size_t)p->g.batch * p->g.heads * p->g.tokens * sizeof(float);
  return (bytes + 255) & ~size_t(255);
}

int current_device_matches(const swin_attn_plan_s *p) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWIN_ERR_CUDA;
  return dev == p->device ? SWIN_OK : SWIN_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

const char *swin_attn_strerror(int status) {
  switch (status) {
    case SWIN_OK: return "ok";
    case SWIN_ERR_INVALID_ARG: return "invalid argument";
    case SWIN_ERR_UNSUPPORTED: return "unsupported problem (window size for the head_dim, head_dim, dtype, impl, bias rows)";
    case SWIN_ERR_ALIGNMENT: return "pointer misaligned (16 bytes; 4 for bias, dbias and land; 256 for workspace)";
    case SWIN_ERR_WORKSPACE: return "workspace missing or too small";
    case SWIN_ERR_CUDA: return "CUDA runtime error";
    case SWIN_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case SWIN_ERR_DEVICE: return "a kernel recorded a device-side error";
    default: return "unknown status";
  }
}

int swin_attn_window_range(int64_t M, int64_t P, int64_t r, int64_t *L, int64_t *R) {
  if (!L || !R || M < 0 || P < 1 || r < 0 || r >= P) return SWIN_ERR_INVALID_ARG;
  eq4_range(M, P, r, *L, *R);
  return SWIN_OK;
}

int swin_attn_plan(const swin_attn_desc *desc, swin_attn_plan_t *out) {
  if (!out) return SWIN_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = check_desc(desc);
  if (rc) return rc;
  swin_attn_plan_s *p = new (std::nothrow) swin_attn_plan_s;
  if (!p) return SWIN_ERR_CUDA;
  std::memset(p, 0, sizeof(*p));
  p->d = *desc;
  p->g = make_geo(desc);
  p->wait_limit_ns = 1000000000ull;
  p->debug_force_timeout = 0;
  const Geo &g = p->g;
  if (cudaGetDevice(&p->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
    free_plan(p);
    return SWIN_ERR_CUDA;
  }
  // kernel family
  p->large = desc->head_dim == 128;
  const bool tc_ok = p->large ? large_supported(g, desc->dtype) : tc_supported(g, desc->dtype);
  if ((desc->impl == SWIN_IMPL_TC || p->large) && !tc_ok) {
    free_plan(p);
    return SWIN_ERR_UNSUPPORTED;
  }
  p->impl = desc->impl == SWIN_IMPL_AUTO ? (tc_ok ? SWIN_IMPL_TC : SWIN_IMPL_SIMT) : desc->impl;
  if (!p->large && p->impl == SWIN_IMPL_TC && ((g.n + 15) & ~15) + g.n <= 128) set_pack(p->g, 2);
  // work items: (head, image, window group) for the small-window kernels,
  // (head, image, window, query tile) for the head_dim-128 kernels
  p->items = p->large ? (int64_t)g.heads * g.batch * g.nwin * g.nqt : (int64_t)g.heads * g.batch * g.nitem;
  int fwd_bps = 1, bwd_bps = 1;
  if (p->impl == SWIN_IMPL_SIMT) {
    if (simt_occupancy(false, g, desc->dtype, &fwd_bps) || simt_occupancy(true, g, desc->dtype, &bwd_bps)) {
      free_plan(p);
      return SWIN_ERR_CUDA;
    }
  } else {
    fwd_bps = tc_fwd_ctas_per_sm(g);
    bwd_bps = tc_bwd_ctas_per_sm(g);
  }
  p->fwd_items = p->large ? large_fwd_items(g) : p->items;
  p->fwd_ctas = (int)std::min<int64_t>(p->fwd_items, (int64_t)std::max(1, fwd_bps) * p->num_sms);
  p->bwd_ctas = (int)std::min<int64_t>(p->items, (int64_t)std::max(1, bwd_bps) * p->num_sms);
  if (p->impl == SWIN_IMPL_TC && !p->large && g.heads <= p->num_sms) {
    // A whole number of CTAs per head: the Eq. (4) split then gives CTA
    // h*k + j the same windows of every head h, so CTAs of adjacent heads
    // run in step and each 128-byte L2 fill (two heads' 64-byte rows of one
    // token) is used by both. Otherwise they drift apart and the DRAM reads
    // double.
    const int k = p->num_sms / g.heads;
    p->fwd_ctas = p->bwd_ctas = (int)std::min<int64_t>(p->items, (int64_t)k * g.heads);
  }
  // workspace slots: one partial dBias table per (CTA, head it touches)
  const int64_t per_head = p->items / g.heads;
  std::vector<int> slot_base(p->bwd_ctas), slot_head;
  for (int r = 0; r < p->bwd_ctas; ++r) {
    int64_t L, R;
    eq4_range(p->items, p->bwd_ctas, r, L, R);
    slot_base[r] = (int)slot_head.size();
    if (R > L)
      for (int64_t h = L / per_head; h <= (R - 1) / per_head; ++h) slot_head.push_back((int)h);
  }
  p->ws_slots = (int64_t)slot_head.size();
  std::vector<int> head_begin(g.heads + 1);
  for (int h = 0; h <= g.heads; ++h)
    head_begin[h] = (int)(std::lower_bound(slot_head.begin(), slot_head.end(), h) - slot_head.begin());
  // device allocations
  const int64_t nslots = (int64_t)g.nwin * g.n;
  bool ok = cudaMalloc(&p->d_win_src, sizeof(int32_t) * nslots) == cudaSuccess &&
            cudaMalloc(&p->d_region, nslots) == cudaSuccess &&
            cudaMalloc(&p->d_tok_dst, sizeof(int32_t) * g.tokens) == cudaSuccess &&
            (g.n > kMaxRelidxSlots || cudaMalloc(&p->d_relidx, sizeof(int32_t) * g.n * g.n) == cudaSuccess) &&
            cudaMalloc(&p->d_status, sizeof(int)) == cudaSuccess &&
            cudaMalloc(&p->d_slot_base, sizeof(int) * p->bwd_ctas) == cudaSuccess &&
            cudaMalloc(&p->d_head_slot_begin, sizeof(int) * (g.heads + 1)) == cudaSuccess;
  ok = ok && cudaMemset(p->d_status, 0, sizeof(int)) == cudaSuccess &&
       cudaMemcpy(p->d_slot_base, slot_base.data(), sizeof(int) * p->bwd_ctas, cudaMemcpyHostToDevice) == cudaSuccess &&
       cudaMemcpy(p->d_head_slot_begin, head_begin.data(), sizeof(int) * (g.heads + 1), cudaMemcpyHostToDevice) ==
           cudaSuccess;
  if (ok) {
    const int blocks = (int)std::min<int64_t>((nslots + 255) / 256, 4096);
    tables_kernel<<<blocks, 256>>>(g, p->d_win_src, p->d_region, p->d_tok_dst);
    if (p->d_relidx) relidx_kernel<<<(int)std::min<int64_t>(((int64_t)g.n * g.n + 255) / 256, 65535), 256>>>(g, p->d_relidx);
    ok = cudaGetLastError() == cudaSuccess && cudaDeviceSynchronize() == cudaSuccess;
  }
  if (!ok) {
    free_plan(p);
    return SWIN_ERR_CUDA;
  }
  *out = p;
  return SWIN_OK;
}

int swin_attn_plan_get_info(swin_attn_plan_t p, swin_attn_plan_info *info) {
  if (!p || !info) return SWIN_ERR_INVALID_ARG;
  info->windows_per_image = p->g.nwin;
  info->tokens_per_image = p->g.tokens;
  info->slots = p->g.n;
  info->bias_rows = p->g.T;
  info->impl = p->impl;
  info->fwd_ctas = p->fwd_ctas;
  info->bwd_ctas = p->bwd_ctas;
  info->num_sms = p->num_sms;
  info->work_items = p->items;
  info->dbias_slots = p->ws_slots;
  return SWIN_OK;
}

int swin_attn_plan_tables(swin_attn_plan_t p, int32_t *win_src, uint8_t *region, int32_t *tok_dst, int32_t *relidx) {
  if (!p) return SWIN_ERR_INVALID_ARG;
  const int64_t nslots = (int64_t)p->g.nwin * p->g.n;
  bool ok = true;
  if (win_src) ok = ok && cudaMemcpy(win_src, p->d_win_src, 4 * nslots, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (region) ok = ok && cudaMemcpy(region, p->d_region, nslots, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (tok_dst) ok = ok && cudaMemcpy(tok_dst, p->d_tok_dst, 4 * (int64_t)p->g.tokens, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (relidx && !p->d_relidx) return SWIN_ERR_UNSUPPORTED;  // not kept for windows of more than 2048 slots
  if (relidx) ok = ok && cudaMemcpy(relidx, p->d_relidx, 4 * (int64_t)p->g.n * p->g.n, cudaMemcpyDeviceToHost) == cudaSuccess;
  return ok ? SWIN_OK : SWIN_ERR_CUDA;
}

size_t swin_attn_workspace_bytes(swin_attn_plan_t p) {
  if (!p) return 0;
  const size_t bytes = (size_t)p->ws_slots * p->g.T * sizeof(float);
  return delta_bytes(p) + ((bytes + 255) & ~size_t(255));
}

int swin_attn_fwd(swin_attn_plan_t p, const void *q, const void *k, const void *v, const float *bias,
                  const uint8_t *land, void *o, float *lse, swin_stream_t stream) {
  if (!p || !q || !k || !v || !o) return SWIN_ERR_INVALID_ARG;
  if (p->d.has_land && !land) return SWIN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return SWIN_ERR_ALIGNMENT;
  // lse and land are read four slots per load where four slots are
  // consecutive tokens: 16 and 4 bytes
  if ((bias && !aligned4(bias)) || (lse && !aligned16(lse)) || (p->d.has_land && !aligned4(land)))
    return SWIN_ERR_ALIGNMENT;
  int rc = current_device_matches(p);
  if (rc) return rc;
  FwdArgs a;
  a.g = p->g;
  a.q = q;
  a.k = k;
  a.v = v;
  a.bias = bias;
  a.land = p->d.has_land ? land : nullptr;
  a.o = o;
  a.lse = lse;
  a.status = p->d_status;
  a.items = p->fwd_items;
  a.ctas = p->fwd_ctas;
  a.scale = 1.0f / sqrtf((float)p->g.hd);
  a.wait_limit_ns = p->wait_limit_ns;
  a.debug_force_timeout = p->debug_force_timeout;
  if (p->large) return launch_fwd_large(a, stream);
  if (p->impl == SWIN_IMPL_TC) return launch_fwd_tc(a, stream);
  return launch_fwd_simt(a, p->d.dtype, stream);
}

}  // extern "C"

namespace {
// swin_attn_bwd and swin_attn_bwd_o: o (the forward's output) may be NULL.
int bwd_impl(swin_attn_plan_t p, const void *q, const void *k, const void *v, const void *o, const void *dout,
             const float *lse, const float *bias, const uint8_t *land, void *dq, void *dk, void *dv, float *dbias,
             void *workspace, size_t workspace_bytes, swin_stream_t stream) {
  if (!p || !q || !k || !v || !dout || !lse || !dq || !dk || !dv) return SWIN_ERR_INVALID_ARG;
  if (o && !aligned16(o)) return SWIN_ERR_ALIGNMENT;
  if (p->d.has_land && !land) return SWIN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dv))
    return SWIN_ERR_ALIGNMENT;
  if (!aligned16(lse) || (bias && !aligned4(bias)) || (dbias && !aligned4(dbias)) ||
      (p->d.has_land && !aligned4(land)))
    return SWIN_ERR_ALIGNMENT;
  if (dbias || p->large) {  // head_dim-128 plans always keep delta in the workspace
    if (!workspace || workspace_bytes < swin_attn_workspace_bytes(p)) return SWIN_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return SWIN_ERR_ALIGNMENT;
  }
  int rc = current_device_matches(p);
  if (rc) return rc;
  BwdArgs a;
  a.g = p->g;
  a.q = q;
  a.k = k;
  a.v = v;
  a.dout = dout;
  a.lse = lse;
  a.bias = bias;
  a.land = p->d.has_land ? land : nullptr;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.delta = p->large ? static_cast<float *>(workspace) : nullptr;
  a.o = p->large ? o : nullptr;  // the other kernels recompute delta in the pass that needs it
  a.ws = dbias ? reinterpret_cast<float *>(static_cast<char *>(workspace) + delta_bytes(p)) : nullptr;
  a.slot_base = p->d_slot_base;
  a.ws_slots = p->ws_slots;
  a.status = p->d_status;
  a.items = p->items;
  a.ctas = p->bwd_ctas;
  a.scale = 1.0f / sqrtf((float)p->g.hd);
  a.wait_limit_ns = p->wait_limit_ns;
  a.debug_force_timeout = p->debug_force_timeout;
  rc = p->large ? launch_bwd_large(a, stream)
       : p->impl == SWIN_IMPL_TC ? launch_bwd_tc(a, stream) : launch_bwd_simt(a, p->d.dtype, stream);
  if (rc || !dbias) return rc;
  FoldArgs f;
  f.ws = a.ws;
  f.head_slot_begin = p->d_head_slot_begin;
  f.dbias = dbias;
  f.T = p->g.T;
  f.heads = p->g.heads;
  const int total = f.T * f.heads;
  fold_kernel<<<(total + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(f);
  return cudaPeekAtLastError() == cudaSuccess ? SWIN_OK : SWIN_ERR_CUDA;
}
}  // namespace

extern "C" {

int swin_attn_bwd(swin_attn_plan_t p, const void *q, const void *k, const void *v, const void *dout,
                  const float *lse, const float *bias, const uint8_t *land, void *dq, void *dk, void *dv,
                  float *dbias, void *workspace, size_t workspace_bytes, swin_stream_t stream) {
  return bwd_impl(p, q, k, v, nullptr, dout, lse, bias, land, dq, dk, dv, dbias, workspace, workspace_bytes,
                  stream);
}

int swin_attn_bwd_o(swin_attn_plan_t p, const void *q, const void *k, const void *v, const void *o,
                    const void *dout, const float *lse, const float *bias, const uint8_t *land, void *dq, void *dk,
                    void *dv, float *dbias, void *workspace, size_t workspace_bytes, swin_stream_t stream) {
  if (!o) return SWIN_ERR_INVALID_ARG;
  return bwd_impl(p, q, k, v, o, dout, lse, bias, land, dq, dk, dv, dbias, workspace, workspace_bytes, stream);
}

int swin_attn_block_fwd(swin_attn_plan_t p, const void *x, const float *ln_gamma, const float *ln_beta,
                        float ln_eps, const void *w_qkv, const float *b_qkv, const void *w_o, const float *b_o,
                        const float *bias, const uint8_t *land, void *y, swin_stream_t stream) {
  if (!p || !x || !ln_gamma || !ln_beta || !w_qkv || !b_qkv || !w_o || !b_o || !y) return SWIN_ERR_INVALID_ARG;
  if (p->d.has_land && !land) return SWIN_ERR_INVALID_ARG;
  if (!(ln_eps > 0.f) || !std::isfinite(ln_eps)) return SWIN_ERR_INVALID_ARG;
  const int64_t bytes = (int64_t)p->g.batch * p->g.tokens * p->g.C * 2;
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x), ya = reinterpret_cast<uintptr_t>(y);
  if (xa < ya + (uintptr_t)bytes && ya < xa + (uintptr_t)bytes) return SWIN_ERR_INVALID_ARG;  // y overlaps x
  if (!aligned16(x) || !aligned16(y) || !aligned16(w_qkv) || !aligned16(w_o)) return SWIN_ERR_ALIGNMENT;
  if (!aligned4(ln_gamma) || !aligned4(ln_beta) || !aligned4(b_qkv) || !aligned4(b_o) || (bias && !aligned4(bias)) ||
      (p->d.has_land && !aligned4(land)))
    return SWIN_ERR_ALIGNMENT;
  if (p->d.dtype != SWIN_BF16 || p->impl != SWIN_IMPL_TC || p->large) return SWIN_ERR_UNSUPPORTED;
  int rc = current_device_matches(p);
  if (rc) return rc;
  BlockArgs a;
  a.g = p->g;
  a.x = x;
  a.y = y;
  a.gamma = ln_gamma;
  a.beta = ln_beta;
  a.b_qkv = b_qkv;
  a.b_o = b_o;
  a.bias = bias;
  a.land = p->d.has_land ? land : nullptr;
  a.eps = ln_eps;
  a.scale = 1.0f / sqrtf((float)p->g.hd);
  a.status = p->d_status;
  a.items = (int64_t)p->g.batch * p->g.nwin;
  a.ctas = (int)std::min<int64_t>(a.items, (int64_t)p->num_sms);
  a.wait_limit_ns = p->wait_limit_ns;
  a.debug_force_timeout = p->debug_force_timeout;
  if (a.items == 0) return SWIN_OK;
  return launch_block_fwd(a, w_qkv, w_o, stream);
}

int swin_attn_plan_set_debug(swin_attn_plan_t p, uint64_t wait_limit_ns, int force_timeout) {
  if (!p || wait_limit_ns == 0 || (force_timeout != 0 && force_timeout != 1)) return SWIN_ERR_INVALID_ARG;
  p->wait_limit_ns = wait_limit_ns;
  p->debug_force_timeout = force_timeout;
  return SWIN_OK;
}

int swin_attn_status(swin_attn_plan_t p, swin_stream_t stream) {
  if (!p) return SWIN_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SWIN_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, p->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SWIN_ERR_CUDA;
  if (h != kStatusOk && cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess) return SWIN_ERR_CUDA;
  if (h == kStatusTimeout) return SWIN_ERR_TIMEOUT;
  return h == kStatusOk ? SWIN_OK : SWIN_ERR_DEVICE;
}

void swin_attn_plan_destroy(swin_attn_plan_t p) {
  if (!p) return;
  cudaDeviceSynchronize();
  free_plan(p);
}

}  // extern "C"
