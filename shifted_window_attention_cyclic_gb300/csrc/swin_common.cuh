// swin_common.cuh -- geometry, routing and launch parameters shared by the
// CUDA kernels of the SW-MSA library (sm_103a).
//
// Routing (TERRA, Sec. IV.D "Differentiable Token Routes"; BEAST page, Model
// Architecture): slot sigma of window omega sits at rolled position
// p_d = omega_d * w_d + sigma_d; it is a pad when p_d >= G_d in some dim, else
// it is fed by the grid token u_d = (p_d + s_d) mod G_d (the roll by -s,
// inverted). Region bit d = [dim d not periodic, s_d > 0, p_d >= G_d - s_d].
// All kernels and the table builder call slot_route(), so the tables that the
// plan exports are exactly the routing the kernels perform.
#pragma once
#include <cstdint>

#include "../../include/swin_attn.h"

namespace swin {

// Geometry normalised to three dims: a 2-D problem gets a leading dim of
// extent 1 (window 1, shift 0, not periodic), which leaves window/slot
// flattening and bias rows unchanged.
struct Geo {
  int G[3], w[3], s[3], per[3], nw[3];
  int lead;        // 3 - ndim: region bit of normalised dim a is (a - lead)
  int n;           // slots per window
  int nwin;        // windows per image
  int wstep;       // window order inside an (head, image) block: the i-th window is (i * wstep) mod nwin
  // Windows per work item (tensor-core kernels): with pack = 2 the two
  // windows 2k and 2k+1 of that order share one 128-row tile, the first in
  // rows [0, n), the second in rows [offb, offb + n); rows = tile rows used.
  int pack, nitem;  // nitem = ceil(nwin / pack) items per (head, image) block
  int offb, rows;
  int istep;        // (pack * wstep) mod nwin: window step from one item to the next
  int nqt;         // query (= key) tiles of 128 slots per window (head_dim-128 kernels)
  int tb1, tb0;    // extents in dims 1 and 0 of a 128-slot tile that is a grid box (w2 x tb1 x tb0
                   // = 128 slots of whole window rows); 0 when the window's tiles are never boxes
  int tokens;      // tokens per image
  int T;           // bias rows
  int rstride[3];  // prod_{e>d} (2 w_e - 1)
  int heads, hd, C;
  int batch;
  int has_land;
};

// Routing of one slot of one window (window coords already decoded).
struct SlotRoute {
  int src;    // token index inside the image, -1 for a pad
  int reg;    // region bits (0 for pads)
  int rbase;  // sum_d (sigma_d + w_d - 1) * rstride_d  (query side of the bias row)
  int roff;   // sum_d sigma_d * rstride_d                (key side of the bias row)
};

__host__ __device__ __forceinline__ void window_coords(const Geo &g, int omega, int wc[3]) {
  wc[2] = omega % g.nw[2];
  int t = omega / g.nw[2];
  wc[1] = t % g.nw[1];
  wc[0] = t / g.nw[1];
}

__host__ __device__ __forceinline__ SlotRoute slot_route(const Geo &g, const int wc[3], int sigma) {
  int sc[3];
  sc[2] = sigma % g.w[2];
  int t = sigma / g.w[2];
  sc[1] = t % g.w[1];
  sc[0] = t / g.w[1];
  SlotRoute r;
  r.rbase = 0;
  r.roff = 0;
  int src = 0, reg = 0;
  bool pad = false;
  for (int a = 0; a < 3; ++a) {
    int p = wc[a] * g.w[a] + sc[a];
    pad |= p >= g.G[a];
    int u = p + g.s[a];
    if (u >= g.G[a]) u -= g.G[a];
    src = src * g.G[a] + u;
    if (!g.per[a] && g.s[a] > 0 && p >= g.G[a] - g.s[a]) reg |= 1 << (a - g.lead);
    r.rbase += (sc[a] + g.w[a] - 1) * g.rstride[a];
    r.roff += sc[a] * g.rstride[a];
  }
  r.src = pad ? -1 : src;
  r.reg = pad ? 0 : reg;
  return r;
}

// Work items are (head, image, window group), head-major: item = (h * B + b) *
// nitem + k, and the k-th item of an (h, b) block holds windows number
// pack*k .. pack*k + pack - 1 of the order i -> (i * wstep) mod nwin (the
// second one only if pack*k + 1 < nwin).
// wstep is coprime with nwin (a permutation) and near nwin * 0.618, so a
// CTA's contiguous item range mixes windows from every part of the grid:
// the windows at the grid's ends (which wrap or pad and load by rows, the
// slower path) are spread evenly over the CTAs instead of falling in a few
// CTAs' ranges.
struct Item {
  int h, b, omega;
};

__host__ __device__ __forceinline__ Item decode_item(const Geo &g, int64_t it) {
  Item x;
  const int64_t k = it % g.nitem;
  x.omega = (int)((k * g.pack * g.wstep) % g.nwin);  // the item's first window
  int64_t t = it / g.nitem;
  x.b = (int)(t % g.batch);
  x.h = (int)(t / g.batch);
  return x;
}

// Sequential walk over work items in order, one step per item, without
// divisions (a CTA's items are a contiguous range).
struct ItemCursor {
  int h, b, k, omega;
  __host__ __device__ __forceinline__ void init(const Geo &g, int64_t it) {
    const Item x = decode_item(g, it);
    h = x.h;
    b = x.b;
    k = (int)(it % g.nitem);
    omega = x.omega;
  }
  // the item's second window (pack = 2), if the image has it
  __host__ __device__ __forceinline__ bool has2(const Geo &g) const { return g.pack == 2 && 2 * k + 1 < g.nwin; }
  __host__ __device__ __forceinline__ int omega2(const Geo &g) const {
    const int o = omega + g.wstep;
    return o >= g.nwin ? o - g.nwin : o;
  }
  __host__ __device__ __forceinline__ void next(const Geo &g) {
    omega += g.istep;
    if (omega >= g.nwin) omega -= g.nwin;
    if (++k == g.nitem) {
      k = 0;
      omega = 0;
      if (++b == g.batch) {
        b = 0;
        ++h;
      }
    }
  }
};

// Tile row -> slot of its window (u = 0 or 1 for pack = 2), or -1 for a row
// that no window slot uses.
template <int kPack>
__host__ __device__ __forceinline__ int tile_slot(const Geo &g, int row, int &u) {
  u = (kPack == 2 && row >= g.offb) ? 1 : 0;
  const int s = row - u * g.offb;
  return s < g.n ? s : -1;
}

// In-window coordinates of one slot, computed once per thread.
struct SlotCoord {
  int sc[3];
};

__host__ __device__ __forceinline__ SlotCoord slot_coord(const Geo &g, int sigma) {
  SlotCoord c;
  c.sc[2] = sigma % g.w[2];
  const int t = sigma / g.w[2];
  c.sc[1] = t % g.w[1];
  c.sc[0] = t / g.w[1];
  return c;
}

// slot_route() for a slot whose coordinates are already known (no divisions).
__host__ __device__ __forceinline__ SlotRoute route_slot(const Geo &g, const int wc[3], const SlotCoord &c) {
  SlotRoute r;
  r.rbase = 0;
  r.roff = 0;
  int src = 0, reg = 0;
  bool pad = false;
  for (int a = 0; a < 3; ++a) {
    const int p = wc[a] * g.w[a] + c.sc[a];
    pad |= p >= g.G[a];
    int u = p + g.s[a];
    if (u >= g.G[a]) u -= g.G[a];
    src = src * g.G[a] + u;
    if (!g.per[a] && g.s[a] > 0 && p >= g.G[a] - g.s[a]) reg |= 1 << (a - g.lead);
    r.rbase += (c.sc[a] + g.w[a] - 1) * g.rstride[a];
    r.roff += c.sc[a] * g.rstride[a];
  }
  r.src = pad ? -1 : src;
  r.reg = pad ? 0 : reg;
  return r;
}

// TERRA Eq. (4): contiguous range of CTA r among P over M items.
__host__ __device__ __forceinline__ void eq4_range(int64_t M, int64_t P, int64_t r, int64_t &L, int64_t &R) {
  L = (r * M) / P;
  R = ((r + 1) * M) / P;
}

// Device status word values (first error wins).
enum : int { kStatusOk = 0, kStatusTimeout = 1, kStatusBounds = 2 };

// Bounds-checked build (-DSWIN_CHECK_BOUNDS): a raw global access of elements
// [idx, idx + len) of a buffer of `count` elements first checks the range; a
// violation records kStatusBounds in the status word (read by
// swin_attn_status as SWIN_ERR_DEVICE) and the caller skips the access. In
// the normal build the check is a constant true.
__device__ __forceinline__ bool in_bounds(int64_t idx, int64_t len, int64_t count, int *status) {
#ifdef SWIN_CHECK_BOUNDS
  if (idx < 0 || idx + len > count) {
    atomicCAS(status, 0, kStatusBounds);
    return false;
  }
#else
  (void)idx, (void)len, (void)count, (void)status;
#endif
  return true;
}

struct FwdArgs {
  Geo g;
  const void *q, *k, *v;
  const float *bias;
  const uint8_t *land;
  void *o;
  float *lse;
  int *status;
  int64_t items;
  int ctas;
  float scale;  // hd^-1/2
  uint64_t wait_limit_ns;   // bound of every in-kernel wait
  int debug_force_timeout;  // testing hook: one role waits on a barrier nothing arrives at
};

struct BwdArgs {
  Geo g;
  const void *q, *k, *v, *dout;
  const float *lse, *bias;
  const uint8_t *land;
  void *dq, *dk, *dv;
  float *ws;              // [slots][T] partial dBias tables, or nullptr (dbias not wanted)
  float *delta;           // head_dim-128 kernels: [B][heads][tokens] delta_i, or nullptr
  const void *o;          // the forward's output, or nullptr: with head_dim 128, delta = dO . O from it
  int64_t ws_slots;       // slots of ws
  const int *slot_base;   // [ctas] first workspace slot of each CTA
  int *status;
  int64_t items;
  int ctas;
  float scale;
  uint64_t wait_limit_ns;
  int debug_force_timeout;
};

struct FoldArgs {
  const float *ws;
  const int *head_slot_begin;  // [heads + 1] slot range of every head
  float *dbias;                // [T][heads]
  int T, heads;
};

// The attention half of a Swin block (swin_block.cu): LayerNorm + QKV
// projection, SW-MSA, out-projection + residual.
struct BlockArgs {
  Geo g;
  const void *x;
  void *y;
  const float *gamma, *beta, *b_qkv, *b_o, *bias;
  const uint8_t *land;
  float eps, scale;
  int *status;
  int64_t items;  // windows (batch * nwin)
  int ctas;
  uint64_t wait_limit_ns;
  int debug_force_timeout;  // testing hook: every thread first waits on a barrier nothing arrives at
};

// Launchers implemented in the kernel translation units.
int launch_fwd_simt(const FwdArgs &a, int dtype, void *stream);
int launch_block_fwd(const BlockArgs &a, const void *w_qkv, const void *w_o, void *stream);
int launch_bwd_simt(const BwdArgs &a, int dtype, void *stream);
int simt_fwd_smem(const Geo &g);
int simt_bwd_smem(const Geo &g);
int simt_occupancy(bool bwd, const Geo &g, int dtype, int *blocks_per_sm);

}  // namespace swin
