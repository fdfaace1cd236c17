// swin_large.cuh -- shared pieces of the head_dim-128 kernels (windows of any
// size, key-tiled): tile layouts, the CTAs' item schedules, work-item
// decoding, slot routing of a 128-slot tile, its TMA loads (whole-tile boxes,
// boxes of runs of consecutive slots, gather4 rows) and the mask rows.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "swin_tc.cuh"
#include "tc_ptx.cuh"

namespace swin {
namespace lg {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint16_t kBf16One = 0x3F80;     // 1.0
constexpr uint16_t kBf16NegBig = 0xF180;  // -2^100

constexpr int kHd = 128;
constexpr int kHalfBytes = 128 * 128;      // 128 rows x 64 bf16 (one channel half), 128-byte swizzle
constexpr int kTileBytes = 2 * kHalfBytes;  // 128 rows x 128 bf16
constexpr int kMaskBytes = 128 * 32;        // 128 rows x 16 bf16, 32-byte swizzle
constexpr uint32_t kTmemCols = 512;

__device__ __forceinline__ uint32_t sw32(int r, int c) { return r * 32 + ((c ^ ((r >> 2) & 1)) << 4); }

// Item = (h, b, window, tile), tile fastest.
struct LItem {
  int h, b, omega, qt;
};
__device__ __forceinline__ LItem decode(const Geo &g, int64_t it) {
  LItem x;
  x.qt = (int)(it % g.nqt);
  int64_t t = it / g.nqt;
  x.omega = (int)(t % g.nwin);
  t /= g.nwin;
  x.b = (int)(t % g.batch);
  x.h = (int)(t / g.batch);
  return x;
}

// The work items of this CTA: item k is first + k * step, k < count.
// Strided (CTA r takes r, r + ctas, ...): the CTAs running at one time work on
// neighbouring items, tiles of one window and head, whose key/value or query
// tiles then stay in L2 for all of them. Contiguous (TERRA Eq. (4) ranges)
// where the dBias workspace slots follow those ranges.
struct Items {
  int64_t first, step, count;
  __device__ __forceinline__ int64_t operator[](int64_t k) const { return first + k * step; }
};
__device__ __forceinline__ Items strided_items(int64_t items, int ctas) {
  const int64_t r = blockIdx.x;
  return Items{r, ctas, r < items ? (items - 1 - r) / ctas + 1 : 0};
}
__device__ __forceinline__ Items range_items(int64_t items, int ctas) {
  int64_t L, R;
  eq4_range(items, ctas, blockIdx.x, L, R);
  return Items{L, 1, R - L};
}

// Mask row chunk 0 (region codes < 8): query rows carry a one-hot of the
// region code (live queries), key rows 0 in the column of their code if live
// and -2^100 elsewhere; columns 8..15 are constant (0 / -2^100).
__device__ __forceinline__ uint4 mask_chunk(bool live, int reg, bool key) {
  const uint32_t nb2 = (uint32_t)kBf16NegBig | ((uint32_t)kBf16NegBig << 16);
  const uint32_t other = key ? nb2 : 0u;
  const uint32_t hit = !live ? other
                       : key ? ((reg & 1) ? (uint32_t)kBf16NegBig : (uint32_t)kBf16NegBig << 16)
                             : ((reg & 1) ? (uint32_t)kBf16One << 16 : (uint32_t)kBf16One);
  const int t = reg >> 1;
  return make_uint4(t == 0 ? hit : other, t == 1 ? hit : other, t == 2 ? hit : other, t == 3 ? hit : other);
}

// Routes of the four slots 4*lane .. 4*lane+3 of tile `tile` of window omega:
// grid token (or -1 for pads and slots past the window), region bits, and
// the query and key sides of the bias row offset.
struct Quad {
  int src[4], reg[4], roff[4], rbase[4];
};
__device__ __forceinline__ Quad route_quad(const Geo &g, int omega, int tile, int lane) {
  int wc[3];
  window_coords(g, omega, wc);
  Quad q;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int slot = tile * 128 + 4 * lane + j;
    if (slot < g.n) {
      const SlotRoute r = slot_route(g, wc, slot);
      q.src[j] = r.src;
      q.reg[j] = r.reg;
      q.roff[j] = r.roff;
      q.rbase[j] = r.rbase;
    } else {
      q.src[j] = -1;
      q.reg[j] = 0;
      q.roff[j] = 0;
      q.rbase[j] = g.T - 1;  // keeps rbase - roff inside the bias column
    }
  }
  return q;
}

// Land test of the quad's live slots (land may be null).
__device__ __forceinline__ void quad_live(const Quad &q, const uint8_t *land, int64_t tok0, bool (&live)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) live[j] = q.src[j] >= 0 && (!land || __ldg(land + tok0 + q.src[j]) == 0);
}

// The three TMA views of one [B, G0, G1, G2, C] bf16 tensor: 128-slot tile
// boxes (64 channels x w2 x tb1 x tb0), the [B*T, C] row view for gather4 and
// runs of run_len(g) slots along the grid's last dimension (64 channels x
// run_len). (A fourth view per tensor measured slower throughout.)
struct TileMaps {
  CUtensorMap box, rows, run;
};

// Slots per run: 16 where window rows hold 16-slot runs well (w2 a multiple
// of 16, or at least 64), else 8. Measured: 16-slot boxes beat row gathers
// and 32-slot boxes; in windows 30 slots wide 8-slot boxes beat 16-slot ones.
__host__ __device__ __forceinline__ int run_len(const Geo &g) { return g.w[2] % 16 == 0 || g.w[2] >= 64 ? 16 : 8; }

// Whether the run_len slots of the lane's group of quads (run_len / 4 lanes,
// tile rows from 4 x the group's first lane) hold consecutive positions along
// the grid's last dimension within one grid row (no pad, no seam wrap, no
// slot past the window), and the grid coordinates of the group's first slot.
// Such a run loads as one box instead of one gather4 per four rows.
// Warp-collective: every lane of the warp calls it.
struct Run {
  bool run, lead;  // lead: this lane is the group's first (it issues the run's box)
  int c[3];        // grid coordinates (dims 0, 1, 2) of the group's first slot
};
__device__ __forceinline__ Run find_run(const Geo &g, const Quad &q, int lane) {
  const int len = run_len(g), gl = len >> 2, gm = gl - 1;  // lanes per run, and the lane mask within one
  const int s0 = __shfl_sync(0xffffffffu, q.src[0], lane & ~gm);
  const bool step = q.src[0] >= 0 && q.src[0] == s0 + 4 * (lane & gm) && q.src[1] == q.src[0] + 1 &&
                    q.src[2] == q.src[0] + 2 && q.src[3] == q.src[0] + 3;
  const uint32_t bal = __ballot_sync(0xffffffffu, step), all = (1u << gl) - 1u;
  Run r;
  const int x2 = s0 >= 0 ? s0 % g.G[2] : 0, rest = s0 >= 0 ? s0 / g.G[2] : 0;
  r.run = ((bal >> (lane & ~gm)) & all) == all && x2 + len <= g.G[2];
  r.lead = (lane & gm) == 0;
  r.c[2] = x2;
  r.c[1] = rest % g.G[1];
  r.c[0] = rest / g.G[1];
  return r;
}

// One 64-channel half (channels h*128 + 64*half ..) of the lane's quad of
// tile rows into the half-tile at dst_half: the first lane of a run copies it
// as one box, lanes outside runs gather their four rows (pads read token 0).
__device__ __forceinline__ void load_half(uint32_t dst_half, const TileMaps *m, const Run &r, const Quad &q, int b,
                                          int tokens, int h, int half, int lane, int nq4, uint32_t bar) {
  const int ch = h * kHd + 64 * half;
  if (r.run) {
    if (r.lead) tma_load_5d(dst_half + 512u * lane, &m->run, ch, r.c[2], r.c[1], r.c[0], b, bar);
  } else if (lane < nq4) {
    const int r0 = b * tokens;
    tma_gather4(dst_half + 512u * lane, &m->rows, ch, r0 + max(q.src[0], 0), r0 + max(q.src[1], 0),
                r0 + max(q.src[2], 0), r0 + max(q.src[3], 0), bar);
  }
}

// Grid coordinates of the first slot of tile `tile` of window omega when the
// tile is a box of the grid (whole window rows that neither wrap nor pad).
__device__ __forceinline__ bool tile_box(const Geo &g, int omega, int tile, int (&c)[3]) {
  if (g.tb1 == 0 || (tile + 1) * 128 > g.n) return false;
  int wc[3];
  window_coords(g, omega, wc);
  const int s0 = tile * 128;
  const int o[3] = {s0 / (g.w[1] * g.w[2]), (s0 / g.w[2]) % g.w[1], 0};
  const int ext[3] = {g.tb0, g.tb1, g.w[2]};
  bool box = true;
#pragma unroll
  for (int d = 0; d < 3; ++d) {
    c[d] = wc[d] * g.w[d] + g.s[d] + o[d];
    box = box && c[d] + ext[d] <= g.G[d];
  }
  return box;
}

// One 128-slot tile of head h into `dst` (two 64-channel halves): two box
// copies from lane 0 when the tile is a box, else runs and row
// gathers (load_half). Completion is counted on `bar` (32 KB for a full tile
// either way). Warp-collective: `box` is the same on every lane.
__device__ __forceinline__ void load_tile(uint32_t dst, const TileMaps *m, const Geo &g, bool box, const int (&c)[3],
                                          const Quad &q, int b, int h, int lane, int nq4, uint32_t bar) {
  if (box) {
    if (lane == 0) {
      tma_load_5d(dst, &m->box, h * kHd, c[2], c[1], c[0], b, bar);
      tma_load_5d(dst + kHalfBytes, &m->box, h * kHd + 64, c[2], c[1], c[0], b, bar);
    }
  } else {
    const Run r = find_run(g, q, lane);
    load_half(dst, m, r, q, b, g.tokens, h, 0, lane, nq4, bar);
    load_half(dst + kHalfBytes, m, r, q, b, g.tokens, h, 1, lane, nq4, bar);
  }
}

// K-major 128B-swizzled descriptor of k-step kk (16 channels) of a 128-row
// tile held as two 64-channel halves.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
  return smem_desc(tile + (uint32_t)(kk >> 2) * kHalfBytes + 32u * (kk & 3), 16, 1024, kSwizzle128B);
}
// MN-major (channels = N) descriptor of the 16 rows starting at `row` of such
// a tile, as the B operand of a product over the rows (N = 128 channels).
__device__ __forceinline__ uint64_t nmajor_desc(uint32_t tile, int row) {
  return smem_desc(tile + (uint32_t)row * 128u, kHalfBytes, 1024, kSwizzle128B);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Row view [B*T, C] of a bf16 tensor for TMA gather4: box one row high and 64
// channels (128 bytes) wide, 128-byte swizzle (the layout of the operand
// tile halves).
inline bool rows128_map(CUtensorMap *m, const void *base, const Geo &g) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)g.C, (cuuint64_t)g.batch * (cuuint64_t)g.tokens};
  cuuint64_t strides[1] = {dims[0] * 2};
  cuuint32_t box[2] = {64u, 1u};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Box view of the same tensor: (64 channels, w2, tb1, tb0, 1) per copy.
inline bool box128_map(CUtensorMap *m, const void *base, const Geo &g) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  if (g.tb1 == 0) {  // tiles are never boxes: a valid map of the row view stands in (never used)
    return rows128_map(m, base, g);
  }
  const cuuint64_t e = 2;
  cuuint64_t dims[5] = {(cuuint64_t)g.C, (cuuint64_t)g.G[2], (cuuint64_t)g.G[1], (cuuint64_t)g.G[0],
                        (cuuint64_t)g.batch};
  cuuint64_t strides[4] = {dims[0] * e, dims[0] * dims[1] * e, dims[0] * dims[1] * dims[2] * e,
                           dims[0] * dims[1] * dims[2] * dims[3] * e};
  cuuint32_t box[5] = {64u, (cuuint32_t)g.w[2], (cuuint32_t)g.tb1, (cuuint32_t)g.tb0, 1u};
  cuuint32_t es[5] = {1u, 1u, 1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Run view of the same tensor: (64 channels, run_len, 1, 1, 1) per copy.
inline bool run_map(CUtensorMap *m, const void *base, const Geo &g) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  if (g.G[2] < run_len(g)) {  // no run fits in a grid row: a valid map of the row view stands in (never used)
    return rows128_map(m, base, g);
  }
  const cuuint64_t e = 2;
  cuuint64_t dims[5] = {(cuuint64_t)g.C, (cuuint64_t)g.G[2], (cuuint64_t)g.G[1], (cuuint64_t)g.G[0],
                        (cuuint64_t)g.batch};
  cuuint64_t strides[4] = {dims[0] * e, dims[0] * dims[1] * e, dims[0] * dims[1] * dims[2] * e,
                           dims[0] * dims[1] * dims[2] * dims[3] * e};
  cuuint32_t box[5] = {64u, (cuuint32_t)run_len(g), 1u, 1u, 1u};
  cuuint32_t es[5] = {1u, 1u, 1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool tile_maps(TileMaps *t, const void *base, const Geo &g) {
  return box128_map(&t->box, base, g) && run_map(&t->run, base, g) && rows128_map(&t->rows, base, g);
}

}  // namespace lg
}  // namespace swin
