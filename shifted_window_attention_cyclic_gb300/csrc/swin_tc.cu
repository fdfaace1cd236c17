// swin_tc.cu -- tcgen05/TMEM kernels of SW-MSA for bf16, head_dim 32,
// windows of up to 128 slots (sm_103a).
//
// Work items are (head h, image b, window omega); each CTA (one per SM) takes
// a contiguous range of items (TERRA Eq. (4)) and runs them through a
// warp-specialised pipeline over a few shared-memory stages:
//  * gather warps (3): route every slot of the item (cyclic shift, ragged
//    edge, pads) and load the Q, K, V (and dO) rows by TMA, one 5-D box per
//    tensor for windows that neither wrap nor pad, TMA gather4 by rows
//    otherwise; they also write the slot metadata and two K=16 mask tiles:
//    Qm (one-hot of the query's region code) and Km (0 where the key is a
//    live key of that region, -2^100 elsewhere), so that one extra MMA step
//    adds the region/land/pad mask to QK^T.
//  * MMA warp (1 elected thread): tcgen05.mma with fp32 accumulators in TMEM.
//  * softmax warps (2 warpgroups, each half of every row's keys): one thread
//    per TMEM lane (query slot); logits x = S*scale*log2e + bias*log2e with
//    the head's bias tile [slot_i][slot_j] resident in shared memory.
//  * epilogue warps (4): read the accumulators from TMEM and store rows at
//    the slots' grid tokens (the reverse route).
// Forward: S = QK^T (+ mask), P = exp2(x - m_h) per warpgroup half, O = P V
// into two accumulators (one per key half) combined by the epilogue.
// Backward: S and dP = dO V^T, P from the saved log-sum-exp, delta = sum P dP,
// dS = P (dP - delta); dV = P^T dO, dK = dS^T Q, dQ = dS K on the tensor
// cores; dBias accumulated per slot pair in TMEM and folded at head changes.
// Masked keys get exactly zero probability: exp2 of about -3e29 is +0.
//
// Every wait is bounded (globaltimer); on timeout the CTA raises an abort
// flag, every role leaves its loop, copies and MMAs in flight are drained,
// TMEM is freed and the device status word reports a timeout.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "swin_tc.cuh"
#include "tc_ptx.cuh"

namespace swin {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint16_t kBf16One = 0x3F80;   // 1.0
constexpr uint16_t kBf16NegBig = 0xF180;  // -2^100

// Swizzled byte offset of 16-byte chunk c of row r in a 32-byte-row mask tile.
__device__ __forceinline__ uint32_t sw32(int r, int c) { return r * 32 + ((c ^ ((r >> 2) & 1)) << 4); }

__device__ __forceinline__ int round16(int x) { return (x + 15) & ~15; }

// Mask rows of one slot (K = 16 columns, 32-byte swizzle): Qm = one-hot of
// the query's region code (live queries only); Km = 0 in the column of the
// key's region code if the key is live, -2^100 everywhere else. Qm Km^T then
// adds -2^100 to every masked logit. Region codes are below 8, so columns
// 8-15 are constant (Qm 0, Km -2^100) and written once per stage; per item
// only the first 16-byte chunk of each row changes.
__device__ __forceinline__ uint4 mask_row_chunk0(bool live, int reg, bool key) {
  const uint32_t nb2 = (uint32_t)kBf16NegBig | ((uint32_t)kBf16NegBig << 16);
  const uint32_t other = key ? nb2 : 0u;
  const uint32_t hit = !live ? other
                       : key ? ((reg & 1) ? (uint32_t)kBf16NegBig : (uint32_t)kBf16NegBig << 16)
                             : ((reg & 1) ? (uint32_t)kBf16One << 16 : (uint32_t)kBf16One);
  const int t = reg >> 1;
  return make_uint4(t == 0 ? hit : other, t == 1 ? hit : other, t == 2 ? hit : other, t == 3 ? hit : other);
}

// Epilogue store of one 32-channel bf16 row per lane (lane = slot row of the
// warp's 32) to that row's grid token. Written straight from registers, one
// store instruction would touch 32 rows 512 bytes apart; instead the rows go
// through the warp's 2 KB staging area (16-byte chunks swizzled by row) and
// come back four lanes per row, so each store instruction writes 8 whole
// 64-byte rows. `dst` is the row's destination (nullptr: row not stored).
__device__ __forceinline__ void store_rows_bf16(uint8_t *stage, const uint32_t (&w)[16], __nv_bfloat16 *dst,
                                                int lane) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4 *>(stage + lane * 64 + ((c ^ (lane & 3)) << 4)) =
        make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  __syncwarp();
  const uint64_t mine = reinterpret_cast<uint64_t>(dst);
  const int c = lane & 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = 8 * k + (lane >> 2);
    const uint64_t d = __shfl_sync(0xffffffffu, mine, r);
    const uint4 v = *reinterpret_cast<const uint4 *>(stage + r * 64 + ((c ^ (r & 3)) << 4));
    if (d) reinterpret_cast<uint4 *>(d)[c] = v;
  }
  __syncwarp();
}

// One head's bias column (bias*log2e, 0 without a bias) held by the 256
// softmax threads, thread t rows t, t+256, t+512 (at most 735 rows for a
// window of up to 128 slots). It is loaded one head ahead, at kernel entry
// for the first head and right after each head change for the next, so that
// the shared-memory copy made at a head change waits on no load.
struct BiasColumn {
  float v[3];
  __device__ __forceinline__ void load(const float *bias, const Geo &g, int h, int t) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int r = t + 256 * k;
      v[k] = (bias && r < g.T) ? __ldg(bias + (int64_t)r * g.heads + h) * kLog2e : 0.f;
    }
  }
  __device__ __forceinline__ void store(float *col, const Geo &g, int t) const {
#pragma unroll
    for (int k = 0; k < 3; ++k)
      if (t + 256 * k < g.T) col[t + 256 * k] = v[k];
  }
};

// Where one item's mask rows and slot metadata sit in a stage (the operand
// tiles, 128 slot rows x 64 B with 64-byte swizzle, are passed per warp).
struct StageLayout {
  uint32_t bytes;            // stage stride
  uint32_t qm, km;           // mask tiles: 128 rows x 32 B, 32-byte swizzle
  uint32_t src, live, lse2;  // int src[128], uint8 live[128], float lse*log2e[128]
};

// The two TMA views of one [B, G0, G1, G2, C] bf16 tensor that the gather
// warps load from (one head's 32 channels, 64-byte swizzle).
struct TmaSet {
  CUtensorMap box;   // a whole window: (32, w2, w1, w0, 1)
  CUtensorMap rows;  // the [B*T, C] row view for gather4: (32, 1)
};

// Gather warps (three). Lane l of every warp routes slots 4l .. 4l+3 of the
// next item one item ahead; warp 0 also loads their land bytes (and
// log-sum-exps), so that those loads are in flight while the current item is
// issued.
// Warps 1 and 2 bring in the operand tiles (tile_a, and tile_b if ntiles = 2),
// by TMA only. A window that neither wraps nor pads in any dim is one box
// (lane 0 loads it); any other window is gathered by rows: lane l fetches
// the rows of its own four slots with one gather4, pads reading token 0 of
// the image, which the masks discard. Nothing here waits on a copy:
// completion is counted in transaction bytes on the stage's full barrier.
// Warp 0 writes the slot metadata. With kSplitMasks, warp 1 writes the query
// mask rows (Qm) and warp 2 the key mask rows (Km), each loading the land
// bytes it needs; otherwise warp 0 loads them and writes both mask tiles,
// and (given no tiles) no copy waits behind its land loads.
template <int kStages, bool kSplitMasks, int kPack>
__device__ __forceinline__ void gather_role(const Geo &g, const StageLayout &lay, int ntiles, uint32_t tile_a,
                                            uint32_t tile_b, const TmaSet *ma, const TmaSet *mb,
                                            const uint8_t *land, const float *lse, uint8_t *smem, uint32_t sbase,
                                            uint32_t full0, uint32_t empty0, const WaitCtl &ctl, int64_t L,
                                            int64_t count, int pw, int lane) {
  // The one-window forward keeps the gather code from before two-window items
  // existed: measured, the general body below slowed that kernel by 2-4 %
  // (instruction layout; the work is the same), while it runs the backward
  // slightly faster.
  if constexpr (kPack == 1 && !kSplitMasks) {
    const int n = g.n, nq4 = (n + 3) >> 2;
    SlotCoord sc[4];
    int foff[4];  // token offset of slot 4l + j from the window's origin when the window is a box
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int slot = 4 * lane + j;
      sc[j] = slot_coord(g, slot < n ? slot : 0);
      foff[j] = (sc[j].sc[0] * g.G[1] + sc[j].sc[1]) * g.G[2] + sc[j].sc[2];
    }
    struct Prep {
      int h, b, c[3];  // c: the window's first grid coordinate in each dim (a box's corner)
      bool box;
      int src[4];
      uint32_t reg4;
      bool lvec;         // land[0] holds the four land bytes
      uint32_t land[4];  // raw bytes: consumed one item later
      float lse[4];
    };
    auto prep = [&](const ItemCursor &cu, Prep &p) {
      p.h = cu.h;
      p.b = cu.b;
      int wc[3];
      window_coords(g, cu.omega, wc);
      p.box = true;
#pragma unroll
      for (int d = 0; d < 3; ++d) {
        p.c[d] = wc[d] * g.w[d] + g.s[d];
        p.box = p.box && p.c[d] + g.w[d] <= g.G[d];
      }
      const int org = (p.c[0] * g.G[1] + p.c[1]) * g.G[2] + p.c[2];
      const int64_t tok0 = (int64_t)cu.b * g.tokens;
      p.reg4 = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int src = -1, reg = 0;
        if (4 * lane + j < n) {
          if (p.box) {
            src = org + foff[j];
          } else {
            const SlotRoute r = route_slot(g, wc, sc[j]);
            src = r.src;
            reg = r.reg;
          }
        }
        p.src[j] = src;
        p.reg4 |= (uint32_t)reg << (8 * j);
      }
      // land bytes (and LSE values) are read by warp 0 alone, which writes the
      // slot metadata and both mask tiles. The four slots of a lane are four
      // consecutive tokens of one row of a box window when w2 % 4 == 0: then
      // they come as one 4-byte (16-byte) load if it is aligned.
      p.lvec = false;
      if (pw != 0 && !kSplitMasks) return;
      const bool run4 = p.box && (g.w[2] & 3) == 0 && 4 * lane + 3 < n;
      const int64_t lt = tok0 + p.src[0];
      const int64_t lo = ((int64_t)cu.b * g.heads + cu.h) * g.tokens + p.src[0];
      if (land) {
        if (run4 && (lt & 3) == 0) {
          p.lvec = true;
          p.land[0] = in_bounds(lt, 4, (int64_t)g.batch * g.tokens, ctl.status) ? __ldg(reinterpret_cast<const unsigned int *>(land + lt)) : 0u;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) p.land[j] = p.src[j] >= 0 && in_bounds(tok0 + p.src[j], 1, (int64_t)g.batch * g.tokens, ctl.status) ? __ldg(land + tok0 + p.src[j]) : 0u;
        }
      }
      if (lse && pw == 0) {
        if (run4 && (lo & 3) == 0) {
          const float4 l4 = in_bounds(lo, 4, (int64_t)g.batch * g.heads * g.tokens, ctl.status) ? __ldg(reinterpret_cast<const float4 *>(lse + lo)) : make_float4(0.f, 0.f, 0.f, 0.f);
          p.lse[0] = l4.x;
          p.lse[1] = l4.y;
          p.lse[2] = l4.z;
          p.lse[3] = l4.w;
        } else {
          const float *lrow = lse + ((int64_t)cu.b * g.heads + cu.h) * g.tokens;
#pragma unroll
          for (int j = 0; j < 4; ++j) p.lse[j] = p.src[j] >= 0 && in_bounds((lrow - lse) + p.src[j], 1, (int64_t)g.batch * g.heads * g.tokens, ctl.status) ? __ldg(lrow + p.src[j]) : 0.f;
        }
      }
    };
    ItemCursor cur;
    Prep pc, pn;
    if (count > 0) {
      cur.init(g, L);
      prep(cur, pc);
    }
    int64_t it = 0;
    for (; it < count; ++it) {
      const int s = (int)(it % kStages);
      ItemCursor nx = cur;
      nx.next(g);
      if (it + 1 < count) prep(nx, pn);
      if (it >= kStages && !mbar_wait_warp(empty0 + 8u * s, (uint32_t)((it / kStages) - 1) & 1u, ctl)) break;
      const uint32_t st = sbase + s * lay.bytes, full = full0 + 8u * s;
      uint8_t *sp = smem + s * lay.bytes;
      const Prep &p = pc;
      if (lane == 0 && ntiles > 0) mbar_expect_tx(full, (uint32_t)(ntiles * (p.box ? n * 64 : nq4 * 256)));
      __syncwarp();
      const int x = p.h * 32;
      if (ntiles == 0) {
        // warp 0: no operand tiles
      } else if (p.box) {
        if (lane == 0) {
          tma_load_5d(st + tile_a, &ma->box, x, p.c[2], p.c[1], p.c[0], p.b, full);
          if (ntiles > 1) tma_load_5d(st + tile_b, &mb->box, x, p.c[2], p.c[1], p.c[0], p.b, full);
        }
      } else if (lane < nq4) {
        const int r0 = p.b * g.tokens;  // row of token 0 of the image in the [B*T, C] view
        const int r[4] = {r0 + max(p.src[0], 0), r0 + max(p.src[1], 0), r0 + max(p.src[2], 0), r0 + max(p.src[3], 0)};
        tma_gather4(st + tile_a + 256u * lane, &ma->rows, x, r[0], r[1], r[2], r[3], full);
        if (ntiles > 1) tma_gather4(st + tile_b + 256u * lane, &mb->rows, x, r[0], r[1], r[2], r[3], full);
      }
      bool live[4] = {false, false, false, false};
      if (kSplitMasks || pw == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          live[j] = p.src[j] >= 0 && (!land || (p.lvec ? ((p.land[0] >> (8 * j)) & 0xffu) : p.land[j]) == 0);
      }
      if (pw == 0) {
        *reinterpret_cast<int4 *>(sp + lay.src + 16 * lane) = make_int4(p.src[0], p.src[1], p.src[2], p.src[3]);
        *reinterpret_cast<uint32_t *>(sp + lay.live + 4 * lane) =
            (live[0] ? 1u : 0u) | (live[1] ? 0x100u : 0u) | (live[2] ? 0x10000u : 0u) | (live[3] ? 0x1000000u : 0u);
        if (lse)
          *reinterpret_cast<float4 *>(sp + lay.lse2 + 16 * lane) =
              make_float4(live[0] ? p.lse[0] * kLog2e : 0.f, live[1] ? p.lse[1] * kLog2e : 0.f,
                          live[2] ? p.lse[2] * kLog2e : 0.f, live[3] ? p.lse[3] * kLog2e : 0.f);
      }
      if (kSplitMasks ? pw != 0 : pw == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int slot = 4 * lane + j, reg = (int)((p.reg4 >> (8 * j)) & 0xffu);
          if (slot < n) {
            if (!kSplitMasks || pw == 1)
              *reinterpret_cast<uint4 *>(sp + lay.qm + sw32(slot, 0)) = mask_row_chunk0(live[j], reg, false);
            if (!kSplitMasks || pw == 2)
              *reinterpret_cast<uint4 *>(sp + lay.km + sw32(slot, 0)) = mask_row_chunk0(live[j], reg, true);
          }
        }
      }
      fence_proxy_async_smem();  // mask rows are read by the tensor cores
      mbar_arrive_warp(full);
      cur = nx;
      pc = pn;
    }
    // Copies still in flight must land before the CTA exits. Unless a role gave
    // up early these stages were consumed already and the waits return at once.
    volatile int no_abort = 0;
    const WaitCtl dctl{&no_abort, ctl.status, ctl.limit_ns < 50000000ull ? ctl.limit_ns : 50000000ull};
    for (int64_t k = it > kStages ? it - kStages : 0; k < it; ++k)
      mbar_wait_warp(full0 + 8u * (uint32_t)(k % kStages), (uint32_t)(k / kStages) & 1u, dctl);
  } else {
    const int n = g.n, nq4 = (n + 3) >> 2;
    // The lane's tile rows 4l .. 4l+3 belong to window u of the item (the
    // second window starts at row offb, a multiple of 16) and hold its slots
    // s0 .. s0+3.
    const int u = (kPack == 2 && 4 * lane >= g.offb) ? 1 : 0;
    const int s0 = 4 * lane - u * g.offb;
    SlotCoord sc[4];
    int foff[4];  // token offset of slot s0 + j from the window's origin when the window is a box
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int slot = s0 + j;
      sc[j] = slot_coord(g, slot < n ? slot : 0);
      foff[j] = (sc[j].sc[0] * g.G[1] + sc[j].sc[1]) * g.G[2] + sc[j].sc[2];
    }
    struct Prep {
      int h, b, c[3];  // c: the lane's window's first grid coordinate in each dim (a box's corner)
      bool box;        // the lane's window is one box
      bool has;        // the lane's window exists (the item may hold one window only)
      uint32_t tx;     // bytes one tile of the item brings in (both windows)
      int src[4];
      uint32_t reg4;
      bool lvec;         // land[0] holds the four land bytes
      uint32_t land[4];  // raw bytes: consumed one item later
      float lse[4];
    };
    auto prep = [&](const ItemCursor &cu, Prep &p) {
      p.h = cu.h;
      p.b = cu.b;
      int wc[3] = {0, 0, 0};
      p.tx = 0;
      p.has = false;
      p.box = false;
#pragma unroll
      for (int uu = 0; uu < kPack; ++uu) {
        if (uu == 1 && !cu.has2(g)) break;
        int wcu[3], cc[3];
        window_coords(g, uu == 0 ? cu.omega : cu.omega2(g), wcu);
        bool box = true;
#pragma unroll
        for (int d = 0; d < 3; ++d) {
          cc[d] = wcu[d] * g.w[d] + g.s[d];
          box = box && cc[d] + g.w[d] <= g.G[d];
        }
        p.tx += box ? (uint32_t)n * 64u : (uint32_t)nq4 * 256u;
        if (uu == u) {
          p.has = true;
          p.box = box;
#pragma unroll
          for (int d = 0; d < 3; ++d) {
            wc[d] = wcu[d];
            p.c[d] = cc[d];
          }
        }
      }
      const int org = (p.c[0] * g.G[1] + p.c[1]) * g.G[2] + p.c[2];
      const int64_t tok0 = (int64_t)cu.b * g.tokens;
      p.reg4 = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int src = -1, reg = 0;
        if (p.has && s0 + j < n) {
          if (p.box) {
            src = org + foff[j];
          } else {
            const SlotRoute r = route_slot(g, wc, sc[j]);
            src = r.src;
            reg = r.reg;
          }
        }
        p.src[j] = src;
        p.reg4 |= (uint32_t)reg << (8 * j);
      }
      // land bytes (and LSE values) are read by warp 0 alone, which writes the
      // slot metadata and both mask tiles. The four slots of a lane are four
      // consecutive tokens of one row of a box window when w2 % 4 == 0: then
      // they come as one 4-byte (16-byte) load if it is aligned.
      p.lvec = false;
      if (pw != 0 && !kSplitMasks) return;
      const bool run4 = p.box && (g.w[2] & 3) == 0 && s0 + 3 < n;
      const int64_t lt = tok0 + p.src[0];
      const int64_t lo = ((int64_t)cu.b * g.heads + cu.h) * g.tokens + p.src[0];
      if (land) {
        if (run4 && (lt & 3) == 0) {
          p.lvec = true;
          p.land[0] = in_bounds(lt, 4, (int64_t)g.batch * g.tokens, ctl.status) ? __ldg(reinterpret_cast<const unsigned int *>(land + lt)) : 0u;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) p.land[j] = p.src[j] >= 0 && in_bounds(tok0 + p.src[j], 1, (int64_t)g.batch * g.tokens, ctl.status) ? __ldg(land + tok0 + p.src[j]) : 0u;
        }
      }
      if (lse && pw == 0) {
        if (run4 && (lo & 3) == 0) {
          const float4 l4 = in_bounds(lo, 4, (int64_t)g.batch * g.heads * g.tokens, ctl.status) ? __ldg(reinterpret_cast<const float4 *>(lse + lo)) : make_float4(0.f, 0.f, 0.f, 0.f);
          p.lse[0] = l4.x;
          p.lse[1] = l4.y;
          p.lse[2] = l4.z;
          p.lse[3] = l4.w;
        } else {
          const float *lrow = lse + ((int64_t)cu.b * g.heads + cu.h) * g.tokens;
#pragma unroll
          for (int j = 0; j < 4; ++j) p.lse[j] = p.src[j] >= 0 && in_bounds((lrow - lse) + p.src[j], 1, (int64_t)g.batch * g.heads * g.tokens, ctl.status) ? __ldg(lrow + p.src[j]) : 0.f;
        }
      }
    };
    ItemCursor cur;
    Prep pc, pn;
    if (count > 0) {
      cur.init(g, L);
      prep(cur, pc);
    }
    int64_t it = 0;
    for (; it < count; ++it) {
      const int s = (int)(it % kStages);
      ItemCursor nx = cur;
      nx.next(g);
      if (it + 1 < count) prep(nx, pn);
      if (it >= kStages && !mbar_wait_warp(empty0 + 8u * s, (uint32_t)((it / kStages) - 1) & 1u, ctl)) break;
      const uint32_t st = sbase + s * lay.bytes, full = full0 + 8u * s;
      uint8_t *sp = smem + s * lay.bytes;
      const Prep &p = pc;
      if (lane == 0 && ntiles > 0) mbar_expect_tx(full, (uint32_t)ntiles * p.tx);
      __syncwarp();
      const int x = p.h * 32;
      if (ntiles == 0 || !p.has) {
        // warp 0 of the forward (no operand tiles), or no window in these rows
      } else if (p.box) {
        if (s0 == 0) {  // the window's first lane: rows [u * offb, u * offb + n)
          const uint32_t row0 = (uint32_t)(u * g.offb) * 64u;
          tma_load_5d(st + tile_a + row0, &ma->box, x, p.c[2], p.c[1], p.c[0], p.b, full);
          if (ntiles > 1) tma_load_5d(st + tile_b + row0, &mb->box, x, p.c[2], p.c[1], p.c[0], p.b, full);
        }
      } else if (s0 < n) {
        const int r0 = p.b * g.tokens;  // row of token 0 of the image in the [B*T, C] view
        const int r[4] = {r0 + max(p.src[0], 0), r0 + max(p.src[1], 0), r0 + max(p.src[2], 0), r0 + max(p.src[3], 0)};
        tma_gather4(st + tile_a + 256u * lane, &ma->rows, x, r[0], r[1], r[2], r[3], full);
        if (ntiles > 1) tma_gather4(st + tile_b + 256u * lane, &mb->rows, x, r[0], r[1], r[2], r[3], full);
      }
      bool live[4] = {false, false, false, false};
      if (kSplitMasks || pw == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          live[j] = p.src[j] >= 0 && (!land || (p.lvec ? ((p.land[0] >> (8 * j)) & 0xffu) : p.land[j]) == 0);
      }
      if (pw == 0) {
        *reinterpret_cast<int4 *>(sp + lay.src + 16 * lane) = make_int4(p.src[0], p.src[1], p.src[2], p.src[3]);
        *reinterpret_cast<uint32_t *>(sp + lay.live + 4 * lane) =
            (live[0] ? 1u : 0u) | (live[1] ? 0x100u : 0u) | (live[2] ? 0x10000u : 0u) | (live[3] ? 0x1000000u : 0u);
        if (lse)
          *reinterpret_cast<float4 *>(sp + lay.lse2 + 16 * lane) =
              make_float4(live[0] ? p.lse[0] * kLog2e : 0.f, live[1] ? p.lse[1] * kLog2e : 0.f,
                          live[2] ? p.lse[2] * kLog2e : 0.f, live[3] ? p.lse[3] * kLog2e : 0.f);
      }
      if (kSplitMasks ? pw != 0 : pw == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // window u's region codes sit in mask columns 8u .. 8u+7 (chunk u)
          const int row = 4 * lane + j, reg = (int)((p.reg4 >> (8 * j)) & 0xffu);
          if (s0 + j < n) {
            if (!kSplitMasks || pw == 1)
              *reinterpret_cast<uint4 *>(sp + lay.qm + sw32(row, u)) = mask_row_chunk0(live[j], reg, false);
            if (!kSplitMasks || pw == 2)
              *reinterpret_cast<uint4 *>(sp + lay.km + sw32(row, u)) = mask_row_chunk0(live[j], reg, true);
          }
        }
      }
      fence_proxy_async_smem();  // mask rows are read by the tensor cores
      mbar_arrive_warp(full);
      cur = nx;
      pc = pn;
    }
    // Copies still in flight must land before the CTA exits. Unless a role gave
    // up early these stages were consumed already and the waits return at once.
    volatile int no_abort = 0;
    const WaitCtl dctl{&no_abort, ctl.status, ctl.limit_ns < 50000000ull ? ctl.limit_ns : 50000000ull};
    for (int64_t k = it > kStages ? it - kStages : 0; k < it; ++k)
      mbar_wait_warp(full0 + 8u * (uint32_t)(k % kStages), (uint32_t)(k / kStages) & 1u, dctl);
  }
}

// ---------------------------------------------------------------- forward ---
namespace fwd {

constexpr int kStages = 4;
constexpr int kTileBytes = 128 * 64;  // 128 slot rows x 32 bf16
constexpr int kMaskBytes = 128 * 32;  // 128 rows x 16 bf16
constexpr int kQ = 0, kK = kTileBytes, kV = 2 * kTileBytes, kQm = 3 * kTileBytes, kKm = kQm + kMaskBytes;
constexpr int kMeta = kKm + kMaskBytes;  // int32 src[128], uint8 live[128]
constexpr int kStageBytes = kMeta + 1024;
constexpr int kBias = kStages * kStageBytes;  // fp32 [128][kBiasStride]: bias*log2e of the current head
constexpr int kBiasStride = 132;
constexpr int kBarOff = kBias + 128 * kBiasStride * 4;
// barrier indices
constexpr int bFull = 0, bEmpty = kStages, bSFull = 2 * kStages, bPFull = bSFull + 2, bOFull = bPFull + 2,
              bTFree = bOFull + 2, bNever = bTFree + 2, bDrain = bNever + 1, bBsync = bDrain + 1,
              kNumBars = bBsync + 1;
constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem slot (u32), abort flag (int)
// Per-item exchange slots from the softmax to the epilogue warps (slot it % 4):
// float max[4][2][128] and float sum[4][2][128], one value per half row;
// then int roff[128]. Item it may reuse the slot of item it - 4 because S(it)
// is issued only after PV(it - 2), which waits for the epilogue to be done
// with item it - 4.
constexpr int kXchgSlots = 4;
constexpr int kXchg = (kMiscOff + 16 + 127) & ~127;
constexpr int kRoff = kXchg + kXchgSlots * 2 * 2 * 128 * 4;
// the current head's bias column (bias*log2e, up to kMaxBiasRows rows), staged
// once per head by the softmax warps: the table is read by every CTA at once,
// and one load per row and CTA keeps that hot spot cool
constexpr int kMaxBiasRows = 768;
constexpr int kBvec = (kRoff + 512 + 127) & ~127;
constexpr int kOStage = kBvec + kMaxBiasRows * 4;  // 4 epilogue warps x 2 KB store staging (16-byte stores)
constexpr int kSmemBytes = kOStage + 8192 + 1024;    // + alignment slack
static_assert(kStageBytes % 1024 == 0 && kBias % 16 == 0, "stage tiles need 1024-byte alignment");
static_assert(kXchg % 16 == 0 && kOStage % 16 == 0, "vector accesses need 16-byte alignment");
static_assert(kSmemBytes <= 232448, "over the 227 KB of shared memory a CTA may use");

// warps 0-7: two softmax warpgroups, each owning half of every row's columns;
// 8-11: epilogue; 12-14: gather; 15: MMA
constexpr int kSoftmaxWarps = 8, kEpilogueWarp0 = 8, kProducerWarp0 = 12, kMmaWarp = 15;
constexpr int kProducerThreads = (kMmaWarp - kProducerWarp0) * 32;
constexpr int kThreads = (kMmaWarp + 1) * 32;
// TMEM columns: S of item parity b at 128*b, its 16-key group k at +16k, with
// that group's P (bf16 pairs) over its first 8 columns; O of item parity b
// and key half h (the keys of softmax warpgroup h) at 256 + 64*b + 32*h
constexpr uint32_t kTmemCols = 512, kColS = 0, kColO = 256;

// kPack: windows per work item (1 or 2), a compile-time copy per value so
// that the one-window kernel carries no code for the second window.
template <int kPack>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const FwdArgs a, const __grid_constant__ TmaSet tmq, const __grid_constant__ TmaSet tmk,
                  const __grid_constant__ TmaSet tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int idx) { return bars + 8u * idx; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMiscOff + 4);

  const Geo &g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = round16(kPack == 2 ? g.rows : g.n), NG = N >> 4;  // key columns of the tile (both windows)
  int64_t L, R;
  eq4_range(a.items, a.ctas, blockIdx.x, L, R);
  const int64_t count = R - L;
  WaitCtl ctl{abort_flag, a.status, a.wait_limit_ns};
  BiasColumn bcol;  // softmax threads: the first head's column, in flight during the set-up
  if (threadIdx.x < 256 && count > 0) bcol.load(a.bias, g, decode_item(g, L).h, threadIdx.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(bFull + s), kProducerThreads / 32);
      mbar_init(bar(bEmpty + s), 1 + 4);  // MMA commit + epilogue warps (slot metadata read)
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(bar(bSFull + w), 1);
      mbar_init(bar(bPFull + w), kSoftmaxWarps);
      mbar_init(bar(bOFull + w), 1);
      mbar_init(bar(bTFree + w), 4);  // epilogue warps
    }
    mbar_init(bar(bNever), 1);
    mbar_init(bar(bBsync), kSoftmaxWarps);
    mbar_init(bar(bDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  {
    // key side of every slot's bias row offset, for the bias-row builds
    int *roff = reinterpret_cast<int *>(smem + kRoff);
    int wc0[3] = {0, 0, 0};
    if (threadIdx.x < 128) {
      int u;
      const int sg = tile_slot<kPack>(g, threadIdx.x, u);
      roff[threadIdx.x] = sg >= 0 ? slot_route(g, wc0, sg).roff : 0;
    }
  }
  // stage tiles start zeroed: box loads fill only the window's rows, and rows
  // past the last slot must stay finite for the MMAs
  for (int z = threadIdx.x; z < kStages * kStageBytes / 16; z += blockDim.x)
    reinterpret_cast<uint4 *>(smem)[z] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  // A row of window u has its region codes in mask columns 8u .. 8u+7; the
  // other 8 key-mask columns are -2^100 for every item. Rows no window slot
  // uses are pads for every item: -2^100 in every key-mask column, no token
  // (query mask rows stay zero).
  for (int z = threadIdx.x; z < kStages * 128; z += blockDim.x) {
    const int st = z / 128, row = z % 128;
    int u;
    const int sg = tile_slot<kPack>(g, row, u);
    const uint32_t nb2 = (uint32_t)kBf16NegBig | ((uint32_t)kBf16NegBig << 16);
    *reinterpret_cast<uint4 *>(smem + st * kStageBytes + kKm + sw32(row, 1 - u)) = make_uint4(nb2, nb2, nb2, nb2);
    if (sg < 0) {
      *reinterpret_cast<uint4 *>(smem + st * kStageBytes + kKm + sw32(row, u)) = make_uint4(nb2, nb2, nb2, nb2);
      reinterpret_cast<int *>(smem + st * kStageBytes + kMeta)[row] = -1;
    }
  }
  fence_proxy_async_smem();
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kProducerWarp0 && warp < kMmaWarp) {
    // ------------------------------------------------------------ gather ---
    const int pw = warp - kProducerWarp0;
    const StageLayout lay{kStageBytes, kQm, kKm, kMeta, kMeta + 512, 0};
    // warp 0: masks and metadata; warp 1: Q and K; warp 2: V
    gather_role<kStages, false, kPack>(g, lay, pw == 0 ? 0 : pw == 1 ? 2 : 1, pw == 1 ? kQ : kV, kK, pw == 1 ? &tmq : &tmv,
                         &tmk, g.has_land ? a.land : nullptr, nullptr, smem, sbase, bar(bFull), bar(bEmpty), ctl, L,
                         count, pw, lane);
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------- MMA ---
    // Event loop: S(k) is issued as soon as its data has landed and PV(k-2)
    // (same TMEM buffer) has been issued; PV(k) as soon as P(k) is written and
    // the epilogue has read O(k-2). Neither waits behind the other.
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16(128, N, 0, 0);
      const uint32_t idesc_pv = idesc_bf16(128, 32, 0, 1);
      const int ng0 = (NG + 1) >> 1;  // key groups of softmax warpgroup 0
      int64_t ns = 0, npv = 0;
      uint64_t idle_since = 0;
      uint32_t spins = 0;
      while (npv < count) {
        bool progress = false;
        if (ns < count && ns <= npv + 1) {
          const int s = (int)(ns % kStages), wb = (int)(ns & 1);
          if (mbar_test(bar(bFull + s), (uint32_t)(ns / kStages) & 1u)) {
            tc_fence_after();
            const uint32_t st = sbase + s * kStageBytes;
            const uint32_t d = tmem + kColS + 128u * wb;
            mma_ss(d, smem_desc(st + kQ, 16, 512, kSwizzle64B), smem_desc(st + kK, 16, 512, kSwizzle64B), idesc_qk,
                   0);
            mma_ss(d, smem_desc(st + kQ + 32, 16, 512, kSwizzle64B), smem_desc(st + kK + 32, 16, 512, kSwizzle64B),
                   idesc_qk, 1);
            mma_ss(d, smem_desc(st + kQm, 16, 256, kSwizzle32B), smem_desc(st + kKm, 16, 256, kSwizzle32B),
                   idesc_qk, 1);
            mma_commit(bar(bSFull + wb));
            ++ns;
            progress = true;
          }
        }
        if (npv < ns) {
          const int s = (int)(npv % kStages), wb = (int)(npv & 1);
          if (mbar_test(bar(bPFull + wb), (uint32_t)(npv >> 1) & 1u) &&
              (npv < 2 || mbar_test(bar(bTFree + wb), (uint32_t)((npv >> 1) - 1) & 1u))) {
            tc_fence_after();
            const uint32_t st = sbase + s * kStageBytes;
            const uint32_t d = tmem + kColO + 64u * wb, p = tmem + kColS + 128u * wb;
            // keys of warpgroup 0 into O half 0, of warpgroup 1 into O half 1
            for (int kk = 0; kk < NG; ++kk)
              mma_ts(kk < ng0 ? d : d + 32u, p + 16u * kk,
                     smem_desc(st + kV + 1024u * kk, kTileBytes, 512, kSwizzle64B), idesc_pv,
                     (kk == 0 || kk == ng0) ? 0u : 1u);
            mma_commit(bar(bOFull + wb));
            mma_commit(bar(bEmpty + s));
            ++npv;
            progress = true;
          }
        }
        if (progress) {
          spins = 0;
          idle_since = 0;
          continue;
        }
        // nothing ready: sleep on the barrier most likely to complete next
        // (woken at its completion, or after a short hint)
        if (ns < count && ns <= npv + 1)
          mbar_try_wait_hint(bar(bFull + (int)(ns % kStages)), (uint32_t)(ns / kStages) & 1u, 64);
        else if (npv < ns)
          mbar_try_wait_hint(bar(bPFull + (int)(npv & 1)), (uint32_t)(npv >> 1) & 1u, 64);
        if ((++spins & 15u) == 0) {
          if (*abort_flag) break;
          const uint64_t now = globaltimer();
          if (idle_since == 0) {
            idle_since = now;
          } else if (now - idle_since > a.wait_limit_ns) {
            *abort_flag = 1;
            atomicCAS(a.status, 0, kStatusTimeout);
            break;
          }
        }
      }
      // drain every MMA this thread issued before TMEM is released
      mma_commit(bar(bDrain));
      volatile int no_abort = 0;
      WaitCtl drain_ctl{&no_abort, a.status, a.wait_limit_ns};
      mbar_wait(bar(bDrain), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp >= kEpilogueWarp0) {
    // ---------------------------------------------------------- epilogue ---
    // Per item, O row i arrives in two halves: O_h holds the keys of softmax
    // warpgroup h, weighted relative to that half's own row max m_h, with
    // half row sum l_h. With m = max(m_0, m_1) and a_h = exp2(m_h - m):
    // O = (a_0 O_0 + a_1 O_1) / (a_0 l_0 + a_1 l_1), rounded to bf16 and
    // stored at the slot's grid token (the reverse route), and the
    // log-sum-exp (m + log2(a_0 l_0 + a_1 l_1)) * ln 2; land rows store zeros.
    const int q4 = warp & 3, i = q4 * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const float *xmax = reinterpret_cast<const float *>(smem + kXchg);  // [slot][half][128]
    const float *xsum = xmax + kXchgSlots * 256;
    const bool two = ((NG + 1) >> 1) < NG;  // warpgroup 1 owns some keys
    ItemCursor x;
    if (count > 0) x.init(g, L);
    for (int64_t it = 0; it < count; ++it, x.next(g)) {
      const int wb = (int)(it & 1), xs = (int)(it % kXchgSlots), s = (int)(it % kStages);
      if (!mbar_wait_warp(bar(bOFull + wb), (uint32_t)(it >> 1) & 1u, ctl)) break;
      tc_fence_after();
      const uint32_t tO = tmem + lane_addr + kColO + 64u * wb;
      uint32_t o0[16], o1[16], o2[16], o3[16];  // O_0 columns 0-15, 16-31; O_1 columns 0-15, 16-31
      tmem_ld16(tO, o0);
      tmem_ld16(tO + 16, o1);
      tmem_ld16(tO + 32, o2);
      tmem_ld16(tO + 48, o3);
      const uint8_t *sp = smem + s * kStageBytes;
      const int src = reinterpret_cast<const int *>(sp + kMeta)[i];
      const bool live = (sp + kMeta + 512)[i] != 0;
      const float m0 = xmax[xs * 256 + i], m1 = xmax[xs * 256 + 128 + i];
      const float l0 = xsum[xs * 256 + i], l1 = xsum[xs * 256 + 128 + i];
      mbar_arrive_warp(bar(bEmpty + s));  // done with the stage's slot metadata
      tmem_wait_ld_tied(o0, o1);
      tmem_wait_ld_tied(o2, o3);
      tc_fence_before();
      mbar_arrive_warp(bar(bTFree + wb));
      const bool store = src >= 0 && in_bounds(((int64_t)x.b * g.tokens + src) * g.C + (int64_t)x.h * 32, 32, (int64_t)g.batch * g.tokens * g.C, a.status);  // pad rows carry src = -1
      {
        const float m = two ? fmaxf(m0, m1) : m0;
        const float a0 = ex2(m0 - m), a1 = two ? ex2(m1 - m) : 0.f;
        const float l = two ? fmaf(a0, l0, a1 * l1) : l0;
        const float inv = live ? __frcp_rn(l) : 0.f;
        const float c0 = a0 * inv, c1 = a1 * inv;
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint32_t *h0 = e < 16 ? o0 : o1;
          const uint32_t *h1 = e < 16 ? o2 : o3;
          const int o = e & 15;
          float v0 = __uint_as_float(h0[o]) * c0, v1 = __uint_as_float(h0[o + 1]) * c0;
          if (two) {
            v0 = fmaf(__uint_as_float(h1[o]), c1, v0);
            v1 = fmaf(__uint_as_float(h1[o + 1]), c1, v1);
          }
          w[e >> 1] = pack_bf16(v0, v1);
        }
        __nv_bfloat16 *dst = store ? static_cast<__nv_bfloat16 *>(a.o) +
                                         ((int64_t)x.b * g.tokens + src) * g.C + (int64_t)x.h * 32
                                   : nullptr;
        store_rows_bf16(smem + kOStage + 2048 * q4, w, dst, lane);
        if (store && a.lse)
          a.lse[((int64_t)x.b * g.heads + x.h) * g.tokens + src] = live ? (m + __log2f(l)) * kLn2 : -INFINITY;
      }
    }
    tmem_wait_ld();
  } else {
    // ----------------------------------------------------------- softmax ---
    // Thread (grp, i): TMEM lane i (query slot i), 16-column groups [gb, ge)
    // of the item's S row (warpgroup grp's half of the keys), loaded into
    // registers with one wait. (A load and its wait stay in straight-line
    // code: registers that an asynchronous TMEM load is still writing must
    // not be carried around the loop, where the compiler may copy them.)
    // x = S*scale*log2e + bias*log2e (this half of bias row i, in smem); the
    // half row max m_h; p = exp2(x - m_h) -> P (bf16) over the first 8 columns
    // of each of this thread's 16-column S groups (never over columns the
    // other warpgroup may not have read yet); m_h and the half row sum go to
    // the item's exchange slot for the epilogue warps, which put the two
    // halves on one scale. No exchange between the warpgroups.
    const int grp = warp >> 2, q4 = warp & 3, i = q4 * 32 + lane;
    const int ng0 = (NG + 1) >> 1, gb = grp ? ng0 : 0, ge = grp ? NG : ng0;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    float *brow = reinterpret_cast<float *>(smem + kBias) + i * kBiasStride;
    float *xmax = reinterpret_cast<float *>(smem + kXchg);  // [slot][half][128]
    float *xsum = xmax + kXchgSlots * 256;
    const int *roff = reinterpret_cast<const int *>(smem + kRoff);
    const float cs = a.scale * kLog2e;
    const float2 cs2 = make_float2(cs, cs);
    int wc0[3] = {0, 0, 0};
    int ui;
    const int si = tile_slot<kPack>(g, i, ui);  // this row's slot and window
    // With two windows per item, warpgroup grp's key columns are exactly
    // window grp's (the second window starts at column offb = 16 * ng0): a
    // warp whose rows all belong to the other window (or are pads) has only
    // masked keys in its half and writes P = 0 without computing it.
    const bool idle = kPack == 2 && !__any_sync(0xffffffffu, si >= 0 && ui == grp);
    const int rbase = si >= 0 ? slot_route(g, wc0, si).rbase : 0;
    int cur_h = -1;
    const int h_last = count > 0 ? decode_item(g, R - 1).h : 0;  // heads rise by one along the range
    uint32_t bs_phase = 0;
    float *bvec = reinterpret_cast<float *>(smem + kBvec);
    bool ok = true;
    if (a.debug_force_timeout && grp == 0) ok = mbar_wait_warp(bar(bNever), 0, ctl);
    ItemCursor x;
    if (count > 0) x.init(g, L);
    for (int64_t it = 0; ok && it < count; ++it, x.next(g)) {
      if (x.h != cur_h) {
        // head change: this thread alone reads this half of bias row i; the
        // loads are independent so their latencies overlap
        // The head's bias column goes to shared memory first (one load per
        // row and CTA; every CTA reads the table at once, and 64 loads per
        // thread made it an L2 hot spot, about 20 us per head change), then
        // each thread builds its half row from there.
        if (cur_h >= 0) {  // everyone is done with the previous column
          mbar_arrive_warp(bar(bBsync));
          if (!mbar_wait_warp(bar(bBsync), bs_phase & 1u, ctl)) break;
          ++bs_phase;
        }
        bcol.store(bvec, g, grp * 128 + i);  // loaded one head ahead
        mbar_arrive_warp(bar(bBsync));
        if (!mbar_wait_warp(bar(bBsync), bs_phase & 1u, ctl)) break;
        ++bs_phase;
        if (x.h < h_last) bcol.load(a.bias, g, x.h + 1, grp * 128 + i);
#pragma unroll 16
        for (int jj = 0; jj < 64; ++jj) {
          const int j = 16 * gb + jj;
          int uj;
          const bool pair = si >= 0 && tile_slot<kPack>(g, j, uj) >= 0 && uj == ui;  // query and key of one window
          if (j < 16 * ge) brow[j] = pair ? bvec[rbase - roff[j]] : 0.f;
        }
        cur_h = x.h;
      }
      const int wb = (int)(it & 1), xs = (int)(it % kXchgSlots);
      const uint32_t tS = tmem + lane_addr + kColS + 128u * wb;
      if (!mbar_wait_warp(bar(bSFull + wb), (uint32_t)(it >> 1) & 1u, ctl)) break;
      tc_fence_after();
      if (idle) {
        const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          if (gb + k4 < ge) tmem_st8(tS + 16u * (gb + k4), z);
        xmax[xs * 256 + grp * 128 + i] = -1e30f;  // weight exp2(-1e30 - m) = 0 in the epilogue
        xsum[xs * 256 + grp * 128 + i] = 0.f;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(bar(bPFull + wb));
        continue;
      }
      uint32_t sv[4][16];
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4)
        if (gb + k4 < ge) tmem_ld16(tS + 16u * (gb + k4), sv[k4]);
      tmem_wait_ld_tied(sv[0], sv[1]);
      tmem_wait_ld_tied(sv[2], sv[3]);
      // x = S*cs + bias2 (kept in sv), half row max (independent chains)
      float mp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        if (gb + k4 < ge) {
#pragma unroll
          for (int e4 = 0; e4 < 16; e4 += 4) {
            const float4 b4 = *reinterpret_cast<const float4 *>(brow + 16 * (gb + k4) + e4);
            const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sv[k4][e4]), __uint_as_float(sv[k4][e4 + 1])),
                                         cs2, make_float2(b4.x, b4.y));
            const float2 x1 = __ffma2_rn(
                make_float2(__uint_as_float(sv[k4][e4 + 2]), __uint_as_float(sv[k4][e4 + 3])), cs2,
                make_float2(b4.z, b4.w));
            sv[k4][e4] = __float_as_uint(x0.x);
            sv[k4][e4 + 1] = __float_as_uint(x0.y);
            sv[k4][e4 + 2] = __float_as_uint(x1.x);
            sv[k4][e4 + 3] = __float_as_uint(x1.y);
            mp[e4 >> 2] = max3(mp[e4 >> 2], max3(x0.x, x0.y, x1.x), x1.y);
          }
        }
      }
      const float m = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3]));
      // p = exp2(x - m), half row sum, P (bf16) over S
      const float2 negm = make_float2(-m, -m);
      float2 sp2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        if (gb + k4 < ge) {
          uint32_t pv[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float2 xs2 =
                __fadd2_rn(make_float2(__uint_as_float(sv[k4][e]), __uint_as_float(sv[k4][e + 1])), negm);
            const float2 p = make_float2(ex2(xs2.x), ex2(xs2.y));
            sp2[(e >> 1) & 3] = __fadd2_rn(sp2[(e >> 1) & 3], p);
            pv[e >> 1] = pack_bf16(p.x, p.y);
          }
          tmem_st8(tS + 16u * (gb + k4), pv);  // over the first half of its own S group
        }
      }
      const float2 sum2 = __fadd2_rn(__fadd2_rn(sp2[0], sp2[1]), __fadd2_rn(sp2[2], sp2[3]));
      xmax[xs * 256 + grp * 128 + i] = m;
      xsum[xs * 256 + grp * 128 + i] = sum2.x + sum2.y;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(bar(bPFull + wb));
    }
    tmem_wait_st();
    tmem_wait_ld();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace fwd

// --------------------------------------------------------------- backward ---
// Per work item: S = Q K^T + mask and dP = dO V^T into TMEM; one thread per
// query row recomputes P = exp2(S*cs + bias2 - lse2) (pass 1: delta_i =
// sum_j P_ij dP_ij, P to smem for dV), then dS = P (dP - delta) (pass 2: dS to
// smem for dK and dQ, added into the per-head dBias slot-pair accumulator kept
// in TMEM). dV = P^T dO, dK = dS^T Q and dQ = dS K run on the tensor cores;
// the epilogue warps store them at the slots' grid tokens (the inverse route).
// The bias tile of the current head lives in smem (row i is only read by
// thread i); at a head change the TMEM accumulator is folded into bias rows
// in a fixed order and written to the CTA's workspace slot.
namespace bwd {

constexpr int kStages = 2;
constexpr int kTile = 128 * 64, kMask = 128 * 32;
constexpr int kQ = 0, kK = kTile, kV = 2 * kTile, kdO = 3 * kTile, kQm = 4 * kTile, kKm = kQm + kMask;
constexpr int kMeta = kKm + kMask;  // int32 src[128] @0, float lse2[128] @512, uint8 live[128] @1024
constexpr int kStageBytes = kMeta + 2048;
constexpr int kP = kStages * kStageBytes;  // P tile, bf16, [j-atom][i][64 j], 128B swizzle
constexpr int kdS = kP + 32768;            // dS tile, same layout
constexpr int kBias = kdS + 32768;         // fp32 [128][kBiasStride]: bias*log2e, or the dBias fold buffer
constexpr int kBiasStride = 132;
constexpr int kBarOff = kBias + 128 * kBiasStride * 4;
constexpr int bFull = 0, bEmpty = kStages, bSpFull = 2 * kStages, bPFull = bSpFull + 1, bDsFull = bPFull + 1,
              bAccFull = bDsFull + 1, bAccFree = bAccFull + 1, bDsFree = bAccFree + 1, bWsync = bDsFree + 1,
              bDsync = bWsync + 1, bNever = bDsync + 1, bDrain = bNever + 1, bVFree = bDrain + 1,
              kNumBars = bVFree + 2;
constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem slot, abort flag
constexpr int kDeltaOff = (kMiscOff + 16 + 127) & ~127;  // float [2][128]: the two halves of delta_i
constexpr int kRoff = kDeltaOff + 1024;                  // int [128]: key side of every slot's bias row offset
constexpr int kOStage = kRoff + 512;                     // 4 epilogue warps x 2 KB store staging (16-byte stores)
constexpr int kSmemBytes = kOStage + 8192 + 1024;
static_assert(kStageBytes % 1024 == 0 && kP % 1024 == 0 && kdS % 1024 == 0, "operand tiles need 1024-byte alignment");
static_assert(kBias % 16 == 0 && kOStage % 16 == 0, "vector accesses need 16-byte alignment");
static_assert(kSmemBytes <= 232448, "over the 227 KB of shared memory a CTA may use");

// softmax warps 0-7: two warpgroups, each owning half of every row's columns
// gather warps 12-14: 96 threads cover the 128 slot rows (threads 0-31 take two)
constexpr int kSoftmaxThreads = 256, kEpilogueWarp0 = 8, kProducerWarp0 = 12, kMmaWarp = 15;
constexpr int kProducerThreads = (kMmaWarp - kProducerWarp0) * 32;
constexpr int kThreads = (kMmaWarp + 1) * 32;
// dV has two buffers (item parity): dV(it) is issued as soon as P(it) is
// written, while the epilogue may still be draining item it - 1; dK and dQ
// wait for that drain.
constexpr uint32_t kTmemCols = 512, kColS = 0, kColdP = 128, kColdV = 256, kColdK = 288, kColdQ = 320,
                   kColdV1 = 352, kColAcc = 384;

// byte offset of the 16-byte chunk holding j = 8c..8c+7 of row i in a P/dS tile
__device__ __forceinline__ uint32_t pds_chunk(int i, int c) {
  return (c >> 3) * 16384 + (i >> 3) * 1024 + (i & 7) * 128 + (((c & 7) ^ (i & 7)) << 4);
}

template <int kPack>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const BwdArgs a, const __grid_constant__ TmaSet tmq, const __grid_constant__ TmaSet tmk,
                  const __grid_constant__ TmaSet tmv, const __grid_constant__ TmaSet tmdo) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int idx) { return bars + 8u * idx; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMiscOff + 4);

  const Geo &g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = round16(kPack == 2 ? g.rows : g.n), NG = N >> 4;  // key columns of the tile (both windows)
  int64_t L, R;
  eq4_range(a.items, a.ctas, blockIdx.x, L, R);
  const int64_t count = R - L;
  WaitCtl ctl{abort_flag, a.status, a.wait_limit_ns};
  BiasColumn bcol;  // softmax threads: the first head's column, in flight during the set-up
  if (threadIdx.x < 256 && count > 0) bcol.load(a.bias, g, decode_item(g, L).h, threadIdx.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(bFull + s), kProducerThreads / 32);
      mbar_init(bar(bEmpty + s), 1 + 4);  // MMA commit + epilogue warps
    }
    mbar_init(bar(bSpFull), 1);
    mbar_init(bar(bPFull), kSoftmaxThreads / 32);
    mbar_init(bar(bDsFull), kSoftmaxThreads / 32);
    mbar_init(bar(bAccFull), 1);
    mbar_init(bar(bAccFree), 4);
    mbar_init(bar(bDsFree), 1);
    mbar_init(bar(bWsync), kSoftmaxThreads / 32);
    mbar_init(bar(bDsync), kSoftmaxThreads / 32);
    mbar_init(bar(bNever), 1);
    mbar_init(bar(bDrain), 1);
    mbar_init(bar(bVFree), 4);
    mbar_init(bar(bVFree + 1), 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // stage tiles start zeroed: box loads fill only the window's rows, and rows
  // past the last slot must stay finite for the MMAs
  for (int z = threadIdx.x; z < kStages * kStageBytes / 16; z += blockDim.x)
    reinterpret_cast<uint4 *>(smem)[z] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  {
    int *ro = reinterpret_cast<int *>(smem + kRoff);
    int wc0[3] = {0, 0, 0};
    if (threadIdx.x < 128) {
      int u;
      const int sg = tile_slot<kPack>(g, threadIdx.x, u);
      ro[threadIdx.x] = sg >= 0 ? slot_route(g, wc0, sg).roff : 0;
    }
  }
  // A row of window u has its region codes in mask columns 8u .. 8u+7; the
  // other 8 key-mask columns are -2^100 for every item. Rows no window slot
  // uses are pads for every item: -2^100 in every key-mask column, no token
  // (query mask rows stay zero).
  for (int z = threadIdx.x; z < kStages * 128; z += blockDim.x) {
    const int st = z / 128, row = z % 128;
    int u;
    const int sg = tile_slot<kPack>(g, row, u);
    const uint32_t nb2 = (uint32_t)kBf16NegBig | ((uint32_t)kBf16NegBig << 16);
    *reinterpret_cast<uint4 *>(smem + st * kStageBytes + kKm + sw32(row, 1 - u)) = make_uint4(nb2, nb2, nb2, nb2);
    if (sg < 0) {
      *reinterpret_cast<uint4 *>(smem + st * kStageBytes + kKm + sw32(row, u)) = make_uint4(nb2, nb2, nb2, nb2);
      reinterpret_cast<int *>(smem + st * kStageBytes + kMeta)[row] = -1;
    }
  }
  fence_proxy_async_smem();
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kProducerWarp0 && warp < kMmaWarp) {
    // ------------------------------------------------------------ gather ---
    const int pw = warp - kProducerWarp0;
    const StageLayout lay{kStageBytes, kQm, kKm, kMeta, kMeta + 1024, kMeta + 512};
    // warp 0: Q, dO and metadata; warp 1: K and the query masks; warp 2: V and the key masks
    gather_role<kStages, true, kPack>(g, lay, pw == 0 ? 2 : 1, pw == 0 ? kQ : pw == 1 ? kK : kV, kdO,
                               pw == 0 ? &tmq : pw == 1 ? &tmk : &tmv, &tmdo, g.has_land ? a.land : nullptr,
                               pw == 0 ? a.lse : nullptr, smem, sbase, bar(bFull), bar(bEmpty), ctl, L, count, pw,
                               lane);
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------- MMA ---
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16(128, N, 0, 0);
      const uint32_t idesc_mn = idesc_bf16(128, 32, 1, 1);
      const uint32_t idesc_dq = idesc_bf16(128, 32, 0, 1);
      const uint32_t tS = tmem + kColS, tdP = tmem + kColdP;
      auto issue_sdp = [&](int64_t it) -> bool {
        const int s = (int)(it % kStages);
        if (!mbar_wait(bar(bFull + s), (uint32_t)(it / kStages) & 1u, ctl)) return false;
        tc_fence_after();
        const uint32_t st = sbase + s * kStageBytes;
        mma_ss(tS, smem_desc(st + kQ, 16, 512, kSwizzle64B), smem_desc(st + kK, 16, 512, kSwizzle64B), idesc_s, 0);
        mma_ss(tS, smem_desc(st + kQ + 32, 16, 512, kSwizzle64B), smem_desc(st + kK + 32, 16, 512, kSwizzle64B),
               idesc_s, 1);
        mma_ss(tS, smem_desc(st + kQm, 16, 256, kSwizzle32B), smem_desc(st + kKm, 16, 256, kSwizzle32B), idesc_s, 1);
        mma_ss(tdP, smem_desc(st + kdO, 16, 512, kSwizzle64B), smem_desc(st + kV, 16, 512, kSwizzle64B), idesc_s, 0);
        mma_ss(tdP, smem_desc(st + kdO + 32, 16, 512, kSwizzle64B), smem_desc(st + kV + 32, 16, 512, kSwizzle64B),
               idesc_s, 1);
        mma_commit(bar(bSpFull));
        return true;
      };
      bool ok = count > 0 && issue_sdp(0);
      for (int64_t it = 0; ok && it < count; ++it) {
        const int s = (int)(it % kStages);
        const uint32_t st = sbase + s * kStageBytes;
        const int vb = (int)(it & 1);
        if (!mbar_wait(bar(bPFull), (uint32_t)it & 1u, ctl)) break;
        if (it >= 2 && !mbar_wait(bar(bVFree + vb), (uint32_t)((it >> 1) - 1) & 1u, ctl)) break;
        tc_fence_after();
        for (int kk = 0; kk < 8; ++kk)  // dV = P^T dO: M = keys, K = queries
          mma_ss(tmem + (vb ? kColdV1 : kColdV), smem_desc(sbase + kP + 2048u * kk, 16384, 1024, kSwizzle128B),
                 smem_desc(st + kdO + 1024u * kk, kTile, 512, kSwizzle64B), idesc_mn, kk > 0 ? 1u : 0u);
        if (!mbar_wait(bar(bDsFull), (uint32_t)it & 1u, ctl)) break;
        tc_fence_after();
        if (it + 1 < count && !issue_sdp(it + 1)) break;
        if (it >= 1 && !mbar_wait(bar(bAccFree), (uint32_t)(it - 1) & 1u, ctl)) break;
        tc_fence_after();
        for (int kk = 0; kk < 8; ++kk)  // dK = dS^T Q
          mma_ss(tmem + kColdK, smem_desc(sbase + kdS + 2048u * kk, 16384, 1024, kSwizzle128B),
                 smem_desc(st + kQ + 1024u * kk, kTile, 512, kSwizzle64B), idesc_mn, kk > 0 ? 1u : 0u);
        for (int kk = 0; kk < NG; ++kk)  // dQ = dS K: M = queries, K = keys
          mma_ss(tmem + kColdQ, smem_desc(sbase + kdS + 16384u * (kk >> 2) + 32u * (kk & 3), 16, 1024, kSwizzle128B),
                 smem_desc(st + kK + 1024u * kk, kTile, 512, kSwizzle64B), idesc_dq, kk > 0 ? 1u : 0u);
        mma_commit(bar(bAccFull));
        mma_commit(bar(bDsFree));
        mma_commit(bar(bEmpty + s));
      }
      mma_commit(bar(bDrain));
      volatile int no_abort = 0;
      WaitCtl drain_ctl{&no_abort, a.status, a.wait_limit_ns};
      mbar_wait(bar(bDrain), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp >= kEpilogueWarp0) {
    // ---------------------------------------------------------- epilogue ---
    const int q4 = warp & 3, e = q4 * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    ItemCursor x;
    if (count > 0) x.init(g, L);
    for (int64_t it = 0; it < count; ++it, x.next(g)) {
      const int s = (int)(it % kStages);
      if (!mbar_wait_warp(bar(bFull + s), (uint32_t)(it / kStages) & 1u, ctl)) break;
      const int src = reinterpret_cast<const int *>(smem + s * kStageBytes + kMeta)[e];
      mbar_arrive_warp(bar(bEmpty + s));
      if (!mbar_wait_warp(bar(bAccFull), (uint32_t)it & 1u, ctl)) break;
      tc_fence_after();
      // one 32-column accumulator at a time: TMEM -> registers -> bf16 -> grid
      const bool store = src >= 0 && in_bounds(((int64_t)x.b * g.tokens + src) * g.C + (int64_t)x.h * 32, 32, (int64_t)g.batch * g.tokens * g.C, a.status);  // pad rows carry src = -1
      const int64_t off = ((int64_t)x.b * g.tokens + (store ? src : 0)) * g.C + (int64_t)x.h * 32;
      auto drain = [&](uint32_t col, void *base, float mul) {
        uint32_t lo[16], hi[16];
        tmem_ld16(tmem + lane_addr + col, lo);
        tmem_ld16(tmem + lane_addr + col + 16, hi);
        tmem_wait_ld_tied(lo, hi);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          w[e >> 1] = pack_bf16(__uint_as_float(lo[e]) * mul, __uint_as_float(lo[e + 1]) * mul);
          w[8 + (e >> 1)] = pack_bf16(__uint_as_float(hi[e]) * mul, __uint_as_float(hi[e + 1]) * mul);
        }
        store_rows_bf16(smem + kOStage + 2048 * q4, w, store ? static_cast<__nv_bfloat16 *>(base) + off : nullptr,
                        lane);
      };
      // one copy of the drain code for the three accumulators (instruction
      // cache: every role's loop runs on every SM sub-partition at once);
      // the dV buffer is handed back as soon as it is read
      const int vb = (int)(it & 1);
#pragma unroll 1
      for (int t = 0; t < 3; ++t) {
        drain(t == 0 ? (vb ? kColdV1 : kColdV) : t == 1 ? kColdK : kColdQ, t == 0 ? a.dv : t == 1 ? a.dk : a.dq,
              t == 0 ? 1.f : a.scale);
        if (t == 0) {
          tc_fence_before();
          mbar_arrive_warp(bar(bVFree + vb));
        }
      }
      tc_fence_before();
      mbar_arrive_warp(bar(bAccFree));
    }
    tmem_wait_ld();
  } else {
    // ----------------------------------------------------------- softmax ---
    // Warpgroup grp owns the 16-column groups [gb, ge) of every row; lane i
    // of TMEM is query slot i. delta_i is the sum of the two halves (fixed order).
    const int grp = warp >> 2, q4 = warp & 3, i = q4 * 32 + lane, tid = grp * 128 + i;
    const int ng0 = (NG + 1) >> 1, gb = grp ? ng0 : 0, ge = grp ? NG : ng0;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_addr + kColS, tdP = tmem + lane_addr + kColdP, tAcc = tmem + lane_addr + kColAcc;
    float *brow = reinterpret_cast<float *>(smem + kBias) + i * kBiasStride;
    float *dpart = reinterpret_cast<float *>(smem + kDeltaOff);
    const int *roff = reinterpret_cast<const int *>(smem + kRoff);
    const float cs = a.scale * kLog2e;
    const float2 cs2 = make_float2(cs, cs);
    const bool want_db = a.ws != nullptr;
    int wc0[3] = {0, 0, 0};
    int ui;
    const int si = tile_slot<kPack>(g, i, ui);  // this row's slot and window
    // With two windows per item, warpgroup grp's key columns are exactly
    // window grp's: a warp whose rows all belong to the other window (or are
    // pads) has P = dS = 0 in its half; it writes those zeros to the P and
    // dS tiles and adds nothing to delta or dBias.
    const bool idle = kPack == 2 && !__any_sync(0xffffffffu, si >= 0 && ui == grp);
    auto zero_chunks = [&](int tile) {
      for (int c = 2 * gb; c < 2 * ge; ++c)
        *reinterpret_cast<uint4 *>(smem + tile + pds_chunk(i, c)) = make_uint4(0u, 0u, 0u, 0u);
    };
    const SlotRoute ri = slot_route(g, wc0, si >= 0 ? si : 0);
    int cur_h = -1, h_first = -1;
    const int h_last = count > 0 ? decode_item(g, R - 1).h : 0;  // heads rise by one along the range
    uint32_t wsync_phase = 0;
    bool ok = true;
    if (a.debug_force_timeout) ok = mbar_wait_warp(bar(bNever), 0, ctl);
    // Fold the slot-pair dBias accumulator into bias rows (fixed order) and
    // write workspace slot `slot`.
    auto flush = [&](int slot) -> bool {
      for (int gi = gb; gi < ge; ++gi) {
        uint32_t av[16];
        tmem_ld16(tAcc + 16u * gi, av);
        tmem_wait_ld_tied(av);
#pragma unroll
        for (int e = 0; e < 16; ++e) brow[16 * gi + e] = __uint_as_float(av[e]);
      }
      mbar_arrive_warp(bar(bWsync));
      if (!mbar_wait_warp(bar(bWsync), wsync_phase & 1u, ctl)) return false;
      ++wsync_phase;
      const float *acc = reinterpret_cast<const float *>(smem + kBias);
      for (int t = tid; t < g.T; t += kSoftmaxThreads) {
        int dlt[3], rem = t;
        for (int d = 0; d < 3; ++d) {
          dlt[d] = rem / g.rstride[d] - (g.w[d] - 1);
          rem %= g.rstride[d];
        }
        float sum = 0.f;
        for (int i0 = max(0, dlt[0]); i0 < min(g.w[0], g.w[0] + dlt[0]); ++i0)
          for (int i1 = max(0, dlt[1]); i1 < min(g.w[1], g.w[1] + dlt[1]); ++i1)
            for (int i2 = max(0, dlt[2]); i2 < min(g.w[2], g.w[2] + dlt[2]); ++i2) {
              const int qi = (i0 * g.w[1] + i1) * g.w[2] + i2;
              const int kj = ((i0 - dlt[0]) * g.w[1] + (i1 - dlt[1])) * g.w[2] + (i2 - dlt[2]);
              sum += acc[qi * kBiasStride + kj];
              if (kPack == 2) sum += acc[(g.offb + qi) * kBiasStride + g.offb + kj];  // the second window
            }
        if (in_bounds((int64_t)slot * g.T + t, 1, a.ws_slots * g.T, a.status)) a.ws[(int64_t)slot * g.T + t] = sum;
      }
      mbar_arrive_warp(bar(bWsync));
      if (!mbar_wait_warp(bar(bWsync), wsync_phase & 1u, ctl)) return false;
      ++wsync_phase;
      return true;
    };
    ItemCursor x;
    if (count > 0) x.init(g, L);
    for (int64_t it = 0; ok && it < count; ++it, x.next(g)) {
      if (x.h != cur_h) {
        if (cur_h >= 0 && want_db && !flush(a.slot_base[blockIdx.x] + (cur_h - h_first))) break;
        // The head's bias column goes to shared memory first (one load per
        // row and CTA; every CTA reads the table at once, and 64 loads per
        // thread made it an L2 hot spot), staged in the P tile once dV, dK
        // and dQ of the previous item are done with it; each thread then
        // builds its half row from there, and all are done reading before
        // pass 1 writes P.
        float *bvec = reinterpret_cast<float *>(smem + kP);
        if (it >= 1 && !mbar_wait_warp(bar(bDsFree), (uint32_t)(it - 1) & 1u, ctl)) break;
        bcol.store(bvec, g, tid);  // loaded one head ahead
        if (x.h < h_last) bcol.load(a.bias, g, x.h + 1, tid);
        mbar_arrive_warp(bar(bWsync));
        if (!mbar_wait_warp(bar(bWsync), wsync_phase & 1u, ctl)) break;
        ++wsync_phase;
        for (int j = 16 * gb; j < 16 * ge; ++j) {
          int uj;
          const int sj = tile_slot<kPack>(g, j, uj);
          brow[j] = si >= 0 && sj >= 0 && uj == ui ? bvec[ri.rbase - roff[j]] : 0.f;  // query and key of one window
        }
        mbar_arrive_warp(bar(bWsync));
        if (!mbar_wait_warp(bar(bWsync), wsync_phase & 1u, ctl)) break;
        ++wsync_phase;
        if (want_db) {
          uint32_t z[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) z[e] = 0u;
          for (int gi = gb; gi < ge; ++gi) tmem_st16(tAcc + 16u * gi, z);
          tmem_wait_st();
        }
        if (h_first < 0) h_first = x.h;
        cur_h = x.h;
      }
      const int s = (int)(it % kStages);
      if (!mbar_wait_warp(bar(bSpFull), (uint32_t)it & 1u, ctl)) break;
      tc_fence_after();
      if (!mbar_wait_warp(bar(bFull + s), (uint32_t)(it / kStages) & 1u, ctl)) break;
      const uint8_t *sp = smem + s * kStageBytes;
      const float lse2 = reinterpret_cast<const float *>(sp + kMeta + 512)[i];
      const bool live = (sp + kMeta + 1024)[i] != 0;
      // pass 1: P = exp2(S*cs + bias2 - lse2); partial delta = sum_j P dP over
      // this half; P (fp32) back over S in TMEM, P (bf16) to the smem tile.
      float delta = 0.f;
      const float2 nl2 = make_float2(-lse2, -lse2);
      auto p_group = [&](int gi, uint32_t (&sv)[16], uint32_t (&dpv)[16]) {
        uint32_t pb[8];
#pragma unroll
        for (int e4 = 0; e4 < 16; e4 += 4) {
          const float4 b4 = *reinterpret_cast<const float4 *>(brow + 16 * gi + e4);
          const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int e = e4; e < e4 + 4; e += 2) {
            float2 xs = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), cs2,
                                   make_float2(bb[e - e4], bb[e - e4 + 1]));
            xs = __fadd2_rn(xs, nl2);
            const float p0 = live ? ex2(xs.x) : 0.f, p1 = live ? ex2(xs.y) : 0.f;
            delta = fmaf(p0, __uint_as_float(dpv[e]), delta);
            delta = fmaf(p1, __uint_as_float(dpv[e + 1]), delta);
            sv[e] = __float_as_uint(p0);  // P (fp32) overwrites S in the register buffer
            sv[e + 1] = __float_as_uint(p1);
            pb[e >> 1] = pack_bf16(p0, p1);
          }
        }
        tmem_st16(tS + 16u * gi, sv);
        *reinterpret_cast<uint4 *>(smem + kP + pds_chunk(i, 2 * gi)) = make_uint4(pb[0], pb[1], pb[2], pb[3]);
        *reinterpret_cast<uint4 *>(smem + kP + pds_chunk(i, 2 * gi + 1)) = make_uint4(pb[4], pb[5], pb[6], pb[7]);
      };
      if (idle) {
        zero_chunks(kP);
      } else {
        // two groups per TMEM round trip: tcgen05.wait::ld waits for every
        // load in flight, so a double buffer would wait just as often, and
        // the round trips (not the arithmetic) set this pass's length
        uint32_t s0[16], d0[16], s1[16], d1[16];
#pragma unroll 1
        for (int k2 = 0; k2 < 4; k2 += 2) {
          const int g0 = gb + k2, g1 = gb + k2 + 1;
          if (g0 < ge) {
            tmem_ld16(tS + 16u * g0, s0);
            tmem_ld16(tdP + 16u * g0, d0);
            if (g1 < ge) {
              tmem_ld16(tS + 16u * g1, s1);
              tmem_ld16(tdP + 16u * g1, d1);
            }
            tmem_wait_ld_tied(s0, d0);
            p_group(g0, s0, d0);
            if (g1 < ge) {
              tmem_tie(s1, d1);
              p_group(g1, s1, d1);
            }
          }
        }
      }
      dpart[grp * 128 + i] = delta;
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_warp(bar(bPFull));
      mbar_arrive_warp(bar(bDsync));
      if (!mbar_wait_warp(bar(bDsync), (uint32_t)it & 1u, ctl)) break;
      delta = dpart[i] + dpart[128 + i];
      if (it >= 1 && !mbar_wait_warp(bar(bDsFree), (uint32_t)(it - 1) & 1u, ctl)) break;
      tc_fence_after();
      // pass 2: dS = P (dP - delta); dS (bf16) to the smem tile; dBias
      // slot-pair accumulator += dS.
      const float2 nd2 = make_float2(-delta, -delta);
      // 8-column sub-groups (one 16-byte dS chunk each) keep the double
      // buffers of P, dP and the accumulator within the register budget.
      auto ds_sub = [&](int sg, uint32_t (&pv)[8], uint32_t (&dpv)[8], uint32_t (&av)[8]) {
        uint32_t db[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float2 p = make_float2(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1]));
          const float2 d = __fadd2_rn(make_float2(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])), nd2);
          const float2 ds = __fmul2_rn(p, d);
          db[e >> 1] = pack_bf16(ds.x, ds.y);
          const float2 acc = __fadd2_rn(make_float2(__uint_as_float(av[e]), __uint_as_float(av[e + 1])), ds);
          av[e] = __float_as_uint(acc.x);
          av[e + 1] = __float_as_uint(acc.y);
        }
        if (want_db) tmem_st8(tAcc + 8u * sg, av);
        *reinterpret_cast<uint4 *>(smem + kdS + pds_chunk(i, sg)) = make_uint4(db[0], db[1], db[2], db[3]);
      };
      if (idle) {
        zero_chunks(kdS);
      } else {
        uint32_t p0[8], d0[8], a0[8], p1[8], d1[8], a1[8];
        auto load3 = [&](int sg, uint32_t (&pv)[8], uint32_t (&dpv)[8], uint32_t (&av)[8]) {
          tmem_ld8(tS + 8u * sg, pv);
          tmem_ld8(tdP + 8u * sg, dpv);
          if (want_db) {
            tmem_ld8(tAcc + 8u * sg, av);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) av[e] = 0u;
          }
        };
        // two sub-groups per TMEM round trip (se - sb is even)
        const int sb = 2 * gb, se = 2 * ge;
#pragma unroll 1
        for (int k2 = 0; k2 < 8; k2 += 2) {
          const int s0 = sb + k2, s1 = sb + k2 + 1;
          if (s0 < se) {
            load3(s0, p0, d0, a0);
            load3(s1, p1, d1, a1);
            tmem_wait_ld_tied(p0, d0, a0);
            tmem_tie(p1, d1, a1);
            ds_sub(s0, p0, d0, a0);
            ds_sub(s1, p1, d1, a1);
          }
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_warp(bar(bDsFull));
    }
    if (ok && !__any_sync(0xffffffffu, *abort_flag != 0) && cur_h >= 0 && want_db)
      flush(a.slot_base[blockIdx.x] + (cur_h - h_first));
    tmem_wait_st();
    tmem_wait_ld();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace bwd
}  // namespace

bool tc_supported(const Geo &g, int dtype) {
  // gather rows are addressed as int32 rows of the [B*T, C] view
  return dtype == SWIN_BF16 && g.hd == 32 && g.n <= 128 && g.T <= fwd::kMaxBiasRows &&
         (int64_t)g.batch * g.tokens <= INT32_MAX;
}
int tc_fwd_ctas_per_sm(const Geo &) { return 1; }
int tc_bwd_ctas_per_sm(const Geo &) { return 1; }

namespace {

// cuTensorMapEncodeTiled through the runtime's driver entry point.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// Tiled map of a [B, G0, G1, G2, C] bf16 tensor whose box is one window of
// one head: (32 channels, w2, w1, w0, 1), 64-byte swizzle (the layout of the
// kernels' operand tiles).
bool box_tensor_map(CUtensorMap *m, const void *base, const Geo &g) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t e = 2;
  cuuint64_t dims[5] = {(cuuint64_t)g.C, (cuuint64_t)g.G[2], (cuuint64_t)g.G[1], (cuuint64_t)g.G[0],
                        (cuuint64_t)g.batch};
  cuuint64_t strides[4] = {dims[0] * e, dims[0] * dims[1] * e, dims[0] * dims[1] * dims[2] * e,
                           dims[0] * dims[1] * dims[2] * dims[3] * e};
  cuuint32_t box[5] = {32u, (cuuint32_t)g.w[2], (cuuint32_t)g.w[1], (cuuint32_t)g.w[0], 1u};
  cuuint32_t es[5] = {1u, 1u, 1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row view [B*T, C] of the same tensor for TMA gather4: box one row high,
// one head's 32 channels wide.
bool row_tensor_map(CUtensorMap *m, const void *base, const Geo &g) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)g.C, (cuuint64_t)g.batch * (cuuint64_t)g.tokens};
  cuuint64_t strides[1] = {dims[0] * 2};
  cuuint32_t box[2] = {32u, 1u};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Both views of one tensor.
bool tensor_maps(TmaSet *t, const void *base, const Geo &g) {
  return box_tensor_map(&t->box, base, g) && row_tensor_map(&t->rows, base, g);
}

}  // namespace

int launch_fwd_tc(const FwdArgs &a, void *stream) {
  TmaSet mq, mk, mv;
  if (!tensor_maps(&mq, a.q, a.g) || !tensor_maps(&mk, a.k, a.g) || !tensor_maps(&mv, a.v, a.g)) return SWIN_ERR_CUDA;
  auto kern = a.g.pack == 2 ? fwd::fwd_tc_kernel<2> : fwd::fwd_tc_kernel<1>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::kSmemBytes) != cudaSuccess)
    return SWIN_ERR_CUDA;
  kern<<<a.ctas, fwd::kThreads, fwd::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(a, mq, mk, mv);
  return cudaPeekAtLastError() == cudaSuccess ? SWIN_OK : SWIN_ERR_CUDA;
}

int launch_bwd_tc(const BwdArgs &a, void *stream) {
  TmaSet mq, mk, mv, mdo;
  if (!tensor_maps(&mq, a.q, a.g) || !tensor_maps(&mk, a.k, a.g) || !tensor_maps(&mv, a.v, a.g) ||
      !tensor_maps(&mdo, a.dout, a.g))
    return SWIN_ERR_CUDA;
  auto kern = a.g.pack == 2 ? bwd::bwd_tc_kernel<2> : bwd::bwd_tc_kernel<1>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bwd::kSmemBytes) != cudaSuccess)
    return SWIN_ERR_CUDA;
  kern<<<a.ctas, bwd::kThreads, bwd::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(a, mq, mk, mv, mdo);
  return cudaPeekAtLastError() == cudaSuccess ? SWIN_OK : SWIN_ERR_CUDA;
}

}  // namespace swin
