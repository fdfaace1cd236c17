// swin_large.cu -- tcgen05/TMEM forward for head_dim 128 and windows of any
// size (sm_103a): the attention of one window is tiled into 128-slot query
// tiles and 128-slot key tiles, with an online softmax across the key tiles.
//
// This is the regime of the pages' large windows: TERRA runs windows of
// w = 32..128 per side (1 024..16 384 tokens) with Nh = 8 heads of d/Nh = 128
// channels through FlashAttention (Sec. VII.A, Experiment Setup); the BEAST
// page's outer windows hold 1 800 and 64 800 tokens (model configuration
// table). The routing is the one of the small-window kernels (TERRA Sec. IV.D;
// BEAST, Model Architecture): every slot's grid token is computed from its
// window and in-window coordinates, Q, K and V rows are gathered straight from
// the [B, grid, C] tensors by TMA, and O rows are stored at their tokens.
//
// Work item = (head, image, window, query tile of 128 slots); each CTA takes a
// contiguous range of items (TERRA Eq. (4)). Per item the CTA keeps the Q tile
// in shared memory and streams the window's key tiles through two stages:
//  * warp 12 loads the Q tile (TMA gather4, two 64-channel halves) and writes
//    the query mask rows Qm; warp 13 loads K and writes the key mask rows Km
//    and the key side of the bias offsets; warp 14 loads V;
//  * warp 15 issues S = Q K^T + Qm Km^T (8 + 1 MMAs, K = 16 each) and
//    O_h += P_h V (4 MMAs per half h);
//  * softmax warpgroup h (warps 4h .. 4h+3, thread = query row) takes keys
//    [64h, 64h + 64) of every key tile: x = S*scale*log2e + bias*log2e, a
//    running row max m_h and sum l_h, P_h = exp2(x - m_h) in bf16 over S. The
//    running max is only raised when a tile's max exceeds it by more than 8
//    (a factor 256): P stays below 256 and O_h (in TMEM) is rescaled rarely;
//    the final normalisation uses the same max, so the result is exact in
//    real arithmetic;
//  * epilogue warps 8-11 combine the halves, O = (a_0 O_0 + a_1 O_1) /
//    (a_0 l_0 + a_1 l_1) with a_h = exp2(m_h - max(m_0, m_1)), and store the
//    rows (and the log-sum-exp) at the query slots' tokens.
// Masked keys (other region, land, pad) get -2^100 from the mask MMA and so
// exactly zero probability. Every wait is bounded, as in the small kernels.
#include <cuda_bf16.h>

#include "swin_large.cuh"

namespace swin {
namespace lg {
namespace {

constexpr int kStages = 2;                  // key/value stages (= S buffers in TMEM)
constexpr int kQ = 0, kQm = kTileBytes;
constexpr int kStage0 = kQm + kMaskBytes;   // 36 KB, 1024-aligned
constexpr int kK = 0, kV = kTileBytes, kKm = 2 * kTileBytes, kRoff = kKm + kMaskBytes;  // inside a stage
constexpr int kStageBytes = 69 * 1024;      // K, V, Km and int roff[128]
constexpr int kBcol = kStage0 + kStages * kStageBytes;  // bias column of the current head (bias*log2e)
constexpr int kMaxBiasRows = 8192;
constexpr int kXchg = kBcol + kMaxBiasRows * 4;  // float [2 items][2 halves][m, l][128]
constexpr int kBarOff = kXchg + 2 * 2 * 2 * 128 * 4;
constexpr int bQFull = 0, bQFree = 1, bFull = 2, bEmpty = bFull + kStages, bSFull = bEmpty + kStages,
              bPFull = bSFull + kStages, bOFull = bPFull + kStages, bTFree = bOFull + 1, bNever = bTFree + 1,
              bDrain = bNever + 1, bBsync = bDrain + 1, kNumBars = bBsync + 1;
constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem slot (u32), abort flag (int)
constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
static_assert(kStage0 % 1024 == 0 && kStageBytes % 1024 == 0, "operand tiles need 1024-byte alignment");
static_assert(kRoff + 512 <= kStageBytes, "stage layout");
static_assert(kSmemBytes <= 232448, "over the 227 KB of shared memory a CTA may use");

// warps 0-7: softmax (warpgroup h = warp / 4 takes key columns [64h, 64h+64));
// 8-11: epilogue; 12: Q; 13: K (+ key masks, bias offsets); 14: V; 15: MMA
constexpr int kSoftmaxWarps = 8, kEpilogueWarp0 = 8, kQWarp = 12, kKWarp = 13, kVWarp = 14, kMmaWarp = 15;
constexpr int kThreads = 16 * 32;
// TMEM columns: S of key tile t at 128 * (t % 2); O half h at 256 + 128 h
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.f;  // raise the running max only past 2^8

__global__ void __launch_bounds__(kThreads, 1)
    fwd_large_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int idx) { return bars + 8u * idx; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMiscOff + 4);

  const Geo &g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkt = g.nqt;  // key tiles per window = query tiles per window
  int64_t L, R;
  eq4_range(a.items, a.ctas, blockIdx.x, L, R);
  const int64_t count = R - L;
  const int64_t ntiles = count * nkt;  // key tiles this CTA streams, over all its items
  WaitCtl ctl{abort_flag, a.status, a.wait_limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(bQFull), 1);
    mbar_init(bar(bQFree), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(bFull + s), 2);    // K warp, V warp
      mbar_init(bar(bEmpty + s), 1);   // MMA commit after PV of the tile
      mbar_init(bar(bSFull + s), 1);
      mbar_init(bar(bPFull + s), kSoftmaxWarps);
    }
    mbar_init(bar(bOFull), 1);
    mbar_init(bar(bTFree), 4);
    mbar_init(bar(bNever), 1);
    mbar_init(bar(bDrain), 1);
    mbar_init(bar(bBsync), kSoftmaxWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // operand tiles start zeroed (rows past the window stay finite); the
  // constant halves of the mask rows: Qm columns 8-15 = 0, Km columns 8-15 =
  // -2^100
  for (int z = threadIdx.x; z < kBcol / 16; z += blockDim.x) reinterpret_cast<uint4 *>(smem)[z] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  {
    const uint32_t nb2 = (uint32_t)kBf16NegBig | ((uint32_t)kBf16NegBig << 16);
    for (int z = threadIdx.x; z < kStages * 128; z += blockDim.x)
      *reinterpret_cast<uint4 *>(smem + kStage0 + (z / 128) * kStageBytes + kKm + sw32(z % 128, 1)) =
          make_uint4(nb2, nb2, nb2, nb2);
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

  if (warp == kQWarp) {
    // ------------------------------------------------------------ Q tile ---
    for (int64_t it = 0; it < count; ++it) {
      const LItem x = decode(g, L + it);
      const Quad q = route_quad(g, x.omega, x.qt, lane);
      bool live[4];
      quad_live(q, a.land, (int64_t)x.b * g.tokens, live);
      if (it > 0 && !mbar_wait_warp(bar(bQFree), (uint32_t)(it - 1) & 1u, ctl)) break;
      const int rows = min(128, g.n - x.qt * 128), nq4 = (rows + 3) >> 2;
      if (lane == 0) mbar_expect_tx(bar(bQFull), (uint32_t)nq4 * 4u * 256u);
      __syncwarp();
      if (lane < nq4) gather_rows(sbase + kQ, &tmq, q, x.b, g.tokens, x.h, lane, bar(bQFull));
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4 *>(smem + kQm + sw32(4 * lane + j, 0)) = mask_chunk(live[j], q.reg[j], false);
      fence_proxy_async_smem();
      mbar_arrive_warp(bar(bQFull));
    }
  } else if (warp == kKWarp || warp == kVWarp) {
    // -------------------------------------------------------- K, V tiles ---
    const bool kw = warp == kKWarp;
    int64_t t = 0;
    for (; t < ntiles; ++t) {
      const int s = (int)(t % kStages);
      const LItem x = decode(g, L + t / nkt);
      const int kt = (int)(t % nkt);
      const Quad q = route_quad(g, x.omega, kt, lane);
      bool live[4];
      if (kw) quad_live(q, a.land, (int64_t)x.b * g.tokens, live);
      if (t >= kStages && !mbar_wait_warp(bar(bEmpty + s), (uint32_t)((t / kStages) - 1) & 1u, ctl)) break;
      const uint32_t st = sbase + kStage0 + s * kStageBytes;
      uint8_t *sp = smem + kStage0 + s * kStageBytes;
      const int rows = min(128, g.n - kt * 128), nq4 = (rows + 3) >> 2;
      if (lane == 0) mbar_expect_tx(bar(bFull + s), (uint32_t)nq4 * 4u * 256u);
      __syncwarp();
      if (lane < nq4) gather_rows(st + (kw ? kK : kV), kw ? &tmk : &tmv, q, x.b, g.tokens, x.h, lane, bar(bFull + s));
      if (kw) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4 *>(sp + kKm + sw32(4 * lane + j, 0)) = mask_chunk(live[j], q.reg[j], true);
        *reinterpret_cast<int4 *>(sp + kRoff + 16 * lane) = make_int4(q.roff[0], q.roff[1], q.roff[2], q.roff[3]);
        fence_proxy_async_smem();
      }
      mbar_arrive_warp(bar(bFull + s));
    }
    // copies still in flight must land before the CTA exits
    volatile int no_abort = 0;
    const WaitCtl dctl{&no_abort, ctl.status, ctl.limit_ns < 50000000ull ? ctl.limit_ns : 50000000ull};
    for (int64_t k = t > kStages ? t - kStages : 0; k < t; ++k)
      mbar_wait_warp(bar(bFull + (int)(k % kStages)), (uint32_t)(k / kStages) & 1u, dctl);
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------- MMA ---
    // Order: S(0); then for every key tile t: S(t+1) (if it belongs to the
    // same item), PV(t), and at an item's last tile PV(t) before S(t+1), so
    // that the next item's Q tile (loaded once S(t) has freed the buffer)
    // lands while PV(t) runs.
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0), idesc_pv = idesc_bf16(128, 128, 0, 1);
      auto issue_s = [&](int64_t t) -> bool {
        const int s = (int)(t % kStages), kt = (int)(t % nkt);
        const int64_t it = t / nkt;
        if (!mbar_wait(bar(bFull + s), (uint32_t)(t / kStages) & 1u, ctl)) return false;
        if (kt == 0 && !mbar_wait(bar(bQFull), (uint32_t)it & 1u, ctl)) return false;
        tc_fence_after();
        const uint32_t st = sbase + kStage0 + s * kStageBytes, d = tmem + 128u * s;
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(d, kmajor_desc(sbase + kQ, kk), kmajor_desc(st + kK, kk), idesc_s, kk > 0 ? 1u : 0u);
        mma_ss(d, smem_desc(sbase + kQm, 16, 256, kSwizzle32B), smem_desc(st + kKm, 16, 256, kSwizzle32B), idesc_s, 1);
        mma_commit(bar(bSFull + s));
        if (kt == nkt - 1) mma_commit(bar(bQFree));
        return true;
      };
      auto issue_pv = [&](int64_t t) -> bool {
        const int s = (int)(t % kStages), kt = (int)(t % nkt);
        const int64_t it = t / nkt;
        if (!mbar_wait(bar(bPFull + s), (uint32_t)(t / kStages) & 1u, ctl)) return false;
        if (kt == 0 && it > 0 && !mbar_wait(bar(bTFree), (uint32_t)(it - 1) & 1u, ctl)) return false;
        tc_fence_after();
        const uint32_t st = sbase + kStage0 + s * kStageBytes;
        for (int h = 0; h < 2; ++h)
          for (int kk = 0; kk < 4; ++kk) {
            // keys 64h + 16kk ..: P from TMEM, V rows from the stage (channels = N, MN-major)
            mma_ts(tmem + kColO + 128u * h, tmem + 128u * s + 64u * h + 16u * kk, nmajor_desc(st + kV, 64 * h + 16 * kk),
                   idesc_pv, (kt > 0 || kk > 0) ? 1u : 0u);
          }
        mma_commit(bar(bEmpty + s));
        if (kt == nkt - 1) mma_commit(bar(bOFull));
        return true;
      };
      bool ok = ntiles > 0 && issue_s(0);
      for (int64_t t = 0; ok && t < ntiles; ++t) {
        const bool last = (t % nkt) == nkt - 1;
        if (!last && t + 1 < ntiles) ok = issue_s(t + 1);
        ok = ok && issue_pv(t);
        if (ok && last && t + 1 < ntiles) ok = issue_s(t + 1);
      }
      mma_commit(bar(bDrain));
      volatile int no_abort = 0;
      WaitCtl drain_ctl{&no_abort, a.status, a.wait_limit_ns};
      mbar_wait(bar(bDrain), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp >= kEpilogueWarp0) {
    // ---------------------------------------------------------- epilogue ---
    const int q4 = warp & 3, i = q4 * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const float *xc = reinterpret_cast<const float *>(smem + kXchg);
    for (int64_t it = 0; it < count; ++it) {
      const LItem x = decode(g, L + it);
      const int slot = x.qt * 128 + i;
      int wc[3];
      window_coords(g, x.omega, wc);
      const int src = slot < g.n ? slot_route(g, wc, slot).src : -1;
      const bool live = src >= 0 && (!a.land || __ldg(a.land + (int64_t)x.b * g.tokens + src) == 0);
      if (!mbar_wait_warp(bar(bOFull), (uint32_t)it & 1u, ctl)) break;
      tc_fence_after();
      const float *xs = xc + (int)(it & 1) * 512;
      const float m0 = xs[i], l0 = xs[128 + i], m1 = xs[256 + i], l1 = xs[384 + i];
      const float m = fmaxf(m0, m1);
      const float a0 = l0 > 0.f ? ex2(m0 - m) : 0.f, a1 = l1 > 0.f ? ex2(m1 - m) : 0.f;
      const float l = fmaf(a0, l0, a1 * l1);
      const float inv = live && l > 0.f ? __frcp_rn(l) : 0.f;
      const float c0 = a0 * inv, c1 = a1 * inv;
      const bool store = src >= 0 && in_bounds(((int64_t)x.b * g.tokens + src) * g.C + (int64_t)x.h * kHd, kHd,
                                                (int64_t)g.batch * g.tokens * g.C, a.status);
      uint4 *dst = store ? reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.o) +
                                                     ((int64_t)x.b * g.tokens + src) * g.C + (int64_t)x.h * kHd)
                         : nullptr;
#pragma unroll 1
      for (int c = 0; c < 8; c += 2) {  // 32 channels per TMEM round trip
        uint32_t o0[16], o1[16], p0[16], p1[16];
        tmem_ld16(tmem + lane_addr + kColO + 16u * c, o0);
        tmem_ld16(tmem + lane_addr + kColO + 16u * (c + 1), o1);
        tmem_ld16(tmem + lane_addr + kColO + 128u + 16u * c, p0);
        tmem_ld16(tmem + lane_addr + kColO + 128u + 16u * (c + 1), p1);
        tmem_wait_ld_tied(o0, o1);
        tmem_tie(p0, p1);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint32_t *h0 = e < 16 ? o0 : o1;
          const uint32_t *h1 = e < 16 ? p0 : p1;
          const int o = e & 15;
          const float v0 = fmaf(__uint_as_float(h1[o]), c1, __uint_as_float(h0[o]) * c0);
          const float v1 = fmaf(__uint_as_float(h1[o + 1]), c1, __uint_as_float(h0[o + 1]) * c0);
          w[e >> 1] = pack_bf16(v0, v1);
        }
        if (store) {
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[2 * c + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive_warp(bar(bTFree));
      if (store && a.lse)
        a.lse[((int64_t)x.b * g.heads + x.h) * g.tokens + src] = live ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
    tmem_wait_ld();
  } else {
    // ----------------------------------------------------------- softmax ---
    const int grp = warp >> 2, q4 = warp & 3, i = q4 * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    float *bcol = reinterpret_cast<float *>(smem + kBcol);
    float *xc = reinterpret_cast<float *>(smem + kXchg);
    const float cs = a.scale * kLog2e;
    const float2 cs2 = make_float2(cs, cs);
    const bool has_bias = a.bias != nullptr;  // the column is read only with a bias (it holds at most kMaxBiasRows)
    int cur_h = -1, rbase = 0;
    uint32_t bs_phase = 0;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    if (a.debug_force_timeout && grp == 0) ok = mbar_wait_warp(bar(bNever), 0, ctl);
    for (int64_t t = 0; ok && t < ntiles; ++t) {
      const int s = (int)(t % kStages), kt = (int)(t % nkt);
      const int64_t it = t / nkt;
      if (kt == 0) {
        const LItem x = decode(g, L + it);
        if (has_bias && x.h != cur_h) {
          // the head's bias column (bias * log2e) in shared memory; everyone
          // is done with the previous one first
          if (cur_h >= 0) {
            mbar_arrive_warp(bar(bBsync));
            if (!mbar_wait_warp(bar(bBsync), bs_phase & 1u, ctl)) break;
            ++bs_phase;
          }
          for (int r = grp * 128 + i; r < g.T; r += 256) bcol[r] = __ldg(a.bias + (int64_t)r * g.heads + x.h) * kLog2e;
          mbar_arrive_warp(bar(bBsync));
          if (!mbar_wait_warp(bar(bBsync), bs_phase & 1u, ctl)) break;
          ++bs_phase;
          cur_h = x.h;
        }
        const int wc0[3] = {0, 0, 0};
        const int slot = x.qt * 128 + i;
        // a row past the window takes the largest query-side offset, so that
        // rbase - roff stays inside the column for every key (its output is
        // never stored)
        rbase = slot < g.n ? slot_route(g, wc0, slot).rbase : g.T - 1;
        m_run = -INFINITY;
        l_run = 0.f;
      }
      const uint32_t tS = tmem + lane_addr + 128u * s + 64u * grp;
      if (!mbar_wait_warp(bar(bSFull + s), (uint32_t)(t / kStages) & 1u, ctl)) break;
      tc_fence_after();
      uint32_t sv[4][16];
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) tmem_ld16(tS + 16u * k4, sv[k4]);
      const int *roff = reinterpret_cast<const int *>(smem + kStage0 + s * kStageBytes + kRoff) + 64 * grp;
      tmem_wait_ld_tied(sv[0], sv[1]);
      tmem_wait_ld_tied(sv[2], sv[3]);
      // x = S*cs + bias2, tile max
      float mp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
#pragma unroll
        for (int e4 = 0; e4 < 16; e4 += 4) {
          float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
          if (has_bias) {
            const int4 r4 = *reinterpret_cast<const int4 *>(roff + 16 * k4 + e4);
            b0 = bcol[rbase - r4.x];
            b1 = bcol[rbase - r4.y];
            b2 = bcol[rbase - r4.z];
            b3 = bcol[rbase - r4.w];
          }
          const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sv[k4][e4]), __uint_as_float(sv[k4][e4 + 1])), cs2,
                                       make_float2(b0, b1));
          const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sv[k4][e4 + 2]), __uint_as_float(sv[k4][e4 + 3])),
                                       cs2, make_float2(b2, b3));
          sv[k4][e4] = __float_as_uint(x0.x);
          sv[k4][e4 + 1] = __float_as_uint(x0.y);
          sv[k4][e4 + 2] = __float_as_uint(x1.x);
          sv[k4][e4 + 3] = __float_as_uint(x1.y);
          mp[e4 >> 2] = max3(mp[e4 >> 2], max3(x0.x, x0.y, x1.x), x1.y);
        }
      }
      const float mt = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3]));
      // a tile whose keys are all masked for this row (about -2^100 after the
      // mask step) adds nothing; otherwise raise the running max only past 2^8
      const bool any = mt > -1e29f;
      float m_new = m_run;
      if (any && (l_run == 0.f || mt > m_run + kRescaleLog2)) m_new = mt;
      const bool rescale = any && l_run > 0.f && m_new != m_run;
      if (__any_sync(0xffffffffu, rescale)) {
        // O half grp of this row is scaled by exp2(m_run - m_new) once the PV of
        // the previous tile (same item) has completed
        if (!mbar_wait_warp(bar(bEmpty + (int)((t - 1) % kStages)), (uint32_t)((t - 1) / kStages) & 1u, ctl)) break;
        tc_fence_after();
        const float f = rescale ? ex2(m_run - m_new) : 1.f;
        const uint32_t tO = tmem + lane_addr + kColO + 128u * grp;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t ov[16];
          tmem_ld16(tO + 16u * c, ov);
          tmem_wait_ld_tied(ov);
#pragma unroll
          for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
          tmem_st16(tO + 16u * c, ov);
        }
        tmem_wait_st();
        l_run *= f;
      }
      m_run = m_new;
      const float msub = any ? m_run : 0.f;
      const float2 negm = make_float2(-msub, -msub);
      float2 sp2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        uint32_t pv[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float2 xs2 = __fadd2_rn(make_float2(__uint_as_float(sv[k4][e]), __uint_as_float(sv[k4][e + 1])), negm);
          const float2 p = any ? make_float2(ex2(xs2.x), ex2(xs2.y)) : make_float2(0.f, 0.f);
          sp2[(e >> 1) & 3] = __fadd2_rn(sp2[(e >> 1) & 3], p);
          pv[e >> 1] = pack_bf16(p.x, p.y);
        }
        tmem_st8(tS + 16u * k4, pv);
      }
      const float2 sum2 = __fadd2_rn(__fadd2_rn(sp2[0], sp2[1]), __fadd2_rn(sp2[2], sp2[3]));
      l_run += sum2.x + sum2.y;
      if (kt == nkt - 1) {
        float *xs = xc + (int)(it & 1) * 512 + grp * 256;
        xs[i] = m_run;
        xs[128 + i] = l_run;
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(bar(bPFull + s));
    }
    tmem_wait_st();
    tmem_wait_ld();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace
}  // namespace lg

bool large_supported(const Geo &g, int dtype) {
  return dtype == SWIN_BF16 && g.hd == lg::kHd && (int64_t)g.batch * g.tokens <= INT32_MAX;
}
int large_max_bias_rows() { return lg::kMaxBiasRows; }

int launch_fwd_large(const FwdArgs &a, void *stream) {
  if (a.bias && a.g.T > lg::kMaxBiasRows) return SWIN_ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  if (!lg::rows128_map(&mq, a.q, a.g) || !lg::rows128_map(&mk, a.k, a.g) || !lg::rows128_map(&mv, a.v, a.g))
    return SWIN_ERR_CUDA;
  if (cudaFuncSetAttribute(lg::fwd_large_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lg::kSmemBytes) !=
      cudaSuccess)
    return SWIN_ERR_CUDA;
  lg::fwd_large_kernel<<<a.ctas, lg::kThreads, lg::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(a, mq, mk, mv);
  return cudaPeekAtLastError() == cudaSuccess ? SWIN_OK : SWIN_ERR_CUDA;
}

}  // namespace swin
