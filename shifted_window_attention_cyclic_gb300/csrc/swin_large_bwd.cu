// swin_large_bwd.cu -- tcgen05/TMEM backward for head_dim 128 and windows of
// any size (sm_103a), deterministic, two kernels over 128-slot tiles:
//
//  * bwdq_kernel, one query tile per item, two sweeps over the window's key
//    tiles. Sweep 1 recomputes S = Q K^T + mask and dP = dO V^T and
//    accumulates delta_i = sum_j P_ij dP_ij (P = exp2(S*scale*log2e +
//    bias*log2e - lse*log2e) from the forward's log-sum-exp); delta goes to
//    the workspace. Sweep 2 recomputes S and dP, forms dS = P (dP - delta) in
//    bf16 over S in TMEM and accumulates dQ += dS K on the tensor cores
//    (A from TMEM); the epilogue stores dQ * hd^-1/2 at the query tokens.
//    Given the forward's output O, delta_kernel first writes delta_i =
//    sum_c dO_ic O_ic instead and the kernel runs sweep 2 alone.
//  * bwdkv_kernel, one key tile per item, one sweep over the window's query
//    tiles with the keys as the MMA rows: S^T = K Q^T + mask and dP^T = V dO^T,
//    P^T and dS^T (bf16) over them in TMEM, dV += P^T dO and dK += dS^T Q (A
//    from TMEM, B the query tiles as MN-major operands); the dBias of the
//    CTA's head accumulates per bias row in shared memory (atomic adds, or
//    per-diagonal sums where a warp's keys and 16 queries have bias offsets
//    stepping by one) and is written to the CTA's workspace slot at head
//    changes; the epilogue stores dV and dK * hd^-1/2 at the key tokens.
// By default delta is the textbook softmax derivative sum, recomputed from P
// and dP, so this backward reads neither O nor an fp32 copy of it; the form
// from O (TERRA's FlashAttention-style backward) saves sweep 1 and carries
// O's bf16 rounding. Routing, masks and the bias column are those of the
// forward. Whole-row tiles load as 5-D boxes, others as boxes of runs of
// consecutive slots and gather4 rows. Items are strided over the CTAs
// (neighbouring tiles of one window stay in L2), except in the key-tile
// kernel with dBias, whose workspace slots follow contiguous item ranges;
// that kernel takes two query-tile stages when there is neither bias nor
// dBias, one otherwise.
#include <cuda_bf16.h>

#include "swin_large.cuh"

namespace swin {
namespace lg {
namespace {

constexpr int kSoftmaxWarps = 8, kEpilogueWarp0 = 8, kMmaWarp = 15;
constexpr int kThreads = 16 * 32;

// ------------------------------------------------------------ query tiles ---
namespace bq {
constexpr int kStages = 2;
constexpr int kQ = 0, kdO = kTileBytes, kQm = 2 * kTileBytes;  // resident per item
constexpr int kStage0 = kQm + kMaskBytes;                       // 68 KB
constexpr int kK = 0, kV = kTileBytes, kKm = 2 * kTileBytes, kRoff = kKm + kMaskBytes;
constexpr int kStageBytes = 69 * 1024;
constexpr int kBcol = kStage0 + kStages * kStageBytes;
constexpr int kMaxBiasRows = 4096;
constexpr int kDx = kBcol + kMaxBiasRows * 4;  // float [2 items][2 halves][128]: delta partials
constexpr int kBarOff = kDx + 2 * 2 * 128 * 4;
constexpr int bQFull = 0, bQFree = 1, bFull = 2, bEmpty = bFull + kStages, bSFull = bEmpty + kStages,
              bPFull = bSFull + 1, bDQFull = bPFull + 1, bTFree = bDQFull + 1, bNever = bTFree + 1,
              bDrain = bNever + 1, bBsync = bDrain + 1, kNumBars = bBsync + 1;
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kSmemBytes = kMiscOff + 16 + 1024;
static_assert(kStage0 % 1024 == 0 && kStageBytes % 1024 == 0 && kRoff + 512 <= kStageBytes, "layout");
static_assert(kSmemBytes <= 232448, "over the 227 KB of shared memory a CTA may use");
constexpr int kQWarp = 12, kKWarp = 13, kVWarp = 14;
constexpr uint32_t kColS = 0, kColdP = 128, kColdQ = 256;

__global__ void __launch_bounds__(kThreads, 1)
    bwdq_kernel(const BwdArgs a, const __grid_constant__ TileMaps tmq, const __grid_constant__ TileMaps tmk,
                const __grid_constant__ TileMaps tmv, const __grid_constant__ TileMaps tmdo) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int idx) { return bars + 8u * idx; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMiscOff + 4);
  const Geo &g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // key tiles per item: two sweeps (delta, then dS and dQ), or one when delta
  // was computed from the forward's output before this kernel
  const bool delta_given = a.o != nullptr;
  const int nkt = g.nqt, per_item = delta_given ? nkt : 2 * nkt;
  const Items its = strided_items(a.items, a.ctas);
  const int64_t count = its.count, ntiles = count * per_item;
  WaitCtl ctl{abort_flag, a.status, a.wait_limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(bQFull), 1);
    mbar_init(bar(bQFree), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(bFull + s), 2);
      mbar_init(bar(bEmpty + s), 1);
    }
    mbar_init(bar(bSFull), 1);
    mbar_init(bar(bPFull), kSoftmaxWarps);
    mbar_init(bar(bDQFull), 1);
    mbar_init(bar(bTFree), 4);
    mbar_init(bar(bNever), 1);
    mbar_init(bar(bDrain), 1);
    mbar_init(bar(bBsync), kSoftmaxWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
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
    // -------------------------------------------------- Q, dO and masks ---
    for (int64_t it = 0; it < count; ++it) {
      const LItem x = decode(g, its[it]);
      const Quad q = route_quad(g, x.omega, x.qt, lane);
      bool live[4];
      quad_live(q, a.land, (int64_t)x.b * g.tokens, live);
      if (it > 0 && !mbar_wait_warp(bar(bQFree), (uint32_t)(it - 1) & 1u, ctl)) break;
      const int rows = min(128, g.n - x.qt * 128), nq4 = (rows + 3) >> 2;
      if (lane == 0) mbar_expect_tx(bar(bQFull), (uint32_t)nq4 * 2u * 1024u);
      __syncwarp();
      int c[3];
      const bool box = tile_box(g, x.omega, x.qt, c);
      load_tile(sbase + kQ, &tmq, g, box, c, q, x.b, x.h, lane, nq4, bar(bQFull));
      load_tile(sbase + kdO, &tmdo, g, box, c, q, x.b, x.h, lane, nq4, bar(bQFull));
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
      const LItem x = decode(g, its[t / per_item]);
      const int kt = (int)((t % per_item) % nkt);
      const Quad q = route_quad(g, x.omega, kt, lane);
      bool live[4];
      if (kw) quad_live(q, a.land, (int64_t)x.b * g.tokens, live);
      if (t >= kStages && !mbar_wait_warp(bar(bEmpty + s), (uint32_t)((t / kStages) - 1) & 1u, ctl)) break;
      const uint32_t st = sbase + kStage0 + s * kStageBytes;
      uint8_t *sp = smem + kStage0 + s * kStageBytes;
      const int rows = min(128, g.n - kt * 128), nq4 = (rows + 3) >> 2;
      if (lane == 0) mbar_expect_tx(bar(bFull + s), (uint32_t)nq4 * 1024u);
      __syncwarp();
      int c[3];
      const bool box = tile_box(g, x.omega, kt, c);
      load_tile(st + (kw ? kK : kV), kw ? &tmk : &tmv, g, box, c, q, x.b, x.h, lane, nq4, bar(bFull + s));
      if (kw) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4 *>(sp + kKm + sw32(4 * lane + j, 0)) = mask_chunk(live[j], q.reg[j], true);
        *reinterpret_cast<int4 *>(sp + kRoff + 16 * lane) = make_int4(q.roff[0], q.roff[1], q.roff[2], q.roff[3]);
        fence_proxy_async_smem();
      }
      mbar_arrive_warp(bar(bFull + s));
    }
    volatile int no_abort = 0;
    const WaitCtl dctl{&no_abort, ctl.status, ctl.limit_ns < 50000000ull ? ctl.limit_ns : 50000000ull};
    for (int64_t k = t > kStages ? t - kStages : 0; k < t; ++k)
      mbar_wait_warp(bar(bFull + (int)(k % kStages)), (uint32_t)(k / kStages) & 1u, dctl);
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------- MMA ---
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0), idesc_dq = idesc_bf16(128, 128, 0, 1);
      bool ok = true;
      for (int64_t t = 0; ok && t < ntiles; ++t) {
        const int s = (int)(t % kStages), u = (int)(t % per_item), kt = u % nkt;
        const int64_t it = t / per_item;
        const bool second = delta_given || u >= nkt;
        ok = mbar_wait(bar(bFull + s), (uint32_t)(t / kStages) & 1u, ctl) &&
             (u != 0 || mbar_wait(bar(bQFull), (uint32_t)it & 1u, ctl)) &&
             (t == 0 || mbar_wait(bar(bPFull), (uint32_t)(t - 1) & 1u, ctl));  // S and dP of t-1 consumed
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = sbase + kStage0 + s * kStageBytes;
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + kColS, kmajor_desc(sbase + kQ, kk), kmajor_desc(st + kK, kk), idesc_s, kk > 0 ? 1u : 0u);
        mma_ss(tmem + kColS, smem_desc(sbase + kQm, 16, 256, kSwizzle32B), smem_desc(st + kKm, 16, 256, kSwizzle32B),
               idesc_s, 1);
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + kColdP, kmajor_desc(sbase + kdO, kk), kmajor_desc(st + kV, kk), idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(bar(bSFull));
        if (u == per_item - 1) mma_commit(bar(bQFree));  // the item's last reads of Q, dO and Qm
        if (!second) {
          mma_commit(bar(bEmpty + s));
          continue;
        }
        // dQ += dS K once dS is written over S (and the epilogue has read dQ of the previous item)
        ok = mbar_wait(bar(bPFull), (uint32_t)t & 1u, ctl) &&
             (kt != 0 || it == 0 || mbar_wait(bar(bTFree), (uint32_t)(it - 1) & 1u, ctl));
        if (!ok) break;
        tc_fence_after();
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + kColdQ, tmem + kColS + 16u * kk, nmajor_desc(st + kK, 16 * kk), idesc_dq,
                 (kt > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(bEmpty + s));
        if (kt == nkt - 1) mma_commit(bar(bDQFull));
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
    for (int64_t it = 0; it < count; ++it) {
      const LItem x = decode(g, its[it]);
      const int slot = x.qt * 128 + i;
      int wc[3];
      window_coords(g, x.omega, wc);
      const int src = slot < g.n ? slot_route(g, wc, slot).src : -1;
      if (!mbar_wait_warp(bar(bDQFull), (uint32_t)it & 1u, ctl)) break;
      tc_fence_after();
      const bool store = src >= 0 && in_bounds(((int64_t)x.b * g.tokens + src) * g.C + (int64_t)x.h * kHd, kHd,
                                                (int64_t)g.batch * g.tokens * g.C, a.status);
      uint4 *dst = store ? reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.dq) +
                                                     ((int64_t)x.b * g.tokens + src) * g.C + (int64_t)x.h * kHd)
                         : nullptr;
#pragma unroll 1
      for (int c = 0; c < 8; c += 2) {
        uint32_t v0[16], v1[16];
        tmem_ld16(tmem + lane_addr + kColdQ + 16u * c, v0);
        tmem_ld16(tmem + lane_addr + kColdQ + 16u * (c + 1), v1);
        tmem_wait_ld_tied(v0, v1);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          w[e >> 1] = pack_bf16(__uint_as_float(v0[e]) * a.scale, __uint_as_float(v0[e + 1]) * a.scale);
          w[8 + (e >> 1)] = pack_bf16(__uint_as_float(v1[e]) * a.scale, __uint_as_float(v1[e + 1]) * a.scale);
        }
        if (store) {
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[2 * c + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive_warp(bar(bTFree));
    }
    tmem_wait_ld();
  } else {
    // ----------------------------------------------------------- softmax ---
    // thread = query row i; warpgroup grp takes keys [64 grp, 64 grp + 64) of
    // every key tile
    const int grp = warp >> 2, q4 = warp & 3, i = q4 * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    float *bcol = reinterpret_cast<float *>(smem + kBcol);
    float *dx = reinterpret_cast<float *>(smem + kDx);
    const float cs = a.scale * kLog2e;
    const bool has_bias = a.bias != nullptr;
    int cur_h = -1, rbase = 0, src = -1;
    bool live = false;
    float lse2 = 0.f, dpart = 0.f, delta = 0.f;
    uint32_t bs_phase = 0;
    bool ok = true;
    if (a.debug_force_timeout) ok = mbar_wait_warp(bar(bNever), 0, ctl);
    for (int64_t t = 0; ok && t < ntiles; ++t) {
      const int s = (int)(t % kStages), u = (int)(t % per_item), kt = u % nkt;
      const int64_t it = t / per_item;
      const bool second = delta_given || u >= nkt;
      const LItem x = decode(g, its[it]);
      if (u == 0) {
        if (has_bias && x.h != cur_h) {
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
        const int slot = x.qt * 128 + i;
        int wc[3];
        window_coords(g, x.omega, wc);
        const SlotRoute r = slot_route(g, wc, slot < g.n ? slot : 0);
        src = slot < g.n ? r.src : -1;
        rbase = slot < g.n ? r.rbase : g.T - 1;
        live = src >= 0 && (!a.land || __ldg(a.land + (int64_t)x.b * g.tokens + src) == 0);
        lse2 = live ? __ldg(a.lse + ((int64_t)x.b * g.heads + x.h) * g.tokens + src) * kLog2e : 0.f;
        dpart = 0.f;
        if (delta_given) delta = live ? __ldcg(a.delta + ((int64_t)x.b * g.heads + x.h) * g.tokens + src) : 0.f;
      }
      if (!mbar_wait_warp(bar(bSFull), (uint32_t)t & 1u, ctl)) break;
      tc_fence_after();
      const int *roff = reinterpret_cast<const int *>(smem + kStage0 + s * kStageBytes + kRoff) + 64 * grp;
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        const uint32_t col = 64u * grp + 32u * c2;
        uint32_t sv0[16], sv1[16], dv0[16], dv1[16];
        tmem_ld16(tmem + lane_addr + kColS + col, sv0);
        tmem_ld16(tmem + lane_addr + kColS + col + 16, sv1);
        tmem_ld16(tmem + lane_addr + kColdP + col, dv0);
        tmem_ld16(tmem + lane_addr + kColdP + col + 16, dv1);
        tmem_wait_ld_tied(sv0, sv1);
        tmem_tie(dv0, dv1);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t *sv = hh ? sv1 : sv0;
          const uint32_t *dv = hh ? dv1 : dv0;
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float b0 = 0.f, b1 = 0.f;
            if (has_bias) {
              const int2 r2 = *reinterpret_cast<const int2 *>(roff + 32 * c2 + 16 * hh + e);
              b0 = bcol[rbase - r2.x];
              b1 = bcol[rbase - r2.y];
            }
            const float x0 = fmaf(__uint_as_float(sv[e]), cs, b0) - lse2;
            const float x1 = fmaf(__uint_as_float(sv[e + 1]), cs, b1) - lse2;
            const float p0 = live ? ex2(x0) : 0.f, p1 = live ? ex2(x1) : 0.f;
            const float d0 = __uint_as_float(dv[e]), d1 = __uint_as_float(dv[e + 1]);
            if (!second) {
              dpart = fmaf(p0, d0, dpart);
              dpart = fmaf(p1, d1, dpart);
            } else {
              pk[e >> 1] = pack_bf16(p0 * (d0 - delta), p1 * (d1 - delta));
            }
          }
          if (second) tmem_st8(tmem + lane_addr + kColS + col + 16u * hh, pk);  // dS over the first half of S's group
        }
      }
      if (second) tmem_wait_st();
      if (!second && kt == nkt - 1) {
        // delta_i = the two key halves' partial sums, in a fixed order
        float *d2 = dx + (int)(it & 1) * 256;
        d2[grp * 128 + i] = dpart;
        mbar_arrive_warp(bar(bBsync));
        if (!mbar_wait_warp(bar(bBsync), bs_phase & 1u, ctl)) break;
        ++bs_phase;
        delta = d2[i] + d2[128 + i];
        if (grp == 0 && src >= 0) a.delta[((int64_t)x.b * g.heads + x.h) * g.tokens + src] = live ? delta : 0.f;
      }
      tc_fence_before();
      mbar_arrive_warp(bar(bPFull));
    }
    tmem_wait_st();
    tmem_wait_ld();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}
}  // namespace bq

// ---------------------------------------------------------- delta from O ---
// delta_i = sum_c dO_ic O_ic over each head's 128 channels (the softmax
// derivative's row sum, FlashAttention's form): one warp per token, lanes
// over 16-byte chunks of the token's C channels, 16 lanes per head and pass.
__global__ void __launch_bounds__(256) delta_kernel(const BwdArgs a) {
  const Geo &g = a.g;
  const int64_t tok = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= (int64_t)g.batch * g.tokens) return;
  const int64_t b = tok / g.tokens, t = tok % g.tokens;
  const uint4 *o = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.o) + tok * g.C);
  const uint4 *d = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.dout) + tok * g.C);
  const int chunks = g.C >> 3;  // 16-byte chunks per token (16 per head)
  for (int c0 = 0; c0 < chunks; c0 += 32) {
    const int c = c0 + lane;
    float s = 0.f;
    if (c < chunks) {
      const uint4 x = __ldg(o + c), y = __ldg(d + c);
      const uint32_t xa[4] = {x.x, x.y, x.z, x.w}, ya[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s = fmaf(__uint_as_float(xa[e] << 16), __uint_as_float(ya[e] << 16), s);
        s = fmaf(__uint_as_float(xa[e] & 0xFFFF0000u), __uint_as_float(ya[e] & 0xFFFF0000u), s);
      }
    }
#pragma unroll
    for (int m = 8; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    if ((lane & 15) == 0 && c < chunks) a.delta[(b * g.heads + (c >> 4)) * g.tokens + t] = s;
  }
}

// -------------------------------------------------------------- key tiles ---
namespace bkv {
constexpr int kK = 0, kV = kTileBytes, kKm = 2 * kTileBytes;  // resident per item
constexpr int kStage = kKm + kMaskBytes;                         // one query-tile stage
constexpr int kQ = 0, kdO = kTileBytes, kQm = 2 * kTileBytes, kLse = kQm + kMaskBytes, kDelta = kLse + 512,
              kRbase = kDelta + 512;
constexpr int kStageBytes = 70 * 1024;
constexpr int kMaxBiasRows = 8192;
static_assert(kStage % 1024 == 0 && kStageBytes % 1024 == 0 && kRbase + 512 <= kStageBytes, "layout");
// Shared memory with kQS query-tile stages. One stage leaves room for the
// head's bias column, the dBias accumulator and the diagonal-sum scratch; two
// stages (a launch with neither bias nor dBias) load the next query tile
// while this one is computed.
template <int kQS>
struct Lay {
  static constexpr int kBcol = kStage + kQS * kStageBytes;
  static constexpr int kBacc = kBcol + kMaxBiasRows * 4;  // float dBias accumulator of the current head
  // float [8 warps][32 keys][17]: one warp's dS of 16 queries, staged for the diagonal sums
  static constexpr int kDiag = kBacc + kMaxBiasRows * 4;
  static constexpr int kBarOff = kQS == 1 ? kDiag + 8 * 32 * 17 * 4 : kStage + kQS * kStageBytes;
  // stage s: bFull + s (its query tile landed), bEmpty + s (its MMAs are done)
  static constexpr int bKVFull = 0, bKVFree = 1, bFull = 2, bEmpty = bFull + kQS, bSFull = bEmpty + kQS,
                       bPFull = bSFull + 1, bDKVFull = bSFull + 2, bTFree = bSFull + 3, bNever = bSFull + 4,
                       bDrain = bSFull + 5, bBsync = bSFull + 6, kNumBars = bSFull + 7;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "over the 227 KB of shared memory a CTA may use");
};
constexpr int kKVWarp = 12, kQWarp = 13, kdOWarp = 14;
constexpr uint32_t kColS = 0, kColdP = 128, kColdV = 256, kColdK = 384;

template <int kQS>
__global__ void __launch_bounds__(kThreads, 1)
    bwdkv_kernel(const BwdArgs a, const __grid_constant__ TileMaps tmq, const __grid_constant__ TileMaps tmk,
                 const __grid_constant__ TileMaps tmv, const __grid_constant__ TileMaps tmdo) {
  using L_ = Lay<kQS>;
  constexpr int kBcol = L_::kBcol, kBacc = L_::kBacc, kDiag = L_::kDiag, kBarOff = L_::kBarOff,
                kMiscOff = L_::kMiscOff;
  constexpr int bKVFull = L_::bKVFull, bKVFree = L_::bKVFree, bFull = L_::bFull, bEmpty = L_::bEmpty,
                bSFull = L_::bSFull, bPFull = L_::bPFull, bDKVFull = L_::bDKVFull, bTFree = L_::bTFree,
                bNever = L_::bNever, bDrain = L_::bDrain, bBsync = L_::bBsync;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int idx) { return bars + 8u * idx; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMiscOff + 4);
  const Geo &g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqt = g.nqt;
  // (the dBias workspace slots of a launch with dBias follow the contiguous ranges)
  const Items its = kQS == 2 ? strided_items(a.items, a.ctas) : range_items(a.items, a.ctas);
  const int64_t count = its.count, ntiles = count * nqt;  // query tiles streamed over all items
  WaitCtl ctl{abort_flag, a.status, a.wait_limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(bKVFull), 1);
    mbar_init(bar(bKVFree), 1);
    for (int s = 0; s < kQS; ++s) {
      mbar_init(bar(bFull + s), 2);
      mbar_init(bar(bEmpty + s), 1);
    }
    mbar_init(bar(bSFull), 1);
    mbar_init(bar(bPFull), kSoftmaxWarps);
    mbar_init(bar(bDKVFull), 1);
    mbar_init(bar(bTFree), 4);
    mbar_init(bar(bNever), 1);
    mbar_init(bar(bDrain), 1);
    mbar_init(bar(bBsync), kSoftmaxWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int z = threadIdx.x; z < kBarOff / 16; z += blockDim.x) reinterpret_cast<uint4 *>(smem)[z] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  {
    // the constant half of the key mask rows (columns 8-15: -2^100)
    const uint32_t nb2 = (uint32_t)kBf16NegBig | ((uint32_t)kBf16NegBig << 16);
    if (threadIdx.x < 128) *reinterpret_cast<uint4 *>(smem + kKm + sw32(threadIdx.x, 1)) = make_uint4(nb2, nb2, nb2, nb2);
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

  if (warp == kKVWarp) {
    // --------------------------------------------- K, V and key mask rows ---
    for (int64_t it = 0; it < count; ++it) {
      const LItem x = decode(g, its[it]);  // x.qt is the key tile here
      const Quad q = route_quad(g, x.omega, x.qt, lane);
      bool live[4];
      quad_live(q, a.land, (int64_t)x.b * g.tokens, live);
      if (it > 0 && !mbar_wait_warp(bar(bKVFree), (uint32_t)(it - 1) & 1u, ctl)) break;
      const int rows = min(128, g.n - x.qt * 128), nq4 = (rows + 3) >> 2;
      if (lane == 0) mbar_expect_tx(bar(bKVFull), (uint32_t)nq4 * 2u * 1024u);
      __syncwarp();
      int c[3];
      const bool box = tile_box(g, x.omega, x.qt, c);
      load_tile(sbase + kK, &tmk, g, box, c, q, x.b, x.h, lane, nq4, bar(bKVFull));
      load_tile(sbase + kV, &tmv, g, box, c, q, x.b, x.h, lane, nq4, bar(bKVFull));
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4 *>(smem + kKm + sw32(4 * lane + j, 0)) = mask_chunk(live[j], q.reg[j], true);
      fence_proxy_async_smem();
      mbar_arrive_warp(bar(bKVFull));
    }
  } else if (warp == kQWarp || warp == kdOWarp) {
    // ---------------------------------- query tiles (Q, dO, masks, meta) ---
    const bool qw = warp == kQWarp;
    int64_t t = 0;
    for (; t < ntiles; ++t) {
      const int s = (int)(t % kQS);
      const LItem x = decode(g, its[t / nqt]);
      const int qt = (int)(t % nqt);
      const Quad q = route_quad(g, x.omega, qt, lane);
      bool live[4];
      float lse2[4], dl[4];
      if (qw) {
        quad_live(q, a.land, (int64_t)x.b * g.tokens, live);
        const int64_t base = ((int64_t)x.b * g.heads + x.h) * g.tokens;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // dead queries (land, pads) get lse2 = +inf: P = exp2(x - inf) = 0
          lse2[j] = live[j] ? __ldg(a.lse + base + q.src[j]) * kLog2e : INFINITY;
          dl[j] = live[j] ? __ldcg(a.delta + base + q.src[j]) : 0.f;
        }
      }
      if (t >= kQS && !mbar_wait_warp(bar(bEmpty + s), (uint32_t)((t / kQS) - 1) & 1u, ctl)) break;
      uint8_t *sp = smem + kStage + s * kStageBytes;
      const int rows = min(128, g.n - qt * 128), nq4 = (rows + 3) >> 2;
      if (lane == 0) mbar_expect_tx(bar(bFull + s), (uint32_t)nq4 * 1024u);
      __syncwarp();
      int c[3];
      const bool box = tile_box(g, x.omega, qt, c);
      load_tile(sbase + kStage + s * kStageBytes + (qw ? kQ : kdO), qw ? &tmq : &tmdo, g, box, c, q, x.b, x.h, lane,
                nq4, bar(bFull + s));
      if (qw) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4 *>(sp + kQm + sw32(4 * lane + j, 0)) = mask_chunk(live[j], q.reg[j], false);
        *reinterpret_cast<float4 *>(sp + kLse + 16 * lane) = make_float4(lse2[0], lse2[1], lse2[2], lse2[3]);
        *reinterpret_cast<float4 *>(sp + kDelta + 16 * lane) = make_float4(dl[0], dl[1], dl[2], dl[3]);
        *reinterpret_cast<int4 *>(sp + kRbase + 16 * lane) = make_int4(q.rbase[0], q.rbase[1], q.rbase[2], q.rbase[3]);
        fence_proxy_async_smem();
      }
      mbar_arrive_warp(bar(bFull + s));
    }
    // copies still in flight must land before the CTA exits
    volatile int no_abort = 0;
    const WaitCtl dctl{&no_abort, ctl.status, ctl.limit_ns < 50000000ull ? ctl.limit_ns : 50000000ull};
    for (int64_t k = t > kQS ? t - kQS : 0; k < t; ++k)
      mbar_wait_warp(bar(bFull + (int)(k % kQS)), (uint32_t)(k / kQS) & 1u, dctl);
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------- MMA ---
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0), idesc_acc = idesc_bf16(128, 128, 0, 1);
      bool ok = true;
      for (int64_t t = 0; ok && t < ntiles; ++t) {
        const int qt = (int)(t % nqt), s = (int)(t % kQS);
        const int64_t it = t / nqt;
        const uint32_t st = sbase + kStage + s * kStageBytes;
        ok = mbar_wait(bar(bFull + s), (uint32_t)(t / kQS) & 1u, ctl) &&
             (qt != 0 || mbar_wait(bar(bKVFull), (uint32_t)it & 1u, ctl)) &&
             (t == 0 || mbar_wait(bar(bPFull), (uint32_t)(t - 1) & 1u, ctl));
        if (!ok) break;
        tc_fence_after();
        // S^T = K Q^T + mask (keys are the rows), dP^T = V dO^T
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + kColS, kmajor_desc(sbase + kK, kk), kmajor_desc(st + kQ, kk), idesc_s, kk > 0 ? 1u : 0u);
        mma_ss(tmem + kColS, smem_desc(sbase + kKm, 16, 256, kSwizzle32B), smem_desc(st + kQm, 16, 256, kSwizzle32B),
               idesc_s, 1);
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + kColdP, kmajor_desc(sbase + kV, kk), kmajor_desc(st + kdO, kk), idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(bar(bSFull));
        if (qt == nqt - 1) mma_commit(bar(bKVFree));  // the item's last reads of K, V and the key masks
        ok = mbar_wait(bar(bPFull), (uint32_t)t & 1u, ctl) &&
             (qt != 0 || it == 0 || mbar_wait(bar(bTFree), (uint32_t)(it - 1) & 1u, ctl));
        if (!ok) break;
        tc_fence_after();
        // dV += P^T dO, dK += dS^T Q (A from TMEM, the query rows of dO and Q as MN-major B)
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + kColdV, tmem + kColS + 16u * kk, nmajor_desc(st + kdO, 16 * kk), idesc_acc,
                 (qt > 0 || kk > 0) ? 1u : 0u);
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + kColdK, tmem + kColdP + 16u * kk, nmajor_desc(st + kQ, 16 * kk), idesc_acc,
                 (qt > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(bEmpty + s));
        if (qt == nqt - 1) mma_commit(bar(bDKVFull));
      }
      mma_commit(bar(bDrain));
      volatile int no_abort = 0;
      WaitCtl drain_ctl{&no_abort, a.status, a.wait_limit_ns};
      mbar_wait(bar(bDrain), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp >= kEpilogueWarp0) {
    // ---------------------------------------------------------- epilogue ---
    const int q4 = warp & 3, j = q4 * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    for (int64_t it = 0; it < count; ++it) {
      const LItem x = decode(g, its[it]);
      const int slot = x.qt * 128 + j;
      int wc[3];
      window_coords(g, x.omega, wc);
      const int src = slot < g.n ? slot_route(g, wc, slot).src : -1;
      if (!mbar_wait_warp(bar(bDKVFull), (uint32_t)it & 1u, ctl)) break;
      tc_fence_after();
      const bool store = src >= 0 && in_bounds(((int64_t)x.b * g.tokens + src) * g.C + (int64_t)x.h * kHd, kHd,
                                                (int64_t)g.batch * g.tokens * g.C, a.status);
      const int64_t off = ((int64_t)x.b * g.tokens + (store ? src : 0)) * g.C + (int64_t)x.h * kHd;
#pragma unroll 1
      for (int acc = 0; acc < 2; ++acc) {  // dV, then dK * hd^-1/2
        const uint32_t col = acc ? kColdK : kColdV;
        const float mul = acc ? a.scale : 1.f;
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(acc ? a.dk : a.dv) + off);
#pragma unroll 1
        for (int c = 0; c < 8; c += 2) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tmem + lane_addr + col + 16u * c, v0);
          tmem_ld16(tmem + lane_addr + col + 16u * (c + 1), v1);
          tmem_wait_ld_tied(v0, v1);
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            w[e >> 1] = pack_bf16(__uint_as_float(v0[e]) * mul, __uint_as_float(v0[e + 1]) * mul);
            w[8 + (e >> 1)] = pack_bf16(__uint_as_float(v1[e]) * mul, __uint_as_float(v1[e + 1]) * mul);
          }
          if (store) {
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[2 * c + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive_warp(bar(bTFree));
    }
    tmem_wait_ld();
  } else {
    // ----------------------------------------------------------- softmax ---
    // thread = key row j; warpgroup grp takes queries [64 grp, 64 grp + 64)
    // of every query tile
    const int grp = warp >> 2, q4 = warp & 3, j = q4 * 32 + lane, tid = grp * 128 + j;
    float *diag = reinterpret_cast<float *>(smem + kDiag) + warp * (32 * 17);
    bool keys_run = false;  // this warp's 32 keys are window slots whose bias offsets step by one
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    float *bcol = reinterpret_cast<float *>(smem + kBcol);
    float *bacc = reinterpret_cast<float *>(smem + kBacc);
    const float cs = a.scale * kLog2e;
    // (the host picks two query stages only without bias and dBias)
    const bool has_bias = kQS == 1 && a.bias != nullptr, want_db = kQS == 1 && a.ws != nullptr;
    int cur_h = -1, h_first = -1, roff = 0;
    uint32_t bs_phase = 0;
    bool ok = true;
    auto bsync = [&]() -> bool {
      mbar_arrive_warp(bar(bBsync));
      const bool r = mbar_wait_warp(bar(bBsync), bs_phase & 1u, ctl);
      ++bs_phase;
      return r;
    };
    // the CTA's dBias of head cur_h into its workspace slot, accumulator cleared
    auto flush = [&]() {
      float *dstw = a.ws + (int64_t)(a.slot_base[blockIdx.x] + (cur_h - h_first)) * g.T;
      for (int r = tid; r < g.T; r += 256) {
        if (in_bounds((int64_t)(a.slot_base[blockIdx.x] + (cur_h - h_first)) * g.T + r, 1, a.ws_slots * g.T, a.status))
          dstw[r] = bacc[r];
        bacc[r] = 0.f;
      }
    };
    if (a.debug_force_timeout) ok = mbar_wait_warp(bar(bNever), 0, ctl);
    for (int64_t t = 0; ok && t < ntiles; ++t) {
      const int qt = (int)(t % nqt);
      const int64_t it = t / nqt;
      if (qt == 0) {
        const LItem x = decode(g, its[it]);
        if (x.h != cur_h) {
          if (cur_h >= 0) {
            if (!bsync()) break;  // every accumulation and bias read of the previous head is done
            if (want_db) flush();
          }
          if (has_bias)
            for (int r = tid; r < g.T; r += 256) bcol[r] = __ldg(a.bias + (int64_t)r * g.heads + x.h) * kLog2e;
          if (!bsync()) break;
          if (h_first < 0) h_first = x.h;
          cur_h = x.h;
        }
        const int slot = x.qt * 128 + j;
        const int wc0[3] = {0, 0, 0};
        roff = slot < g.n ? slot_route(g, wc0, slot).roff : 0;
        // (the shuffle runs on every lane: a full-mask shuffle that some lanes
        // skip never completes)
        const int roff0 = __shfl_sync(0xffffffffu, roff, 0);
        keys_run = __all_sync(0xffffffffu, slot < g.n && roff == roff0 + lane);
      }
      if (!mbar_wait_warp(bar(bSFull), (uint32_t)t & 1u, ctl)) break;
      tc_fence_after();
      const uint8_t *sp = smem + kStage + (int)(t % kQS) * kStageBytes;
      const float *lse2 = reinterpret_cast<const float *>(sp + kLse) + 64 * grp;
      const float *dl = reinterpret_cast<const float *>(sp + kDelta) + 64 * grp;
      const int *rb = reinterpret_cast<const int *>(sp + kRbase) + 64 * grp;
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        const uint32_t col = 64u * grp + 32u * c2;
        uint32_t sv0[16], sv1[16], dv0[16], dv1[16];
        tmem_ld16(tmem + lane_addr + kColS + col, sv0);
        tmem_ld16(tmem + lane_addr + kColS + col + 16, sv1);
        tmem_ld16(tmem + lane_addr + kColdP + col, dv0);
        tmem_ld16(tmem + lane_addr + kColdP + col + 16, dv1);
        tmem_wait_ld_tied(sv0, sv1);
        tmem_tie(dv0, dv1);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t *sv = hh ? sv1 : sv0;
          const uint32_t *dv = hh ? dv1 : dv0;
          const int c0 = 32 * c2 + 16 * hh;  // first query column of these 16, within this warpgroup's half
          // 16 queries whose bias offsets step by one, against a warp of such
          // keys: the 512 dS values fall on 47 bias rows, one per diagonal
          // (query - key); they are staged and summed per diagonal, so each
          // lane adds two sums instead of 16 values
          const int rq = rb[c0 + (lane & 15)];
          const bool diag_sum = want_db && keys_run && __all_sync(0xffffffffu, rq == rb[c0] + (lane & 15));
          uint32_t pk[8], dk8[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const int c = c0 + e;  // query column within this warpgroup's half
            const float2 l2 = *reinterpret_cast<const float2 *>(lse2 + c);
            const float2 d2 = *reinterpret_cast<const float2 *>(dl + c);
            const int2 r2 = *reinterpret_cast<const int2 *>(rb + c);
            const float b0 = has_bias ? bcol[r2.x - roff] : 0.f, b1 = has_bias ? bcol[r2.y - roff] : 0.f;
            const float p0 = ex2(fmaf(__uint_as_float(sv[e]), cs, b0) - l2.x);
            const float p1 = ex2(fmaf(__uint_as_float(sv[e + 1]), cs, b1) - l2.y);
            const float ds0 = p0 * (__uint_as_float(dv[e]) - d2.x), ds1 = p1 * (__uint_as_float(dv[e + 1]) - d2.y);
            if (diag_sum) {
              diag[lane * 17 + e] = ds0;
              diag[lane * 17 + e + 1] = ds1;
            } else if (want_db) {
              if (ds0 != 0.f) atomicAdd(bacc + (r2.x - roff), ds0);
              if (ds1 != 0.f) atomicAdd(bacc + (r2.y - roff), ds1);
            }
            pk[e >> 1] = pack_bf16(p0, p1);
            dk8[e >> 1] = pack_bf16(ds0, ds1);
          }
          if (diag_sum) {
            // lane t: diagonal t - 31 (queries i <= t, key i + 31 - t) and
            // diagonal t + 1 (queries i > t, key i - t - 1); one of the two per i
            __syncwarp();
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const bool lo = i <= lane;
              const float v = diag[(lo ? i + 31 - lane : i - lane - 1) * 17 + i];
              if (lo) sa += v;
              else sb += v;
            }
            const int base = rb[c0] - (roff - lane);  // bias row of query c0 against this warp's first key
            if (sa != 0.f) atomicAdd(bacc + base + lane - 31, sa);
            if (lane < 15 && sb != 0.f) atomicAdd(bacc + base + lane + 1, sb);
            __syncwarp();
          }
          tmem_st8(tmem + lane_addr + kColS + col + 16u * hh, pk);    // P^T over S^T
          tmem_st8(tmem + lane_addr + kColdP + col + 16u * hh, dk8);  // dS^T over dP^T
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(bar(bPFull));
    }
    if (ok && !__any_sync(0xffffffffu, *abort_flag != 0) && cur_h >= 0 && want_db && bsync()) flush();
    tmem_wait_st();
    tmem_wait_ld();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}
}  // namespace bkv

}  // namespace
}  // namespace lg

int large_bwd_max_bias_rows() { return lg::bq::kMaxBiasRows; }

int launch_bwd_large(const BwdArgs &a, void *stream) {
  if ((a.bias && a.g.T > lg::bq::kMaxBiasRows) || (a.ws && a.g.T > lg::bkv::kMaxBiasRows)) return SWIN_ERR_UNSUPPORTED;
  lg::TileMaps mq, mk, mv, mdo;
  if (!lg::tile_maps(&mq, a.q, a.g) || !lg::tile_maps(&mk, a.k, a.g) || !lg::tile_maps(&mv, a.v, a.g) ||
      !lg::tile_maps(&mdo, a.dout, a.g))
    return SWIN_ERR_CUDA;
  // two query stages in the key-tile kernel when neither the bias column nor
  // the dBias accumulator needs its shared memory
  const bool two = a.bias == nullptr && a.ws == nullptr;
  auto kv = two ? lg::bkv::bwdkv_kernel<2> : lg::bkv::bwdkv_kernel<1>;
  const int kv_smem = two ? lg::bkv::Lay<2>::kSmemBytes : lg::bkv::Lay<1>::kSmemBytes;
  if (cudaFuncSetAttribute(lg::bq::bwdq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lg::bq::kSmemBytes) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, kv_smem) != cudaSuccess)
    return SWIN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.o) {
    const int64_t toks = (int64_t)a.g.batch * a.g.tokens;
    lg::delta_kernel<<<(unsigned)((toks + 7) / 8), 256, 0, s>>>(a);
  }
  lg::bq::bwdq_kernel<<<a.ctas, lg::kThreads, lg::bq::kSmemBytes, s>>>(a, mq, mk, mv, mdo);
  kv<<<a.ctas, lg::kThreads, kv_smem, s>>>(a, mq, mk, mv, mdo);
  return cudaPeekAtLastError() == cudaSuccess ? SWIN_OK : SWIN_ERR_CUDA;
}

}  // namespace swin
