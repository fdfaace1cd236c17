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
// Work item = (head, image, window, pair of query tiles of 128 slots); the
// items are strided over the CTAs (CTA r takes r, r + ctas, ...), so the CTAs
// running together stream the same window's key/value tiles from L2. Both
// query tiles stay
// in shared memory and every key tile of the window, streamed through two
// stages, serves both (half the key/value loads per FLOP of one tile per item):
//  * warp 12 loads the two Q tiles (TMA gather4, two 64-channel halves each)
//    and writes their query mask rows; warps 13 and 8 load K (one channel
//    half each, by gather4 rows, or in windows of at least kRunMinKeyTiles
//    key tiles by boxes of runs of consecutive slots where a run lies in one
//    grid row; 13 also writes the key mask rows and, into a four-slot int16
//    ring, the key side of the bias offsets with the 16-key chunks whose
//    offsets step by one marked), warps 14 and 9 load V. A stage's key half
//    is released after the tile's last S, its value half after its last PV;
//  * warp 15 issues, per key tile, S_A and S_B = Q K^T + Qm Km^T (8 + 1 MMAs
//    each, N = 128) into one TMEM buffer per query tile and O_A, O_B += P V
//    (8 MMAs each), in the order PV_A, S_A of the next tile, PV_B, S_B of the
//    next tile, so that the two query tiles' chains interleave on the
//    tensor pipe;
//  * softmax warpgroup X (warps 4X .. 4X+3, thread = query row of tile X)
//    takes full rows of 128 keys: a first pass over S gives an upper bound of
//    the tile's row max (max S * scale*log2e + the head's largest bias); the
//    running max m is raised to it only when it exceeds m by more than 8 (a
//    factor 256), O (in TMEM) then rescaled, which is rare; the second pass
//    forms x = S*scale*log2e + bias*log2e (a marked chunk reads its 16 bias
//    values at fixed distances from one address), P = exp2(x - m) <= 256 in
//    bf16 over S and the running sum l. The final O / l uses the same m, so the
//    result is exact in real arithmetic. After the item's last key tile the
//    warpgroup itself stores O / l (and the log-sum-exp) at the query tokens.
// Masked keys (other region, land, pad) get -2^100 from the mask MMA and so
// exactly zero probability. Every wait is bounded, as in the small kernels.
#include <cuda_bf16.h>

#include "swin_large.cuh"

namespace swin {
namespace lg {
namespace {

constexpr int kStages = 2;  // key/value stages
constexpr int kQA = 0, kQB = kTileBytes, kQmA = 2 * kTileBytes, kQmB = kQmA + kMaskBytes;
constexpr int kStage0 = kQmB + kMaskBytes;  // 72 KB, 1024-aligned
constexpr int kK = 0, kV = kTileBytes, kKm = 2 * kTileBytes;  // inside a stage
constexpr int kStageBytes = 68 * 1024;
// key side of the bias offsets, int16 [kRoffSlots][128], a ring written with
// the key tiles: slot t mod 4 is rewritten with key tile t + 4, which cannot
// start before the softmax of tile t has finished (see the barriers below)
constexpr int kRoffSlots = 4;
// Key/value tiles load their runs of consecutive slots as boxes only in
// windows of at least this many key tiles. Measured with the strided item
// schedule: faster at 32-507 tiles (-8 % forward time at 32, -5 % at 128).
// Windows of 8 tiles (1 024 slots) gather every row; runs measured no faster
// there with contiguous item ranges.
constexpr int kRunMinKeyTiles = 32;
constexpr int kRoff = kStage0 + kStages * kStageBytes;
constexpr int kBcol = kRoff + kRoffSlots * 256;  // bias column of the current head (bias*log2e)
constexpr int kMaxBiasRows = 4096;
constexpr int kBmax = kBcol + kMaxBiasRows * 4;         // float [8]: per-warp maxima of the column
constexpr int kBarOff = kBmax + 64;
// per query tile X (0 = A, 1 = B): bSFull + X, bPFull + X, bPVDone + X
// stage s: bKFull/bKEmpty for its key tile (+ key mask rows), bVFull/bVEmpty
// for its value tile; the key half is released after the last S of the tile,
// the value half after the last PV
constexpr int bQFull = 0, bQFree = 1, bKFull = 2, bVFull = bKFull + kStages, bKEmpty = bVFull + kStages,
              bVEmpty = bKEmpty + kStages, bSFull = bVEmpty + kStages,
              bPFull = bSFull + 2, bPVDone = bPFull + 2, bNever = bPVDone + 2, bDrain = bNever + 1,
              bBsync = bDrain + 1, kNumBars = bBsync + 1;
constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem slot (u32), abort flag (int)
constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
static_assert(kStage0 % 1024 == 0 && kStageBytes % 1024 == 0 && kKm + kMaskBytes <= kStageBytes, "layout");
static_assert(kSmemBytes <= 232448, "over the 227 KB of shared memory a CTA may use");

// warps 0-7: softmax (warpgroup X = warp / 4 owns query tile X of the item);
// 12: Q; 13 and 8: K (channels 0-63, + key masks and bias offsets; 64-127);
// 14 and 9: V (the same halves); 15: MMA. Four warps issue the key/value row
// gathers: one warp's gather issue alone took longer than the item's MMAs.
constexpr int kSoftmaxWarps = 8, kQWarp = 12, kKWarp = 13, kVWarp = 14, kKWarp2 = 8, kVWarp2 = 9, kMmaWarp = 15;
constexpr int kThreads = 16 * 32;
// TMEM columns: S of query tile X at 128 X; O of query tile X at 256 + 128 X
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.f;  // raise the running max only past 2^8

// Item = (h, b, window, pair of query tiles 2p and 2p+1), pair fastest.
__device__ __forceinline__ LItem decode_pair(const Geo &g, int64_t it) {
  const int nqp = (g.nqt + 1) >> 1;
  LItem x;
  x.qt = 2 * (int)(it % nqp);
  int64_t t = it / nqp;
  x.omega = (int)(t % g.nwin);
  t /= g.nwin;
  x.b = (int)(t % g.batch);
  x.h = (int)(t / g.batch);
  return x;
}

// kRuns: key/value tiles load runs of slots as boxes (windows of at least
// kRunMinKeyTiles key tiles); otherwise every row by gather4.
template <bool kRuns>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_large_kernel(const FwdArgs a, const __grid_constant__ TileMaps tmq, const __grid_constant__ TileMaps tmk,
                     const __grid_constant__ TileMaps tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int idx) { return bars + 8u * idx; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMiscOff + 4);

  const Geo &g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkt = g.nqt;  // key tiles per window
  const Items its = strided_items(a.items, a.ctas);
  const int64_t count = its.count;
  const int64_t ntiles = count * nkt;  // key tiles this CTA streams, over all its items
  WaitCtl ctl{abort_flag, a.status, a.wait_limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(bQFull), 1);
    mbar_init(bar(bQFree), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(bKFull + s), 2);   // the two key gather warps
      mbar_init(bar(bVFull + s), 2);   // the two value gather warps
      mbar_init(bar(bKEmpty + s), 1);  // MMA commit after the tile's last S
      mbar_init(bar(bVEmpty + s), 1);  // MMA commit after the tile's last PV
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(bSFull + x), 1);
      mbar_init(bar(bPFull + x), 4);
      mbar_init(bar(bPVDone + x), 1);
    }
    mbar_init(bar(bNever), 1);
    mbar_init(bar(bDrain), 1);
    mbar_init(bar(bBsync), kSoftmaxWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // operand tiles start zeroed (rows past the window stay finite); the
  // constant halves of the mask rows: Qm columns 8-15 = 0, Km columns 8-15 =
  // -2^100
  for (int z = threadIdx.x; z < kRoff / 16; z += blockDim.x) reinterpret_cast<uint4 *>(smem)[z] = make_uint4(0u, 0u, 0u, 0u);
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
    // ----------------------------------------------------------- Q tiles ---
    for (int64_t it = 0; it < count; ++it) {
      const LItem x = decode_pair(g, its[it]);
      const bool has_b = x.qt + 1 < g.nqt;
      const Quad qa = route_quad(g, x.omega, x.qt, lane);
      const Quad qb = route_quad(g, x.omega, has_b ? x.qt + 1 : x.qt, lane);
      bool la[4], lb[4];
      quad_live(qa, a.land, (int64_t)x.b * g.tokens, la);
      quad_live(qb, a.land, (int64_t)x.b * g.tokens, lb);
      if (it > 0 && !mbar_wait_warp(bar(bQFree), (uint32_t)(it - 1) & 1u, ctl)) break;
      const int rows_a = min(128, g.n - x.qt * 128), nqa = (rows_a + 3) >> 2;
      const int rows_b = has_b ? min(128, g.n - (x.qt + 1) * 128) : 0, nqb = (rows_b + 3) >> 2;
      if (lane == 0) mbar_expect_tx(bar(bQFull), (uint32_t)(nqa + nqb) * 1024u);
      __syncwarp();
      // row gathers (measured faster here than tile boxes or runs, unlike in the backward)
      const Run rows_only{false, false, {0, 0, 0}};
      for (int hf = 0; hf < 2; ++hf)
        load_half(sbase + kQA + hf * kHalfBytes, &tmq, rows_only, qa, x.b, g.tokens, x.h, hf, lane, nqa, bar(bQFull));
      for (int hf = 0; has_b && hf < 2; ++hf)
        load_half(sbase + kQB + hf * kHalfBytes, &tmq, rows_only, qb, x.b, g.tokens, x.h, hf, lane, nqb, bar(bQFull));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        *reinterpret_cast<uint4 *>(smem + kQmA + sw32(4 * lane + j, 0)) = mask_chunk(la[j], qa.reg[j], false);
        *reinterpret_cast<uint4 *>(smem + kQmB + sw32(4 * lane + j, 0)) = mask_chunk(has_b && lb[j], qb.reg[j], false);
      }
      fence_proxy_async_smem();
      mbar_arrive_warp(bar(bQFull));
    }
  } else if (warp == kKWarp || warp == kVWarp || warp == kKWarp2 || warp == kVWarp2) {
    // -------------------------------------------------------- K, V tiles ---
    const bool kw = warp == kKWarp || warp == kKWarp2;
    const int half = (warp == kKWarp2 || warp == kVWarp2) ? 1 : 0;  // channel half this warp loads
    const int full_b = kw ? bKFull : bVFull, empty_b = kw ? bKEmpty : bVEmpty;
    int64_t t = 0;
    for (; t < ntiles; ++t) {
      const int s = (int)(t % kStages);
      const LItem x = decode_pair(g, its[t / nkt]);
      const int kt = (int)(t % nkt);
      const Quad q = route_quad(g, x.omega, kt, lane);
      const bool meta = warp == kKWarp;  // writes the key mask rows and bias offsets
      bool live[4];
      if (meta) quad_live(q, a.land, (int64_t)x.b * g.tokens, live);
      if (t >= kStages && !mbar_wait_warp(bar(empty_b + s), (uint32_t)((t / kStages) - 1) & 1u, ctl)) break;
      const uint32_t st = sbase + kStage0 + s * kStageBytes;
      uint8_t *sp = smem + kStage0 + s * kStageBytes;
      const int rows = min(128, g.n - kt * 128), nq4 = (rows + 3) >> 2;
      if (lane == 0) mbar_expect_tx(bar(full_b + s), (uint32_t)nq4 * 512u);
      __syncwarp();
      // this warp's channel half of the tile rows (pads read token 0): runs
      // along the grid's last dimension as boxes, other rows by gather4
      if constexpr (kRuns) {
        const Run run = find_run(g, q, lane);
        load_half(st + (kw ? kK : kV) + half * kHalfBytes, kw ? &tmk : &tmv, run, q, x.b, g.tokens, x.h, half, lane,
                  nq4, bar(full_b + s));
      } else if (lane < nq4) {
        const int r0 = x.b * g.tokens;
        tma_gather4(st + (kw ? kK : kV) + half * kHalfBytes + 512u * lane, kw ? &tmk.rows : &tmv.rows,
                    x.h * kHd + 64 * half, r0 + max(q.src[0], 0), r0 + max(q.src[1], 0), r0 + max(q.src[2], 0),
                    r0 + max(q.src[3], 0), bar(full_b + s));
      }
      if (meta) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4 *>(sp + kKm + sw32(4 * lane + j, 0)) = mask_chunk(live[j], q.reg[j], true);
        // key side of the bias offsets as negated byte offsets into the column.
        // A 16-key chunk (lanes 4c .. 4c+3) whose keys are all slots of the
        // window with offsets stepping by one is marked regular by bit 0 of its
        // first entry: the softmax then reads its 16 bias values at fixed
        // distances from one address.
        const bool lane_reg = kt * 128 + 4 * lane + 3 < g.n && q.roff[1] == q.roff[0] + 1 &&
                              q.roff[2] == q.roff[0] + 2 && q.roff[3] == q.roff[0] + 3;
        const int lead = __shfl_sync(0xffffffffu, q.roff[0], lane & ~3);
        const uint32_t bal = __ballot_sync(0xffffffffu, lane_reg && q.roff[0] == lead + 4 * (lane & 3));
        const int flag = (lane & 3) == 0 && ((bal >> (lane & ~3)) & 0xFu) == 0xFu ? 1 : 0;
        auto h16 = [](int v) { return (uint32_t)v & 0xFFFFu; };
        *reinterpret_cast<uint2 *>(smem + kRoff + (int)(t % kRoffSlots) * 256 + 8 * lane) =
            make_uint2(h16((-4 * q.roff[0]) | flag) | (h16(-4 * q.roff[1]) << 16),
                       h16(-4 * q.roff[2]) | (h16(-4 * q.roff[3]) << 16));
        fence_proxy_async_smem();
      }
      mbar_arrive_warp(bar(full_b + s));
    }
    // copies still in flight must land before the CTA exits
    volatile int no_abort = 0;
    const WaitCtl dctl{&no_abort, ctl.status, ctl.limit_ns < 50000000ull ? ctl.limit_ns : 50000000ull};
    for (int64_t k = t > kStages ? t - kStages : 0; k < t; ++k)
      mbar_wait_warp(bar(full_b + (int)(k % kStages)), (uint32_t)(k / kStages) & 1u, dctl);
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------- MMA ---
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0), idesc_pv = idesc_bf16(128, 128, 0, 1);
      uint32_t ns[2] = {0u, 0u};  // S of query tile X issued so far (the phase of its barriers)
      // S_X(t) = Q_X K^T + mask into S buffer X
      auto issue_s = [&](int xq, int64_t t) -> bool {
        const int s = (int)(t % kStages), kt = (int)(t % nkt);
        const int64_t it = t / nkt;
        if (xq == 0) {
          if (!mbar_wait(bar(bKFull + s), (uint32_t)(t / kStages) & 1u, ctl)) return false;
          if (kt == 0 && !mbar_wait(bar(bQFull), (uint32_t)it & 1u, ctl)) return false;
          tc_fence_after();
        }
        const uint32_t st = sbase + kStage0 + s * kStageBytes, d = tmem + 128u * xq;
        const uint32_t qt = sbase + (xq ? kQB : kQA), qm = sbase + (xq ? kQmB : kQmA);
        for (int kk = 0; kk < 8; ++kk) mma_ss(d, kmajor_desc(qt, kk), kmajor_desc(st + kK, kk), idesc_s, kk > 0 ? 1u : 0u);
        mma_ss(d, smem_desc(qm, 16, 256, kSwizzle32B), smem_desc(st + kKm, 16, 256, kSwizzle32B), idesc_s, 1);
        mma_commit(bar(bSFull + xq));
        ++ns[xq];
        return true;
      };
      // O_X += P_X V once P_X(t) is written
      auto issue_pv = [&](int xq, int64_t t, uint32_t n) -> bool {
        const int s = (int)(t % kStages), kt = (int)(t % nkt);
        if (!mbar_wait(bar(bPFull + xq), (n - 1) & 1u, ctl)) return false;
        if (xq == 0 && !mbar_wait(bar(bVFull + s), (uint32_t)(t / kStages) & 1u, ctl)) return false;
        tc_fence_after();
        const uint32_t st = sbase + kStage0 + s * kStageBytes;
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + kColO + 128u * xq, tmem + 128u * xq + 16u * kk, nmajor_desc(st + kV, 16 * kk), idesc_pv,
                 (kt > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(bPVDone + xq));
        return true;
      };
      bool ok = true;
      for (int64_t t = 0; ok && t < ntiles; ++t) {
        const int kt = (int)(t % nkt);
        const LItem x = decode_pair(g, its[t / nkt]);
        const bool has_b = x.qt + 1 < g.nqt;
        if (kt == 0) {  // the item's first S's (its Q tiles came in after the previous item's last S's)
          ok = issue_s(0, t) && (!has_b || issue_s(1, t));
          if (!ok) break;
          mma_commit(bar(bKEmpty + (int)(t % kStages)));
          if (kt == nkt - 1) mma_commit(bar(bQFree));
        }
        // PV_A(t), S_A(t+1), PV_B(t), S_B(t+1): S of the next tile of the same item
        // is issued as soon as its query tile's P of this tile has been read
        const bool next = kt + 1 < nkt;
        ok = issue_pv(0, t, ns[0]) && (!next || issue_s(0, t + 1));
        if (ok && has_b) ok = issue_pv(1, t, ns[1]);
        if (!ok) break;
        mma_commit(bar(bVEmpty + (int)(t % kStages)));
        if (next) {
          if (has_b && !issue_s(1, t + 1)) break;
          mma_commit(bar(bKEmpty + (int)((t + 1) % kStages)));
          if (kt + 1 == nkt - 1) mma_commit(bar(bQFree));  // the item's last reads of its Q tiles
        }
      }
      mma_commit(bar(bDrain));
      volatile int no_abort = 0;
      WaitCtl drain_ctl{&no_abort, a.status, a.wait_limit_ns};
      mbar_wait(bar(bDrain), 0, drain_ctl);
    }
    __syncwarp();
  } else if (warp < kSoftmaxWarps) {
    // ----------------------------------------------------------- softmax ---
    const int xq = warp >> 2, q4 = warp & 3, i = q4 * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_addr + 128u * xq, tO = tmem + lane_addr + kColO + 128u * xq;
    float *bcol = reinterpret_cast<float *>(smem + kBcol);
    const uint32_t bcol_u32 = sbase + kBcol;
    float *bmx = reinterpret_cast<float *>(smem + kBmax);
    const float cs = a.scale * kLog2e;
    const bool has_bias = a.bias != nullptr;
    int cur_h = -1, rbase = 0, src = -1;
    bool live = false, mine = false;
    float bmax2 = 0.f, m_run = -INFINITY, l_run = 0.f;
    uint32_t bs_phase = 0, nt = 0;  // key tiles of this warpgroup's query tiles so far (barrier phases)
    bool ok = true;
    auto bsync = [&]() -> bool {
      mbar_arrive_warp(bar(bBsync));
      const bool r = mbar_wait_warp(bar(bBsync), bs_phase & 1u, ctl);
      ++bs_phase;
      return r;
    };
    if (a.debug_force_timeout && xq == 0) ok = mbar_wait_warp(bar(bNever), 0, ctl);
    for (int64_t t = 0; ok && t < ntiles; ++t) {
      const int kt = (int)(t % nkt);
      const LItem x = decode_pair(g, its[t / nkt]);
      if (kt == 0) {
        if (has_bias && x.h != cur_h) {
          // the head's bias column (bias * log2e) and its largest value
          if (cur_h >= 0 && !bsync()) break;
          float mx = -INFINITY;
          for (int r = xq * 128 + i; r < g.T; r += 256) {
            const float b = __ldg(a.bias + (int64_t)r * g.heads + x.h) * kLog2e;
            bcol[r] = b;
            mx = fmaxf(mx, b);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (lane == 0) bmx[warp] = mx;
          if (!bsync()) break;
          bmax2 = bmx[0];
#pragma unroll
          for (int w = 1; w < 8; ++w) bmax2 = fmaxf(bmax2, bmx[w]);
          cur_h = x.h;
        }
        const int qt = x.qt + xq;
        mine = qt < g.nqt;  // warpgroup B has no tile in the last pair of an odd tile count
        const int slot = qt * 128 + i;
        int wc[3];
        window_coords(g, x.omega, wc);
        const SlotRoute r = slot_route(g, wc, mine && slot < g.n ? slot : 0);
        src = mine && slot < g.n ? r.src : -1;
        rbase = mine && slot < g.n ? r.rbase : g.T - 1;
        live = src >= 0 && (!a.land || __ldg(a.land + (int64_t)x.b * g.tokens + src) == 0);
        m_run = -INFINITY;
        l_run = 0.f;
      }
      if (!mine) continue;
      if (!mbar_wait_warp(bar(bSFull + xq), nt & 1u, ctl)) break;
      tc_fence_after();
      const int16_t *roff = reinterpret_cast<const int16_t *>(smem + kRoff + (int)(t % kRoffSlots) * 256);
      // pass 1: an upper bound of the tile's row max from S alone
      float ms = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t sv[4][16];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) tmem_ld16(tS + 64u * c + 16u * k4, sv[k4]);
        tmem_wait_ld_tied(sv[0], sv[1]);
        tmem_wait_ld_tied(sv[2], sv[3]);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
#pragma unroll
          for (int e = 0; e < 16; e += 2)
            ms = max3(ms, __uint_as_float(sv[k4][e]), __uint_as_float(sv[k4][e + 1]));
      }
      // keys all masked for this row (about -2^100 after the mask step): no contribution
      const bool any = ms > -1e29f;
      const float mt = ms * cs + bmax2;
      float m_new = m_run;
      if (any && (l_run == 0.f || mt > m_run + kRescaleLog2)) m_new = mt;
      const bool rescale = any && l_run > 0.f && m_new != m_run;
      if (__any_sync(0xffffffffu, rescale)) {
        // O of this row is scaled by exp2(m_run - m_new) once the PV of the
        // previous tile has completed
        if (!mbar_wait_warp(bar(bPVDone + xq), (nt - 1) & 1u, ctl)) break;
        tc_fence_after();
        const float f = rescale ? ex2(m_run - m_new) : 1.f;
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
      // pass 2: x = S*cs + bias2, P = exp2(x - m) over S, row sum
      const float msub = any ? m_run : 0.f;
      float2 sp2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t sv[4][16];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) tmem_ld16(tS + 64u * c + 16u * k4, sv[k4]);
        tmem_wait_ld_tied(sv[0], sv[1]);
        tmem_wait_ld_tied(sv[2], sv[3]);
        // x - m = S*cs + (bias2 - m) for the 64 keys, in place: the shared-memory
        // bias reads run back to back (no TMEM store between them)
        const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(-msub, -msub);
        if (has_bias) {
          const uint32_t brow = bcol_u32 + 4u * (uint32_t)rbase;  // this row's end of the column
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int v = roff[64 * c + 16 * k4];  // the same entry for every lane
            if (v & 1) {
              // regular chunk: key e's value sits 4e bytes below the first key's
              float bv[16];
              lds_f32_desc16(brow + (uint32_t)(v - 1) - 60u, bv);
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                const float2 x = __fadd2_rn(
                    __ffma2_rn(make_float2(__uint_as_float(sv[k4][e]), __uint_as_float(sv[k4][e + 1])), cs2,
                               make_float2(bv[e], bv[e + 1])),
                    nm2);
                sv[k4][e] = __float_as_uint(x.x);
                sv[k4][e + 1] = __float_as_uint(x.y);
              }
              continue;
            }
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
              const uint2 w = *reinterpret_cast<const uint2 *>(roff + 64 * c + 16 * k4 + e);
              const int4 r4 = make_int4((int)(int16_t)(w.x & 0xFFFFu), (int)w.x >> 16, (int)(int16_t)(w.y & 0xFFFFu),
                                        (int)w.y >> 16);
              const float2 b01 = make_float2(lds_f32(brow + r4.x), lds_f32(brow + r4.y));
              const float2 b23 = make_float2(lds_f32(brow + r4.z), lds_f32(brow + r4.w));
              const float2 x0 = __fadd2_rn(
                  __ffma2_rn(make_float2(__uint_as_float(sv[k4][e]), __uint_as_float(sv[k4][e + 1])), cs2, b01), nm2);
              const float2 x1 = __fadd2_rn(
                  __ffma2_rn(make_float2(__uint_as_float(sv[k4][e + 2]), __uint_as_float(sv[k4][e + 3])), cs2, b23),
                  nm2);
              sv[k4][e] = __float_as_uint(x0.x);
              sv[k4][e + 1] = __float_as_uint(x0.y);
              sv[k4][e + 2] = __float_as_uint(x1.x);
              sv[k4][e + 3] = __float_as_uint(x1.y);
            }
          }
        } else {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const float2 x =
                  __ffma2_rn(make_float2(__uint_as_float(sv[k4][e]), __uint_as_float(sv[k4][e + 1])), cs2, nm2);
              sv[k4][e] = __float_as_uint(x.x);
              sv[k4][e + 1] = __float_as_uint(x.y);
            }
          }
        }
        // P = exp2(x - m) in bf16 over S, row sum
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          uint32_t pv[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float2 p = any ? make_float2(ex2(__uint_as_float(sv[k4][e])), ex2(__uint_as_float(sv[k4][e + 1])))
                                 : make_float2(0.f, 0.f);
            sp2[(e >> 1) & 1] = __fadd2_rn(sp2[(e >> 1) & 1], p);
            pv[e >> 1] = pack_bf16(p.x, p.y);
          }
          tmem_st8(tS + 64u * c + 16u * k4, pv);
        }
      }
      const float2 sum2 = __fadd2_rn(sp2[0], sp2[1]);
      l_run += sum2.x + sum2.y;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(bar(bPFull + xq));
      ++nt;
      if (kt == nkt - 1) {
        // epilogue of the item: O / l at the query tokens, the log-sum-exp
        if (!mbar_wait_warp(bar(bPVDone + xq), (nt - 1) & 1u, ctl)) break;
        tc_fence_after();
        const float inv = live && l_run > 0.f ? __frcp_rn(l_run) : 0.f;
        const bool store = src >= 0 && in_bounds(((int64_t)x.b * g.tokens + src) * g.C + (int64_t)x.h * kHd, kHd,
                                                  (int64_t)g.batch * g.tokens * g.C, a.status);
        uint4 *dst = store ? reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.o) +
                                                       ((int64_t)x.b * g.tokens + src) * g.C + (int64_t)x.h * kHd)
                           : nullptr;
#pragma unroll 1
        for (int c = 0; c < 8; c += 2) {
          uint32_t o0[16], o1[16];
          tmem_ld16(tO + 16u * c, o0);
          tmem_ld16(tO + 16u * (c + 1), o1);
          tmem_wait_ld_tied(o0, o1);
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            w[e >> 1] = pack_bf16(__uint_as_float(o0[e]) * inv, __uint_as_float(o0[e + 1]) * inv);
            w[8 + (e >> 1)] = pack_bf16(__uint_as_float(o1[e]) * inv, __uint_as_float(o1[e + 1]) * inv);
          }
          if (store) {
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[2 * c + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
        if (store && a.lse)
          a.lse[((int64_t)x.b * g.heads + x.h) * g.tokens + src] = live ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
      }
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
int64_t large_fwd_items(const Geo &g) { return (int64_t)g.heads * g.batch * g.nwin * ((g.nqt + 1) / 2); }

int launch_fwd_large(const FwdArgs &a, void *stream) {
  if (a.bias && a.g.T > lg::kMaxBiasRows) return SWIN_ERR_UNSUPPORTED;
  lg::TileMaps mq, mk, mv;
  if (!lg::tile_maps(&mq, a.q, a.g) || !lg::tile_maps(&mk, a.k, a.g) || !lg::tile_maps(&mv, a.v, a.g))
    return SWIN_ERR_CUDA;
  auto kern = a.g.nqt >= lg::kRunMinKeyTiles ? lg::fwd_large_kernel<true> : lg::fwd_large_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lg::kSmemBytes) !=
      cudaSuccess)
    return SWIN_ERR_CUDA;
  kern<<<a.ctas, lg::kThreads, lg::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(a, mq, mk, mv);
  return cudaPeekAtLastError() == cudaSuccess ? SWIN_OK : SWIN_ERR_CUDA;
}

}  // namespace swin
