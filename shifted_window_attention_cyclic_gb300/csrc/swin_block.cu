// swin_block.cu -- the attention half of a Swin block in one kernel (sm_103a):
// LayerNorm and the QKV projection as its prologue, shifted-window attention
// per head, the out-projection and the residual add as its epilogue (TERRA,
// Fig. 4: "Layernorm", "Window Attention"; Sec. III: W-MSA / SW-MSA blocks).
// For bf16, head_dim 32, windows of up to 128 slots and C = heads * 32 a
// multiple of 64 up to 256. Q, K, V and O never leave the SM: per window only
// X is read (twice: for the LayerNorm and, from L2, for the residual) and Y
// written.
//
// One CTA per SM takes a contiguous range of windows (TERRA Eq. (4)), in the
// plan's spread order; per window, all 256 threads run the phases in order:
//  * route: slot -> grid token (cyclic shift, ragged edge, pads), region and
//    land -> the K = 16 mask rows Qm / Km (one extra MMA step adds -2^100 to
//    every masked logit, as in the attention kernels), key side of the bias
//    offsets;
//  * LayerNorm: X of a window that is a box of the grid arrives as 5-D TMA
//    boxes straight into the tile, other windows' rows by 16-byte loads; two
//    threads per row, mean and biased variance in fp32 from registers, Xn =
//    (x - mean) * rstd * gamma + beta in bf16 into a 128-byte-swizzled
//    K-major tile (in place);
//  * per head h: [Q|K|V]_h = Xn W_qkv,h^T (tcgen05, N = 96, fp32 in TMEM),
//    + b_qkv, to bf16 tiles; S = Q K^T + mask; softmax over the slot's keys
//    by both warpgroups (keys 0-63 and 64-127, each its own max, sum and PV
//    accumulator) with the head's bias column (x = S*scale*log2e +
//    bias*log2e, P = exp2(x - max) in bf16 over S); O = P V (A from TMEM);
//    O / l (0 for dead queries) to a bf16 tile; Y += O W_o,h^T (N = C,
//    accumulated over the heads in TMEM). The next head's W_qkv rows are
//    fetched by one 4-D TMA copy while this head's attention runs; W_o's
//    columns once the previous head's out-projection has completed.
//  * epilogue: Y + b_o + X at the slot's token, in bf16 (pads write nothing);
//    for box windows X is reloaded into the tile during the last head and y
//    leaves as TMA box stores.
// Every wait is bounded; on timeout all threads leave together (the result
// of the wait is agreed with a CTA-wide AND), drain the copies and MMAs in
// flight, free TMEM, and the status word reports the timeout.
#include <cuda_bf16.h>

#include "swin_large.cuh"

namespace swin {
namespace blk {
namespace {

using namespace ptx;
using lg::kBf16NegBig;
using lg::kLog2e;
using lg::mask_chunk;
using lg::sw32;

constexpr int kThreads = 256;
constexpr int kHdB = 32;       // head_dim
constexpr int kMaxC = 256;     // channels
constexpr int kMaxBias = 8192;  // floats of the staged bias columns (heads x rows)

// shared memory (bytes from a 1024-aligned base)
constexpr int kXn = 0;                        // bf16 [C/64][128][64] SW128: LayerNorm(X)
constexpr int kWqkv = kXn + 4 * 16384;        // bf16 [C/64][96][64] SW128: rows of W_qkv for head h
constexpr int kWo = kWqkv + 4 * 12288;        // bf16 [C][32] SW64: columns h*32.. of W_o
constexpr int kQ = kWo + kMaxC * 64;          // bf16 [128][32] SW64 each
constexpr int kK = kQ + 8192, kV = kK + 8192, kO = kV + 8192;
constexpr int kQm = kO + 8192, kKm = kQm + 4096;  // [128][16] SW32
constexpr int kBcol = kKm + 4096;             // float [heads][T]: bias * log2e
constexpr int kRoff = kBcol + kMaxBias * 4;   // int [128]: key side of the bias offsets, as -4 * offset (bytes)
constexpr int kSrc = kRoff + 512;             // int [128]: source token of each slot, -1 for pads
constexpr int kRb = kSrc + 512;               // int [128]: query side of the bias offsets
constexpr int kXch = kRb + 512;               // float [2][128]: second warpgroup's row max and sum
constexpr int kPar = kXch + 1024;             // float gamma[256], beta[256], b_o[256], b_qkv[768]
constexpr int kBarOff = kPar + (3 * kMaxC + 3 * kMaxC) * 4;
constexpr int bW = 0, bWo = 1, bQKV = 2, bS = 3, bO = 4, bY = 5, bDrain = 6, bX = 7, bNever = 8, kNumBars = 9;
constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem slot, abort flag
constexpr int kSmemBytes = kMiscOff + 16 + 1024;
static_assert(kSmemBytes <= 232448, "over the 227 KB of shared memory a CTA may use");
static_assert(kWqkv % 1024 == 0 && kWo % 1024 == 0 && kQ % 1024 == 0 && kQm % 1024 == 0, "layout");

// TMEM columns: QKV (96) at 0, O (32) at 96, S (128) at 128, Y (C) at 256;
// the second key half's O at 64 (the V columns, read before the PV product)
constexpr uint32_t kColQKV = 0, kColO1 = 64, kColO = 96, kColS = 128, kColY = 256;

// 16-byte chunk c of row r in a 64-byte-row tile with 64-byte swizzle
__device__ __forceinline__ uint32_t sw64(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }
// 16-byte chunk c of row r in a 128-byte-row tile with 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// TMA box store of shared memory into a 5-D tensor map (bulk group), and the
// bulk-group waits (.read: the source may be overwritten; plain: complete)
__device__ __forceinline__ void tma_store_5d(const void *tmap, uint32_t src, int c0, int c1, int c2, int c3, int c4) {
  asm volatile("cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(tmap),
               "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__global__ void __launch_bounds__(kThreads, 1)
    block_kernel(const BlockArgs a, const __grid_constant__ CUtensorMap wqkv_map,
                 const __grid_constant__ CUtensorMap wo_map, const __grid_constant__ CUtensorMap x_map,
                 const __grid_constant__ CUtensorMap y_map) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  auto bar = [&](int idx) { return bars + 8u * idx; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMiscOff + 4);
  const Geo &g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = g.C, H = g.heads, nkb = C >> 6;
  int64_t L, R;
  eq4_range(a.items, a.ctas, blockIdx.x, L, R);
  const int64_t count = R - L, total_heads = count * H;
  WaitCtl ctl{abort_flag, a.status, a.wait_limit_ns};
  float *bcol = reinterpret_cast<float *>(smem + kBcol);
  int *roff = reinterpret_cast<int *>(smem + kRoff);
  int *srcs = reinterpret_cast<int *>(smem + kSrc);
  int *rbs = reinterpret_cast<int *>(smem + kRb);
  float *xch = reinterpret_cast<float *>(smem + kXch);
  float *gam = reinterpret_cast<float *>(smem + kPar), *bet = gam + kMaxC, *bo = bet + kMaxC, *bqkv = bo + kMaxC;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // parameters and every head's bias column, once per CTA
  for (int c = tid; c < C; c += kThreads) {
    gam[c] = __ldg(a.gamma + c);
    bet[c] = __ldg(a.beta + c);
    bo[c] = __ldg(a.b_o + c);
  }
  for (int c = tid; c < 3 * C; c += kThreads) bqkv[c] = __ldg(a.b_qkv + c);
  for (int z = tid; z < H * g.T; z += kThreads) {
    const int h = z / g.T, r = z % g.T;
    bcol[z] = a.bias ? __ldg(a.bias + (int64_t)r * H + h) * kLog2e : 0.f;
  }
  // constant halves of the mask rows: Qm columns 8-15 = 0, Km columns 8-15 = -2^100
  if (tid < 128) {
    const uint32_t nb2 = (uint32_t)kBf16NegBig | ((uint32_t)kBf16NegBig << 16);
    *reinterpret_cast<uint4 *>(smem + kQm + sw32(tid, 1)) = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(smem + kKm + sw32(tid, 1)) = make_uint4(nb2, nb2, nb2, nb2);
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), lg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // weights of head h: W_qkv rows {q, k, v} x (h*32 .. h*32+31), all C columns
  // (C/64 blocks of 64), and W_o columns h*32 .. h*32+31 (all C rows)
  uint32_t n_wqkv = 0, n_wo = 0;  // copies issued (thread 0): the drain waits for the last of each
  auto load_wqkv = [&](int h) {
    ++n_wqkv;
    // one copy: (64 channels) x (32 rows of head h) x (q, k, v) x (C/64 channel
    // blocks), landing as [block][q|k|v][row][64 channels], the MMA's B layout
    mbar_expect_tx(bar(bW), (uint32_t)(3 * nkb * 4096));
    tma_load_4d(sbase + kWqkv, &wqkv_map, 0, h * kHdB, 0, 0, bar(bW));
    mbar_arrive(bar(bW));  // the phase completes once this arrival and the bytes are in
  };
  auto load_wo = [&](int h) {
    ++n_wo;
    mbar_expect_tx(bar(bWo), (uint32_t)(C * 64));
    tma_load_2d(sbase + kWo, &wo_map, h * kHdB, 0, bar(bWo));
    mbar_arrive(bar(bWo));
  };
  // a window that neither wraps nor pads is a box of the grid: X arrives, and
  // y leaves, as one 5-D TMA box per 64-channel block (the Xn tile's layout)
  auto window_box = [&](int omega, int (&c)[3]) -> bool {
    int wc[3];
    window_coords(g, omega, wc);
    bool box = true;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
      c[d] = wc[d] * g.w[d] + g.s[d];
      box = box && c[d] + g.w[d] <= g.G[d];
    }
    return box;
  };
  uint32_t n_x = 0;  // X box loads issued (thread 0; every thread counts the waits alike)
  auto load_x = [&](const int (&c)[3], int b) {
    ++n_x;
    mbar_expect_tx(bar(bX), (uint32_t)(nkb * g.n * 128));
    for (int kb = 0; kb < nkb; ++kb)
      tma_load_5d(sbase + kXn + kb * 16384, &x_map, kb * 64, c[2], c[1], c[0], b, bar(bX));
    mbar_arrive(bar(bX));
  };
  // every thread waits (bounded), then the CTA agrees on the outcome
  auto cta_wait = [&](int b, uint32_t parity, bool ok) -> bool {
    if (ok) ok = mbar_wait(bar(b), parity, ctl);
    return __syncthreads_and(ok) != 0;
  };

  const float cs = a.scale * kLog2e;
  const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
  const int row = (warp & 3) * 32 + lane;  // TMEM lane = slot of this thread in the TMEM phases
  const uint32_t idesc_qkv = idesc_bf16(128, 96, 0, 0), idesc_pv = idesc_bf16(128, 32, 0, 1),
                 idesc_y = idesc_bf16(128, (uint32_t)C, 0, 0);
  const int ng = (g.n + 15) >> 4;  // 16-key groups of S
  const uint32_t idesc_s = idesc_bf16(128, (uint32_t)(16 * ng), 0, 0);
  uint32_t hc = 0;  // heads done in this CTA (phase of every per-head barrier)
  uint32_t xph = 0;  // X box loads waited for so far (phase of bX)
  bool ok = true;
  if (tid == 0 && total_heads > 0) {
    load_wqkv(0);
    load_wo(0);
  }

  // testing hook: the bounded wait runs out on a barrier nothing arrives at
  if (a.debug_force_timeout) ok = cta_wait(bNever, 0, true);
  for (int64_t it = 0; ok && it < count; ++it) {
    const int64_t item = L + it;
    // windows in the plan's spread order (the i-th is (i * wstep) mod nwin):
    // wrapping and padded windows (row loads) fall evenly over the CTAs
    const int omega = (int)(((item % g.nwin) * (int64_t)g.wstep) % g.nwin), b = (int)(item / g.nwin);
    int bc[3];
    const bool box = window_box(omega, bc);
    if (tid == 0) {
      // the previous window's y stores have read the region (before this
      // window's X box or LayerNorm writes it; the route's barrier orders
      // the other threads' writes after this wait)
      bulk_wait_read0();
      if (box) load_x(bc, b);
    }
    // ------------------------------------------------------------- route ---
    int rbase = g.T - 1, src = -1;
    bool live = false;
    if (tid < 128) {
      int reg = 0, ro = 0;
      if (tid < g.n) {
        int wc[3];
        window_coords(g, omega, wc);
        const SlotRoute r = slot_route(g, wc, tid);
        src = r.src;
        reg = r.reg;
        rbase = r.rbase;
        ro = r.roff;
        live = src >= 0 && (!a.land || __ldg(a.land + (int64_t)b * g.tokens + src) == 0);
      }
      srcs[tid] = src;
      roff[tid] = -4 * ro;  // negated byte offset into a bias column
      rbs[tid] = rbase;
      *reinterpret_cast<uint4 *>(smem + kQm + sw32(tid, 0)) = mask_chunk(live, reg, false);
      *reinterpret_cast<uint4 *>(smem + kKm + sw32(tid, 0)) = mask_chunk(live, reg, true);
    }
    __syncthreads();
    if (box) {
      ok = cta_wait(bX, xph & 1u, true);
      ++xph;
      if (!ok) break;
    }
    // --------------------------------------------------------- LayerNorm ---
    {
      const int r = tid >> 1, half = tid & 1, cw = C >> 1;  // this thread: channels [half*cw, half*cw + cw)
      const int s = srcs[r];
      uint4 xv[16];
      const uint4 *xp = s >= 0 ? reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.x) +
                                                                 ((int64_t)b * g.tokens + s) * C + half * cw)
                               : nullptr;
      float sum = 0.f;
      // a box window's rows are already in the tile (read in place), others
      // come from L2/HBM
      if (box) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c0 = half * cw + 8 * j;
          xv[j] = (s >= 0 && 8 * j < cw)
                      ? *reinterpret_cast<const uint4 *>(smem + kXn + (c0 >> 6) * 16384 + sw128(r, (c0 & 63) >> 3))
                      : make_uint4(0u, 0u, 0u, 0u);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) xv[j] = (xp && 8 * j < cw) ? __ldg(xp + j) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        sum += bf_lo(xv[j].x) + bf_hi(xv[j].x) + bf_lo(xv[j].y) + bf_hi(xv[j].y) + bf_lo(xv[j].z) +
               bf_hi(xv[j].z) + bf_lo(xv[j].w) + bf_hi(xv[j].w);
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      const float mean = sum / (float)C;
      float sq = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (8 * j < cw) {
          const uint32_t w4[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float d0 = bf_lo(w4[e]) - mean, d1 = bf_hi(w4[e]) - mean;
            sq = fmaf(d0, d0, fmaf(d1, d1, sq));
          }
        }
      }
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      const float rstd = rsqrtf(sq / (float)C + a.eps);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (8 * j < cw) {
          const int c0 = half * cw + 8 * j;  // first channel of this 16-byte chunk
          const uint32_t w4[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
          uint32_t o4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = c0 + 2 * e;
            const float y0 = (bf_lo(w4[e]) - mean) * rstd * gam[c] + bet[c];
            const float y1 = (bf_hi(w4[e]) - mean) * rstd * gam[c + 1] + bet[c + 1];
            o4[e] = s >= 0 ? pack_bf16(y0, y1) : 0u;
          }
          *reinterpret_cast<uint4 *>(smem + kXn + (c0 >> 6) * 16384 + sw128(r, (c0 & 63) >> 3)) =
              make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    float m_own = 0.f, l_own = 0.f;  // this warpgroup's row max and sum over its key half
    bool any_own = false;
    for (int h = 0; h < H; ++h, ++hc) {
      const uint32_t ph = hc & 1u;
      // ---------------------------------------------- QKV_h = Xn W_qkv,h^T ---
      bool ok0 = true;
      if (tid == 0) {
        ok0 = mbar_wait(bar(bW), ph, ctl);
        if (ok0) {
          tc_fence_after();
          for (int kk = 0; kk < 4 * nkb; ++kk)
            mma_ss(tmem + kColQKV,
                   smem_desc(sbase + kXn + (kk >> 2) * 16384 + 32u * (kk & 3), 16, 1024, kSwizzle128B),
                   smem_desc(sbase + kWqkv + (kk >> 2) * 12288 + 32u * (kk & 3), 16, 1024, kSwizzle128B),
                   idesc_qkv, kk > 0 ? 1u : 0u);
          mma_commit(bar(bQKV));
          // W_o's columns of this head once the previous out-projection has read W_o
          if (hc > 0) {
            ok0 = mbar_wait(bar(bY), (hc - 1) & 1u, ctl);
            if (ok0) load_wo(h);
          }
        }
      }
      ok = cta_wait(bQKV, ph, ok0);
      if (!ok) break;
      tc_fence_after();
      // the next head's W_qkv rows (this head's product has read them)
      if (tid == 0 && (int64_t)hc + 1 < total_heads) load_wqkv(h + 1 < H ? h + 1 : 0);
      // the window's last QKV product has read Xn: X comes back into the
      // region for the epilogue's residual
      if (tid == 0 && box && h == H - 1) load_x(bc, b);
      // -------------------------------------- + b_qkv, bf16 Q / K / V tiles ---
      {
        const int part = warp < 4 ? 0 : 2;  // warps 0-3: Q then K; warps 4-7: V
        for (int p = part; p < (warp < 4 ? 2 : 3); ++p) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tmem + lane_addr + kColQKV + 32u * p, v0);
          tmem_ld16(tmem + lane_addr + kColQKV + 32u * p + 16u, v1);
          tmem_wait_ld_tied(v0, v1);
          const float *bb = bqkv + p * C + h * kHdB;
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            w[e >> 1] = pack_bf16(__uint_as_float(v0[e]) + bb[e], __uint_as_float(v0[e + 1]) + bb[e + 1]);
            w[8 + (e >> 1)] =
                pack_bf16(__uint_as_float(v1[e]) + bb[16 + e], __uint_as_float(v1[e + 1]) + bb[16 + e + 1]);
          }
          uint8_t *tile = smem + (p == 0 ? kQ : p == 1 ? kK : kV);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4 *>(tile + sw64(row, q)) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      // ------------------------------------------------------ S = Q K^T + mask ---
      if (tid == 0) {
        tc_fence_after();
        mma_ss(tmem + kColS, smem_desc(sbase + kQ, 16, 512, kSwizzle64B), smem_desc(sbase + kK, 16, 512, kSwizzle64B),
               idesc_s, 0u);
        mma_ss(tmem + kColS, smem_desc(sbase + kQ + 32, 16, 512, kSwizzle64B),
               smem_desc(sbase + kK + 32, 16, 512, kSwizzle64B), idesc_s, 1u);
        mma_ss(tmem + kColS, smem_desc(sbase + kQm, 16, 256, kSwizzle32B),
               smem_desc(sbase + kKm, 16, 256, kSwizzle32B), idesc_s, 1u);
        mma_commit(bar(bS));
      }
      ok = cta_wait(bS, ph, true);
      if (!ok) break;
      tc_fence_after();
      // ------------------------------------------------------------ softmax ---
      // warpgroup grp takes keys [64 grp, 64 grp + 64) of every row: its own
      // max m, P = exp2(x - m) in bf16 over its S columns and its sum l; the
      // O epilogue puts the two halves on one scale
      {
        const int grp = warp >> 2, kb0 = 4 * grp, nk = min(ng - kb0, 4);
        any_own = false;
        m_own = 0.f;
        l_own = 0.f;
        if (nk > 0) {
          uint32_t sv[4][16];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (k < nk) tmem_ld16(tmem + lane_addr + kColS + 16u * (kb0 + k), sv[k]);
          tmem_wait_ld_tied(sv[0], sv[1]);
          tmem_tie(sv[2], sv[3]);
          // the row's end of the head's bias column; keys step back by their offsets
          const uint32_t brow = sbase + kBcol + 4u * (uint32_t)(h * g.T + rbs[row]);
          const int *ro = roff + 16 * kb0;
          float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (k < nk) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float x = fmaf(__uint_as_float(sv[k][e]), cs, lds_f32(brow + (uint32_t)ro[16 * k + e]));
                sv[k][e] = __float_as_uint(x);
                mq[e & 3] = fmaxf(mq[e & 3], x);
              }
            }
          }
          const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
          // keys all masked in this half (about -2^100 after the mask step): no weight
          any_own = mx > -1e29f;
          m_own = any_own ? mx : 0.f;
          float lq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (k < nk) {
              uint32_t pv[8];
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                const float p0 = any_own ? ex2(__uint_as_float(sv[k][e]) - m_own) : 0.f;
                const float p1 = any_own ? ex2(__uint_as_float(sv[k][e + 1]) - m_own) : 0.f;
                lq[(e >> 1) & 3] += p0 + p1;
                pv[e >> 1] = pack_bf16(p0, p1);
              }
              tmem_st8(tmem + lane_addr + kColS + 16u * (kb0 + k), pv);
            }
          }
          l_own = (lq[0] + lq[1]) + (lq[2] + lq[3]);
          tmem_wait_st();
        }
        if (grp == 1) {
          xch[row] = any_own ? m_own : -INFINITY;
          xch[128 + row] = l_own;
        }
      }
      tc_fence_before();
      __syncthreads();
      // ---------------------------------------------------------- O = P V ---
      // keys 0-63 into O (columns 96..127), keys 64-127 into O1 (64..95)
      if (tid == 0) {
        tc_fence_after();
        for (int kk = 0; kk < ng; ++kk)
          mma_ts(tmem + (kk < 4 ? kColO : kColO1), tmem + kColS + 16u * kk,
                 smem_desc(sbase + kV + 1024u * kk, 8192, 512, kSwizzle64B), idesc_pv, (kk & 3) ? 1u : 0u);
        mma_commit(bar(bO));
      }
      ok = cta_wait(bO, ph, true);
      if (!ok) break;
      tc_fence_after();
      // ------------------------------------------------- O / l -> bf16 tile ---
      if (warp < 4) {
        const float m1 = xch[row], l1 = xch[128 + row];
        const bool any1 = ng > 4 && m1 != -INFINITY;
        const float m = any_own ? (any1 ? fmaxf(m_own, m1) : m_own) : (any1 ? m1 : 0.f);
        const float s0 = any_own ? ex2(m_own - m) : 0.f, s1 = any1 ? ex2(m1 - m) : 0.f;
        const float lsum = l_own * s0 + l1 * s1;
        const float inv = live && lsum > 0.f ? 1.f / lsum : 0.f;
        const float a0 = s0 * inv, a1 = s1 * inv;
        uint32_t o0[16], o1[16], q0[16], q1[16];
        tmem_ld16(tmem + lane_addr + kColO, o0);
        tmem_ld16(tmem + lane_addr + kColO + 16u, o1);
        if (ng > 4) {
          tmem_ld16(tmem + lane_addr + kColO1, q0);
          tmem_ld16(tmem + lane_addr + kColO1 + 16u, q1);
        }
        tmem_wait_ld_tied(o0, o1);
        tmem_tie(q0, q1);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          float v0 = __uint_as_float(o0[e]) * a0, v1 = __uint_as_float(o0[e + 1]) * a0;
          float u0 = __uint_as_float(o1[e]) * a0, u1 = __uint_as_float(o1[e + 1]) * a0;
          if (ng > 4) {
            v0 = fmaf(__uint_as_float(q0[e]), a1, v0);
            v1 = fmaf(__uint_as_float(q0[e + 1]), a1, v1);
            u0 = fmaf(__uint_as_float(q1[e]), a1, u0);
            u1 = fmaf(__uint_as_float(q1[e + 1]), a1, u1);
          }
          w[e >> 1] = pack_bf16(v0, v1);
          w[8 + (e >> 1)] = pack_bf16(u0, u1);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4 *>(smem + kO + sw64(row, q)) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      // ------------------------------------------------ Y += O W_o,h^T ---
      ok0 = true;
      if (tid == 0) {
        ok0 = mbar_wait(bar(bWo), ph, ctl);
        if (ok0) {
          tc_fence_after();
          for (int kk = 0; kk < 2; ++kk)
            mma_ss(tmem + kColY, smem_desc(sbase + kO + 32u * kk, 16, 512, kSwizzle64B),
                   smem_desc(sbase + kWo + 32u * kk, 16, 512, kSwizzle64B), idesc_y, (h > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(bY));
        }
      }
      // the next head's first wait (bQKV) or the epilogue's (bY) agrees on ok0
      if (!ok0) *abort_flag = 1;
    }
    if (!ok) break;
    // ------------------------------------------- Y + b_o + X at the tokens ---
    ok = cta_wait(bY, (hc - 1) & 1u, true);
    if (!ok) break;
    if (box) {
      ok = cta_wait(bX, xph & 1u, true);  // X back in the region
      ++xph;
      if (!ok) break;
    }
    tc_fence_after();
    if (box) {
      // y = Y + b_o + X in bf16 over X in the tile (row = slot), then one box
      // store per 64-channel block
      const int cw = C >> 1, c0 = (warp < 4 ? 0 : cw);
      const bool real = row < g.n;
      for (int k = 0; k < cw / 16; ++k) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_addr + kColY + (uint32_t)(c0 + 16 * k), v);
        tmem_wait_ld_tied(v);
        if (real) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int cc = c0 + 16 * k + 8 * q;  // first channel of this 16-byte chunk
            uint4 *ptr = reinterpret_cast<uint4 *>(smem + kXn + (cc >> 6) * 16384 + sw128(row, (cc & 63) >> 3));
            const uint4 xq = *ptr;
            const uint32_t xw[4] = {xq.x, xq.y, xq.z, xq.w};
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(v[8 * q + 2 * e]) + bo[cc + 2 * e] + bf_lo(xw[e]),
                               __uint_as_float(v[8 * q + 2 * e + 1]) + bo[cc + 2 * e + 1] + bf_hi(xw[e]));
            *ptr = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        for (int kb = 0; kb < nkb; ++kb) tma_store_5d(&y_map, sbase + kXn + kb * 16384, kb * 64, bc[2], bc[1], bc[0], b);
        bulk_commit();
      }
    } else {
      const int cw = C >> 1, c0 = (warp < 4 ? 0 : cw);  // warps 0-3: first half of the channels
      const int s = srcs[row];
      const bool store = s >= 0 && in_bounds(((int64_t)b * g.tokens + s) * C + c0, cw,
                                             (int64_t)g.batch * g.tokens * C, a.status);
      const int64_t base = ((int64_t)b * g.tokens + (s >= 0 ? s : 0)) * C + c0;
      const uint4 *xr = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.x) + base);
      uint4 *yr = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.y) + base);
      for (int k = 0; k < cw / 16; ++k) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_addr + kColY + (uint32_t)(c0 + 16 * k), v);
        tmem_wait_ld_tied(v);
        if (store) {
          const uint4 x0 = __ldg(xr + 2 * k), x1 = __ldg(xr + 2 * k + 1);
          const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int c = c0 + 16 * k + 2 * e;
            w[e] = pack_bf16(__uint_as_float(v[2 * e]) + bo[c] + bf_lo(xw[e]),
                             __uint_as_float(v[2 * e + 1]) + bo[c + 1] + bf_hi(xw[e]));
          }
          yr[2 * k] = make_uint4(w[0], w[1], w[2], w[3]);
          yr[2 * k + 1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (tid == 0) bulk_wait0();  // every y box store complete before the CTA leaves

  // drain: MMAs in flight, then weight copies still in flight
  if (tid == 0) {
    volatile int no_abort = 0;
    WaitCtl dctl{&no_abort, a.status, a.wait_limit_ns < 50000000ull ? a.wait_limit_ns : 50000000ull};
    mma_commit(bar(bDrain));
    mbar_wait(bar(bDrain), 0, dctl);
    // the last copy of each weight tile may still be landing (its phase is
    // then the only one not yet waited for); earlier ones were consumed
    if (n_wqkv > 0) mbar_wait(bar(bW), (n_wqkv - 1) & 1u, dctl);
    if (n_wo > 0) mbar_wait(bar(bWo), (n_wo - 1) & 1u, dctl);
    if (n_x > 0) mbar_wait(bar(bX), (n_x - 1) & 1u, dctl);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, lg::kTmemCols);
}

}  // namespace
}  // namespace blk

int launch_block_fwd(const BlockArgs &a, const void *w_qkv, const void *w_o, void *stream) {
  const Geo &g = a.g;
  if (g.hd != blk::kHdB || g.n > 128 || g.C % 64 != 0 || g.C > blk::kMaxC || g.heads * g.T > blk::kMaxBias)
    return SWIN_ERR_UNSUPPORTED;
  PFN_cuTensorMapEncodeTiled_v12000 enc = lg::tensor_map_encoder();
  if (!enc) return SWIN_ERR_CUDA;
  CUtensorMap mq, mo;
  {
    // W_qkv [3C][C] as (channel in block, row in part, part, channel block)
    const cuuint64_t C2 = (cuuint64_t)g.C * 2;
    cuuint64_t dims[4] = {64, (cuuint64_t)g.C, 3, (cuuint64_t)(g.C / 64)};
    cuuint64_t strides[3] = {C2, C2 * (cuuint64_t)g.C, 128};
    cuuint32_t box[4] = {64u, 32u, 3u, (cuuint32_t)(g.C / 64)};
    cuuint32_t es[4] = {1u, 1u, 1u, 1u};
    if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(w_qkv), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SWIN_ERR_CUDA;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)g.C, (cuuint64_t)g.C};
    cuuint64_t strides[1] = {(cuuint64_t)g.C * 2};
    cuuint32_t box[2] = {32u, (cuuint32_t)g.C};
    cuuint32_t es[2] = {1u, 1u};
    if (enc(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w_o), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SWIN_ERR_CUDA;
  }
  // x and y as [B, G0, G1, G2, C] boxes of (64 channels, a whole window), 128-byte swizzle
  CUtensorMap mx, my;
  {
    const cuuint64_t e = 2;
    cuuint64_t dims[5] = {(cuuint64_t)g.C, (cuuint64_t)g.G[2], (cuuint64_t)g.G[1], (cuuint64_t)g.G[0],
                          (cuuint64_t)g.batch};
    cuuint64_t strides[4] = {dims[0] * e, dims[0] * dims[1] * e, dims[0] * dims[1] * dims[2] * e,
                             dims[0] * dims[1] * dims[2] * dims[3] * e};
    cuuint32_t box[5] = {64u, (cuuint32_t)g.w[2], (cuuint32_t)g.w[1], (cuuint32_t)g.w[0], 1u};
    cuuint32_t es[5] = {1u, 1u, 1u, 1u, 1u};
    for (int t = 0; t < 2; ++t)
      if (enc(t ? &my : &mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, t ? a.y : const_cast<void *>(a.x), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SWIN_ERR_CUDA;
  }
  if (cudaFuncSetAttribute(blk::block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, blk::kSmemBytes) !=
      cudaSuccess)
    return SWIN_ERR_CUDA;
  blk::block_kernel<<<a.ctas, blk::kThreads, blk::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(a, mq, mo, mx, my);
  return cudaPeekAtLastError() == cudaSuccess ? SWIN_OK : SWIN_ERR_CUDA;
}

}  // namespace swin
