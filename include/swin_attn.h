/*
 * swin_attn.h -- C ABI of a single-GPU (GB300, sm_103a) library for
 * shifted-window multi-head self-attention (SW-MSA) over a lat-lon(-depth)
 * token grid: cyclic shift, ragged edge windows, periodic longitude seam,
 * shift-boundary (region) mask, land mask, relative-position bias, softmax,
 * PV and the reverse routing back to the grid; forward and backward.
 *
 * Where the operation is defined (page title, section):
 *  - "TERRA: A Hierarchical Parallel Training and Memory Orchestration
 *    Framework for High-Resolution AI-based Earth Modeling", Sec. IV.D
 *    "Differentiable Token Routes": window coordinate and in-window offset of
 *    a token follow from its global grid coordinate; a window shift changes
 *    the coordinate; the backward applies the inverse route. Sec. V.A, Eq. (4):
 *    ragged contiguous window ranges (used here to split work over CTAs).
 *  - "4D Parallelism Unlocks Exascale Bayesian Neural Networks for
 *    High-Fidelity Atmospheric Modeling", Model Architecture: the domain is
 *    rolled by floor(window/2) between attention layers; Swin-style window
 *    attention with a relative-position bias.
 *
 * Definition computed (all dims outermost first; G grid, w window, s shift):
 *   rolled position p_d = (u_d - s_d) mod G_d of the token at coordinate u;
 *   window floor(p_d / w_d), slot p_d mod w_d (ceil(G_d / w_d) windows per dim,
 *   the last one may be short: its missing slots are pads);
 *   region bit d = [dim d not periodic and s_d > 0 and p_d >= G_d - s_d];
 *   key j is visible to query i iff same window, same region bits, j not land;
 *   s_ij = hd^-1/2 q_i.k_j + bias[row(i,j), h],
 *   row(i,j) = sum_d (sig_i,d - sig_j,d + w_d - 1) * prod_{e>d} (2 w_e - 1);
 *   O_i = softmax over visible j of s_ij, times V; land queries give O = 0.
 *
 * Conventions for every entry point:
 *  - Returns SWIN_OK (0) or a negative status; nothing is launched when an
 *    argument check fails.
 *  - Tensors are owned by the caller, device-resident, contiguous. Every
 *    q/k/v/o/dout/dq/dk/dv pointer and lse must be 16-byte aligned, land,
 *    bias and dbias 4-byte aligned: the tensor-core kernels read four
 *    consecutive LSE values, or land bytes, with one load. fwd and bwd
 *    return SWIN_ERR_ALIGNMENT (launching nothing) for any pointer that
 *    breaks this rule; buffer sizes are the caller's to keep.
 *  - q, k, v, o, dout, dq, dk, dv: [B, grid..., C] channel-last, C = heads *
 *    head_dim, head h in channels [h*hd, (h+1)*hd); element type = desc.dtype.
 *  - bias, dbias: float32 [rows][heads], rows = prod(2 w_d - 1).
 *  - lse: float32 [B][heads][grid...] natural-log log-sum-exp per query
 *    (-inf for land queries).
 *  - land: uint8 [B, grid...], nonzero = land.
 *  - fwd/bwd allocate nothing and are asynchronous on `stream`.
 */
#ifndef SWIN_ATTN_H
#define SWIN_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define SWIN_OK 0
#define SWIN_ERR_INVALID_ARG (-1) /* NULL/inconsistent argument or descriptor */
#define SWIN_ERR_UNSUPPORTED (-2) /* head_dim not 16/32/128, window too large for head_dim, ... */
#define SWIN_ERR_ALIGNMENT (-3)   /* a pointer breaks its alignment rule (see Conventions) */
#define SWIN_ERR_WORKSPACE (-4)   /* workspace NULL or smaller than required */
#define SWIN_ERR_CUDA (-5)        /* a CUDA runtime call or launch failed */
#define SWIN_ERR_TIMEOUT (-6)     /* a kernel gave up a bounded wait (device status word) */
#define SWIN_ERR_DEVICE (-7)      /* a kernel recorded another device-side error */

/* Element types of q, k, v, o, dout, dq, dk, dv. */
#define SWIN_F32 0
#define SWIN_BF16 1

/* Kernel family. AUTO picks the tensor-core path for bf16 with head_dim 32 or 128. */
#define SWIN_IMPL_AUTO 0
#define SWIN_IMPL_SIMT 1   /* fp32 FFMA kernels (head_dim 16/32, windows up to 128 slots) */
#define SWIN_IMPL_TC 2     /* tcgen05/TMEM kernels (bf16; head_dim 32 with windows up to 128
                              slots, or head_dim 128 with windows of any size) */

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *swin_stream_t;

/* Opaque plan. Owns its device-side tables and status word. */
typedef struct swin_attn_plan_s *swin_attn_plan_t;

typedef struct {
  int32_t ndim;        /* 2: (lat, lon); 3: (depth, lat, lon) */
  int32_t impl;        /* SWIN_IMPL_* */
  int64_t batch;       /* B >= 1 */
  int32_t grid[3];     /* G_d >= 1, outermost first; batch * prod(G) < 2^31 */
  int32_t window[3];   /* w_d >= 1; prod(w) <= 128, or <= 65536 with head_dim 128 */
  int32_t shift[3];    /* 0 <= s_d < w_d, s_d < G_d (or 0); all zero = W-MSA */
  int32_t periodic[3]; /* 1 = cyclic neighbour (no region bit), 0 = region-masked */
  int32_t heads;       /* >= 1 */
  int32_t head_dim;    /* 16 or 32; or 128 (bf16, tensor cores): windows of any size, split
                          into 128-slot query and key tiles with an online softmax */
  int32_t dtype;       /* SWIN_F32 or SWIN_BF16 */
  int32_t has_land;    /* 1 = a land mask is passed to fwd/bwd */
} swin_attn_desc;

/* Sizes and launch shapes of a plan (all counts, no pointers). */
typedef struct {
  int64_t windows_per_image;
  int64_t tokens_per_image;
  int32_t slots;       /* n = prod(w) */
  int32_t bias_rows;   /* prod(2 w_d - 1) */
  int32_t impl;        /* resolved SWIN_IMPL_SIMT or SWIN_IMPL_TC */
  int32_t fwd_ctas;    /* persistent CTAs of the forward kernel */
  int32_t bwd_ctas;    /* persistent CTAs of the backward kernel */
  int32_t num_sms;
  int64_t work_items;  /* heads * B * ceil(windows_per_image / k): one head and k windows each, k = 2 on
                          the tensor-core path when two windows fit one 128-slot tile, else 1 */
  int64_t dbias_slots; /* partial dBias tables in the workspace */
} swin_attn_plan_info;

/* Validate `desc` and build a plan on the current CUDA device: routing tables
 * (win_src, region, tok_dst, relidx) are computed on the device by the same
 * routing function the kernels use, and the work partition is fixed.
 * Synchronous; allocates device memory owned by the plan.
 * Errors: INVALID_ARG (NULL, bad sizes, shift >= window), UNSUPPORTED
 * (slots > 128 without head_dim 128, slots > 65536, head_dim, dtype, impl not
 * available for the dtype or head_dim), CUDA. */
int swin_attn_plan(const swin_attn_desc *desc, swin_attn_plan_t *out);

/* Copy `plan`'s sizes into *info (host). Errors: INVALID_ARG. */
int swin_attn_plan_get_info(swin_attn_plan_t plan, swin_attn_plan_info *info);

/* Copy the routing tables of one image to HOST buffers (any may be NULL):
 *   win_src [nwin][n] int32: grid token feeding slot s of window w, -1 = pad;
 *   region  [nwin][n] uint8: region bits of that token (bit d for dim d), 0 for pads;
 *   tok_dst [N] int32: w*n + s of every token (the inverse route);
 *   relidx  [n][n] int32: bias row of the slot pair (query i, key j); kept by
 *           the plan for windows of up to 2048 slots only (UNSUPPORTED above).
 * Synchronous. Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
int swin_attn_plan_tables(swin_attn_plan_t plan, int32_t *win_src, uint8_t *region,
                          int32_t *tok_dst, int32_t *relidx);

/* Bytes of device workspace swin_attn_bwd needs: the partial dBias tables,
 * and for head_dim 128 also delta_i = sum_j P_ij dP_ij of every query. */
size_t swin_attn_workspace_bytes(swin_attn_plan_t plan);

/* Forward. q, k, v, o as above; bias may be NULL (zero bias); land required
 * iff desc.has_land; lse may be NULL (inference) else receives the float32
 * log-sum-exp. Pad slots write nothing; every grid token is written once.
 * head_dim 128: a non-NULL bias needs at most 4096 bias rows (UNSUPPORTED).
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED, CUDA (launch). */
int swin_attn_fwd(swin_attn_plan_t plan, const void *q, const void *k, const void *v,
                  const float *bias, const uint8_t *land, void *o, float *lse,
                  swin_stream_t stream);

/* Backward of L = sum(O * dout): writes dq, dk, dv (every token) and
 * OVERWRITES dbias (may be NULL: not computed). lse is the forward's output
 * for the same inputs (required). delta_i = sum_j P_ij dP_ij is recomputed
 * in-kernel, so O is not an input. workspace: device, >=
 * swin_attn_workspace_bytes(plan) bytes, 256-byte aligned, contents ignored
 * (not needed when dbias is NULL, except with head_dim 128, whose backward
 * keeps delta there). head_dim 128: a non-NULL bias needs at most 4096 bias
 * rows and a non-NULL dbias at most 8192 (UNSUPPORTED); its dBias is summed
 * per CTA with shared-memory atomic adds, so it may differ between calls in
 * the last bits (the other outputs, and dBias of head_dim 16/32, do not).
 * When swin_attn_status then reports SWIN_ERR_TIMEOUT, every output of the
 * call is undefined.
 * Errors: INVALID_ARG, ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA. */
int swin_attn_bwd(swin_attn_plan_t plan, const void *q, const void *k, const void *v,
                  const void *dout, const float *lse, const float *bias,
                  const uint8_t *land, void *dq, void *dk, void *dv, float *dbias,
                  void *workspace, size_t workspace_bytes, swin_stream_t stream);

/* Backward that also receives the forward's output o (same type, layout and
 * alignment as q; o of the same inputs). With head_dim 128, delta_i is then
 * sum over the head's channels of dout_ic * o_ic (FlashAttention's form of
 * the softmax derivative's row sum, which TERRA's FlashAttention backward
 * uses), computed by a small kernel before the query-tile kernel, which then
 * sweeps the key tiles once instead of twice. It differs from swin_attn_bwd's
 * delta by the rounding of o to the storage type. Other head dims ignore o
 * (their kernels recompute delta in the pass that needs it at no extra cost)
 * and give swin_attn_bwd's results. Other arguments, results and errors as
 * swin_attn_bwd; o NULL is INVALID_ARG, misaligned ALIGNMENT. */
int swin_attn_bwd_o(swin_attn_plan_t plan, const void *q, const void *k, const void *v, const void *o,
                    const void *dout, const float *lse, const float *bias, const uint8_t *land, void *dq,
                    void *dk, void *dv, float *dbias, void *workspace, size_t workspace_bytes,
                    swin_stream_t stream);

/* Backward for callers that cannot allocate device memory. No counterpart on
 * the pages: it exists for callers whose host code has no device allocator
 * of its own (for example a C or Fortran model that only receives tensors),
 * or whose device memory all belongs to a pool they may not touch while
 * stepping, and who therefore cannot provide swin_attn_bwd's workspace.
 * Same arguments, results and errors as swin_attn_bwd without the
 * workspace: the partial dBias tables go to a fixed device array inside this
 * library (SWIN_NOALLOC_MAX_WORKSPACE_BYTES, held on every GPU that loads the
 * library until the process exits). Nothing is allocated by any call.
 *  - With dbias != NULL, plans whose swin_attn_workspace_bytes() exceeds
 *    the array are rejected with SWIN_ERR_WORKSPACE (nothing is launched).
 *    With dbias == NULL the array is not used and any plan is accepted.
 *  - The first call in a CUDA context (per device, and again after
 *    cudaDeviceReset or in another context on that device) looks up the
 *    array's device address in that context; make that first call before
 *    any stream capture.
 *  - All calls share the one array: calls that can overlap on the GPU (other
 *    streams, other threads) race on it; serialise them. Each call writes
 *    every partial table it reads; when swin_attn_status reports
 *    SWIN_ERR_TIMEOUT, that call's outputs (dbias included) are undefined.
 * Errors: those of swin_attn_bwd, WORKSPACE as above, CUDA. */
#define SWIN_NOALLOC_MAX_WORKSPACE_BYTES ((size_t)4 << 20)
int swin_attn_bwd_noalloc(swin_attn_plan_t plan, const void *q, const void *k, const void *v,
                          const void *dout, const float *lse, const float *bias,
                          const uint8_t *land, void *dq, void *dk, void *dv, float *dbias,
                          swin_stream_t stream);

/* The attention half of a Swin block in one kernel: LayerNorm and the QKV
 * projection as its prologue, SW-MSA as above, the out-projection and the
 * residual add as its epilogue, so that Q, K, V and O never go to device
 * memory (TERRA, Fig. 4 "Layernorm ... Window Attention ... MLP" and Sec. III;
 * BEAST page, "Model Architecture"). Per token t of image b:
 *   Xn = (x - mean) / sqrt(var + ln_eps) * ln_gamma + ln_beta
 *        (mean and biased variance over the C channels of x),
 *   [q | k | v] = bf16(Xn) W_qkv^T + b_qkv, each rounded to bf16,
 *   o = SW-MSA(q, k, v; bias, land) of the plan's geometry, rounded to bf16,
 *   y = x + o W_o^T + b_o, rounded to bf16.
 * x, y: bf16 [B, grid..., C], 16-byte aligned, y must not overlap x; every
 * grid token is written once. w_qkv: bf16 [3C][C] row-major (rows 0..C-1
 * give q, C..2C-1 k, 2C..3C-1 v; head h owns rows h*32..h*32+31 of each);
 * w_o: bf16 [C][C] row-major (row = output channel); both 16-byte aligned.
 * ln_gamma, ln_beta, b_o: float32 [C]; b_qkv: float32 [3C]; bias as above
 * (may be NULL); all 4-byte aligned. ln_eps > 0 and finite.
 * Supported plans: bf16, head_dim 32, at most 128 slots per window, C a
 * multiple of 64 up to 256, heads * bias rows <= 8192 (else UNSUPPORTED).
 * Forward only (no autograd through the projections here).
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED, CUDA (launch). */
int swin_attn_block_fwd(swin_attn_plan_t plan, const void *x, const float *ln_gamma, const float *ln_beta,
                        float ln_eps, const void *w_qkv, const float *b_qkv, const void *w_o,
                        const float *b_o, const float *bias, const uint8_t *land, void *y,
                        swin_stream_t stream);

/* Testing hook for the failure path of the tensor-core kernels (the fused
 * block's included). Every wait inside those kernels gives up after
 * `wait_limit_ns` (default 1 s) and then records SWIN_ERR_TIMEOUT in the
 * status word. force_timeout = 1 makes one role of the next launches wait on
 * a barrier that nothing arrives at, so the bounded wait runs out on purpose
 * (the kernel then drains and exits).
 * Errors: INVALID_ARG (NULL plan, zero limit, force_timeout not 0/1). */
int swin_attn_plan_set_debug(swin_attn_plan_t plan, uint64_t wait_limit_ns, int force_timeout);

/* Synchronise `stream`, read and clear the plan's device status word.
 * Returns SWIN_OK, SWIN_ERR_TIMEOUT, SWIN_ERR_DEVICE or SWIN_ERR_CUDA. */
int swin_attn_status(swin_attn_plan_t plan, swin_stream_t stream);

/* Free the plan's device memory (synchronises the device). NULL is a no-op. */
void swin_attn_plan_destroy(swin_attn_plan_t plan);

/* Static message for a status code. */
const char *swin_attn_strerror(int status);

/* TERRA Sec. V.A, Eq. (4): rank r of P ranks owns the contiguous window-index
 * range [floor(r*M/P), floor((r+1)*M/P)). Host-only, used for the CTA work
 * split. Errors: INVALID_ARG (M < 0, P < 1, r outside [0, P), NULL). */
int swin_attn_window_range(int64_t M, int64_t P, int64_t r, int64_t *L, int64_t *R);

/* TERRA Sec. V.A, Eq. (3): the fixed (two-dimensional round-robin) window
 * assignment over an m x n mesh pads each input dimension until every rank
 * owns the same number of whole windows. For one dimension of `extent` input
 * points, `stride` input points per token (patch size times sampling factor,
 * p*alpha), `window` tokens per window and `ranks` mesh ranks along that
 * dimension (m or n): *padded = ceil(extent / q) * q, q = stride*window*ranks.
 * ranks = 1 gives the least padding to whole windows, the padding that the
 * ragged assignment of Eq. (4) keeps. Host-only arithmetic; the attention
 * kernels never pad (pad slots of ragged windows are masked instead).
 * Errors: INVALID_ARG (extent, stride, window or ranks below 1, NULL, or a
 * result above INT64_MAX). */
int swin_attn_fixed_padded_extent(int64_t extent, int64_t stride, int64_t window, int64_t ranks,
                                  int64_t *padded);

#ifdef __cplusplus
}
#endif

#endif /* SWIN_ATTN_H */
