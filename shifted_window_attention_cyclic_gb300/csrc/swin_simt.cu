// swin_simt.cu -- fp32 FFMA kernels of SW-MSA (forward and backward).
//
// These serve the fp32 path (FFMA, not TF32: the fp32 path has to stay within
// 1e-5 of an fp64 result) and any shape the tensor-core kernels do not take.
// Both are persistent: CTA r walks the contiguous head-major work-item range
// of TERRA Eq. (4) (Sec. V.A), one (head, image, window) item at a time, with
// one thread per window slot. The shift, the ragged partition and the
// reverse route are fused into the row loads and stores (slot_route), so no
// permuted copy of any activation exists.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "swin_common.cuh"

namespace swin {
namespace {

constexpr int kThreads = 128;  // one thread per slot, n <= 128

// ---- row I/O: HD contiguous elements of one (token, head) ---------------
template <typename T, int HD>
struct RowIO;

template <int HD>
struct RowIO<float, HD> {
  static __device__ __forceinline__ void load(const float *p, float *out) {
    const float4 *p4 = reinterpret_cast<const float4 *>(p);
#pragma unroll
    for (int c = 0; c < HD / 4; ++c) {
      float4 x = __ldg(p4 + c);
      out[4 * c] = x.x;
      out[4 * c + 1] = x.y;
      out[4 * c + 2] = x.z;
      out[4 * c + 3] = x.w;
    }
  }
  static __device__ __forceinline__ void store(float *p, const float *in, float mul) {
    float4 *p4 = reinterpret_cast<float4 *>(p);
#pragma unroll
    for (int c = 0; c < HD / 4; ++c)
      p4[c] = make_float4(in[4 * c] * mul, in[4 * c + 1] * mul, in[4 * c + 2] * mul, in[4 * c + 3] * mul);
  }
};

template <int HD>
struct RowIO<__nv_bfloat16, HD> {
  static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float *out) {
    const uint4 *p4 = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int c = 0; c < HD / 8; ++c) {
      uint4 x = __ldg(p4 + c);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        out[8 * c + 2 * e] = __uint_as_float(w[e] << 16);
        out[8 * c + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float *in, float mul) {
    uint4 *p4 = reinterpret_cast<uint4 *>(p);
#pragma unroll
    for (int c = 0; c < HD / 8; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h = __floats2bfloat162_rn(in[8 * c + 2 * e] * mul, in[8 * c + 2 * e + 1] * mul);
        w[e] = *reinterpret_cast<uint32_t *>(&h);
      }
      p4[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
};

template <int HD>
__device__ __forceinline__ float dot_row(const float *a, const float *b_smem) {
  const float4 *b4 = reinterpret_cast<const float4 *>(b_smem);
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < HD / 4; ++c) {
    float4 x = b4[c];
    acc = fmaf(a[4 * c], x.x, acc);
    acc = fmaf(a[4 * c + 1], x.y, acc);
    acc = fmaf(a[4 * c + 2], x.z, acc);
    acc = fmaf(a[4 * c + 3], x.w, acc);
  }
  return acc;
}

template <int HD>
__device__ __forceinline__ void axpy_row(float *acc, float p, const float *b_smem) {
  const float4 *b4 = reinterpret_cast<const float4 *>(b_smem);
#pragma unroll
  for (int c = 0; c < HD / 4; ++c) {
    float4 x = b4[c];
    acc[4 * c] = fmaf(p, x.x, acc[4 * c]);
    acc[4 * c + 1] = fmaf(p, x.y, acc[4 * c + 1]);
    acc[4 * c + 2] = fmaf(p, x.z, acc[4 * c + 2]);
    acc[4 * c + 3] = fmaf(p, x.w, acc[4 * c + 3]);
  }
}

__host__ __device__ inline int round4(int x) { return (x + 3) & ~3; }

// ---- forward --------------------------------------------------------------
// smem: K, V tiles [128][HD] fp32, bias column [T], key codes [128], key offsets [128].
template <int HD>
__host__ __device__ inline int fwd_smem_bytes(int T) {
  return (2 * kThreads * HD + round4(T)) * 4 + 2 * kThreads * 4;
}

template <typename T, int HD>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(const FwdArgs a) {
  extern __shared__ float4 smem4[];
  float *sK = reinterpret_cast<float *>(smem4);
  float *sV = sK + kThreads * HD;
  float *sB = sV + kThreads * HD;
  int *sCode = reinterpret_cast<int *>(sB + round4(a.g.T));
  int *sRoff = sCode + kThreads;
  const Geo &g = a.g;
  const int tid = threadIdx.x;
  int64_t L, R;
  eq4_range(a.items, a.ctas, blockIdx.x, L, R);
  int cur_h = -1;
  for (int64_t it = L; it < R; ++it) {
    const Item x = decode_item(g, it);
    if (x.h != cur_h) {
      for (int t = tid; t < g.T; t += kThreads) sB[t] = a.bias ? a.bias[(int64_t)t * g.heads + x.h] : 0.f;
      cur_h = x.h;
    }
    int wc[3];
    window_coords(g, x.omega, wc);
    SlotRoute r = {-1, 0, 0, 0};
    bool live = false;
    float q[HD];
    int64_t tok = 0;
    if (tid < g.n) {
      r = slot_route(g, wc, tid);
      if (r.src >= 0 && !in_bounds((int64_t)x.b * g.tokens + r.src, 1, (int64_t)g.batch * g.tokens, a.status)) r.src = -1;
      if (r.src >= 0) {
        tok = (int64_t)x.b * g.tokens + r.src;
        const bool land = g.has_land && a.land[tok];
        live = !land;
        const int64_t off = tok * g.C + (int64_t)x.h * HD;
        RowIO<T, HD>::load(static_cast<const T *>(a.q) + off, q);
        RowIO<T, HD>::load(static_cast<const T *>(a.k) + off, sK + tid * HD);
        RowIO<T, HD>::load(static_cast<const T *>(a.v) + off, sV + tid * HD);
      }
      sCode[tid] = live ? r.reg : -1;
      sRoff[tid] = r.roff;
    }
    __syncthreads();
    if (r.src >= 0) {
      float acc[HD];
#pragma unroll
      for (int c = 0; c < HD; ++c) acc[c] = 0.f;
      float m = -INFINITY, l = 0.f, lse = -INFINITY, inv = 0.f;
      if (live) {
        for (int j = 0; j < g.n; ++j) {
          if (sCode[j] != r.reg) continue;
          const float s = dot_row<HD>(q, sK + j * HD) * a.scale + sB[r.rbase - sRoff[j]];
          if (s > m) {
            const float corr = expf(m - s);
            l *= corr;
#pragma unroll
            for (int c = 0; c < HD; ++c) acc[c] *= corr;
            m = s;
          }
          const float p = expf(s - m);
          l += p;
          axpy_row<HD>(acc, p, sV + j * HD);
        }
        inv = 1.f / l;
        lse = m + logf(l);
      }
      RowIO<T, HD>::store(static_cast<T *>(a.o) + tok * g.C + (int64_t)x.h * HD, acc, inv);
      if (a.lse) a.lse[((int64_t)x.b * g.heads + x.h) * g.tokens + r.src] = lse;
    }
    __syncthreads();
  }
}

// ---- backward -------------------------------------------------------------
// smem: Q, K, V, dO tiles [128][HD]; lse, delta [128]; bias column [T];
// key codes, query codes, key offsets, query bases [128]; partial dBias
// [128][129] accumulated over the CTA's windows of one head.
constexpr int kPartStride = kThreads + 1;

template <int HD>
__host__ __device__ inline int bwd_smem_bytes(int T) {
  return (4 * kThreads * HD + 2 * kThreads + round4(T)) * 4 + 4 * kThreads * 4 + kThreads * kPartStride * 4;
}

// Fold the per-slot-pair partial sums into bias rows, in a fixed order, and
// write them to workspace slot `slot`; then clear the partial.
__device__ void flush_partial(const Geo &g, float *sPart, float *ws, int slot) {
  __syncthreads();
  for (int t = threadIdx.x; t < g.T; t += blockDim.x) {
    int dlt[3], rem = t;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      dlt[a] = rem / g.rstride[a] - (g.w[a] - 1);
      rem %= g.rstride[a];
    }
    float sum = 0.f;
    for (int i0 = max(0, dlt[0]); i0 < min(g.w[0], g.w[0] + dlt[0]); ++i0)
      for (int i1 = max(0, dlt[1]); i1 < min(g.w[1], g.w[1] + dlt[1]); ++i1)
        for (int i2 = max(0, dlt[2]); i2 < min(g.w[2], g.w[2] + dlt[2]); ++i2) {
          const int i = (i0 * g.w[1] + i1) * g.w[2] + i2;
          const int j = ((i0 - dlt[0]) * g.w[1] + (i1 - dlt[1])) * g.w[2] + (i2 - dlt[2]);
          sum += sPart[i * kPartStride + j];
        }
    ws[(int64_t)slot * g.T + t] = sum;
  }
  __syncthreads();
  for (int x = threadIdx.x; x < kThreads * kPartStride; x += blockDim.x) sPart[x] = 0.f;
  __syncthreads();
}

template <typename T, int HD>
__global__ void __launch_bounds__(kThreads) bwd_simt_kernel(const BwdArgs a) {
  extern __shared__ float4 smem4[];
  float *sQ = reinterpret_cast<float *>(smem4);
  float *sK = sQ + kThreads * HD;
  float *sV = sK + kThreads * HD;
  float *sdO = sV + kThreads * HD;
  float *sLse = sdO + kThreads * HD;
  float *sDelta = sLse + kThreads;
  float *sB = sDelta + kThreads;
  int *sKcode = reinterpret_cast<int *>(sB + round4(a.g.T));
  int *sQcode = sKcode + kThreads;
  int *sRoff = sQcode + kThreads;
  int *sRbase = sRoff + kThreads;
  float *sPart = reinterpret_cast<float *>(sRbase + kThreads);
  const Geo &g = a.g;
  const int tid = threadIdx.x;
  for (int x = tid; x < kThreads * kPartStride; x += kThreads) sPart[x] = 0.f;
  int64_t L, R;
  eq4_range(a.items, a.ctas, blockIdx.x, L, R);
  if (L >= R) return;
  const int h_first = decode_item(g, L).h;
  int cur_h = -1;
  for (int64_t it = L; it < R; ++it) {
    const Item x = decode_item(g, it);
    if (x.h != cur_h) {
      if (cur_h >= 0 && a.ws) flush_partial(g, sPart, a.ws, a.slot_base[blockIdx.x] + (cur_h - h_first));
      for (int t = tid; t < g.T; t += kThreads) sB[t] = a.bias ? a.bias[(int64_t)t * g.heads + x.h] : 0.f;
      cur_h = x.h;
    }
    int wc[3];
    window_coords(g, x.omega, wc);
    SlotRoute r = {-1, 0, 0, 0};
    bool live = false;
    int64_t tok = 0;
    if (tid < g.n) {
      r = slot_route(g, wc, tid);
      if (r.src >= 0 && !in_bounds((int64_t)x.b * g.tokens + r.src, 1, (int64_t)g.batch * g.tokens, a.status)) r.src = -1;
      if (r.src >= 0) {
        tok = (int64_t)x.b * g.tokens + r.src;
        live = !(g.has_land && a.land[tok]);
        const int64_t off = tok * g.C + (int64_t)x.h * HD;
        RowIO<T, HD>::load(static_cast<const T *>(a.q) + off, sQ + tid * HD);
        RowIO<T, HD>::load(static_cast<const T *>(a.k) + off, sK + tid * HD);
        RowIO<T, HD>::load(static_cast<const T *>(a.v) + off, sV + tid * HD);
        RowIO<T, HD>::load(static_cast<const T *>(a.dout) + off, sdO + tid * HD);
        sLse[tid] = live ? a.lse[((int64_t)x.b * g.heads + x.h) * g.tokens + r.src] : 0.f;
      }
      sKcode[tid] = live ? r.reg : -1;
      sQcode[tid] = live ? r.reg : -2;
      sRoff[tid] = r.roff;
      sRbase[tid] = r.rbase;
    }
    __syncthreads();
    // Pass A: this thread is query i = tid.
    float delta = 0.f;
    if (live) {
      float qi[HD], doi[HD], dq[HD];
#pragma unroll
      for (int c = 0; c < HD; ++c) {
        qi[c] = sQ[tid * HD + c];
        doi[c] = sdO[tid * HD + c];
        dq[c] = 0.f;
      }
      const float lse = sLse[tid];
      for (int j = 0; j < g.n; ++j) {
        if (sKcode[j] != r.reg) continue;
        const float s = dot_row<HD>(qi, sK + j * HD) * a.scale + sB[r.rbase - sRoff[j]];
        delta = fmaf(expf(s - lse), dot_row<HD>(doi, sV + j * HD), delta);
      }
      for (int j = 0; j < g.n; ++j) {
        if (sKcode[j] != r.reg) continue;
        const float s = dot_row<HD>(qi, sK + j * HD) * a.scale + sB[r.rbase - sRoff[j]];
        const float p = expf(s - lse);
        const float ds = p * (dot_row<HD>(doi, sV + j * HD) - delta);
        axpy_row<HD>(dq, ds, sK + j * HD);
        sPart[tid * kPartStride + j] += ds;
      }
      RowIO<T, HD>::store(static_cast<T *>(a.dq) + tok * g.C + (int64_t)x.h * HD, dq, a.scale);
    } else if (r.src >= 0) {
      float z[HD];
#pragma unroll
      for (int c = 0; c < HD; ++c) z[c] = 0.f;
      RowIO<T, HD>::store(static_cast<T *>(a.dq) + tok * g.C + (int64_t)x.h * HD, z, 1.f);
    }
    if (tid < g.n) sDelta[tid] = delta;
    __syncthreads();
    // Pass B: this thread is key j = tid.
    if (r.src >= 0) {
      float dk[HD], dv[HD];
#pragma unroll
      for (int c = 0; c < HD; ++c) dk[c] = dv[c] = 0.f;
      if (live) {
        float kj[HD], vj[HD];
#pragma unroll
        for (int c = 0; c < HD; ++c) {
          kj[c] = sK[tid * HD + c];
          vj[c] = sV[tid * HD + c];
        }
        for (int i = 0; i < g.n; ++i) {
          if (sQcode[i] != r.reg) continue;
          const float s = dot_row<HD>(kj, sQ + i * HD) * a.scale + sB[sRbase[i] - r.roff];
          const float p = expf(s - sLse[i]);
          const float ds = p * (dot_row<HD>(vj, sdO + i * HD) - sDelta[i]);
          axpy_row<HD>(dk, ds, sQ + i * HD);
          axpy_row<HD>(dv, p, sdO + i * HD);
        }
      }
      RowIO<T, HD>::store(static_cast<T *>(a.dk) + tok * g.C + (int64_t)x.h * HD, dk, a.scale);
      RowIO<T, HD>::store(static_cast<T *>(a.dv) + tok * g.C + (int64_t)x.h * HD, dv, 1.f);
    }
    __syncthreads();
  }
  if (a.ws) flush_partial(g, sPart, a.ws, a.slot_base[blockIdx.x] + (cur_h - h_first));
}

template <typename T, int HD>
int launch_fwd_t(const FwdArgs &a, cudaStream_t st) {
  const int smem = fwd_smem_bytes<HD>(a.g.T);
  auto kern = fwd_simt_kernel<T, HD>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SWIN_ERR_CUDA;
  kern<<<a.ctas, kThreads, smem, st>>>(a);
  return cudaPeekAtLastError() == cudaSuccess ? SWIN_OK : SWIN_ERR_CUDA;
}

template <typename T, int HD>
int launch_bwd_t(const BwdArgs &a, cudaStream_t st) {
  const int smem = bwd_smem_bytes<HD>(a.g.T);
  auto kern = bwd_simt_kernel<T, HD>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SWIN_ERR_CUDA;
  kern<<<a.ctas, kThreads, smem, st>>>(a);
  return cudaPeekAtLastError() == cudaSuccess ? SWIN_OK : SWIN_ERR_CUDA;
}

}  // namespace

int simt_fwd_smem(const Geo &g) { return g.hd == 16 ? fwd_smem_bytes<16>(g.T) : fwd_smem_bytes<32>(g.T); }
int simt_bwd_smem(const Geo &g) { return g.hd == 16 ? bwd_smem_bytes<16>(g.T) : bwd_smem_bytes<32>(g.T); }

int launch_fwd_simt(const FwdArgs &a, int dtype, void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (a.g.hd == 16)
    return dtype == SWIN_BF16 ? launch_fwd_t<__nv_bfloat16, 16>(a, st) : launch_fwd_t<float, 16>(a, st);
  return dtype == SWIN_BF16 ? launch_fwd_t<__nv_bfloat16, 32>(a, st) : launch_fwd_t<float, 32>(a, st);
}

int launch_bwd_simt(const BwdArgs &a, int dtype, void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (a.g.hd == 16)
    return dtype == SWIN_BF16 ? launch_bwd_t<__nv_bfloat16, 16>(a, st) : launch_bwd_t<float, 16>(a, st);
  return dtype == SWIN_BF16 ? launch_bwd_t<__nv_bfloat16, 32>(a, st) : launch_bwd_t<float, 32>(a, st);
}

int simt_occupancy(bool bwd, const Geo &g, int dtype, int *blocks_per_sm) {
  cudaError_t e;
  const int smem = bwd ? simt_bwd_smem(g) : simt_fwd_smem(g);
  const void *fn;
  if (g.hd == 16)
    fn = bwd ? (dtype == SWIN_BF16 ? (const void *)bwd_simt_kernel<__nv_bfloat16, 16> : (const void *)bwd_simt_kernel<float, 16>)
             : (dtype == SWIN_BF16 ? (const void *)fwd_simt_kernel<__nv_bfloat16, 16> : (const void *)fwd_simt_kernel<float, 16>);
  else
    fn = bwd ? (dtype == SWIN_BF16 ? (const void *)bwd_simt_kernel<__nv_bfloat16, 32> : (const void *)bwd_simt_kernel<float, 32>)
             : (dtype == SWIN_BF16 ? (const void *)fwd_simt_kernel<__nv_bfloat16, 32> : (const void *)fwd_simt_kernel<float, 32>);
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return SWIN_ERR_CUDA;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, kThreads, smem);
  return e == cudaSuccess ? SWIN_OK : SWIN_ERR_CUDA;
}

}  // namespace swin
