// G1: one-pass safe softmax of the rows of a row-major fp32 matrix.
//
// The running pair (m, l) of the online normaliser (curionode "The Online
// Softmax.", introduction; roadmapper "Online softmax", "The recurrence")
// is evaluated in base 2 with log2(e) folded into the scale once and exp2 for
// every exponential, the rescale factor included (roadmapper "Things that
// break": mixing bases is one of the listed failures).
//
// Register-resident path (cols <= 16384): one CTA of 256 threads per row.
// Each thread loads its slice of the row once with 16-byte streaming loads,
// keeps it in registers, forms its own partial state (m_t, l_t, p_t) and the
// CTA merges the 256 partial states with the pairwise identity (warp shuffles,
// then one shared-memory round) -- the merge the curionode page calls
// associative, used here in place of a second pass over HBM. The weights p
// are then rescaled in registers and written once: 4 bytes read and 4 bytes
// written per element.
//
// Streaming path (rows longer than 16384, or not 16-byte aligned): each
// thread runs the recurrence over its chunks of the row as they arrive, the
// CTA merges the states, then the row is read a second time to write y
// (2 reads + 1 write per element).
//
// Internal state is in base 2: for a thread whose largest input is xm,
// M = xm * c with c = scale * log2(e) carried as c_hi + c_lo, and each weight
// is 2^(x*c - M), the exponent formed with two FMAs so that only its final
// rounding matters. ABI outputs are natural: m = fl32(scale * max x) and
// l = sum exp(scale * x - m).

#include <cfloat>
#include <cstdint>

#include "device_common.cuh"
#include "oss_internal.h"

namespace oss {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct ScaleConsts {
  float scale;  // natural-unit scale (for m)
  float c_hi;   // scale * log2(e), leading float
  float c_lo;   // scale * log2(e) - c_hi
  float e_hi;   // log2(e), leading float
  float e_lo;   // log2(e) - e_hi
};

// Base-2 maximum belonging to a raw maximum xm (>= the base-2 image of every
// other x of the same slice, since c > 0 and rounding is monotone).
__device__ __forceinline__ float base2_of(float xm, const ScaleConsts& k) {
  return fmaf(xm, k.c_hi, xm * k.c_lo);
}

// 2^(x*c - M). The inner FMA forms x*c_hi - M from the exact product, so the
// cancellation against M happens before any rounding and the result is
// rounded at its own (small) magnitude; the outer FMA adds x*c_lo. Rounding
// the other way round (x*c_lo - M first) would cost half an ulp of M, which
// for large logits (M ~ 5000) is 2.4e-4 in the exponent.
__device__ __forceinline__ float weight(float x, float M, const ScaleConsts& k) {
  return ex2(fmaf(x, k.c_lo, fmaf(x, k.c_hi, -M)));
}

// Merge partial state (xa, la) with (xb, lb); x* are raw maxima, l* sums of
// weights relative to base2_of(x*). An empty side has x = -inf, l = 0.
__device__ __forceinline__ void merge_state(float& xa, float& la, float xb, float lb,
                                            const ScaleConsts& k) {
  const float xm = fmaxf(xa, xb);
  if (xm == neg_inf()) return;  // both empty: stays (-inf, 0)
  const float Mm = base2_of(xm, k);
  const float fa = (xa == neg_inf()) ? 0.f : ex2(base2_of(xa, k) - Mm);
  const float fb = (xb == neg_inf()) ? 0.f : ex2(base2_of(xb, k) - Mm);
  la = la * fa + lb * fb;
  xa = xm;
}

// CTA-wide merge of every thread's (xm, ls). Returns the row state in all threads.
__device__ __forceinline__ void cta_merge(float& xm, float& ls, const ScaleConsts& k,
                                          float2* sh /* [kWarps] */) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float xo = __shfl_xor_sync(0xffffffffu, xm, off);
    const float lo = __shfl_xor_sync(0xffffffffu, ls, off);
    merge_state(xm, ls, xo, lo, k);
  }
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) sh[warp] = make_float2(xm, ls);
  __syncthreads();
  float2 s = sh[0];
  xm = s.x;
  ls = s.y;
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    s = sh[w];
    merge_state(xm, ls, s.x, s.y, k);
  }
}

// m and l of a finished row, in natural units.
__device__ __forceinline__ void write_ml(float xm, float ls, const ScaleConsts& k,
                                         int64_t row, float* m_out, float* l_out) {
  if (xm == neg_inf()) {
    if (m_out) m_out[row] = neg_inf();
    if (l_out) l_out[row] = 0.f;
    return;
  }
  const float m_nat = k.scale * xm;
  // ls is relative to M = base2_of(xm); convert to m_nat * log2(e):
  // l = ls * 2^(M - m_nat * log2 e), the difference formed to ~2^-40.
  const float M = base2_of(xm, k);
  const float hi = m_nat * k.e_hi;
  const float err = fmaf(m_nat, k.e_hi, -hi);
  const float delta = ((M - hi) - err) - m_nat * k.e_lo;
  if (m_out) m_out[row] = m_nat;
  if (l_out) l_out[row] = ls * ex2(delta);
}

template <int NV>
__global__ void __launch_bounds__(kThreads, (NV <= 8) ? 4 : 2)
softmax_rows_reg_kernel(const float* __restrict__ x, float* __restrict__ y,
                        float* __restrict__ m_out, float* __restrict__ l_out,
                        int64_t rows, int cols, int64_t ld_x, int64_t ld_y, ScaleConsts k) {
  __shared__ float2 sh[kWarps];
  const int nfull = cols >> 2;  // complete 16-byte chunks
  const int tail = cols & 3;
  const int tid = threadIdx.x;

  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float* xr = x + row * ld_x;
    float* yr = y + row * ld_y;
    float4 v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int c4 = tid + i * kThreads;
      if (c4 < nfull) {
        v[i] = ld_stream(reinterpret_cast<const float4*>(xr) + c4);
      } else {
        v[i] = make_float4(neg_inf(), neg_inf(), neg_inf(), neg_inf());
        if (c4 == nfull && tail) {
          const float* p = xr + 4 * c4;
          v[i].x = p[0];
          if (tail > 1) v[i].y = p[1];
          if (tail > 2) v[i].z = p[2];
        }
      }
    }
    // thread-local maximum of the raw inputs (exact)
    float xm = neg_inf();
#pragma unroll
    for (int i = 0; i < NV; ++i)
      xm = fmaxf(xm, fmaxf(fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w)));
    // thread-local weights relative to the thread's own maximum
    const float Mt = (xm == neg_inf()) ? 0.f : base2_of(xm, k);
    float ls = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      v[i].x = weight(v[i].x, Mt, k);
      v[i].y = weight(v[i].y, Mt, k);
      v[i].z = weight(v[i].z, Mt, k);
      v[i].w = weight(v[i].w, Mt, k);
      ls += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    }
    const float xm_t = xm;
    cta_merge(xm, ls, k, sh);
    // per-thread factor: 2^(M_t - M_row) / l_row (0 for an empty row or slice)
    float f = 0.f;
    if (xm_t != neg_inf() && ls > 0.f)
      f = ex2(base2_of(xm_t, k) - base2_of(xm, k)) * (1.0f / ls);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int c4 = tid + i * kThreads;
      const float4 o = make_float4(v[i].x * f, v[i].y * f, v[i].z * f, v[i].w * f);
      if (c4 < nfull) {
        st_stream(reinterpret_cast<float4*>(yr) + c4, o);
      } else if (c4 == nfull && tail) {
        float* p = yr + 4 * c4;
        p[0] = o.x;
        if (tail > 1) p[1] = o.y;
        if (tail > 2) p[2] = o.z;
      }
    }
    if (tid == 0) write_ml(xm, ls, k, row, m_out, l_out);
    __syncthreads();  // sh is reused by the next row
  }
}

// Rows too long for registers, or rows that are not 16-byte aligned: each
// thread runs the recurrence over its chunks of the row as they arrive
// (16-byte chunks when aligned, single elements otherwise), the CTA merges the
// states, then the row is read a second time to write y (2 reads + 1 write).
template <bool kVec>
__global__ void __launch_bounds__(kThreads)
softmax_rows_stream_kernel(const float* __restrict__ x, float* __restrict__ y,
                           float* __restrict__ m_out, float* __restrict__ l_out,
                           int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                           ScaleConsts k) {
  __shared__ float2 sh[kWarps];
  constexpr int W = kVec ? 4 : 1;
  const int64_t nchunks = (cols + W - 1) / W;
  const int tid = threadIdx.x;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float* xr = x + row * ld_x;
    float* yr = y + row * ld_y;
    float xm = neg_inf(), ls = 0.f;
    for (int64_t c = tid; c < nchunks; c += kThreads) {
      float v[W];
      if (kVec && (c + 1) * W <= cols) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(xr) + c);
        v[0] = f.x;
        if (kVec) { v[1 % W] = f.y; v[2 % W] = f.z; v[3 % W] = f.w; }
      } else {
#pragma unroll
        for (int e = 0; e < W; ++e) v[e] = (c * W + e < cols) ? xr[c * W + e] : neg_inf();
      }
      float bm = v[0];
#pragma unroll
      for (int e = 1; e < W; ++e) bm = fmaxf(bm, v[e]);
      const float xn = fmaxf(xm, bm);
      if (xn == neg_inf()) continue;  // nothing visible yet: no -inf - -inf
      const float Mn = base2_of(xn, k);
      const float corr = (xm == neg_inf()) ? 0.f : ex2(base2_of(xm, k) - Mn);
      float add = 0.f;
#pragma unroll
      for (int e = 0; e < W; ++e) add += weight(v[e], Mn, k);
      ls = ls * corr + add;
      xm = xn;
    }
    cta_merge(xm, ls, k, sh);
    const float M = (xm == neg_inf()) ? 0.f : base2_of(xm, k);
    const float inv = (ls > 0.f) ? 1.0f / ls : 0.f;
    for (int64_t c = tid; c < nchunks; c += kThreads) {
      if (kVec && (c + 1) * W <= cols) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(xr) + c);
        const float4 o = make_float4(weight(f.x, M, k) * inv, weight(f.y, M, k) * inv,
                                     weight(f.z, M, k) * inv, weight(f.w, M, k) * inv);
        st_stream(reinterpret_cast<float4*>(yr) + c, o);
      } else {
        for (int e = 0; e < W; ++e)
          if (c * W + e < cols) yr[c * W + e] = weight(xr[c * W + e], M, k) * inv;
      }
    }
    if (tid == 0) write_ml(xm, ls, k, row, m_out, l_out);
    __syncthreads();
  }
}

int grid_for(int64_t rows, int ctas_per_sm) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t cap = static_cast<int64_t>(sms) * ctas_per_sm * 64;
  return static_cast<int>(rows < cap ? rows : cap);
}

}  // namespace

void split_constant(double c, float* hi, float* lo) {
  *hi = static_cast<float>(c);
  *lo = static_cast<float>(c - static_cast<double>(*hi));
}

cudaError_t launch_softmax_rows(const float* x, float* y, float* m, float* l, int64_t rows,
                                int64_t cols, int64_t ld_x, int64_t ld_y, float scale,
                                cudaStream_t stream) {
  const double kLog2e = 1.4426950408889634074;
  ScaleConsts k;
  k.scale = scale;
  split_constant(static_cast<double>(scale) * kLog2e, &k.c_hi, &k.c_lo);
  split_constant(kLog2e, &k.e_hi, &k.e_lo);

  const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                   (ld_x & 3) == 0 && (ld_y & 3) == 0;
  if (!vec) {
    softmax_rows_stream_kernel<false><<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, cols, ld_x, ld_y, k);
    return cudaGetLastError();
  }
  const int64_t chunks = (cols + 3) / 4;
  const int nv = static_cast<int>((chunks + kThreads - 1) / kThreads);
  const int c = static_cast<int>(cols);
  if (nv <= 1) {
    softmax_rows_reg_kernel<1><<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
  } else if (nv <= 2) {
    softmax_rows_reg_kernel<2><<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
  } else if (nv <= 4) {
    softmax_rows_reg_kernel<4><<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
  } else if (nv <= 8) {
    softmax_rows_reg_kernel<8><<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
  } else if (nv <= 16) {
    softmax_rows_reg_kernel<16><<<grid_for(rows, 2), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
  } else {
    softmax_rows_stream_kernel<true><<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, cols, ld_x, ld_y, k);
  }
  return cudaGetLastError();
}

}  // namespace oss
