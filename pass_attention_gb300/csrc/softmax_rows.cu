// G1: one-pass safe softmax of the rows of a row-major fp32 matrix.
//
// The running pair (m, l) of the online normaliser (curionode "The Online
// Softmax.", introduction; roadmapper "Online softmax", "The recurrence")
// is evaluated in base 2 with log2(e) folded into the scale once and exp2 for
// every exponential, the rescale factor included (roadmapper "Things that
// break": mixing bases is one of the listed failures).
//
// Register-resident path: rows of up to 2048 fp32 (16384 16-bit) elements go
// to the grouped kernel below, where a group of 32-256 threads owns a row and
// a CTA works on several rows at once; longer fp32 rows of up to 16384
// elements take one CTA of 256 threads per row. In both, each thread loads
// its slice of the row once with 16-byte streaming loads,
// keeps it in registers, forms its own partial state (m_t, l_t, p_t) and the
// row's threads merge their partial states with the merge identity (warp shuffles,
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

#include <cuda_fp16.h>

#include <atomic>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <limits>

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
// for large logits (M ~ 5000) is 2.4e-4 in the exponent. The host splits c
// so that c_hi and c_lo are both > 0 (make_consts): a masked entry x = -inf
// then gives -inf in both FMAs and a weight of exactly 0. (With c_lo <= 0,
// which nearest rounding of c_hi gives for scale 0.1, -inf * c_lo would be
// +inf or NaN and the weight NaN.)
__device__ __forceinline__ float weight(float x, float M, const ScaleConsts& k) {
  return ex2(fmaf(x, k.c_lo, fmaf(x, k.c_hi, -M)));
}

// weight() of two elements with packed (two-lane) FMAs: the same two
// roundings per element.
__device__ __forceinline__ float2 weight2(float2 x, float2 negM, const ScaleConsts& k) {
  const float2 t = __ffma2_rn(x, make_float2(k.c_hi, k.c_hi), negM);
  const float2 e = __ffma2_rn(x, make_float2(k.c_lo, k.c_lo), t);
  return make_float2(ex2(e.x), ex2(e.y));
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// CTA-wide merge of every thread's (xm, ls) -- xm a raw maximum, ls the sum
// of weights relative to base2_of(xm), (-inf, 0) for an empty slice; returns
// the row state in all threads. The merge identity in its n-ary form: the warp's maximum first
// (shuffles of the raw maxima), each thread's sum scaled to it (one ex2), the
// scaled sums added by shuffles; then the warps' states through shared
// memory, the row maximum first and each warp sum scaled once. Folding the
// states in pairwise gives the same (max, sum) with 2 * (5 + kWarps - 1)
// exponentials per thread instead of 1 + kWarps; for 16-bit rows, with twice
// the elements per byte, that difference was 8 % of the kernel's time.
__device__ __forceinline__ void cta_merge(float& xm, float& ls, const ScaleConsts& k,
                                               float2* sh /* [kWarps] */) {
  float xw = xm;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) xw = fmaxf(xw, __shfl_xor_sync(0xffffffffu, xw, off));
  float lw = (xm == neg_inf()) ? 0.f : ls * ex2(base2_of(xm, k) - base2_of(xw, k));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = make_float2(xw, lw);
  __syncthreads();
  float x = sh[0].x;
#pragma unroll
  for (int w = 1; w < kWarps; ++w) x = fmaxf(x, sh[w].x);
  float l = 0.f;
  if (x != neg_inf()) {
    const float M = base2_of(x, k);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float2 s = sh[w];
      if (s.x != neg_inf()) l += s.y * ex2(base2_of(s.x, k) - M);
    }
  }
  xm = x;
  ls = l;
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

// ---------------------------------------------------------------------------
// Thread-block clusters: the launch constants of the cluster-resident kernel
// and the helpers every cluster-aware kernel uses. A kernel launched without
// a cluster sees each CTA as a cluster of one.
// ---------------------------------------------------------------------------

constexpr int kClThreads = 512;
constexpr int kClUnroll = 4;  // chunks each thread loads before using them
constexpr int kClWarps = kClThreads / 32;
constexpr int kClMaxCtas = 8;
constexpr int kClPiece = 16384;                       // bytes per bulk copy
constexpr unsigned long long kClTimeoutNs = 2000000000ull;  // bounded wait on the copies
constexpr int64_t kClDoubleCap = int64_t(48) << 10;   // rows this short: one CTA, two buffers
constexpr int64_t kClSingleCap = int64_t(200) << 10;  // longer rows: one buffer per CTA

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t c;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(c));
  return c;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t c;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(c));
  return c;
}
// every thread of every CTA of the cluster; orders shared-memory writes
// (local and remote) before the barrier with reads after it
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// The same barrier when only warp 0 has written anything the cluster reads
// after it: the other warps arrive without a release fence.
__device__ __forceinline__ void cluster_sync_warp0_wrote() {
  if (threadIdx.x < 32)
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  else
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// (a, b) into the same shared-memory slot of CTA `rank` of the cluster
__device__ __forceinline__ void st_peer_f2(const void* slot, uint32_t rank, float a, float b) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(slot)), "r"(rank));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity, for at most timeout_ns.
// Returns false on a give-up, which is recorded in the error word; the caller
// carries on (every CTA of the cluster must still reach the same cluster
// barriers) but waits and copies no more, so a failed launch ends after
// about one timeout rather than one per row.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned int* err,
                                                  uint64_t timeout_ns) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try(bar, parity)) return true;
    if ((n & 63u) == 0 && timer_ns() - t0 > timeout_ns) {
      report_error(err, kKernelSoftmaxRows | (1u << 8));
      return false;
    }
  }
}

// n-ary merge of the n <= 32 (max, sum) states s[0..n), by one warp: lane w
// takes state w, the lanes' maximum by shuffles, then each sum scaled to it
// (one ex2) and the scaled sums added by shuffles. Every warp that calls it
// gets the same result.
__device__ __forceinline__ float2 merge_states_warp(const float2* s, int n, const ScaleConsts& k) {
  const int lane = threadIdx.x & 31;
  const float2 e = (lane < n) ? s[lane] : make_float2(neg_inf(), 0.f);
  float x = e.x;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  float l = (e.x == neg_inf()) ? 0.f : e.y * ex2(base2_of(e.x, k) - base2_of(x, k));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  return make_float2(x, l);
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
                           ScaleConsts k, int64_t slice_chunks) {
  __shared__ float2 sh[kWarps];
  __shared__ float2 cstate[2][kClMaxCtas];
  constexpr int W = kVec ? 4 : 1;
  const int64_t nchunks = (cols + W - 1) / W;
  const int tid = threadIdx.x;
  // in a cluster of C CTAs, CTA r streams chunks [r * slice, (r + 1) * slice)
  const uint32_t C = cluster_size();
  const uint32_t rank = cluster_rank();
  const int64_t c_lo = static_cast<int64_t>(rank) * slice_chunks;
  const int64_t c_hi = (c_lo + slice_chunks < nchunks) ? c_lo + slice_chunks : nchunks;
  if (C > 1) cluster_sync_all();  // every peer has started before any writes to it
  int sbuf = 0;
  for (int64_t row = cluster_id(); row < rows; row += cluster_count()) {
    const float* xr = x + row * ld_x;
    float* yr = y + row * ld_y;
    float xm = neg_inf(), ls = 0.f;
    for (int64_t c = c_lo + tid; c < c_hi; c += kThreads) {
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
    if (C > 1) {  // the cluster's CTA states, through distributed shared memory
      if (tid == 0)
        for (uint32_t r = 0; r < C; ++r) st_peer_f2(&cstate[sbuf][rank], r, xm, ls);
      cluster_sync_warp0_wrote();
      const float2 st = merge_states_warp(cstate[sbuf], static_cast<int>(C), k);
      xm = st.x;
      ls = st.y;
      sbuf ^= 1;
    }
    const float M = (xm == neg_inf()) ? 0.f : base2_of(xm, k);
    const float inv = (ls > 0.f) ? 1.0f / ls : 0.f;
    for (int64_t c = c_lo + tid; c < c_hi; c += kThreads) {
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
    if (rank == 0 && tid == 0) write_ml(xm, ls, k, row, m_out, l_out);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Multi-pass comparators. Each pass is its own kernel over the whole matrix,
// so every pass reads x from HBM again (the curionode page's point: the safe
// softmax reads the vector three times, the online normaliser twice before
// the final write, os_softmax_rows once). Between passes m[] holds the raw
// row maximum and l[] the sum relative to its base-2 image; the write pass
// converts both to the natural-unit outputs.
// ---------------------------------------------------------------------------

template <bool kVec>
__device__ __forceinline__ int load_chunk(const float* xr, int64_t c, int64_t cols, float (&v)[4]) {
  if (kVec && (c + 1) * 4 <= cols) {
    const float4 f = __ldcs(reinterpret_cast<const float4*>(xr) + c);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    return 4;
  }
  const int64_t base = c * (kVec ? 4 : 1);
#pragma unroll
  for (int e = 0; e < 4; ++e)
    v[e] = (e < (kVec ? 4 : 1) && base + e < cols) ? xr[base + e] : neg_inf();
  return kVec ? 4 : 1;
}

// pass "max": m[r] = max_j x[r, j] (raw)
template <bool kVec>
__global__ void __launch_bounds__(kThreads)
softmax_pass_max(const float* __restrict__ x, float* __restrict__ m_out, int64_t rows,
                 int64_t cols, int64_t ld_x) {
  __shared__ float sh[kWarps];
  const int64_t nchunks = kVec ? (cols + 3) / 4 : cols;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float* xr = x + row * ld_x;
    float xm = neg_inf();
    for (int64_t c = threadIdx.x; c < nchunks; c += kThreads) {
      float v[4];
      load_chunk<kVec>(xr, c, cols, v);
      xm = fmaxf(xm, fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) xm = fmaxf(xm, __shfl_xor_sync(0xffffffffu, xm, off));
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = xm;
    __syncthreads();
    if (threadIdx.x == 0) {
      float r = sh[0];
      for (int w = 1; w < kWarps; ++w) r = fmaxf(r, sh[w]);
      m_out[row] = r;
    }
    __syncthreads();
  }
}

// pass "sum": l[r] = sum_j 2^(x c - M_r), M_r = base-2 image of m[r]
template <bool kVec>
__global__ void __launch_bounds__(kThreads)
softmax_pass_sum(const float* __restrict__ x, const float* __restrict__ m_in,
                 float* __restrict__ l_out, int64_t rows, int64_t cols, int64_t ld_x,
                 ScaleConsts k) {
  __shared__ float sh[kWarps];
  const int64_t nchunks = kVec ? (cols + 3) / 4 : cols;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float* xr = x + row * ld_x;
    const float xm = m_in[row];
    const float M = (xm == neg_inf()) ? 0.f : base2_of(xm, k);
    float ls = 0.f;
    for (int64_t c = threadIdx.x; c < nchunks; c += kThreads) {
      float v[4];
      load_chunk<kVec>(xr, c, cols, v);
      ls += (weight(v[0], M, k) + weight(v[1], M, k)) + (weight(v[2], M, k) + weight(v[3], M, k));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = ls;
    __syncthreads();
    if (threadIdx.x == 0) {
      float r = 0.f;
      for (int w = 0; w < kWarps; ++w) r += sh[w];
      l_out[row] = r;
    }
    __syncthreads();
  }
}

// pass "online": the running (max, sum) pair over the row, then the merge of
// the threads' pairs: m[r] raw maximum, l[r] relative sum
template <bool kVec>
__global__ void __launch_bounds__(kThreads)
softmax_pass_online(const float* __restrict__ x, float* __restrict__ m_out,
                    float* __restrict__ l_out, int64_t rows, int64_t cols, int64_t ld_x,
                    ScaleConsts k) {
  __shared__ float2 sh[kWarps];
  const int64_t nchunks = kVec ? (cols + 3) / 4 : cols;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float* xr = x + row * ld_x;
    float xm = neg_inf(), ls = 0.f;
    for (int64_t c = threadIdx.x; c < nchunks; c += kThreads) {
      float v[4];
      load_chunk<kVec>(xr, c, cols, v);
      const float xn = fmaxf(xm, fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])));
      if (xn == neg_inf()) continue;  // nothing visible yet: no -inf - -inf
      const float Mn = base2_of(xn, k);
      const float corr = (xm == neg_inf()) ? 0.f : ex2(base2_of(xm, k) - Mn);
      ls = ls * corr + ((weight(v[0], Mn, k) + weight(v[1], Mn, k)) +
                        (weight(v[2], Mn, k) + weight(v[3], Mn, k)));
      xm = xn;
    }
    cta_merge(xm, ls, k, sh);
    if (threadIdx.x == 0) {
      m_out[row] = xm;
      l_out[row] = ls;
    }
    __syncthreads();
  }
}

// pass "write": y = 2^(x c - M) / l, then m and l converted to natural units
template <bool kVec>
__global__ void __launch_bounds__(kThreads)
softmax_pass_write(const float* __restrict__ x, float* __restrict__ y, float* __restrict__ m_io,
                   float* __restrict__ l_io, int64_t rows, int64_t cols, int64_t ld_x,
                   int64_t ld_y, ScaleConsts k) {
  const int64_t nchunks = kVec ? (cols + 3) / 4 : cols;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float* xr = x + row * ld_x;
    float* yr = y + row * ld_y;
    const float xm = m_io[row];
    const float ls = l_io[row];
    const float M = (xm == neg_inf()) ? 0.f : base2_of(xm, k);
    const float inv = (ls > 0.f) ? 1.0f / ls : 0.f;
    for (int64_t c = threadIdx.x; c < nchunks; c += kThreads) {
      float v[4];
      const int n = load_chunk<kVec>(xr, c, cols, v);
      if (kVec && n == 4 && (c + 1) * 4 <= cols) {
        st_stream(reinterpret_cast<float4*>(yr) + c,
                  make_float4(weight(v[0], M, k) * inv, weight(v[1], M, k) * inv,
                              weight(v[2], M, k) * inv, weight(v[3], M, k) * inv));
      } else {
        const int64_t base = c * (kVec ? 4 : 1);
        for (int e = 0; e < (kVec ? 4 : 1); ++e)
          if (base + e < cols) yr[base + e] = weight(v[e], M, k) * inv;
      }
    }
    __syncthreads();  // every thread has read m_io / l_io of this row
    if (threadIdx.x == 0) write_ml(xm, ls, k, row, m_io, l_io);
  }
}

// ---------------------------------------------------------------------------
// 16-bit rows (bf16 or fp16 in and out; m, l fp32). The same recurrence and
// merge; elements are widened to fp32 exactly, every weight is formed in fp32
// and y is rounded to the row's type once, to nearest even.
// kType: 1 = bf16, 2 = fp16.
// ---------------------------------------------------------------------------

template <int kType>
__device__ __forceinline__ float h16_lo(uint32_t w) {
  if (kType == 1) return __uint_as_float(w << 16);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
template <int kType>
__device__ __forceinline__ float h16_hi(uint32_t w) {
  if (kType == 1) return __uint_as_float(w & 0xffff0000u);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
template <int kType>
__device__ __forceinline__ float h16_one(uint16_t b) {
  return h16_lo<kType>(b);
}
// two fp32 -> one word of two 16-bit values (lo in the low half), RN
template <int kType>
__device__ __forceinline__ uint32_t h16_pack(float lo, float hi) {
  uint32_t w;
  if (kType == 1)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
  return w;
}
template <int kType>
__device__ __forceinline__ uint16_t h16_round(float f) {
  return static_cast<uint16_t>(h16_pack<kType>(f, 0.f) & 0xffffu);
}
// -inf twice, in the type's bits
template <int kType>
__device__ __forceinline__ uint32_t h16_neg_inf2() {
  return kType == 1 ? 0xff80ff80u : 0xfc00fc00u;
}

template <int kType>
__device__ __forceinline__ float max8(const uint4& v) {
  const float a = fmaxf(fmaxf(h16_lo<kType>(v.x), h16_hi<kType>(v.x)),
                        fmaxf(h16_lo<kType>(v.y), h16_hi<kType>(v.y)));
  const float b = fmaxf(fmaxf(h16_lo<kType>(v.z), h16_hi<kType>(v.z)),
                        fmaxf(h16_lo<kType>(v.w), h16_hi<kType>(v.w)));
  return fmaxf(a, b);
}
template <int kType>
__device__ __forceinline__ float sum8(const uint4& v, float M, const ScaleConsts& k) {
  const float a = (weight(h16_lo<kType>(v.x), M, k) + weight(h16_hi<kType>(v.x), M, k)) +
                  (weight(h16_lo<kType>(v.y), M, k) + weight(h16_hi<kType>(v.y), M, k));
  const float b = (weight(h16_lo<kType>(v.z), M, k) + weight(h16_hi<kType>(v.z), M, k)) +
                  (weight(h16_lo<kType>(v.w), M, k) + weight(h16_hi<kType>(v.w), M, k));
  return a + b;
}
template <int kType>
__device__ __forceinline__ uint32_t out2(uint32_t w, float M, float inv, const ScaleConsts& k) {
  return h16_pack<kType>(weight(h16_lo<kType>(w), M, k) * inv, weight(h16_hi<kType>(w), M, k) * inv);
}
template <int kType>
__device__ __forceinline__ uint4 out8(const uint4& v, float M, float inv, const ScaleConsts& k) {
  return make_uint4(out2<kType>(v.x, M, inv, k), out2<kType>(v.y, M, inv, k),
                    out2<kType>(v.z, M, inv, k), out2<kType>(v.w, M, inv, k));
}

// ---------------------------------------------------------------------------
// Grouped rows: one kernel for fp32, bf16 and fp16 rows that are 16-byte
// aligned and fit in registers. A group of TPR threads (8, 16, 32, 64, 128 or
// 256) owns one row at a time, so a CTA of 256 threads works on 256 / TPR
// rows and short rows keep as many bytes in flight per SM as long ones. A chunk is
// 16 bytes: 4 fp32 or 8 16-bit elements; each thread holds NV chunks.
//
// Per row: the thread's maximum, its weights 2^(x*c - M_t) (packed FMAs, one
// ex2 per element), the merge of the group's (max, sum) states in n-ary form
// (warp shuffles, then shared memory between the group's warps), then each
// weight scaled by 2^(M_t - M_row) / l_row and written once. With kPrefetch
// the grid is persistent and the next row's chunks are loaded into registers
// before the current row is reduced, so a group's loads overlap its own
// arithmetic and stores.
// kKind: 0 = fp32, 1 = bf16, 2 = fp16.
// ---------------------------------------------------------------------------

template <int kKind>
struct RowElem {
  static constexpr int kEpc = (kKind == 0) ? 4 : 8;  // elements per 16-byte chunk
  static constexpr int kSize = (kKind == 0) ? 4 : 2;  // bytes per element
};

template <int kKind>
__device__ __forceinline__ uint32_t neg_inf_word() {
  return (kKind == 0) ? 0xff800000u : h16_neg_inf2<kKind>();
}

// The 16-byte chunks of a row of n elements whose first element lies `s`
// elements past a 16-byte boundary (0 <= s < kEpc; 0 for an aligned row):
// chunk c holds the elements [c * kEpc - s, (c + 1) * kEpc - s), so every
// chunk sits on the 16-byte grid and ceil((n + s) / kEpc) chunks cover the
// row. Every chunk that holds an element of the row is loaded as one 16-byte
// access; in the partial first and last chunks the elements outside the row
// are then replaced by -inf. (Those extra bytes share a 16-byte granule, and
// so a page, with the row's own first or last element: the load reads bytes
// outside the row but never faults, and nothing outside the row is written.)
// Chunks wholly outside the row are not read.
template <int kKind>
__device__ __forceinline__ int phase_of(const void* row) {
  return static_cast<int>((reinterpret_cast<uintptr_t>(row) & 15u) / RowElem<kKind>::kSize);
}

// Rows on the 16-byte grid (phase 0): chunk c is elements [c * kEpc,
// (c + 1) * kEpc); nfull whole chunks, then a last chunk of `tail` elements.
template <int kKind>
__device__ __forceinline__ uint4 load_chunk16_grid(const char* xr, int c, int nfull, int tail) {
  if (c < nfull) return __ldcs(reinterpret_cast<const uint4*>(xr) + c);
  uint32_t wd[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) wd[h] = neg_inf_word<kKind>();
  if (c == nfull && tail) {
    if (kKind == 0) {
      const uint32_t* p = reinterpret_cast<const uint32_t*>(xr) + 4 * c;
#pragma unroll
      for (int e = 0; e < 3; ++e)
        if (e < tail) wd[e] = p[e];
    } else {
      const uint16_t* p = reinterpret_cast<const uint16_t*>(xr) + 8 * c;
#pragma unroll
      for (int e = 0; e < 7; ++e)
        if (e < tail)
          wd[e >> 1] = (e & 1) ? ((wd[e >> 1] & 0xffffu) | (uint32_t(p[e]) << 16))
                               : ((wd[e >> 1] & 0xffff0000u) | uint32_t(p[e]));
    }
  }
  return make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

template <int kKind>
__device__ __forceinline__ void store_chunk16_grid(char* yr, int c, int nfull, int tail, const uint4& o) {
  if (c < nfull) {
    __stcs(reinterpret_cast<uint4*>(yr) + c, o);
  } else if (c == nfull && tail) {
    const uint32_t wd[4] = {o.x, o.y, o.z, o.w};
    if (kKind == 0) {
      uint32_t* p = reinterpret_cast<uint32_t*>(yr) + 4 * c;
#pragma unroll
      for (int e = 0; e < 3; ++e)
        if (e < tail) p[e] = wd[e];
    } else {
      uint16_t* p = reinterpret_cast<uint16_t*>(yr) + 8 * c;
#pragma unroll
      for (int e = 0; e < 7; ++e)
        if (e < tail) p[e] = static_cast<uint16_t>((e & 1) ? (wd[e >> 1] >> 16) : (wd[e >> 1] & 0xffffu));
    }
  }
}

// Chunk c's 16-byte granule when it holds any element of the row, else all
// -inf (a predicated load: several of them issue back to back).
template <int kKind>
__device__ __forceinline__ uint4 ld_granule(const char* xr, int c, int n, int s) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  const int first = c * kEpc - s;
  const uint32_t ninf = neg_inf_word<kKind>();
  uint4 v = make_uint4(ninf, ninf, ninf, ninf);
  if (first < n && first + kEpc > 0) v = __ldcs(reinterpret_cast<const uint4*>(xr + first * kEsz));
  return v;
}

// A loaded granule of chunk c with the elements outside the row replaced by
// -inf (whole chunks pass unchanged).
template <int kKind>
__device__ __forceinline__ uint4 fix_granule(uint4 v, int c, int n, int s) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  const int first = c * kEpc - s;
  if (first >= 0 && first + kEpc <= n) return v;
  const uint32_t ninf = neg_inf_word<kKind>();
  uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < kEpc; ++e) {
    const int j = first + e;
    if (j < 0 || j >= n) {
      if (kKind == 0)
        wd[e] = ninf;
      else
        wd[e >> 1] = (e & 1) ? ((wd[e >> 1] & 0xffffu) | (ninf & 0xffff0000u))
                             : ((wd[e >> 1] & 0xffff0000u) | (ninf & 0xffffu));
    }
  }
  return make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

template <int kKind>
__device__ __forceinline__ uint4 load_chunk16(const char* xr, int c, int n, int s) {
  return fix_granule<kKind>(ld_granule<kKind>(xr, c, n, s), c, n, s);
}

// Chunk c of y (the same phase s as x's row), written for its elements in
// [0, n) only.
template <int kKind>
__device__ __forceinline__ void store_chunk16(char* yr, int c, int n, int s, const uint4& o) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  const int first = c * kEpc - s;
  if (first >= 0 && first + kEpc <= n) {
    __stcs(reinterpret_cast<uint4*>(yr + first * kEsz), o);
    return;
  }
  if (first >= n || first + kEpc <= 0) return;
  const uint32_t wd[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
  for (int e = 0; e < kEpc; ++e) {
    const int j = first + e;
    if (j >= 0 && j < n) {
      if (kKind == 0)
        reinterpret_cast<uint32_t*>(yr)[j] = wd[e];
      else
        reinterpret_cast<uint16_t*>(yr)[j] =
            static_cast<uint16_t>((e & 1) ? (wd[e >> 1] >> 16) : (wd[e >> 1] & 0xffffu));
    }
  }
}

// the chunk's elements widened to fp32 (exact), as pairs
template <int kKind>
__device__ __forceinline__ void unpack_chunk16(const uint4& v, float2* w /* [kEpc / 2] */) {
  if (kKind == 0) {
    w[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
    w[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
  } else {
    w[0] = make_float2(h16_lo<kKind>(v.x), h16_hi<kKind>(v.x));
    w[1] = make_float2(h16_lo<kKind>(v.y), h16_hi<kKind>(v.y));
    w[2] = make_float2(h16_lo<kKind>(v.z), h16_hi<kKind>(v.z));
    w[3] = make_float2(h16_lo<kKind>(v.w), h16_hi<kKind>(v.w));
  }
}

// the chunk's weights times f, in the row's type (one rounding for 16-bit)
template <int kKind>
__device__ __forceinline__ uint4 pack_chunk16(const float2* w, float2 f) {
  if (kKind == 0) {
    const float2 a = __fmul2_rn(w[0], f);
    const float2 b = __fmul2_rn(w[1], f);
    return make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(b.x),
                      __float_as_uint(b.y));
  } else {
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float2 q = __fmul2_rn(w[h], f);
      o[h] = h16_pack<kKind>(q.x, q.y);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__device__ __forceinline__ void group_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Merge of the (xm, ls) states of the TPR threads that own one row; returns
// the row state in all of them. The n-ary form of cta_merge: shuffles within
// the group, then (TPR > 32) the TPR / 32 warp states through sh[] (one entry
// per warp of the CTA) behind a barrier of the group's own threads. Every
// lane of a warp must call it (all shuffles use the full mask).
template <int TPR>
__device__ __forceinline__ void group_merge(float& xm, float& ls, const ScaleConsts& k,
                                            float2* sh, int g) {
  // a group narrower than a warp shuffles within its own aligned lanes
  constexpr int kTop = (TPR < 32 ? TPR : 32) / 2;
  float xw = xm;
#pragma unroll
  for (int off = kTop; off > 0; off >>= 1) xw = fmaxf(xw, __shfl_xor_sync(0xffffffffu, xw, off));
  float lw = (xm == neg_inf()) ? 0.f : ls * ex2(base2_of(xm, k) - base2_of(xw, k));
#pragma unroll
  for (int off = kTop; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
  if (TPR <= 32) {
    xm = xw;
    ls = lw;
    return;
  }
  constexpr int kW = TPR / 32;
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = make_float2(xw, lw);
  if (TPR == kThreads)
    __syncthreads();
  else
    group_barrier(1 + g, TPR);
  const float2* s = sh + g * kW;
  float x = s[0].x;
#pragma unroll
  for (int w = 1; w < kW; ++w) x = fmaxf(x, s[w].x);
  float l = 0.f;
  if (x != neg_inf()) {
    const float M = base2_of(x, k);
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const float2 e = s[w];
      if (e.x != neg_inf()) l += e.y * ex2(base2_of(e.x, k) - M);
    }
  }
  xm = x;
  ls = l;
}

// kExtra: one more chunk slot per thread (NV + 1), for rows off the 16-byte
// grid, which need one chunk more than an aligned row; only the group's
// first thread ever finds its extra chunk inside the row.
template <int kKind, int TPR, int NV, bool kPrefetch, int kMinBlocks, bool kExtra>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
softmax_rows_grouped_kernel(const void* __restrict__ x, void* __restrict__ y,
                            float* __restrict__ m_out, float* __restrict__ l_out, int64_t rows,
                            int cols, int64_t ld_x, int64_t ld_y, ScaleConsts k) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  constexpr int kGroups = kThreads / TPR;
  constexpr int kSlots = NV + (kExtra ? 1 : 0);
  // two sets of per-warp states: a warp may start the next row's merge
  // while the group's slower warps still read this row's, and a set is not
  // written again until every warp of the group has passed the barrier
  // of the row in between
  __shared__ float2 sh[2][kWarps];
  const int tid = threadIdx.x;
  const int g = tid / TPR;
  const int t = tid % TPR;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kGroups;
  // Groups narrower than a warp share their warp's shuffles, so the warp
  // walks its rows together: the loop runs on the row of the warp's first
  // group, and a group whose own row is past the end takes part as an empty
  // row (no loads or stores).
  constexpr int kPerWarp = (TPR < 32) ? 32 / TPR : 1;
  const int lead = g % kPerWarp;
  const uint4 pad = make_uint4(neg_inf_word<kKind>(), neg_inf_word<kKind>(), neg_inf_word<kKind>(),
                               neg_inf_word<kKind>());
  int64_t wrow = static_cast<int64_t>(blockIdx.x) * kGroups + g - lead;
  const char* xb = static_cast<const char*>(x);
  char* yb = static_cast<char*>(y);

  // Rows on the grid use the plain chunking; rows off it (kExtra) load each
  // granule first and mask the partial chunks after, so that a thread's
  // loads issue back to back.
  const int nfull = cols / kEpc;
  const int tail = cols % kEpc;
  auto load = [&](const char* xr, int c, int s) {
    if constexpr (kExtra)
      return ld_granule<kKind>(xr, c, cols, s);
    else
      return load_chunk16_grid<kKind>(xr, c, nfull, tail);
  };
  auto fix = [&](const uint4& v, int c, int s) {
    if constexpr (kExtra)
      return fix_granule<kKind>(v, c, cols, s);
    else
      return v;
  };
  uint4 nx[kSlots];
  int nx_s = 0;  // the phase of the row held in nx
  if (kPrefetch && wrow + lead < rows) {
    const char* xr = xb + (wrow + lead) * ld_x * kEsz;
    nx_s = phase_of<kKind>(xr);
#pragma unroll
    for (int i = 0; i < kSlots; ++i) nx[i] = load(xr, t + i * TPR, nx_s);
  }
  int buf = 0;
  for (; wrow < rows; wrow += stride) {
    const int64_t row = wrow + lead;
    const bool active = row < rows;
    float2 w[kSlots][kEpc / 2];
    if (kPrefetch) {
#pragma unroll
      for (int i = 0; i < kSlots; ++i)
        unpack_chunk16<kKind>(active ? fix(nx[i], t + i * TPR, nx_s) : pad, w[i]);
      const int64_t next = row + stride;
      if (next < rows) {
        const char* xr = xb + next * ld_x * kEsz;
        nx_s = phase_of<kKind>(xr);
#pragma unroll
        for (int i = 0; i < kSlots; ++i) nx[i] = load(xr, t + i * TPR, nx_s);
      }
    } else {
      const char* xr = xb + row * ld_x * kEsz;
      const int s = phase_of<kKind>(xr);
      uint4 v[kSlots];
#pragma unroll
      for (int i = 0; i < kSlots; ++i) v[i] = active ? load(xr, t + i * TPR, s) : pad;
#pragma unroll
      for (int i = 0; i < kSlots; ++i) unpack_chunk16<kKind>(fix(v[i], t + i * TPR, s), w[i]);
    }
    float xa = neg_inf(), xc = neg_inf();
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
#pragma unroll
      for (int h = 0; h < kEpc / 2; h += 2) {
        xa = fmax3(xa, w[i][h].x, w[i][h].y);
        if (h + 1 < kEpc / 2) xc = fmax3(xc, w[i][h + 1].x, w[i][h + 1].y);
      }
    }
    float xm = fmaxf(xa, xc);
    const float Mt = (xm == neg_inf()) ? 0.f : base2_of(xm, k);
    const float2 negM = make_float2(-Mt, -Mt);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
#pragma unroll
      for (int h = 0; h < kEpc / 2; ++h) {
        w[i][h] = weight2(w[i][h], negM, k);
        acc = __fadd2_rn(acc, w[i][h]);
      }
    }
    float ls = acc.x + acc.y;
    const float xm_t = xm;
    group_merge<TPR>(xm, ls, k, sh[buf], g);
    float f = 0.f;
    if (xm_t != neg_inf() && ls > 0.f)
      f = ex2(base2_of(xm_t, k) - base2_of(xm, k)) * (1.0f / ls);
    const float2 f2 = make_float2(f, f);
    if (active) {
      char* yr = yb + row * ld_y * kEsz;
      const int s = phase_of<kKind>(yr);  // x's row has the same phase
#pragma unroll
      for (int i = 0; i < kSlots; ++i) {
        if constexpr (kExtra)
          store_chunk16<kKind>(yr, t + i * TPR, cols, s, pack_chunk16<kKind>(w[i], f2));
        else
          store_chunk16_grid<kKind>(yr, t + i * TPR, nfull, tail, pack_chunk16<kKind>(w[i], f2));
      }
      if (t == 0) write_ml(xm, ls, k, row, m_out, l_out);
    }
    buf ^= 1;
  }
}

// ---------------------------------------------------------------------------
// Cluster-resident rows: rows too long for registers (more than 16384
// elements) but short enough to fit in the shared memory of a thread-block
// cluster of C <= 8 CTAs. CTA r of a cluster holds slice r of the row, copied
// in by bulk asynchronous copies; each CTA reduces its slice to a (max, sum)
// state, the CTAs exchange their states through distributed shared memory and
// merge them (the merge identity of partial results), and each CTA then
// writes its slice once. One HBM read and one write per element, where the
// streaming kernel reads the row twice.
// ---------------------------------------------------------------------------

// Issue the copies of one row's slice (n elements at xr, phase s) into
// `buf_a` (thread 0 only), in the chunks of load_chunk16: the whole 16-byte
// chunks by bulk copies that complete on `bar_a`, the partial first and last
// chunks by plain loads, padded with -inf. The barrier is told to expect
// `extra` bytes more than are copied (0 but in the test hook, which makes the
// wait run out).
template <int kKind>
__device__ __forceinline__ void issue_slice(const char* xr, uint4* buf, uint32_t buf_a, uint32_t bar_a,
                                            int n, int s, uint32_t extra) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  const int nch = (n > 0) ? (n + s + kEpc - 1) / kEpc : 0;
  const int ca = (s == 0) ? 0 : 1;   // the first whole chunk
  const int cb = (n + s) / kEpc;     // one past the last whole chunk
  const uint32_t bulk = (n > 0 && cb > ca) ? static_cast<uint32_t>(cb - ca) * 16u : 0u;
  // the buffer's previous contents were last touched through the generic
  // proxy; order that before the copies' asynchronous writes
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (bulk + extra > 0) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_a),
                 "r"(bulk + extra)
                 : "memory");
    const char* src = xr + (ca * kEpc - s) * kEsz;  // 16-byte aligned
    const uint32_t dst = buf_a + static_cast<uint32_t>(ca) * 16u;
    for (uint32_t off = 0; off < bulk; off += kClPiece) {
      const uint32_t size = (bulk - off < kClPiece) ? (bulk - off) : kClPiece;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
              "r"(dst + off), "l"(src + off), "r"(size), "r"(bar_a)
          : "memory");
    }
  } else {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_a) : "memory");
  }
  if (n > 0) {
    if (s != 0) buf[0] = load_chunk16<kKind>(xr, 0, n, s);
    if (cb < nch && !(s != 0 && cb == 0)) buf[cb] = load_chunk16<kKind>(xr, cb, n, s);
  }
}

// kDouble: two slice buffers; the next row's copies are issued as soon as
// the current row's have landed, so they are in flight while the current row
// is reduced and written.
template <int kKind, bool kDouble>
__global__ void __launch_bounds__(kClThreads, 2)
softmax_rows_cluster_kernel(const void* __restrict__ x, void* __restrict__ y,
                            float* __restrict__ m_out, float* __restrict__ l_out, int64_t rows,
                            int64_t cols, int64_t ld_x, int64_t ld_y, ScaleConsts k,
                            int slice_elems, unsigned int* err, uint32_t fault_tx,
                            uint64_t timeout_ns) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  extern __shared__ __align__(128) uint4 slices[];  // this CTA's slice buffer(s), 16-byte chunks
  __shared__ float2 wstate[kClWarps];
  __shared__ float2 cstate[2][kClMaxCtas];         // the cluster's CTA states, by row parity
  __shared__ __align__(8) uint64_t bars[2];

  const int tid = threadIdx.x;
  const uint32_t C = cluster_size();
  const uint32_t rank = cluster_rank();
  const int64_t lo = static_cast<int64_t>(rank) * slice_elems;
  const int64_t left = cols - lo;
  const int n = static_cast<int>(left <= 0 ? 0 : (left < slice_elems ? left : slice_elems));
  // a slice whose rows are not 16-byte aligned spans one chunk more
  const int stride_chunks = (slice_elems / kEpc + 1 + 7) / 8 * 8;  // second buffer 128-byte aligned
  const int64_t row0 = cluster_id();
  const int64_t rstep = cluster_count();
  const char* xb = static_cast<const char*>(x);

  if (tid == 0) {
    for (int b = 0; b < (kDouble ? 2 : 1); ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[b])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // every CTA of the cluster has started (its shared memory may be written
  // by peers from here on) and the barriers' initialisation is visible
  cluster_sync_all();
  if (kDouble && tid == 0 && row0 < rows) {
    const char* xr0 = xb + (row0 * ld_x + lo) * kEsz;
    issue_slice<kKind>(xr0, slices, smem_u32(slices), smem_u32(&bars[0]), n, phase_of<kKind>(xr0),
                       fault_tx);
  }

  uint32_t parity = 0u;  // bit b: the phase parity to wait for on buffer b
  int sbuf = 0;  // cstate set
  int it = 0;
  bool live = true;  // false once this thread gave up on a wait: no more waits or copies
  for (int64_t row = row0; row < rows; row += rstep, ++it) {
    const int b = kDouble ? (it & 1) : 0;
    uint4* slice = slices + b * stride_chunks;
    const uint32_t bar_a = smem_u32(&bars[b]);
    const char* xr = xb + (row * ld_x + lo) * kEsz;
    char* yr = static_cast<char*>(y) + (row * ld_y + lo) * kEsz;
    const int s = phase_of<kKind>(xr);  // y's slice has the same phase
    const int nch = (n > 0) ? (n + s + kEpc - 1) / kEpc : 0;
    if (!kDouble && tid == 0 && live)
      issue_slice<kKind>(xr, slice, smem_u32(slice), bar_a, n, s, it == 0 ? fault_tx : 0u);
    if (live) live = mbar_wait_bounded(bar_a, (parity >> b) & 1u, err, timeout_ns);
    parity ^= 1u << b;
    __syncthreads();  // the tail chunk, written by thread 0
    if (kDouble && tid == 0 && live && row + rstep < rows) {
      // the other buffer was read out before the end of the previous row
      uint4* other = slices + (b ^ 1) * stride_chunks;
      const char* xn = xb + ((row + rstep) * ld_x + lo) * kEsz;
      issue_slice<kKind>(xn, other, smem_u32(other), smem_u32(&bars[b ^ 1]), n, phase_of<kKind>(xn), 0u);
    }

    // The thread's (max, sum) over its chunks, by the online recurrence:
    // each step loads kClUnroll chunks (tid, tid + T, ...), takes their
    // maximum, rescales the running sum once if it rose, then adds the
    // step's weights relative to the running maximum.
    const uint4 pad = make_uint4(neg_inf_word<kKind>(), neg_inf_word<kKind>(), neg_inf_word<kKind>(),
                                 neg_inf_word<kKind>());
    float xm = neg_inf();
    float2 negM = make_float2(0.f, 0.f);
    float2 acc = make_float2(0.f, 0.f);
    for (int c0 = tid; c0 < nch; c0 += kClThreads * kClUnroll) {
      float2 w[kClUnroll][kEpc / 2];
#pragma unroll
      for (int u = 0; u < kClUnroll; ++u)
        unpack_chunk16<kKind>((c0 + u * kClThreads < nch) ? slice[c0 + u * kClThreads] : pad, w[u]);
      float cm = xm;
#pragma unroll
      for (int u = 0; u < kClUnroll; ++u)
#pragma unroll
        for (int h = 0; h < kEpc / 2; ++h) cm = fmax3(cm, w[u][h].x, w[u][h].y);
      if (cm != xm) {  // a larger (finite) maximum: rescale what is summed so far
        const float Mn = base2_of(cm, k);
        if (xm != neg_inf()) {
          const float r = ex2(-negM.x - Mn);
          acc = __fmul2_rn(acc, make_float2(r, r));
        }
        xm = cm;
        negM = make_float2(-Mn, -Mn);
      }
#pragma unroll
      for (int u = 0; u < kClUnroll; ++u)
#pragma unroll
        for (int h = 0; h < kEpc / 2; ++h) acc = __fadd2_rn(acc, weight2(w[u][h], negM, k));
    }
    float ls = acc.x + acc.y;

    // the CTA's state: warp maxima and scaled sums by shuffles, then the
    // warp states through shared memory
    float xw = xm;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) xw = fmaxf(xw, __shfl_xor_sync(0xffffffffu, xw, off));
    float lw = (xm == neg_inf()) ? 0.f : ls * ex2(base2_of(xm, k) - base2_of(xw, k));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
    if ((tid & 31) == 0) wstate[tid >> 5] = make_float2(xw, lw);
    __syncthreads();
    float2 st = merge_states_warp(wstate, kClWarps, k);
    if (C > 1) {
      if (tid == 0)
        for (uint32_t r = 0; r < C; ++r) st_peer_f2(&cstate[sbuf][rank], r, st.x, st.y);
      cluster_sync_warp0_wrote();
      st = merge_states_warp(cstate[sbuf], static_cast<int>(C), k);
      sbuf ^= 1;
    }
    xm = st.x;
    ls = st.y;

    // y = 2^(x*c - M_row) / l, formed again from x (an empty row gives 0)
    const bool nonempty = (xm != neg_inf()) && ls > 0.f;
    const float Mr = nonempty ? base2_of(xm, k) : 0.f;
    const float2 negMr = make_float2(-Mr, -Mr);
    const float inv = nonempty ? 1.0f / ls : 0.f;
    const float2 f2 = make_float2(inv, inv);
    for (int c0 = tid; c0 < nch; c0 += kClThreads * kClUnroll) {
      uint4 v[kClUnroll];
#pragma unroll
      for (int u = 0; u < kClUnroll; ++u) v[u] = (c0 + u * kClThreads < nch) ? slice[c0 + u * kClThreads] : pad;
#pragma unroll
      for (int u = 0; u < kClUnroll; ++u) {
        if (c0 + u * kClThreads < nch) {
          float2 w[kEpc / 2];
          unpack_chunk16<kKind>(v[u], w);
#pragma unroll
          for (int h = 0; h < kEpc / 2; ++h) w[h] = weight2(w[h], negMr, k);
          store_chunk16<kKind>(yr, c0 + u * kClThreads, n, s, pack_chunk16<kKind>(w, f2));
        }
      }
    }
    if (rank == 0 && tid == 0) write_ml(xm, ls, k, row, m_out, l_out);
    __syncthreads();  // the slice is read out before its buffer is refilled
  }
}

// Long or unaligned 16-bit rows: the recurrence over the row as it streams
// (8-element chunks when aligned, single elements otherwise), the CTA merge,
// then a second read of the row for the write (2 reads + 1 write).
template <int kType, bool kVec>
__global__ void __launch_bounds__(kThreads)
softmax_rows16_stream_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
                             float* __restrict__ m_out, float* __restrict__ l_out, int64_t rows,
                             int64_t cols, int64_t ld_x, int64_t ld_y, ScaleConsts k,
                             int64_t slice_chunks) {
  __shared__ float2 sh[kWarps];
  __shared__ float2 cstate[2][kClMaxCtas];
  constexpr int W = kVec ? 8 : 1;
  const int64_t nchunks = (cols + W - 1) / W;
  const int tid = threadIdx.x;
  // in a cluster of C CTAs, CTA r streams chunks [r * slice, (r + 1) * slice)
  const uint32_t C = cluster_size();
  const uint32_t rank = cluster_rank();
  const int64_t c_lo = static_cast<int64_t>(rank) * slice_chunks;
  const int64_t c_hi = (c_lo + slice_chunks < nchunks) ? c_lo + slice_chunks : nchunks;
  if (C > 1) cluster_sync_all();  // every peer has started before any writes to it
  int sbuf = 0;
  for (int64_t row = cluster_id(); row < rows; row += cluster_count()) {
    const uint16_t* xr = x + row * ld_x;
    uint16_t* yr = y + row * ld_y;
    float xm = neg_inf(), ls = 0.f;
    for (int64_t c = c_lo + tid; c < c_hi; c += kThreads) {
      if (kVec && (c + 1) * W <= cols) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr) + c);
        const float xn = fmaxf(xm, max8<kType>(v));
        if (xn == neg_inf()) continue;  // nothing visible yet: no -inf - -inf
        const float Mn = base2_of(xn, k);
        const float corr = (xm == neg_inf()) ? 0.f : ex2(base2_of(xm, k) - Mn);
        ls = ls * corr + sum8<kType>(v, Mn, k);
        xm = xn;
      } else {
        for (int64_t j = c * W; j < cols && j < (c + 1) * W; ++j) {
          const float xv = h16_one<kType>(xr[j]);
          const float xn = fmaxf(xm, xv);
          if (xn == neg_inf()) continue;
          const float Mn = base2_of(xn, k);
          const float corr = (xm == neg_inf()) ? 0.f : ex2(base2_of(xm, k) - Mn);
          ls = ls * corr + weight(xv, Mn, k);
          xm = xn;
        }
      }
    }
    cta_merge(xm, ls, k, sh);
    if (C > 1) {  // the cluster's CTA states, through distributed shared memory
      if (tid == 0)
        for (uint32_t r = 0; r < C; ++r) st_peer_f2(&cstate[sbuf][rank], r, xm, ls);
      cluster_sync_warp0_wrote();
      const float2 st = merge_states_warp(cstate[sbuf], static_cast<int>(C), k);
      xm = st.x;
      ls = st.y;
      sbuf ^= 1;
    }
    const float M = (xm == neg_inf()) ? 0.f : base2_of(xm, k);
    const float inv = (ls > 0.f) ? 1.0f / ls : 0.f;
    for (int64_t c = c_lo + tid; c < c_hi; c += kThreads) {
      if (kVec && (c + 1) * W <= cols) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr) + c);
        __stcs(reinterpret_cast<uint4*>(yr) + c, out8<kType>(v, M, inv, k));
      } else {
        for (int64_t j = c * W; j < cols && j < (c + 1) * W; ++j)
          yr[j] = h16_round<kType>(weight(h16_one<kType>(xr[j]), M, k) * inv);
      }
    }
    if (rank == 0 && tid == 0) write_ml(xm, ls, k, row, m_out, l_out);
    __syncthreads();
  }
}

int sm_count() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

int grid_for(int64_t rows, int ctas_per_sm) {
  const int64_t cap = static_cast<int64_t>(sm_count()) * ctas_per_sm * 64;
  return static_cast<int>(rows < cap ? rows : cap);
}

}  // namespace

namespace {

// c (> 0) as hi + lo with hi the float below c and lo = c - hi > 0, both
// positive (the device code relies on it for masked entries, see weight()).
// Where c is a float itself, hi is the float just below it and lo that
// spacing; lo is never 0 (for c below the smallest normal it is set to the
// smallest subnormal, an error of 2^-149 in c).
void split_positive(double c, float* hi, float* lo) {
  float h = static_cast<float>(c);
  if (static_cast<double>(h) >= c) h = std::nextafter(h, 0.0f);
  float l = static_cast<float>(c - static_cast<double>(h));
  if (!(l > 0.0f)) l = std::numeric_limits<float>::denorm_min();
  *hi = h;
  *lo = l;
}

ScaleConsts make_consts(float scale) {
  const double kLog2e = 1.4426950408889634074;
  ScaleConsts k;
  k.scale = scale;
  split_positive(static_cast<double>(scale) * kLog2e, &k.c_hi, &k.c_lo);
  split_positive(kLog2e, &k.e_hi, &k.e_lo);
  return k;
}

}  // namespace

// Launch of a streaming kernel (`width` elements per chunk): a CTA per row
// while the rows fill the GPU (eight CTAs per SM); with fewer rows each row is
// cut into C contiguous slices, one per CTA of a cluster of C <= 8, as long
// as every CTA keeps at least 16 chunks per thread. The slices' states meet
// through distributed shared memory. A failed cluster launch falls back to a
// CTA per row.
template <typename T, typename Kernel>
void launch_stream(Kernel kernel, const T* x, T* y, float* m, float* l, int64_t rows, int64_t cols,
                   int64_t ld_x, int64_t ld_y, const ScaleConsts& k, int width, cudaStream_t stream) {
  const int64_t nchunks = (cols + width - 1) / width;
  const int64_t resident = static_cast<int64_t>(sm_count()) * 8;
  int64_t c = 1;
  if (rows < resident) {
    c = resident / rows;
    const int64_t by_work = nchunks / (int64_t(kThreads) * 16);
    if (c > by_work) c = by_work;
    if (c > kClMaxCtas) c = kClMaxCtas;
    if (c < 1) c = 1;
  }
  if (c > 1) {
    const int64_t slice = (nchunks + c - 1) / c;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned int>(c);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.gridDim = dim3(static_cast<unsigned int>(rows * c), 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, x, y, m, l, rows, cols, ld_x, ld_y, k, slice) == cudaSuccess)
      return;
    cudaGetLastError();
  }
  kernel<<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, cols, ld_x, ld_y, k, nchunks);
}

// Launch of softmax_rows_grouped_kernel: persistent (one wave of kMinBlocks
// CTAs per SM) when it prefetches, else up to 64 waves of a grid-stride loop.
template <int kKind, int TPR, int NV, bool kPrefetch, int kMinBlocks, bool kExtra = false>
void launch_grouped(const void* x, void* y, float* m, float* l, int64_t rows, int cols,
                    int64_t ld_x, int64_t ld_y, const ScaleConsts& k, cudaStream_t stream) {
  constexpr int kGroups = kThreads / TPR;
  const int64_t need = (rows + kGroups - 1) / kGroups;
  const int64_t cap = static_cast<int64_t>(sm_count()) * kMinBlocks * (kPrefetch ? 1 : 64);
  const int g = static_cast<int>(need < cap ? need : cap);
  softmax_rows_grouped_kernel<kKind, TPR, NV, kPrefetch, kMinBlocks, kExtra>
      <<<g, kThreads, 0, stream>>>(x, y, m, l, rows, cols, ld_x, ld_y, k);
}

// Every row of x starts at the same offset from a 16-byte boundary as the
// same row of y (the chunks of load_chunk16 then line up for both).
bool same_phase(const void* x, const void* y, int64_t ld_x, int64_t ld_y, int esz) {
  const int64_t dx = static_cast<int64_t>(reinterpret_cast<uintptr_t>(x) & 15u);
  const int64_t dy = static_cast<int64_t>(reinterpret_cast<uintptr_t>(y) & 15u);
  return dx == dy && ((ld_x - ld_y) * esz) % 16 == 0;
}

struct ClusterCfg {
  int ctas;
  int slice_elems;
  size_t smem;
};

template <int kKind, bool kDouble>
cudaLaunchConfig_t cluster_launch_cfg(const ClusterCfg& cc, cudaLaunchAttribute* attr,
                                      cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cc.ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kClThreads, 1, 1);
  cfg.gridDim = dim3(cc.ctas, 1, 1);
  cfg.dynamicSmemBytes = cc.smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of `ctas` CTAs that can be resident at once (0 when none can),
// cached per device, cluster size and shared-memory size in 8 KB steps.
template <int kKind, bool kDouble>
int resident_clusters(const ClusterCfg& cc) {
  static std::atomic<int> cache[64][kClMaxCtas + 1][32];  // resident + 1; 0 = not asked yet
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t kb8 = (cc.smem + 8191) >> 13;
  const bool cached = dev >= 0 && dev < 64 && kb8 < 32;
  if (cached) {
    const int v = cache[dev][cc.ctas][kb8].load();
    if (v > 0) return v - 1;
  }
  auto kernel = softmax_rows_cluster_kernel<kKind, kDouble>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 210 << 10) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_launch_cfg<kKind, kDouble>(cc, attr, nullptr);
  int resident = 0;
  if (cudaOccupancyMaxActiveClusters(&resident, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    resident = 0;
  }
  if (cached) cache[dev][cc.ctas][kb8].store(resident + 1);
  return resident;
}

// The cluster for a row of `cols` elements: slices of at most `cap` bytes
// (in each of two buffers when kDouble), at most kClMaxCtas of them, and
// among the cluster sizes that hold the row the one that keeps the most SMs
// busy (clusters resident at once x CTAs per cluster; a GPC's SMs need not
// divide into clusters evenly), the smallest on a tie.
template <int kKind, bool kDouble>
bool pick_cluster(int64_t cols, int64_t cap, int max_ctas, ClusterCfg* out) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  if (cap <= 0) return false;
  const int64_t cmin = (cols * kEsz + cap - 1) / cap;
  int best_used = 0;
  for (int64_t c = cmin < 1 ? 1 : cmin; c <= max_ctas; ++c) {
    int64_t per = (cols + c - 1) / c;
    per = (per + kEpc - 1) / kEpc * kEpc;
    if (per * kEsz > cap) continue;
    const int64_t chunks = per / kEpc + 1;  // + 1: a slice not 16-byte aligned spans one more
    const int64_t stride = (chunks + 7) / 8 * 8;
    ClusterCfg cc{static_cast<int>(c), static_cast<int>(per),
                  static_cast<size_t>((kDouble ? stride + chunks : chunks) * 16)};
    const int used = resident_clusters<kKind, kDouble>(cc) * cc.ctas;
    if (used > best_used) {
      best_used = used;
      *out = cc;
    }
  }
  return best_used > 0;
}

// Launch of softmax_rows_cluster_kernel, as many clusters as can be resident
// at once (each loops over its rows).
template <int kKind, bool kDouble>
bool launch_cluster_rows_as(const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                            int64_t ld_x, int64_t ld_y, const ScaleConsts& k, const ClusterCfg& cc,
                            unsigned int* err, const RowsFault& fault, cudaStream_t stream) {
  // the chunks (and the bulk copies of the whole ones) sit on the 16-byte
  // grid: x's and y's rows in step, elements aligned, slices whole chunks
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  if (!same_phase(x, y, ld_x, ld_y, kEsz) || (reinterpret_cast<uintptr_t>(x) % kEsz) != 0 ||
      cc.slice_elems % kEpc != 0)
    return false;
  const int resident = resident_clusters<kKind, kDouble>(cc);
  if (resident < 1) return false;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_launch_cfg<kKind, kDouble>(cc, attr, stream);
  const int64_t nclusters = rows < resident ? rows : resident;
  cfg.gridDim = dim3(static_cast<unsigned int>(nclusters * cc.ctas), 1, 1);
  const int64_t c64 = cols;
  const uint64_t timeout = fault.timeout_ns > 0 ? static_cast<uint64_t>(fault.timeout_ns) : kClTimeoutNs;
  return cudaLaunchKernelEx(&cfg, softmax_rows_cluster_kernel<kKind, kDouble>, x, y, m, l, rows, c64,
                            ld_x, ld_y, k, cc.slice_elems, err, fault.extra_tx, timeout) == cudaSuccess;
}

// Rows held in a cluster's shared memory. A row of at most kClDoubleCap
// bytes takes one CTA with two buffers (its next row's copies in flight
// while it reduces the current one); a longer row takes one buffer of at
// most 200 KB in each of up to eight CTAs. False, launching nothing, when the
// row is longer. (Measured on the GB300 with 2^28-element matrices: two
// buffers won only when the row fit one CTA; for longer rows the extra CTAs
// they need cost more than the overlap gained.)
template <int kKind>
bool launch_cluster_rows(const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                         int64_t ld_x, int64_t ld_y, const ScaleConsts& k, unsigned int* err,
                         const RowsFault& fault, cudaStream_t stream) {
  ClusterCfg cc;
  if (pick_cluster<kKind, true>(cols, kClDoubleCap, 1, &cc))
    return launch_cluster_rows_as<kKind, true>(x, y, m, l, rows, cols, ld_x, ld_y, k, cc, err, fault,
                                               stream);
  if (pick_cluster<kKind, false>(cols, kClSingleCap, kClMaxCtas, &cc))
    return launch_cluster_rows_as<kKind, false>(x, y, m, l, rows, cols, ld_x, ld_y, k, cc, err, fault,
                                                stream);
  return false;
}

cudaError_t launch_softmax_rows(const float* x, float* y, float* m, float* l, int64_t rows,
                                int64_t cols, int64_t ld_x, int64_t ld_y, float scale,
                                unsigned int* err_word, const RowsFault& fault, cudaStream_t stream) {
  const ScaleConsts k = make_consts(scale);

  const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                   (ld_x & 3) == 0 && (ld_y & 3) == 0;
  if (!vec) {
    // Rows off the 16-byte grid, x and y in step: 16-byte chunks on the grid
    // with the partial first and last chunks masked, in the configuration of
    // an aligned row of the same length plus one chunk slot per thread.
    // Otherwise stream.
    const int64_t chunks = (cols + 3) / 4;
    const int c = static_cast<int>(cols);
    if (!same_phase(x, y, ld_x, ld_y, 4)) {
      launch_stream(softmax_rows_stream_kernel<false>, x, y, m, l, rows, cols, ld_x, ld_y, k, 1, stream);
    } else if (chunks <= 8) {
      launch_grouped<0, 8, 1, true, 4, true>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    } else if (chunks <= 16) {
      launch_grouped<0, 16, 1, true, 4, true>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    } else if (chunks <= 32) {
      launch_grouped<0, 32, 1, true, 4, true>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    } else if (chunks <= 64) {
      launch_grouped<0, 32, 2, false, 6, true>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    } else if (chunks <= 128) {
      launch_grouped<0, 32, 4, false, 4, true>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    } else if (chunks <= 256) {
      launch_grouped<0, 64, 4, false, 4, true>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    } else if (chunks <= 512) {
      launch_grouped<0, 128, 4, false, 4, true>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    } else if (chunks <= 1024) {
      launch_grouped<0, 256, 4, false, 4, true>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    } else if (chunks <= 2048) {
      launch_grouped<0, 256, 8, false, 2, true>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    } else if (!launch_cluster_rows<0>(x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, stream)) {
      launch_stream(softmax_rows_stream_kernel<false>, x, y, m, l, rows, cols, ld_x, ld_y, k, 1, stream);
    }
    return cudaGetLastError();
  }
  const int64_t chunks = (cols + 3) / 4;
  const int nv = static_cast<int>((chunks + kThreads - 1) / kThreads);
  const int c = static_cast<int>(cols);
  // Rows of up to 2048 elements: several rows per CTA, each thread holding
  // up to four 16-byte chunks (configurations measured on the GB300 at
  // 2^28 elements per matrix; prefetching helped only the shortest rows).
  if (chunks <= 8) {
    launch_grouped<0, 8, 1, true, 8>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 16) {
    launch_grouped<0, 16, 1, true, 8>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 32) {
    launch_grouped<0, 32, 1, true, 8>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 64) {
    launch_grouped<0, 32, 2, false, 6>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 128) {
    launch_grouped<0, 32, 4, false, 6>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 256) {
    launch_grouped<0, 64, 4, false, 6>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 512) {
    launch_grouped<0, 128, 4, false, 5>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (nv <= 4) {
    softmax_rows_reg_kernel<4><<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
  } else if (nv <= 8) {
    softmax_rows_reg_kernel<8><<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
  } else if (nv <= 16) {
    softmax_rows_reg_kernel<16><<<grid_for(rows, 2), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
  } else {
    if (!launch_cluster_rows<0>(x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, stream))
      launch_stream(softmax_rows_stream_kernel<true>, x, y, m, l, rows, cols, ld_x, ld_y, k, 4, stream);
  }
  return cudaGetLastError();
}

// The 16-bit configurations by the aligned chunk count of a row; kExtra
// adds the slot that a row off the 16-byte grid needs.
template <int kType, bool kExtra>
void dispatch_rows16_table(const uint16_t* x, uint16_t* y, float* m, float* l, int64_t rows,
                           int64_t cols, int64_t chunks, int64_t ld_x, int64_t ld_y,
                           const ScaleConsts& k, unsigned int* err_word, const RowsFault& fault,
                           cudaStream_t stream) {
  const int c = static_cast<int>(cols);
  // Rows of up to 16384 elements: persistent CTAs with the next row's chunks
  // prefetched into registers (the widening of fp16 costs a conversion per
  // element, and without the prefetch that arithmetic stalled the loads);
  // 256 / TPR rows per CTA for rows of up to 4096 elements (groups of 8 and
  // 16 threads, without the prefetch, for rows of up to 128).
  if (chunks <= 8) {
    launch_grouped<kType, 8, 1, false, kExtra ? 4 : 8, kExtra>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 16) {
    launch_grouped<kType, 16, 1, false, kExtra ? 4 : 8, kExtra>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 32) {
    launch_grouped<kType, 32, 1, true, kExtra ? 4 : 6, kExtra>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 64) {
    launch_grouped<kType, 32, 2, true, kExtra ? 3 : 5, kExtra>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 128) {
    launch_grouped<kType, 32, 4, true, kExtra ? 2 : 3, kExtra>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 256) {
    launch_grouped<kType, 64, 4, true, kExtra ? 2 : 3, kExtra>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 512) {
    launch_grouped<kType, 128, 4, true, kExtra ? 2 : 3, kExtra>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 1024) {
    launch_grouped<kType, 256, 4, true, kExtra ? 2 : 3, kExtra>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (chunks <= 2048) {
    launch_grouped<kType, 256, 8, kExtra ? false : true, 2, kExtra>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  } else if (!launch_cluster_rows<kType>(x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, stream)) {
    // 16-byte accesses only for rows on the grid
    launch_stream(softmax_rows16_stream_kernel<kType, !kExtra>, x, y, m, l, rows, cols, ld_x, ld_y, k,
                  kExtra ? 1 : 8, stream);
  }
}

template <int kType>
void dispatch_rows16(const uint16_t* x, uint16_t* y, float* m, float* l, int64_t rows,
                     int64_t cols, int64_t ld_x, int64_t ld_y, const ScaleConsts& k,
                     unsigned int* err_word, const RowsFault& fault, cudaStream_t stream) {
  const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                   (ld_x & 7) == 0 && (ld_y & 7) == 0;
  if (!vec && !same_phase(x, y, ld_x, ld_y, 2)) {
    launch_stream(softmax_rows16_stream_kernel<kType, false>, x, y, m, l, rows, cols, ld_x, ld_y, k, 1, stream);
    return;
  }
  // rows off the 16-byte grid (x and y in step) take the configuration of an
  // aligned row of the same length with one more chunk slot per thread
  const int64_t chunks = (cols + 7) / 8;
  if (vec)
    dispatch_rows16_table<kType, false>(x, y, m, l, rows, cols, chunks, ld_x, ld_y, k, err_word, fault, stream);
  else
    dispatch_rows16_table<kType, true>(x, y, m, l, rows, cols, chunks, ld_x, ld_y, k, err_word, fault, stream);
}

cudaError_t launch_softmax_rows16(const uint16_t* x, uint16_t* y, float* m, float* l,
                                  int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                                  float scale, int dtype, unsigned int* err_word,
                                  const RowsFault& fault, cudaStream_t stream) {
  const ScaleConsts k = make_consts(scale);
  if (dtype == 1)
    dispatch_rows16<1>(x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, stream);
  else
    dispatch_rows16<2>(x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, stream);
  return cudaGetLastError();
}

cudaError_t launch_softmax_rows_multipass(const float* x, float* y, float* m, float* l,
                                          int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                                          float scale, int passes, cudaStream_t stream) {
  const ScaleConsts k = make_consts(scale);
  const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                   (ld_x & 3) == 0 && (ld_y & 3) == 0;
  const int g = grid_for(rows, 4);
  if (vec) {
    if (passes == 3) {
      softmax_pass_max<true><<<g, kThreads, 0, stream>>>(x, m, rows, cols, ld_x);
      softmax_pass_sum<true><<<g, kThreads, 0, stream>>>(x, m, l, rows, cols, ld_x, k);
    } else {
      softmax_pass_online<true><<<g, kThreads, 0, stream>>>(x, m, l, rows, cols, ld_x, k);
    }
    softmax_pass_write<true><<<g, kThreads, 0, stream>>>(x, y, m, l, rows, cols, ld_x, ld_y, k);
  } else {
    if (passes == 3) {
      softmax_pass_max<false><<<g, kThreads, 0, stream>>>(x, m, rows, cols, ld_x);
      softmax_pass_sum<false><<<g, kThreads, 0, stream>>>(x, m, l, rows, cols, ld_x, k);
    } else {
      softmax_pass_online<false><<<g, kThreads, 0, stream>>>(x, m, l, rows, cols, ld_x, k);
    }
    softmax_pass_write<false><<<g, kThreads, 0, stream>>>(x, y, m, l, rows, cols, ld_x, ld_y, k);
  }
  return cudaGetLastError();
}

}  // namespace oss
