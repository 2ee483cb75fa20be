// Device and host helpers shared by the row-softmax kernels (G1): the
// base-2 exponent arithmetic of the online normaliser, the merge of
// per-thread (max, sum) states, the 16-byte chunking of a row, 16-bit
// element conversions, thread-block-cluster primitives, and the launch
// paths the dispatch in softmax_rows.cu chooses between.
//
// Internal state is in base 2: for a thread whose largest input is xm,
// M = xm * c with c = scale * log2(e) carried as c_hi + c_lo, and each weight
// is 2^(x*c - M), the exponent formed with two FMAs so that only its final
// rounding matters. ABI outputs are natural: m = fl32(scale * max x) and
// l = sum exp(scale * x - m).
#pragma once

#include <cuda_fp16.h>

#include <atomic>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <limits>

#include "device_common.cuh"
#include "oss_internal.h"

namespace oss {

struct ScaleConsts {
  float scale;  // natural-unit scale (for m)
  float c_hi;   // scale * log2(e), leading float
  float c_lo;   // scale * log2(e) - c_hi
  float e_hi;   // log2(e), leading float
  float e_lo;   // log2(e) - e_hi
};

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

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

inline int sm_count() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

inline int grid_for(int64_t rows, int ctas_per_sm) {
  const int64_t cap = static_cast<int64_t>(sm_count()) * ctas_per_sm * 64;
  return static_cast<int>(rows < cap ? rows : cap);
}


// c (> 0) as hi + lo with hi the float below c and lo = c - hi > 0, both
// positive (the device code relies on it for masked entries, see weight()).
// Where c is a float itself, hi is the float just below it and lo that
// spacing; lo is never 0 (for c below the smallest normal it is set to the
// smallest subnormal, an error of 2^-149 in c).
inline void split_positive(double c, float* hi, float* lo) {
  float h = static_cast<float>(c);
  if (static_cast<double>(h) >= c) h = std::nextafter(h, 0.0f);
  float l = static_cast<float>(c - static_cast<double>(h));
  if (!(l > 0.0f)) l = std::numeric_limits<float>::denorm_min();
  *hi = h;
  *lo = l;
}

inline ScaleConsts make_consts(float scale) {
  const double kLog2e = 1.4426950408889634074;
  ScaleConsts k;
  k.scale = scale;
  split_positive(static_cast<double>(scale) * kLog2e, &k.c_hi, &k.c_lo);
  split_positive(kLog2e, &k.e_hi, &k.e_lo);
  return k;
}


// Every row of x starts at the same offset from a 16-byte boundary as the
// same row of y (the chunks of load_chunk16 then line up for both).
inline bool same_phase(const void* x, const void* y, int64_t ld_x, int64_t ld_y, int esz) {
  const int64_t dx = static_cast<int64_t>(reinterpret_cast<uintptr_t>(x) & 15u);
  const int64_t dy = static_cast<int64_t>(reinterpret_cast<uintptr_t>(y) & 15u);
  return dx == dy && ((ld_x - ld_y) * esz) % 16 == 0;
}

}  // namespace

// Launch paths in their own translation units. Each returns false, launching
// nothing, for rows it does not take (the caller then tries the next path).
// kind: 0 = fp32, 1 = bf16, 2 = fp16. `on_grid`: x's and y's rows are
// 16-byte aligned (else they share an offset from the 16-byte grid).

// softmax_grouped.cu: several rows per CTA, rows held in registers (fp32 up
// to 2048 elements on the grid or 8192 off it; 16-bit up to 16384).
bool grouped_rows(int kind, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                  int64_t ld_x, int64_t ld_y, const ScaleConsts& k, bool on_grid, cudaStream_t stream);

// softmax_cluster.cu: a row per thread-block cluster, held in its registers
// (softmax_cluster_regs.cu: aligned rows of up to 131072 16-bit or 65536
// fp32 elements) or in its shared memory (up to 1.6 MB).
bool cluster_rows(int kind, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                  int64_t ld_x, int64_t ld_y, const ScaleConsts& k, unsigned int* err,
                  const RowsFault& fault, cudaStream_t stream);

// softmax_wide.cu: rows the cluster path does not hold (over 1.6 MB), a
// group of rows at a time over the whole GPU (cooperative launch), slice
// states merged at a grid barrier through the workspace `ws` (at least
// wide_workspace_bytes() bytes); x is read once from HBM and once more from
// L2. Returns false (launching nothing) without a workspace.
bool wide_rows(int kind, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
               int64_t ld_x, int64_t ld_y, const ScaleConsts& k, bool on_grid, void* ws,
               int64_t ws_bytes, unsigned int* err, cudaStream_t stream);
int64_t wide_workspace_bytes();

// softmax_flat.cu: short rows (at most 512 bytes, or 1 KB off the 16-byte
// grid; fp32 rows on the grid only where the grouped kernel would leave lanes
// idle) of a matrix whose x rows lie back to back, tiles of whole rows staged
// in shared memory; x and y at any offset from the grid, y at any leading
// dimension.
bool flat_rows(int kind, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
               int64_t ld_x, int64_t ld_y, const ScaleConsts& k, unsigned int* err,
               const RowsFault& fault, cudaStream_t stream);

}  // namespace oss
