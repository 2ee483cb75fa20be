// G3: split-KV decode partials, and G4: the fixed-tree merge of partials.
//
// Split-KV decode kernels run the online-softmax recurrence over separate
// chunks of the keys and merge the partial softmaxes afterwards with the same
// correction identity, which spares them float atomics (metalworking "Online
// Softmax", closing note). The pairwise identity is associative, so partials
// may be merged in any order or tree (curionode "The Online Softmax.", "One
// pass, exactly"); G4 uses one fixed tree so every run gives the same bits.
//
// G3 is a streaming GEMV: every key and value row is read once from HBM
// (256 B each at D = 128) and used for one dot product and one AXPY on the
// FMA pipe. A CTA (4 warps) owns one (batch, head, split); each warp takes 8
// keys at a time, lane i holding dims [4i, 4i+4) of q, k, v and O. Scores are
// formed in base 2 (q is pre-multiplied by scale * log2(e)); per 8-key group:
//   m_new = max(m, max t);  c = 2^(m - m_new);  p = 2^(t - m_new);
//   l = l*c + sum p;        O = O*c + sum p v.
// The four warp states are merged through shared memory at the end.

#include <cstdint>

#include "device_common.cuh"
#include "oss_internal.h"

namespace oss {
namespace {

constexpr int kDecodeThreads = 128;
constexpr int kDecodeWarps = kDecodeThreads / 32;
constexpr int kKeysPerWarpStep = 8;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

__device__ __forceinline__ uint2 ld_stream_u2(const uint2* p) { return __ldcs(p); }

__global__ void __launch_bounds__(kDecodeThreads)
decode_splitkv_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                      const uint16_t* __restrict__ v, const int32_t* __restrict__ kv_len,
                      int H, int Lmax, int num_splits, float c,
                      float* __restrict__ part_m, float* __restrict__ part_l,
                      float* __restrict__ part_o) {
  constexpr int D = 128;
  const int split = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int L = kv_len[b];
  L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
  const int chunk = (L + num_splits - 1) / num_splits;
  const int lo = min(L, split * chunk);
  const int hi = min(L, lo + chunk);

  const size_t bh = static_cast<size_t>(b) * H + h;
  // q slice, pre-scaled into base-2 units
  const uint2 qw = reinterpret_cast<const uint2*>(q + bh * D)[lane];
  const float q0 = bf16_lo(qw.x) * c, q1 = bf16_hi(qw.x) * c;
  const float q2 = bf16_lo(qw.y) * c, q3 = bf16_hi(qw.y) * c;

  const uint2* kp = reinterpret_cast<const uint2*>(k + bh * static_cast<size_t>(Lmax) * D) + lane;
  const uint2* vp = reinterpret_cast<const uint2*>(v + bh * static_cast<size_t>(Lmax) * D) + lane;

  float m = neg_inf(), l = 0.f;
  float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;

  for (int base = lo + warp * kKeysPerWarpStep; base < hi;
       base += kDecodeWarps * kKeysPerWarpStep) {
    uint2 kr[kKeysPerWarpStep], vr[kKeysPerWarpStep];
#pragma unroll
    for (int j = 0; j < kKeysPerWarpStep; ++j) {
      const int key = base + j;
      if (key < hi) {
        kr[j] = ld_stream_u2(kp + static_cast<size_t>(key) * (D / 4));
        vr[j] = ld_stream_u2(vp + static_cast<size_t>(key) * (D / 4));
      } else {
        kr[j] = make_uint2(0u, 0u);
        vr[j] = make_uint2(0u, 0u);
      }
    }
    float t[kKeysPerWarpStep];
#pragma unroll
    for (int j = 0; j < kKeysPerWarpStep; ++j) {
      float s = q0 * bf16_lo(kr[j].x);
      s = fmaf(q1, bf16_hi(kr[j].x), s);
      s = fmaf(q2, bf16_lo(kr[j].y), s);
      s = fmaf(q3, bf16_hi(kr[j].y), s);
      t[j] = s;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
      for (int j = 0; j < kKeysPerWarpStep; ++j) t[j] += __shfl_xor_sync(0xffffffffu, t[j], off);
    }
    float mx = neg_inf();
#pragma unroll
    for (int j = 0; j < kKeysPerWarpStep; ++j) {
      if (base + j >= hi) t[j] = neg_inf();
      mx = fmaxf(mx, t[j]);
    }
    // key `base` is always inside the chunk, so mx and m_new are finite
    const float m_new = fmaxf(m, mx);
    const float corr = ex2(m - m_new);  // 0 on the first group (m = -inf)
    float psum = 0.f;
    o0 *= corr; o1 *= corr; o2 *= corr; o3 *= corr;
#pragma unroll
    for (int j = 0; j < kKeysPerWarpStep; ++j) {
      const float p = ex2(t[j] - m_new);
      psum += p;
      o0 = fmaf(p, bf16_lo(vr[j].x), o0);
      o1 = fmaf(p, bf16_hi(vr[j].x), o1);
      o2 = fmaf(p, bf16_lo(vr[j].y), o2);
      o3 = fmaf(p, bf16_hi(vr[j].y), o3);
    }
    l = fmaf(l, corr, psum);
    m = m_new;
  }

  // merge the four warp states (pairwise identity, fixed order)
  __shared__ float sh_m[kDecodeWarps], sh_l[kDecodeWarps];
  __shared__ float4 sh_o[kDecodeWarps][32];
  if (lane == 0) {
    sh_m[warp] = m;
    sh_l[warp] = l;
  }
  sh_o[warp][lane] = make_float4(o0, o1, o2, o3);
  __syncthreads();
  if (warp != 0) return;
  float M = neg_inf();
#pragma unroll
  for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, sh_m[w]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f;
  if (M != neg_inf()) {
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float f = ex2(sh_m[w] - M);  // 0 for an empty warp (m = -inf)
      const float4 ow = sh_o[w][lane];
      acc.x = fmaf(ow.x, f, acc.x);
      acc.y = fmaf(ow.y, f, acc.y);
      acc.z = fmaf(ow.z, f, acc.z);
      acc.w = fmaf(ow.w, f, acc.w);
      lsum = fmaf(sh_l[w], f, lsum);
    }
  }
  const size_t pidx = bh * num_splits + split;
  reinterpret_cast<float4*>(part_o + pidx * D)[lane] = acc;
  if (lane == 0) {
    part_m[pidx] = (M == neg_inf()) ? neg_inf() : M * kLn2;
    part_l[pidx] = lsum;
  }
}

// One warp per group; partials staged in shared memory and merged level by
// level: (0,1),(2,3),... then (0,2),(4,6),... -- an odd slot is carried up.
// Warps per CTA (blockDim.x / 32) are chosen on the host to fit shared memory.
constexpr int kMergeMaxWarps = 4;
constexpr size_t kMergeSmemBudget = 200 * 1024;

__global__ void __launch_bounds__(kMergeMaxWarps * 32)
merge_partials_kernel(const float* __restrict__ part_m, const float* __restrict__ part_l,
                      const float* __restrict__ part_o, int64_t groups, int S, int D,
                      int finalize, void* __restrict__ o_out, float* __restrict__ m_out,
                      float* __restrict__ l_out, float* __restrict__ lse_out) {
  extern __shared__ float4 smem4[];
  const int warps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int D4 = D >> 2;
  // per warp: 64 maxima + 64 sums, then S x D partial outputs
  float4* mine = smem4 + static_cast<size_t>(warp) * (32 + static_cast<size_t>(S) * D4);
  float* sm = reinterpret_cast<float*>(mine);
  float4* so = mine + 32;

  for (int64_t g = static_cast<int64_t>(blockIdx.x) * warps + warp; g < groups;
       g += static_cast<int64_t>(gridDim.x) * warps) {
    float* s_m = sm;       // base-2 maxima
    float* s_l = sm + 64;  // sums
    for (int s = lane; s < S; s += 32) {
      const float mv = part_m[g * S + s];
      s_m[s] = (mv == neg_inf()) ? neg_inf() : mv * kLog2e;
      s_l[s] = part_l[g * S + s];
    }
    const float4* src = reinterpret_cast<const float4*>(part_o + g * S * D);
    for (int i = lane; i < S * D4; i += 32) so[i] = src[i];
    __syncwarp();
    for (int stride = 1; stride < S; stride <<= 1) {
      for (int i = 0; i + stride < S; i += 2 * stride) {
        const int j = i + stride;
        const float mi = s_m[i], mj = s_m[j];
        const float mm = fmaxf(mi, mj);
        float fi = 0.f, fj = 0.f;
        if (mm != neg_inf()) {
          fi = ex2(mi - mm);
          fj = ex2(mj - mm);
        }
        const float li = s_l[i], lj = s_l[j];
        for (int d = lane; d < D4; d += 32) {
          const float4 a = so[i * D4 + d], bq = so[j * D4 + d];
          so[i * D4 + d] = make_float4(fmaf(a.x, fi, bq.x * fj), fmaf(a.y, fi, bq.y * fj),
                                       fmaf(a.z, fi, bq.z * fj), fmaf(a.w, fi, bq.w * fj));
        }
        __syncwarp();
        if (lane == 0) {
          s_m[i] = mm;
          s_l[i] = fmaf(li, fi, lj * fj);
        }
        __syncwarp();
      }
    }
    const float M = s_m[0], Ls = s_l[0];
    const bool empty = (M == neg_inf()) || !(Ls > 0.f);
    const float inv = empty ? 0.f : 1.0f / Ls;
    for (int d = lane; d < D4; d += 32) {
      const float4 a = so[d];
      if (finalize) {
        uint32_t w0, w1;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w0) : "f"(a.y * inv), "f"(a.x * inv));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w1) : "f"(a.w * inv), "f"(a.z * inv));
        reinterpret_cast<uint2*>(o_out)[g * D4 + d] = make_uint2(w0, w1);
      } else {
        reinterpret_cast<float4*>(o_out)[g * D4 + d] = a;
      }
    }
    if (lane == 0) {
      const float m_nat = empty ? neg_inf() : M * kLn2;
      if (m_out) m_out[g] = m_nat;
      if (l_out) l_out[g] = empty ? 0.f : Ls;
      if (lse_out) lse_out[g] = empty ? neg_inf() : m_nat + logf(Ls);
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_decode_splitkv(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  const int32_t* kv_len, int B, int H, int Lmax, int D,
                                  int num_splits, float scale, float* part_m, float* part_l,
                                  float* part_o, cudaStream_t stream) {
  if (D != 128) return cudaErrorNotSupported;
  const float c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  dim3 grid(num_splits, H, B);
  decode_splitkv_kernel<<<grid, kDecodeThreads, 0, stream>>>(q, k, v, kv_len, H, Lmax, num_splits,
                                                             c, part_m, part_l, part_o);
  return cudaGetLastError();
}

cudaError_t launch_merge_partials(const float* part_m, const float* part_l, const float* part_o,
                                  int64_t groups, int num_splits, int D, int finalize,
                                  void* o_out, float* m_out, float* l_out, float* lse_out,
                                  cudaStream_t stream) {
  const size_t per_warp = sizeof(float4) * (32 + static_cast<size_t>(num_splits) * (D / 4));
  int warps = static_cast<int>(kMergeSmemBudget / per_warp);
  warps = warps < 1 ? 1 : (warps > kMergeMaxWarps ? kMergeMaxWarps : warps);
  const size_t smem = per_warp * warps;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(merge_partials_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t need = (groups + warps - 1) / warps;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  const int grid = static_cast<int>(need < cap ? need : cap);
  merge_partials_kernel<<<grid, warps * 32, smem, stream>>>(
      part_m, part_l, part_o, groups, num_splits, D, finalize, o_out, m_out, l_out, lse_out);
  return cudaGetLastError();
}

}  // namespace oss
