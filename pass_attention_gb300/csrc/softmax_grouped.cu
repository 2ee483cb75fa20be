// G1, grouped rows: one kernel for fp32, bf16 and fp16 rows short enough
// for registers. A group of TPR threads (8, 16, 32, 64, 128 or 256) owns one
// row at a time, so a CTA of 256 threads works on 256 / TPR rows and short
// rows keep as many bytes in flight per SM as long ones. A chunk is 16 bytes
// (4 fp32 or 8 16-bit elements, on the 16-byte grid: see load_chunk16); each
// thread holds NV chunks, NV + 1 for rows off the grid.
//
// Per row: the thread's maximum, its weights 2^(x*c - M_t) (packed FMAs, one
// ex2 per element), the merge of the group's (max, sum) states in n-ary form
// (warp shuffles, then shared memory between the group's warps), then each
// weight scaled by 2^(M_t - M_row) / l_row and written once. With kPrefetch
// the grid is persistent and the next row's chunks are loaded into registers
// before the current row is reduced, so a group's loads overlap its own
// arithmetic and stores.
// kKind: 0 = fp32, 1 = bf16, 2 = fp16.

#include "softmax_common.cuh"

namespace oss {
namespace {

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

// kExtra: rows may lie off the 16-byte grid (the chunking of ld_granule /
// fix_granule instead of the plain one). kSlot: one more chunk slot per
// thread (NV + 1), for such rows when the one chunk more they need does not
// fit TPR * NV; only the group's first thread ever finds its extra chunk
// inside the row.
template <int kKind, int TPR, int NV, bool kPrefetch, int kMinBlocks, bool kExtra, bool kSlot>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
softmax_rows_grouped_kernel(const void* __restrict__ x, void* __restrict__ y,
                            float* __restrict__ m_out, float* __restrict__ l_out, int64_t rows,
                            int cols, int64_t ld_x, int64_t ld_y, ScaleConsts k) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  constexpr int kGroups = kThreads / TPR;
  constexpr int kSlots = NV + (kSlot ? 1 : 0);
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

// Launch of softmax_rows_grouped_kernel: persistent (one wave of kMinBlocks
// CTAs per SM) when it prefetches, else up to 64 waves of a grid-stride loop.
template <int kKind, int TPR, int NV, bool kPrefetch, int kMinBlocks, bool kExtra = false,
          bool kSlot = kExtra>
void launch_grouped(const void* x, void* y, float* m, float* l, int64_t rows, int cols,
                    int64_t ld_x, int64_t ld_y, const ScaleConsts& k, cudaStream_t stream) {
  constexpr int kGroups = kThreads / TPR;
  const int64_t need = (rows + kGroups - 1) / kGroups;
  const int64_t cap = static_cast<int64_t>(sm_count()) * kMinBlocks * (kPrefetch ? 1 : 64);
  const int g = static_cast<int>(need < cap ? need : cap);
  softmax_rows_grouped_kernel<kKind, TPR, NV, kPrefetch, kMinBlocks, kExtra, kSlot>
      <<<g, kThreads, 0, stream>>>(x, y, m, l, rows, cols, ld_x, ld_y, k);
}

// A row off the 16-byte grid in the configuration (TPR, NV) of an aligned
// row of the same length: with the extra chunk slot only when its one chunk
// more does not fit TPR * NV (kMinSlot CTAs per SM then, kMin otherwise).
template <int kKind, int TPR, int NV, bool kPrefetch, int kMin, int kMinSlot>
void launch_off_grid(int64_t chunks, const void* x, void* y, float* m, float* l, int64_t rows,
                     int cols, int64_t ld_x, int64_t ld_y, const ScaleConsts& k, cudaStream_t stream) {
  if (chunks + 1 > int64_t(TPR) * NV)
    launch_grouped<kKind, TPR, NV, kPrefetch, kMinSlot, true, true>(x, y, m, l, rows, cols, ld_x, ld_y, k, stream);
  else
    launch_grouped<kKind, TPR, NV, kPrefetch, kMin, true, false>(x, y, m, l, rows, cols, ld_x, ld_y, k, stream);
}

// fp32 rows: the configurations (threads per row / chunks per thread /
// prefetch / CTAs per SM) measured on the GB300 at 2^28 elements per matrix,
// by the row's chunk count on the 16-byte grid; prefetching helped only the
// shortest rows. Rows off the grid take the same configuration plus one
// chunk slot per thread, with fewer CTAs per SM so that nothing spills.
bool grouped_rows_f32(const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                      int64_t ld_x, int64_t ld_y, const ScaleConsts& k, bool on_grid,
                      cudaStream_t stream) {
  const int64_t chunks = (cols + 3) / 4;
  const int c = static_cast<int>(cols);
  if (on_grid) {
    if (chunks <= 8)
      launch_grouped<0, 8, 1, true, 8>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 16)
      launch_grouped<0, 16, 1, true, 8>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 32)
      launch_grouped<0, 32, 1, true, 8>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 64)
      launch_grouped<0, 32, 2, false, 6>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 128)
      launch_grouped<0, 32, 4, false, 6>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 256)
      launch_grouped<0, 64, 4, false, 6>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 512)
      launch_grouped<0, 128, 4, false, 5>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else
      return false;
    return true;
  }
  if (chunks <= 8)
    launch_off_grid<0, 8, 1, true, 5, 4>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 16)
    launch_off_grid<0, 16, 1, true, 5, 4>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 32)
    launch_off_grid<0, 32, 1, true, 5, 4>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 64)
    launch_off_grid<0, 32, 2, false, 6, 6>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 128)
    launch_off_grid<0, 32, 4, false, 5, 4>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 256)
    launch_off_grid<0, 64, 4, false, 5, 4>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 512)
    launch_off_grid<0, 128, 4, false, 5, 4>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 1024)
    launch_off_grid<0, 256, 4, false, 4, 4>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 2048)
    launch_off_grid<0, 256, 8, false, 2, 2>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else
    return false;
  return true;
}

// 16-bit rows of up to 16384 elements: persistent CTAs with the next row's
// chunks prefetched into registers, or, for the lengths where that measured
// slower, more CTAs per SM without it; 256 / TPR rows per CTA for rows of up
// to 4096 elements (groups of 8 and 16 threads, without the prefetch, for
// rows of up to 128). kExtra: the slot a row off the 16-byte grid needs, with
// fewer CTAs per SM.
template <int kType, bool kExtra>
bool grouped_rows16(const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                    int64_t ld_x, int64_t ld_y, const ScaleConsts& k, cudaStream_t stream) {
  const int64_t chunks = (cols + 7) / 8;
  const int c = static_cast<int>(cols);
  if (!kExtra && chunks > 32 && chunks <= (kType == 1 ? 1024 : 256)) {
    // On the grid these rows ran faster on the GB300 without the prefetch,
    // with more CTAs per SM: bf16 by 3-11%, fp16 of 33-256 chunks by 2-10%
    // (at 512 and 1024 chunks fp16 kept the prefetch, level or up to 0.6%
    // ahead). Rows off the grid lost 5-9% without it, for both types.
    if (chunks <= 64)
      launch_grouped<kType, 32, 2, false, 6>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 128)
      launch_grouped<kType, 32, 4, false, 4>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 256)
      launch_grouped<kType, 64, 4, false, 4>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 512)
      launch_grouped<kType, 128, 4, false, 4>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else
      launch_grouped<kType, 256, 4, false, 4>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    return true;
  }
  if (kExtra) {
    if (chunks <= 8)
      launch_off_grid<kType, 8, 1, false, 5, 4>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 16)
      launch_off_grid<kType, 16, 1, false, 5, 4>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 32)
      launch_off_grid<kType, 32, 1, true, 6, 4>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 64)
      launch_off_grid<kType, 32, 2, true, 4, 3>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 128)
      launch_off_grid<kType, 32, 4, true, 3, 2>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 256)
      launch_off_grid<kType, 64, 4, true, 3, 2>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 512)
      launch_off_grid<kType, 128, 4, true, 3, 2>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 1024)
      launch_off_grid<kType, 256, 4, true, 3, 2>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else if (chunks <= 2048)
      launch_off_grid<kType, 256, 8, false, 2, 2>(chunks, x, y, m, l, rows, c, ld_x, ld_y, k, stream);
    else
      return false;
    return true;
  }
  if (chunks <= 8)
    launch_grouped<kType, 8, 1, false, 8>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 16)
    launch_grouped<kType, 16, 1, false, 8>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 32)
    launch_grouped<kType, 32, 1, true, 6>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 64)
    launch_grouped<kType, 32, 2, true, 5>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 128)
    launch_grouped<kType, 32, 4, true, 3>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 256)
    launch_grouped<kType, 64, 4, true, 3>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 512)
    launch_grouped<kType, 128, 4, true, 3>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 1024)
    launch_grouped<kType, 256, 4, true, 3>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else if (chunks <= 2048)
    launch_grouped<kType, 256, 8, true, 2>(x, y, m, l, rows, c, ld_x, ld_y, k, stream);
  else
    return false;
  return true;
}

}  // namespace

bool grouped_rows(int kind, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                  int64_t ld_x, int64_t ld_y, const ScaleConsts& k, bool on_grid, cudaStream_t stream) {
  if (kind == 0) return grouped_rows_f32(x, y, m, l, rows, cols, ld_x, ld_y, k, on_grid, stream);
  if (kind == 1)
    return on_grid ? grouped_rows16<1, false>(x, y, m, l, rows, cols, ld_x, ld_y, k, stream)
                   : grouped_rows16<1, true>(x, y, m, l, rows, cols, ld_x, ld_y, k, stream);
  return on_grid ? grouped_rows16<2, false>(x, y, m, l, rows, cols, ld_x, ld_y, k, stream)
                 : grouped_rows16<2, true>(x, y, m, l, rows, cols, ld_x, ld_y, k, stream);
}

}  // namespace oss
