// G1: one-pass safe softmax of the rows of a row-major matrix (fp32 here;
// bf16 / fp16 through os_softmax_rows_16bit), and the dispatch between the
// row kernels.
//
// The running pair (m, l) of the online normaliser (curionode "The Online
// Softmax.", introduction; roadmapper "Online softmax", "The recurrence")
// is evaluated in base 2 with log2(e) folded into the scale once and exp2 for
// every exponential, the rescale factor included (roadmapper "Things that
// break": mixing bases is one of the listed failures).
//
// Register-resident paths: each thread loads its slice of the row once with
// 16-byte streaming loads, keeps it in registers, forms its own partial state
// (m_t, l_t, p_t), and the row's threads merge their partial states with the
// merge identity (warp shuffles, then one shared-memory round) -- the merge
// the curionode page calls associative, used here in place of a second pass
// over HBM. The weights p are then rescaled in registers and written once:
// one read and one write per element. This file holds the kernel for aligned
// fp32 rows of 2049..16384 elements (a CTA of 256 threads per row);
// softmax_grouped.cu the kernel for shorter rows (several per CTA) and for
// 16-bit rows; softmax_cluster_regs.cu the kernel for rows held in a
// thread-block cluster's registers, softmax_cluster.cu the one for rows held
// in a cluster's shared memory.
//
// Streaming path (rows beyond those, or whose x and y are not in step on
// the 16-byte grid): each thread runs the recurrence over its chunks of the
// row as they arrive, the CTA (or cluster) merges the states, then the row is
// read a second time to write y (2 reads + 1 write per element). The
// multi-pass comparators are here too.

#include "softmax_common.cuh"

namespace oss {
namespace {

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

}  // namespace

// The dispatch. Rows of a matrix whose x rows lie back to back are staged
// in shared memory by tiles (y at any layout) when they are at most 512 bytes
// long, or at most 1 KB and off the 16-byte grid (fp32 rows on the grid only
// when they would leave a fifth or more of the grouped kernel's lanes idle).
// Otherwise, rows
// whose x and y are not in step on the 16-byte grid are streamed. Aligned fp32
// rows of 2049..16384 elements take a CTA each with the row in registers (the
// kernel the headline workload runs); other rows of up to 2048 fp32 (16384
// 16-bit, 8192 fp32 off the grid) elements go to the grouped kernel, longer
// ones of up to 1.6 MB to a cluster (its registers for aligned rows of up to
// 131072 16-bit or 65536 fp32 elements, else its shared memory), and the rest
// are streamed.
cudaError_t launch_softmax_rows(const float* x, float* y, float* m, float* l, int64_t rows,
                                int64_t cols, int64_t ld_x, int64_t ld_y, float scale,
                                unsigned int* err_word, const RowsFault& fault, void* ws,
                                int64_t ws_bytes, cudaStream_t stream) {
  const ScaleConsts k = make_consts(scale);
  if (flat_rows(0, x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, stream))
    return cudaGetLastError();
  const bool on_grid = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                       (ld_x & 3) == 0 && (ld_y & 3) == 0;
  if (!on_grid && !same_phase(x, y, ld_x, ld_y, 4)) {
    launch_stream(softmax_rows_stream_kernel<false>, x, y, m, l, rows, cols, ld_x, ld_y, k, 1, stream);
    return cudaGetLastError();
  }
  const int64_t chunks = (cols + 3) / 4;
  const int nv = static_cast<int>((chunks + kThreads - 1) / kThreads);
  const int c = static_cast<int>(cols);
  if (on_grid && chunks > 512 && nv <= 16) {
    if (nv <= 4)
      softmax_rows_reg_kernel<4><<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
    else if (nv <= 8)
      softmax_rows_reg_kernel<8><<<grid_for(rows, 4), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
    else
      softmax_rows_reg_kernel<16><<<grid_for(rows, 2), kThreads, 0, stream>>>(x, y, m, l, rows, c, ld_x, ld_y, k);
  } else if (!grouped_rows(0, x, y, m, l, rows, cols, ld_x, ld_y, k, on_grid, stream) &&
             !cluster_rows(0, x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, stream) &&
             !wide_rows(0, x, y, m, l, rows, cols, ld_x, ld_y, k, on_grid, ws, ws_bytes, err_word,
                        stream)) {
    if (on_grid)
      launch_stream(softmax_rows_stream_kernel<true>, x, y, m, l, rows, cols, ld_x, ld_y, k, 4, stream);
    else
      launch_stream(softmax_rows_stream_kernel<false>, x, y, m, l, rows, cols, ld_x, ld_y, k, 1, stream);
  }
  return cudaGetLastError();
}

namespace {

template <int kType>
void dispatch_rows16(const uint16_t* x, uint16_t* y, float* m, float* l, int64_t rows,
                     int64_t cols, int64_t ld_x, int64_t ld_y, const ScaleConsts& k,
                     unsigned int* err_word, const RowsFault& fault, void* ws, int64_t ws_bytes,
                     cudaStream_t stream) {
  if (flat_rows(kType, x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, stream)) return;
  const bool on_grid = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                       (ld_x & 7) == 0 && (ld_y & 7) == 0;
  if (!on_grid && !same_phase(x, y, ld_x, ld_y, 2)) {
    launch_stream(softmax_rows16_stream_kernel<kType, false>, x, y, m, l, rows, cols, ld_x, ld_y, k, 1, stream);
    return;
  }
  if (grouped_rows(kType, x, y, m, l, rows, cols, ld_x, ld_y, k, on_grid, stream) ||
      cluster_rows(kType, x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, stream) ||
      wide_rows(kType, x, y, m, l, rows, cols, ld_x, ld_y, k, on_grid, ws, ws_bytes, err_word, stream))
    return;
  // 16-byte accesses only for rows on the grid
  if (on_grid)
    launch_stream(softmax_rows16_stream_kernel<kType, true>, x, y, m, l, rows, cols, ld_x, ld_y, k, 8, stream);
  else
    launch_stream(softmax_rows16_stream_kernel<kType, false>, x, y, m, l, rows, cols, ld_x, ld_y, k, 1, stream);
}

}  // namespace

cudaError_t launch_softmax_rows16(const uint16_t* x, uint16_t* y, float* m, float* l,
                                  int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                                  float scale, int dtype, unsigned int* err_word,
                                  const RowsFault& fault, void* ws, int64_t ws_bytes,
                                  cudaStream_t stream) {
  const ScaleConsts k = make_consts(scale);
  if (dtype == 1)
    dispatch_rows16<1>(x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, ws, ws_bytes, stream);
  else
    dispatch_rows16<2>(x, y, m, l, rows, cols, ld_x, ld_y, k, err_word, fault, ws, ws_bytes, stream);
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
