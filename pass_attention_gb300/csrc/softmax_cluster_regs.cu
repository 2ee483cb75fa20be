// G1, rows held in a cluster's registers.
//
// Aligned rows of 18433..131072 16-bit or 20481..65536 fp32 elements: a
// thread-block cluster of C <= 8 CTAs of 256 threads holds one row, CTA r
// holding slice r (at most 256 * 8 chunks of 16 bytes, NV chunks a thread).
// Each thread widens its chunks, forms its weights 2^(x*c - M_t) once (one
// ex2 per element) and keeps them in registers while the next row's chunks
// are loaded into registers behind them. The CTA merges its threads' (max,
// sum) states; thread 0 sends the CTA's state to every CTA of the cluster by
// asynchronous stores into distributed shared memory that complete on the
// receiver's mbarrier; each CTA merges the C states in rank order (the merge
// identity of partial results) and writes its weights times
// 2^(M_t - M_row) / l_row. One HBM read and one write per element.
//
// Against the shared-memory cluster kernel (softmax_cluster.cu): one
// exponential per element instead of two, and an exchange on mbarriers
// instead of a cluster barrier. The cluster barrier's release and acquire
// cost each CTA about a microsecond a row, which set the pace of these rows;
// with asynchronous stores only the receiving thread waits, and no fence is
// needed (GB300, 2^28 elements, fraction of the copy peak: bf16 rows of 65536
// and 131072 columns 0.75 and 0.73 on the shared-memory kernel, 0.80 and 0.78
// here with a cluster barrier, 0.95 with the mbarrier exchange; fp32 rows of
// 32768 and 65536 0.81 / 0.77 -> 0.89 / 0.88 -> 0.95 / 0.98).

#include <atomic>

#include "cluster_exchange.cuh"

namespace oss {

namespace {

constexpr int kCrMaxNv = 8;  // chunks a thread at most: 2048 chunks a CTA

// The CTA's (max, sum) in every thread: warp shuffles, then the warp states
// through sh[] behind one CTA barrier.
__device__ __forceinline__ void cta_state(float& xm, float& ls, const ScaleConsts& k, float2* sh) {
  float xw = xm;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) xw = fmaxf(xw, __shfl_xor_sync(0xffffffffu, xw, off));
  float lw = (xm == neg_inf()) ? 0.f : ls * ex2(base2_of(xm, k) - base2_of(xw, k));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = make_float2(xw, lw);
  __syncthreads();
  const float2 s = merge_states_warp(sh, kWarps, k);
  xm = s.x;
  ls = s.y;
}

// slice_elems: elements per CTA (a multiple of 128 bytes, at most
// 256 * NV chunks); the last CTA holds what is left of the row. fault_tx:
// bytes every CTA's first row expects beyond the C states (0 but in the test
// hook, which makes the wait run out). A thread that gave up on a wait
// neither waits nor sends again, so a peer waiting for its state gives up in
// turn, and every CTA still meets the final cluster barrier.
template <int kKind, int NV>
__global__ void __launch_bounds__(kThreads, 2)
softmax_rows_clreg_kernel(const void* __restrict__ x, void* __restrict__ y, float* __restrict__ m_out,
                          float* __restrict__ l_out, int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                          ScaleConsts k, int slice_elems, unsigned int* err, uint32_t fault_tx,
                          uint64_t timeout_ns) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  // per-warp states of the CTA merge, the cluster's CTA states and their
  // mbarriers, each in two sets by row parity: a set is written again two
  // rows later, after every reader of the earlier row has passed a barrier
  // (the CTA's, or, for a peer's store, the receipt of this CTA's state for
  // the row in between)
  __shared__ float2 sh[2][kWarps];
  __shared__ float2 cstate[2][kClMaxCtas];
  __shared__ __align__(8) uint64_t xbar[2];
  const int tid = threadIdx.x;
  const uint32_t C = cluster_size();
  const uint32_t rank = cluster_rank();
  const int64_t lo = static_cast<int64_t>(rank) * slice_elems;
  const int64_t left = cols - lo;
  const int n = static_cast<int>(left <= 0 ? 0 : (left < slice_elems ? left : slice_elems));
  const int nfull = n / kEpc;
  const int tail = n % kEpc;
  const int nch = nfull + (tail ? 1 : 0);
  const int64_t rstep = cluster_count();
  int64_t row = cluster_id();
  const char* xb = static_cast<const char*>(x) + lo * kEsz;
  char* yb = static_cast<char*>(y) + lo * kEsz;

  uint4 nx[NV];
  if (row < rows) {
    const char* xr = xb + row * ld_x * kEsz;
#pragma unroll
    for (int i = 0; i < NV; ++i) nx[i] = load_chunk16_grid<kKind>(xr, tid + i * kThreads, nfull, tail);
  }
  if (tid == 0) {
    for (int b = 0; b < 2; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&xbar[b])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // every CTA of the cluster has started and initialised its barriers: its
  // shared memory may be stored into by peers from here on
  cluster_sync_all();

  bool live = true;
  for (int it = 0; row < rows; row += rstep, ++it) {
    const int b = it & 1;
    float2 w[NV][kEpc / 2];
#pragma unroll
    for (int i = 0; i < NV; ++i) unpack_chunk16<kKind>(nx[i], w[i]);
    const int64_t next = row + rstep;
    if (next < rows) {
      const char* xr = xb + next * ld_x * kEsz;
#pragma unroll
      for (int i = 0; i < NV; ++i) nx[i] = load_chunk16_grid<kKind>(xr, tid + i * kThreads, nfull, tail);
    }
    float xa = neg_inf(), xc = neg_inf();
#pragma unroll
    for (int i = 0; i < NV; ++i) {
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
    // a block of chunks that no lane of the warp holds is skipped (its
    // padding is never stored)
    const int wbase = tid & ~31;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      if (i * kThreads + wbase >= nch) continue;
#pragma unroll
      for (int h = 0; h < kEpc / 2; ++h) {
        w[i][h] = weight2(w[i][h], negM, k);
        acc = __fadd2_rn(acc, w[i][h]);
      }
    }
    float ls = acc.x + acc.y;
    const float xm_t = xm;
    cta_state(xm, ls, k, sh[b]);

    const uint32_t bar = smem_u32(&xbar[b]);
    if (tid == 0 && live) send_state(cstate[b], &xbar[b], C, rank, xm, ls, it == 0 ? fault_tx : 0u);
    if (live) live = wait_states_bounded(bar, (it >> 1) & 1, err, timeout_ns);
    const float2 st = merge_states_warp(cstate[b], static_cast<int>(C), k);
    xm = st.x;
    ls = st.y;

    float f = 0.f;
    if (xm_t != neg_inf() && ls > 0.f) f = ex2(base2_of(xm_t, k) - base2_of(xm, k)) * (1.0f / ls);
    const float2 f2 = make_float2(f, f);
    char* yr = yb + row * ld_y * kEsz;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      store_chunk16_grid<kKind>(yr, tid + i * kThreads, nfull, tail, pack_chunk16<kKind>(w[i], f2));
    if (rank == 0 && tid == 0) write_ml(xm, ls, k, row, m_out, l_out);
  }
  // no CTA leaves while a peer may still store into its shared memory
  cluster_sync_all();
}

template <int kKind, int NV>
cudaLaunchConfig_t clreg_cfg(int ctas, unsigned int grid, cudaLaunchAttribute* attr, cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of `ctas` CTAs that can be resident at once (0 when none can),
// cached per device and cluster size.
template <int kKind, int NV>
int clreg_resident(int ctas) {
  static std::atomic<int> cache[64][kClMaxCtas + 1];  // resident + 1; 0 = not asked yet
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cached = dev >= 0 && dev < 64;
  if (cached) {
    const int v = cache[dev][ctas].load();
    if (v > 0) return v - 1;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = clreg_cfg<kKind, NV>(ctas, static_cast<unsigned int>(ctas), attr, nullptr);
  int resident = 0;
  if (cudaOccupancyMaxActiveClusters(&resident, softmax_rows_clreg_kernel<kKind, NV>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    resident = 0;
  }
  if (cached) cache[dev][ctas].store(resident + 1);
  return resident;
}

template <int kKind, int NV>
bool launch_clreg(const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols, int64_t ld_x,
                  int64_t ld_y, const ScaleConsts& k, int ctas, int64_t per, unsigned int* err,
                  const RowsFault& fault, cudaStream_t stream) {
  const int resident = clreg_resident<kKind, NV>(ctas);
  if (resident < 1) return false;
  const int64_t nclusters = rows < resident ? rows : resident;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg =
      clreg_cfg<kKind, NV>(ctas, static_cast<unsigned int>(nclusters * ctas), attr, stream);
  const uint64_t timeout = fault.timeout_ns > 0 ? static_cast<uint64_t>(fault.timeout_ns) : kClTimeoutNs;
  return cudaLaunchKernelEx(&cfg, softmax_rows_clreg_kernel<kKind, NV>, x, y, m, l, rows, cols, ld_x, ld_y, k,
                            static_cast<int>(per), err, fault.extra_tx, timeout) == cudaSuccess;
}

// The row over the fewest CTAs of 2048 chunks that hold it (C), slices of
// ceil(cols / C) elements rounded up to 128 bytes, and the fewest chunks a
// thread that hold a slice (NV = 5..8): the same cluster as eight chunks a
// thread, without blocks of chunks that hold nothing. (GB300, bf16 rows of
// 100000 columns, C = 7: 0.81 of the copy peak with eight chunks a thread,
// 0.86 with seven.)
template <int kKind>
bool clreg_rows(const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols, int64_t ld_x,
                int64_t ld_y, const ScaleConsts& k, unsigned int* err, const RowsFault& fault,
                cudaStream_t stream) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int64_t kCap = int64_t(kThreads) * kCrMaxNv * kEpc;  // elements a CTA
  constexpr int64_t kAlign = 128 / RowElem<kKind>::kSize;
  const int64_t c = (cols + kCap - 1) / kCap;
  if (c < 2 || c > kClMaxCtas) return false;
  const int64_t per = ((cols + c - 1) / c + kAlign - 1) / kAlign * kAlign;
  if ((c - 1) * per >= cols) return false;  // the last CTA would hold nothing
  const int64_t chunks = per / kEpc;
  const int nv = static_cast<int>((chunks + kThreads - 1) / kThreads);
  const int ctas = static_cast<int>(c);
  switch (nv) {
    case 5: return launch_clreg<kKind, 5>(x, y, m, l, rows, cols, ld_x, ld_y, k, ctas, per, err, fault, stream);
    case 6: return launch_clreg<kKind, 6>(x, y, m, l, rows, cols, ld_x, ld_y, k, ctas, per, err, fault, stream);
    case 7: return launch_clreg<kKind, 7>(x, y, m, l, rows, cols, ld_x, ld_y, k, ctas, per, err, fault, stream);
    case 8: return launch_clreg<kKind, 8>(x, y, m, l, rows, cols, ld_x, ld_y, k, ctas, per, err, fault, stream);
    default: return false;
  }
}

}  // namespace

bool cluster_reg_rows(int kind, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                      int64_t ld_x, int64_t ld_y, const ScaleConsts& k, unsigned int* err,
                      const RowsFault& fault, cudaStream_t stream) {
  const int epc = (kind == 0) ? 4 : 8;
  const bool on_grid = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                       ld_x % epc == 0 && ld_y % epc == 0;
  if (!on_grid) return false;
  // fp32 rows of at most 80 KB stay with the shared-memory kernel, which
  // holds them in one CTA without an exchange (fp32 17000 columns: 0.96 of
  // the copy peak there, 0.92 here)
  if (kind == 0) return cols > 20480 && clreg_rows<0>(x, y, m, l, rows, cols, ld_x, ld_y, k, err, fault, stream);
  // 16-bit rows of at most 36 KB likewise (one CTA there, with two buffers;
  // here two CTAs of five chunks a thread, a fifth of them empty: bf16 16400
  // columns 0.785 there, 0.714 here; 20000 0.757 there, 0.846 here)
  if (cols <= 18432) return false;
  if (kind == 1) return clreg_rows<1>(x, y, m, l, rows, cols, ld_x, ld_y, k, err, fault, stream);
  return clreg_rows<2>(x, y, m, l, rows, cols, ld_x, ld_y, k, err, fault, stream);
}

}  // namespace oss
