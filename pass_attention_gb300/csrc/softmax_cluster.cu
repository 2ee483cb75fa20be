// G1, cluster-resident rows.
//
// Cluster-resident rows: rows too long for registers (more than 16384
// elements) but short enough to fit in the shared memory of a thread-block
// cluster of C <= 8 CTAs, where the register path (softmax_cluster_regs.cu)
// does not take them. CTA r of a cluster holds slice r of the row, copied in
// by bulk asynchronous copies; each CTA reduces its slice to a (max, sum)
// state, the CTAs exchange their states through distributed shared memory on
// mbarriers (cluster_exchange.cuh) and merge them (the merge identity of
// partial results), and each CTA then writes its slice once. One HBM read and
// one write per element, where the streaming kernel reads the row twice.
//
// The exchange was a cluster barrier, warp 0 arriving with release, until
// the mbarrier form measured faster everywhere it applies (GB300, 2^28
// elements, fraction of the copy peak: fp32 rows of 98304, 131072, 204800 and
// 409600 columns 0.884 / 0.870 / 0.837 / 0.658 -> 0.952 / 0.929 / 0.927 /
// 0.689; bf16 262144 0.745 -> 0.771, fp16 262144 0.717 -> 0.755, bf16 819200
// 0.558 -> 0.582; rows held by one CTA unchanged).

#include "cluster_exchange.cuh"

namespace oss {
namespace {

// A chunk widened to fp32 as unpack_chunk16 does, but fp16 by a
// mixed-precision add of zero (PTX add.f32.f16: exact; -0 becomes +0, which
// no softmax quantity can tell apart) instead of the conversion
// __half2float uses. Measured on the GB300 (2^28-element matrices): fp16 rows
// of 32768 columns 0.80 -> 0.84 of the copy peak here, 131072 0.71 -> 0.72;
// the other row kernels were no faster that way (staged rows of 128 columns
// 2% slower), so only this kernel takes it.
__device__ __forceinline__ float f16_add_widen(uint32_t bits16) {
  float d;
  asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(d) : "h"(static_cast<unsigned short>(bits16)), "f"(0.0f));
  return d;
}
template <int kKind>
__device__ __forceinline__ void unpack_chunk16_cl(const uint4& v, float2* w /* [kEpc / 2] */) {
  if constexpr (kKind == 2) {
    w[0] = make_float2(f16_add_widen(v.x & 0xffffu), f16_add_widen(v.x >> 16));
    w[1] = make_float2(f16_add_widen(v.y & 0xffffu), f16_add_widen(v.y >> 16));
    w[2] = make_float2(f16_add_widen(v.z & 0xffffu), f16_add_widen(v.z >> 16));
    w[3] = make_float2(f16_add_widen(v.w & 0xffffu), f16_add_widen(v.w >> 16));
  } else {
    unpack_chunk16<kKind>(v, w);
  }
}

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
template <int kKind, bool kDouble, int kThr>
__global__ void __launch_bounds__(kThr, 1024 / kThr)
softmax_rows_cluster_kernel(const void* __restrict__ x, void* __restrict__ y,
                            float* __restrict__ m_out, float* __restrict__ l_out, int64_t rows,
                            int64_t cols, int64_t ld_x, int64_t ld_y, ScaleConsts k,
                            int slice_elems, unsigned int* err, uint32_t fault_tx,
                            uint64_t timeout_ns) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  extern __shared__ __align__(128) uint4 slices[];  // this CTA's slice buffer(s), 16-byte chunks
  __shared__ float2 wstate[kThr / 32];
  __shared__ float2 cstate[2][kClMaxCtas];         // the cluster's CTA states, by row parity
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ __align__(8) uint64_t xbar[2];  // the states' barriers, by exchange parity

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
    for (int b = 0; b < 2; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&xbar[b])) : "memory");
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
  int xe = 0;  // exchanges so far: slot set and barrier xe & 1, parity (xe >> 1) & 1
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
    for (int c0 = tid; c0 < nch; c0 += kThr * kClUnroll) {
      float2 w[kClUnroll][kEpc / 2];
#pragma unroll
      for (int u = 0; u < kClUnroll; ++u)
        unpack_chunk16_cl<kKind>((c0 + u * kThr < nch) ? slice[c0 + u * kThr] : pad, w[u]);
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
    float2 st = merge_states_warp(wstate, kThr / 32, k);
    if (C > 1) {
      const int xs = xe & 1;
      if (tid == 0 && live) send_state(cstate[xs], &xbar[xs], C, rank, st.x, st.y, 0u);
      if (live) live = wait_states_bounded(smem_u32(&xbar[xs]), (xe >> 1) & 1, err, timeout_ns);
      st = merge_states_warp(cstate[xs], static_cast<int>(C), k);
      ++xe;
    }
    xm = st.x;
    ls = st.y;

    // y = 2^(x*c - M_row) / l, formed again from x (an empty row gives 0)
    const bool nonempty = (xm != neg_inf()) && ls > 0.f;
    const float Mr = nonempty ? base2_of(xm, k) : 0.f;
    const float2 negMr = make_float2(-Mr, -Mr);
    const float inv = nonempty ? 1.0f / ls : 0.f;
    const float2 f2 = make_float2(inv, inv);
    for (int c0 = tid; c0 < nch; c0 += kThr * kClUnroll) {
      uint4 v[kClUnroll];
#pragma unroll
      for (int u = 0; u < kClUnroll; ++u) v[u] = (c0 + u * kThr < nch) ? slice[c0 + u * kThr] : pad;
#pragma unroll
      for (int u = 0; u < kClUnroll; ++u) {
        if (c0 + u * kThr < nch) {
          float2 w[kEpc / 2];
          unpack_chunk16_cl<kKind>(v[u], w);
#pragma unroll
          for (int h = 0; h < kEpc / 2; ++h) {
            if constexpr (kKind == 1) {
              // bf16 y: the exponent from c_hi alone (one FMA, not weight2's
              // two). Dropping c_lo (< one fp32 ulp of c) moves y by at most
              // |x c| 2^-24 ln 2 relative before its rounding to 8 bits: under
              // 5e-4 even for logits of 10^4, against a rounding step of
              // 2^-8. m and l, from the exact form above, are unchanged.
              // (GB300, 2^28 elements: 32768 columns 0.830 -> 0.856 of the
              // copy peak, 20000 0.737 -> 0.758.)
              const float2 t = __ffma2_rn(w[h], make_float2(k.c_hi, k.c_hi), negMr);
              w[h] = make_float2(ex2(t.x), ex2(t.y));
            } else {
              w[h] = weight2(w[h], negMr, k);
            }
          }
          store_chunk16<kKind>(yr, c0 + u * kThr, n, s, pack_chunk16<kKind>(w, f2));
        }
      }
    }
    if (rank == 0 && tid == 0) write_ml(xm, ls, k, row, m_out, l_out);
    __syncthreads();  // the slice is read out before its buffer is refilled
  }
  // no CTA leaves while a peer may still store into its shared memory
  if (C > 1) cluster_sync_all();
}

struct ClusterCfg {
  int ctas;
  int slice_elems;
  size_t smem;
};

template <int kKind, bool kDouble, int kThr>
cudaLaunchConfig_t cluster_launch_cfg(const ClusterCfg& cc, cudaLaunchAttribute* attr,
                                      cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cc.ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThr, 1, 1);
  cfg.gridDim = dim3(cc.ctas, 1, 1);
  cfg.dynamicSmemBytes = cc.smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of `ctas` CTAs that can be resident at once (0 when none can),
// cached per device, cluster size and shared-memory size in 8 KB steps.
template <int kKind, bool kDouble, int kThr>
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
  auto kernel = softmax_rows_cluster_kernel<kKind, kDouble, kThr>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 210 << 10) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_launch_cfg<kKind, kDouble, kThr>(cc, attr, nullptr);
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
template <int kKind, bool kDouble, int kThr>
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
    const int used = resident_clusters<kKind, kDouble, kThr>(cc) * cc.ctas;
    if (used > best_used) {
      best_used = used;
      *out = cc;
    }
  }
  return best_used > 0;
}

// Launch of softmax_rows_cluster_kernel, as many clusters as can be resident
// at once (each loops over its rows).
template <int kKind, bool kDouble, int kThr>
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
  const int resident = resident_clusters<kKind, kDouble, kThr>(cc);
  if (resident < 1) return false;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_launch_cfg<kKind, kDouble, kThr>(cc, attr, stream);
  const int64_t nclusters = rows < resident ? rows : resident;
  cfg.gridDim = dim3(static_cast<unsigned int>(nclusters * cc.ctas), 1, 1);
  const int64_t c64 = cols;
  const uint64_t timeout = fault.timeout_ns > 0 ? static_cast<uint64_t>(fault.timeout_ns) : kClTimeoutNs;
  return cudaLaunchKernelEx(&cfg, softmax_rows_cluster_kernel<kKind, kDouble, kThr>, x, y, m, l, rows, c64,
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
  if (pick_cluster<kKind, true, kClThreads>(cols, kClDoubleCap, 1, &cc))
    return launch_cluster_rows_as<kKind, true, kClThreads>(x, y, m, l, rows, cols, ld_x, ld_y, k, cc,
                                                           err, fault, stream);
  // fp32 rows of 32768 to 131072 elements: CTAs of 256 threads, up to four an
  // SM, overlap their rows' copy waits and exchanges better (GB300, 2^28
  // elements, fraction of the copy peak: 32768 columns 0.770 -> 0.805, 65536
  // 0.755 -> 0.776, 131072 0.847 -> 0.870); 16-bit rows, shorter fp32 rows and
  // longer ones ran slower that way (bf16 and fp16 at 32768 by 6-8%, fp32 at
  // 20000 by 8%, at 262144 by 3%, at 409600 by 7%)
  if constexpr (kKind == 0) {
    if (cols >= 32768 && cols <= 131072 && pick_cluster<kKind, false, kClThreads / 2>(cols, kClSingleCap, kClMaxCtas, &cc))
      return launch_cluster_rows_as<kKind, false, kClThreads / 2>(x, y, m, l, rows, cols, ld_x, ld_y, k,
                                                                  cc, err, fault, stream);
  }
  if (pick_cluster<kKind, false, kClThreads>(cols, kClSingleCap, kClMaxCtas, &cc))
    return launch_cluster_rows_as<kKind, false, kClThreads>(x, y, m, l, rows, cols, ld_x, ld_y, k, cc,
                                                            err, fault, stream);
  return false;
}

}  // namespace

// softmax_cluster_regs.cu: aligned rows short enough for a cluster's
// registers (16-bit 18433..131072 elements, fp32 20481..65536), with one
// exponential per element and the states exchanged on mbarriers; false,
// launching nothing, for other rows.
bool cluster_reg_rows(int kind, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                      int64_t ld_x, int64_t ld_y, const ScaleConsts& k, unsigned int* err,
                      const RowsFault& fault, cudaStream_t stream);

bool cluster_rows(int kind, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                  int64_t ld_x, int64_t ld_y, const ScaleConsts& k, unsigned int* err,
                  const RowsFault& fault, cudaStream_t stream) {
  if (cluster_reg_rows(kind, x, y, m, l, rows, cols, ld_x, ld_y, k, err, fault, stream)) return true;
  if (kind == 0) return launch_cluster_rows<0>(x, y, m, l, rows, cols, ld_x, ld_y, k, err, fault, stream);
  if (kind == 1) return launch_cluster_rows<1>(x, y, m, l, rows, cols, ld_x, ld_y, k, err, fault, stream);
  return launch_cluster_rows<2>(x, y, m, l, rows, cols, ld_x, ld_y, k, err, fault, stream);
}

}  // namespace oss
