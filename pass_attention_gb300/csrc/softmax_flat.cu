// G1, short rows of a dense matrix, staged through shared memory.
//
// Rows of at most 1 KB whose x rows lie back to back (leading dimension =
// row length), so that any run of whole rows is one contiguous byte range.
// A CTA takes tiles of R consecutive rows. The tile's bytes arrive by bulk
// asynchronous copies of the 16-byte granules that cover them, into one of
// three shared-memory buffers, so each CTA has two tiles in flight while it
// works on a third: short rows then keep as many bytes in flight per SM as
// long ones, whatever their offset from the 16-byte grid. A granule that a
// tile shares with its neighbour is copied by both; only the matrix's own
// partial first and last granules, which reach outside x, are read with plain
// 16-byte loads (the bytes outside x share a granule, and so a page, with an
// element of x, and are never used).
//
// A group of G threads (1 to 32) owns a row at a time and reads it from
// shared memory in 16-byte chunks on the grid of its offset s (chunk c holds
// the elements [c * E - s, (c + 1) * E - s), E elements to a chunk, the
// partial first and last chunks padded with -inf), NV chunks a thread. G is
// the narrowest group that holds the row, so that a warp works on 32 / G rows
// at once and the per-row work (the merge of the group's (max, sum) states
// by shuffles, the scale factor, m and l) is shared by as many rows as
// possible; with scalar accesses and groups of 16, that per-row work and one
// shared-memory load and one store per element left the kernel bound by
// instruction issue at half the copy peak for 16-bit rows. y is written in
// 16-byte chunks when its rows have x's offsets, element by element
// otherwise, so y needs neither x's alignment nor its leading dimension.
// When y is laid out like x (the same offsets, rows back to back), a tile of
// y is one byte range with x's alignment: the groups write their y chunks
// into the tile's buffer in place of x (whole chunks as 16-byte stores; at a
// row boundary a granule holds two rows, and each group writes only its own
// elements) and one bulk copy sends the tile's whole granules out; only the
// tile's partial first and last granules are stored element by element.
// Rows off the 16-byte grid then cost no divergent per-element stores.
// kKind: 0 = fp32, 1 = bf16, 2 = fp16.

#include <atomic>

#include "softmax_common.cuh"

namespace oss {
namespace {

constexpr int kFlBufs = 3;                  // tile buffers per CTA
constexpr int kFlMinBlocks = 4;             // CTAs per SM
constexpr int64_t kFlTileBytes = 14 << 10;  // x bytes per tile, at most
constexpr int64_t kFlMaxRowBytes = 1024;    // the longest row taken
constexpr int64_t kFlGridRowBytes = 512;    // the longest taken when every row is on the grid
constexpr int kFlNvA = 4;                   // 16-byte chunks a thread holds: 4, 6
constexpr int kFlNvB = 6;                   // or 8 (the eight-chunk kernels: two
constexpr int kFlNvC = 8;                   // CTAs an SM, tiles of twice the bytes)

template <int kKind>
__device__ __forceinline__ void flat_store(unsigned char* yr, int j, float v) {
  if constexpr (kKind == 0)
    reinterpret_cast<float*>(yr)[j] = v;
  else
    reinterpret_cast<uint16_t*>(yr)[j] = h16_round<kKind>(v);
}

// Thread 0: the copies of tile `tile` (rows [tile * R, tile * R + nr)) into
// the buffer at shared address buf_a, completing on bar_a. [x0, x1) is the
// whole matrix. The buffer holds the granules [ga, gb) that cover the tile;
// those wholly inside x come by bulk copies, the matrix's partial first and
// last granules by plain loads stored at once. The barrier expects `extra`
// bytes more than are copied (0 but in the test hook, which makes the wait
// run out).
__device__ __forceinline__ void issue_tile(uintptr_t x0, uintptr_t x1, int64_t row_bytes, int64_t R,
                                           int64_t rows, int64_t tile, unsigned char* buf,
                                           uint32_t buf_a, uint32_t bar_a, uint32_t extra) {
  const int64_t r0 = tile * R;
  const int64_t nr = (rows - r0 < R) ? rows - r0 : R;
  const uintptr_t a = x0 + static_cast<uintptr_t>(r0 * row_bytes);
  const uintptr_t b = a + static_cast<uintptr_t>(nr * row_bytes);
  const uintptr_t ga = a & ~uintptr_t(15);
  const uintptr_t gb = (b + 15) & ~uintptr_t(15);
  const uintptr_t in0 = (x0 + 15) & ~uintptr_t(15);  // x's first whole granule
  const uintptr_t in1 = x1 & ~uintptr_t(15);         // one past its last whole granule
  const uintptr_t lo = ga > in0 ? ga : in0;
  const uintptr_t hi = gb < in1 ? gb : in1;
  const uint32_t bulk = hi > lo ? static_cast<uint32_t>(hi - lo) : 0u;
  // the buffer was last read through the generic proxy; order that before
  // the copies' asynchronous writes
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (bulk + extra > 0) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_a),
                 "r"(bulk + extra)
                 : "memory");
    const uint32_t dst = buf_a + static_cast<uint32_t>(lo - ga);
    for (uint32_t off = 0; off < bulk; off += kClPiece) {
      const uint32_t size = (bulk - off < kClPiece) ? (bulk - off) : kClPiece;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
              "r"(dst + off), "l"(lo + off), "r"(size), "r"(bar_a)
          : "memory");
    }
  } else {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_a) : "memory");
  }
  // x's partial first granule (in the buffer when this is the first tile)
  // and partial last granule (when it is the last), once if they are one
  const uintptr_t first = x0 & ~uintptr_t(15);
  const uintptr_t last = (x1 - 1) & ~uintptr_t(15);
  const bool head = (x0 & 15) != 0 && ga == first;
  if (head) *reinterpret_cast<uint4*>(buf) = __ldg(reinterpret_cast<const uint4*>(first));
  if ((x1 & 15) != 0 && gb == last + 16 && !(head && last == first))
    *reinterpret_cast<uint4*>(buf + (last - ga)) = __ldg(reinterpret_cast<const uint4*>(last));
}

// y's elements [lo, hi) of the tile from the tile's buffer, element by
// element (the partial granules at the ends of a tile of y).
template <int kKind>
__device__ __forceinline__ void store_elems_from(unsigned char* ybase, const unsigned char* bufbase,
                                                 uintptr_t lo, uintptr_t hi) {
  constexpr int kEsz = RowElem<kKind>::kSize;
  for (uintptr_t a = lo; a < hi; a += kEsz) {
    if (kEsz == 4)
      *reinterpret_cast<uint32_t*>(ybase + a) = *reinterpret_cast<const uint32_t*>(bufbase + a);
    else
      *reinterpret_cast<uint16_t*>(ybase + a) = *reinterpret_cast<const uint16_t*>(bufbase + a);
  }
}

// G threads per row, NV chunks each (a row spans at most G * NV chunks).
// kYInStep: y's rows have x's offsets from the 16-byte grid. kYBulk (with
// kYInStep): y's rows also lie back to back, and tiles of y leave through the
// buffers by bulk copies.
// CTAs per SM for NV chunks a thread (the registers they need) and the
// x bytes a tile holds (eight-chunk kernels take twice the tile, to keep as
// many bytes in flight per SM with half the CTAs).
constexpr int flat_blocks(int nv) { return nv > kFlNvB ? kFlMinBlocks - 2 : nv > kFlNvA ? kFlMinBlocks - 1 : kFlMinBlocks; }
constexpr int64_t flat_tile_bytes(int nv) { return nv > kFlNvB ? 2 * kFlTileBytes : kFlTileBytes; }

template <int kKind, int G, int NV, bool kYInStep, bool kYBulk>
__global__ void __launch_bounds__(kThreads, flat_blocks(NV))
softmax_rows_flat_kernel(const void* __restrict__ x, void* __restrict__ y,
                         float* __restrict__ m_out, float* __restrict__ l_out, int64_t rows,
                         int cols, int64_t ld_y, ScaleConsts k, int64_t R, int64_t tiles,
                         int buf_stride, unsigned int* err, uint32_t fault_tx, uint64_t timeout_ns) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  constexpr int kGroups = kThreads / G;
  constexpr int kPerWarp = (G < 32) ? 32 / G : 1;
  extern __shared__ __align__(128) unsigned char tile_bufs[];
  __shared__ __align__(8) uint64_t bars[kFlBufs];

  const int tid = threadIdx.x;
  const int g = tid / G;
  const int t = tid % G;
  // a warp's groups walk their rows together (the shuffles take the whole
  // warp); a group past the tile's last row runs as an empty row
  const int lead = g % kPerWarp;
  const int64_t row_bytes = static_cast<int64_t>(cols) * kEsz;
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x);
  const uintptr_t x1 = x0 + static_cast<uintptr_t>(rows * row_bytes);
  unsigned char* yb = static_cast<unsigned char*>(y);

  if (tid == 0) {
    for (int b = 0; b < kFlBufs; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[b])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // thread 0's books: buffers with a copy not yet waited for, and the
  // parity of the phase that copy completes
  uint32_t pend = 0u, ppar = 0u;
  if (tid == 0) {
    for (int b = 0; b < kFlBufs; ++b) {
      const int64_t tile = blockIdx.x + static_cast<int64_t>(b) * gridDim.x;
      if (tile < tiles) {
        unsigned char* buf = tile_bufs + b * buf_stride;
        issue_tile(x0, x1, row_bytes, R, rows, tile, buf, smem_u32(buf), smem_u32(&bars[b]),
                   b == 0 ? fault_tx : 0u);
        pend |= 1u << b;
      }
    }
  }
  __syncthreads();  // the granules thread 0 stored

  uint32_t par = 0u;  // bit b: the parity of buffer b's next phase
  bool live = true;   // false once this thread gave up on a wait: no more waits or copies
  int b = 0;
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const uint32_t bar_a = smem_u32(&bars[b]);
    if (live) {
      live = mbar_wait_bounded(bar_a, (par >> b) & 1u, err, timeout_ns);
      pend &= ~(1u << b);  // landed, or given up on for good
    }
    par ^= 1u << b;
    unsigned char* buf = tile_bufs + b * buf_stride;
    const int64_t r0 = tile * R;
    const int nr = static_cast<int>((rows - r0 < R) ? rows - r0 : R);
    const int head = static_cast<int>((x0 + static_cast<uintptr_t>(r0 * row_bytes)) & 15u);

    const uint4 pad = make_uint4(neg_inf_word<kKind>(), neg_inf_word<kKind>(), neg_inf_word<kKind>(),
                                 neg_inf_word<kKind>());
    for (int ib = g - lead; ib < nr; ib += kGroups) {
      const int i = ib + lead;
      const bool active = i < nr;
      const int o = head + i * static_cast<int>(row_bytes);  // the row's byte offset in the buffer
      const int sp = (o & 15) / kEsz;                          // its offset from the grid, in elements
      uint4* rg = reinterpret_cast<uint4*>(buf + (o & ~15));
      const int nch = (cols + sp + kEpc - 1) / kEpc;
      float2 w[NV][kEpc / 2];
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = t + v * G;
        unpack_chunk16<kKind>((active && c < nch) ? fix_granule<kKind>(rg[c], c, cols, sp) : pad, w[v]);
      }
      float xa = neg_inf(), xc = neg_inf();
#pragma unroll
      for (int v = 0; v < NV; ++v) {
#pragma unroll
        for (int h = 0; h < kEpc / 2; h += 2) {
          xa = fmax3(xa, w[v][h].x, w[v][h].y);
          if (h + 1 < kEpc / 2) xc = fmax3(xc, w[v][h + 1].x, w[v][h + 1].y);
        }
      }
      const float xm = fmaxf(xa, xc);
      const float Mt = (xm == neg_inf()) ? 0.f : base2_of(xm, k);
      const float2 negM = make_float2(-Mt, -Mt);
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
#pragma unroll
        for (int h = 0; h < kEpc / 2; ++h) {
          w[v][h] = weight2(w[v][h], negM, k);
          acc = __fadd2_rn(acc, w[v][h]);
        }
      }
      const float ls = acc.x + acc.y;
      // the group's state: the maximum, then each sum scaled to it
      float xw = xm, lw = ls;
      if constexpr (G > 1) {
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) xw = fmaxf(xw, __shfl_xor_sync(0xffffffffu, xw, off));
        lw = (xm == neg_inf()) ? 0.f : ls * ex2(base2_of(xm, k) - base2_of(xw, k));
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
      }
      float f = 0.f;
      if (xm != neg_inf() && lw > 0.f) f = ex2(base2_of(xm, k) - base2_of(xw, k)) * (1.0f / lw);
      const float2 f2 = make_float2(f, f);
      if (active) {
        const int64_t row = r0 + i;
        unsigned char* yr = yb + row * ld_y * kEsz;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          const int c = t + v * G;
          if (c < nch) {
            if constexpr (kYBulk) {
              // y in place of x: whole chunks at once, a chunk shared with a
              // neighbouring row element by element (this row's elements only)
              const uint4 ov = pack_chunk16<kKind>(w[v], f2);
              const int first = c * kEpc - sp;
              if (first >= 0 && first + kEpc <= cols) {
                rg[c] = ov;
              } else {
                const uint32_t wd[4] = {ov.x, ov.y, ov.z, ov.w};
                unsigned char* gp = reinterpret_cast<unsigned char*>(rg + c);
#pragma unroll
                for (int e = 0; e < kEpc; ++e) {
                  const int j = first + e;
                  if (j >= 0 && j < cols) {
                    if (kKind == 0)
                      reinterpret_cast<uint32_t*>(gp)[e] = wd[e];
                    else
                      reinterpret_cast<uint16_t*>(gp)[e] =
                          static_cast<uint16_t>((e & 1) ? (wd[e >> 1] >> 16) : (wd[e >> 1] & 0xffffu));
                  }
                }
              }
            } else if constexpr (kYInStep) {
              store_chunk16<kKind>(reinterpret_cast<char*>(yr), c, cols, sp, pack_chunk16<kKind>(w[v], f2));
            } else {
#pragma unroll
              for (int e = 0; e < kEpc; ++e) {
                const int j = c * kEpc - sp + e;
                if (j >= 0 && j < cols)
                  flat_store<kKind>(yr, j, ((e & 1) ? w[v][e >> 1].y : w[v][e >> 1].x) * f);
              }
            }
          }
        }
        if (t == 0) write_ml(xw, lw, k, row, m_out, l_out);
      }
    }

    if constexpr (kYBulk) {
      // this thread's y writes into the buffer, before the copy reads them
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();  // buffer b is read out (and, kYBulk, holds the tile's y)
    if constexpr (kYBulk) {
      if (tid == 0) {
        // y's tile [ys, ye): the buffer's byte 0 is the granule of ys
        const uintptr_t ys = reinterpret_cast<uintptr_t>(y) + static_cast<uintptr_t>(r0 * row_bytes);
        const uintptr_t ye = ys + static_cast<uintptr_t>(nr * row_bytes);
        const uintptr_t g0 = ys & ~uintptr_t(15);
        const uintptr_t a0 = (ys + 15) & ~uintptr_t(15);
        const uintptr_t a1 = ye & ~uintptr_t(15);
        unsigned char* ybase = reinterpret_cast<unsigned char*>(g0);
        if (a1 > a0) {
          asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(a0),
                       "r"(smem_u32(buf) + static_cast<uint32_t>(a0 - g0)),
                       "r"(static_cast<uint32_t>(a1 - a0))
                       : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          // the partial granules at the ends: this tile's elements only (the
          // rest of each belongs to the neighbouring tile)
          store_elems_from<kKind>(ybase, buf, ys - g0, a0 - g0);
          store_elems_from<kKind>(ybase, buf, a1 - g0, ye - g0);
        } else {
          store_elems_from<kKind>(ybase, buf, ys - g0, ye - g0);
        }
      }
    }
    const int64_t next = tile + static_cast<int64_t>(kFlBufs) * gridDim.x;
    if (tid == 0 && live && next < tiles) {
      unsigned char* nbuf = tile_bufs + b * buf_stride;
      // the bulk copy of y out of this buffer has read it
      if constexpr (kYBulk) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      issue_tile(x0, x1, row_bytes, R, rows, next, nbuf, smem_u32(nbuf), bar_a, 0u);
      pend |= 1u << b;
      ppar = (ppar & ~(1u << b)) | (par & (1u << b));
    }
    b = (b + 1 == kFlBufs) ? 0 : b + 1;
  }
  // after a give-up: the copies still in flight land before the CTA ends
  if (tid == 0)
    for (int c = 0; c < kFlBufs; ++c)
      if ((pend >> c) & 1u) mbar_wait_bounded(smem_u32(&bars[c]), (ppar >> c) & 1u, err, timeout_ns);
  // the bulk copies of y are complete before the CTA ends
  if constexpr (kYBulk)
    if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Tiles of up to kFlTileBytes (fewer rows per tile when the matrix would
// not give every CTA of one wave a tile), one wave of kFlMinBlocks CTAs per
// SM, each walking its tiles.
template <int kKind, int G, int NV, bool kYInStep, bool kYBulk>
void launch_flat(const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                 int64_t ld_y, const ScaleConsts& k, unsigned int* err, const RowsFault& fault,
                 cudaStream_t stream) {
  constexpr int kEsz = RowElem<kKind>::kSize;
  const int64_t row_bytes = cols * kEsz;
  const int64_t cap = static_cast<int64_t>(sm_count()) * flat_blocks(NV);
  // R a multiple of the CTA's groups: a tile of 71 rows for 64 groups took
  // two rounds of the groups, the second with 7 rows, while the CTA's other
  // warps waited at the tile's barrier. Below one round, a tile of one row a
  // group when that stays within twice the tile's bytes (not for the
  // eight-chunk groups, whose rows of 128 and 256 elements lost 2-4% so).
  // GB300, 2^28 elements, fraction of the copy peak: bf16 100 columns 0.600
  // -> 0.686, 200 0.708 -> 0.820, 300 0.644 -> 0.775, 75 0.623 -> 0.746, 33
  // 0.612 -> 0.729; fp32 101 0.767 -> 0.913, 50 0.800 -> 0.891; fp32 100
  // 0.861 -> 0.841.
  constexpr int64_t kGroups = kThreads / G;
  int64_t R = flat_tile_bytes(NV) / row_bytes;
  if (R >= kGroups)
    R = R / kGroups * kGroups;
  else if (NV <= kFlNvB && kGroups * row_bytes <= 2 * flat_tile_bytes(NV))
    R = kGroups;
  const int64_t spread = (rows + cap - 1) / cap;
  if (R > spread) R = spread;
  if (R < 1) R = 1;
  const int64_t tiles = (rows + R - 1) / R;
  const int stride = static_cast<int>((R * row_bytes + 32 + 127) / 128 * 128);
  const int grid = static_cast<int>(tiles < cap ? tiles : cap);
  const uint64_t timeout = fault.timeout_ns > 0 ? static_cast<uint64_t>(fault.timeout_ns) : kClTimeoutNs;
  const size_t smem = static_cast<size_t>(stride) * kFlBufs;
  // above the default limit with the static barriers: raised once per device
  if (smem + sizeof(uint64_t) * kFlBufs > (48u << 10)) {
    constexpr int kMaxDevices = 64;
    static std::atomic<bool> raised[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices || !raised[dev].load(std::memory_order_acquire)) {
      cudaFuncSetAttribute(softmax_rows_flat_kernel<kKind, G, NV, kYInStep, kYBulk>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, 100 << 10);
      if (dev >= 0 && dev < kMaxDevices) raised[dev].store(true, std::memory_order_release);
    }
  }
  softmax_rows_flat_kernel<kKind, G, NV, kYInStep, kYBulk>
      <<<grid, kThreads, smem, stream>>>(
          x, y, m, l, rows, static_cast<int>(cols), ld_y, k, R, tiles, stride, err, fault.extra_tx,
          timeout);
}

template <int kKind, int NV, bool kYInStep, bool kYBulk>
void launch_flat_nv(int G, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                    int64_t ld_y, const ScaleConsts& k, unsigned int* err, const RowsFault& fault,
                    cudaStream_t stream) {
  switch (G) {
    case 1: launch_flat<kKind, 1, NV, kYInStep, kYBulk>(x, y, m, l, rows, cols, ld_y, k, err, fault, stream); break;
    case 2: launch_flat<kKind, 2, NV, kYInStep, kYBulk>(x, y, m, l, rows, cols, ld_y, k, err, fault, stream); break;
    case 4: launch_flat<kKind, 4, NV, kYInStep, kYBulk>(x, y, m, l, rows, cols, ld_y, k, err, fault, stream); break;
    case 8: launch_flat<kKind, 8, NV, kYInStep, kYBulk>(x, y, m, l, rows, cols, ld_y, k, err, fault, stream); break;
    case 16: launch_flat<kKind, 16, NV, kYInStep, kYBulk>(x, y, m, l, rows, cols, ld_y, k, err, fault, stream); break;
    default: launch_flat<kKind, 32, NV, kYInStep, kYBulk>(x, y, m, l, rows, cols, ld_y, k, err, fault, stream); break;
  }
}

// The group for a row spanning `chunks` 16-byte chunks: G threads of NV
// chunks each (G a power of two up to 32, NV 4, 6 or 8), the pair whose
// G * NV slots leave the fewest unused, then the one with fewer threads a row
// (the per-row work -- the group's shuffles, the scale factor, m and l -- is
// repeated by each of its threads). Eight chunks a thread (two CTAs an SM,
// tiles of twice the bytes) for rows off the grid, and on it for groups of
// four threads or more: GB300, 2^28 elements, fraction of the copy peak, bf16
// rows of 100 columns (off the grid, 4 x 4 -> 2 x 8) 0.685 -> 0.788, fp16 100
// 0.691 -> 0.807, fp32 101 0.897 -> 0.963, fp32 50 0.881 -> 0.930; on the
// grid bf16 200 (8 x 4 -> 4 x 8) 0.817 -> 0.863 and fp32 100 0.838 -> 0.869,
// but bf16 120 (4 x 4 -> 2 x 8) 0.826 -> 0.782.
template <int kKind, bool kYInStep, bool kYBulk>
void launch_flat_g(int64_t chunks, bool on_grid, const void* x, void* y, float* m, float* l, int64_t rows,
                   int64_t cols, int64_t ld_y, const ScaleConsts& k, unsigned int* err,
                   const RowsFault& fault, cudaStream_t stream) {
  int best_g = 32, best_nv = kFlNvA;
  int64_t best_waste = -1;
  for (int g = 1; g <= 32; g *= 2) {
    for (int nv : {kFlNvA, kFlNvB, kFlNvC}) {
      if (nv == kFlNvC && on_grid && g < 4) continue;
      const int64_t slots = static_cast<int64_t>(g) * nv;
      if (slots < chunks) continue;
      const int64_t waste = slots - chunks;
      if (best_waste < 0 || waste < best_waste || (waste == best_waste && g < best_g)) {
        best_waste = waste;
        best_g = g;
        best_nv = nv;
      }
    }
  }
  if (best_nv == kFlNvA)
    launch_flat_nv<kKind, kFlNvA, kYInStep, kYBulk>(best_g, x, y, m, l, rows, cols, ld_y, k, err, fault, stream);
  else if (best_nv == kFlNvB)
    launch_flat_nv<kKind, kFlNvB, kYInStep, kYBulk>(best_g, x, y, m, l, rows, cols, ld_y, k, err, fault, stream);
  else
    launch_flat_nv<kKind, kFlNvC, kYInStep, kYBulk>(best_g, x, y, m, l, rows, cols, ld_y, k, err, fault, stream);
}

template <int kKind>
bool flat_rows_as(const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                  int64_t ld_x, int64_t ld_y, const ScaleConsts& k, unsigned int* err,
                  const RowsFault& fault, cudaStream_t stream) {
  constexpr int kEpc = RowElem<kKind>::kEpc;
  constexpr int kEsz = RowElem<kKind>::kSize;
  if ((rows > 1 && ld_x != cols) || cols * kEsz > kFlMaxRowBytes) return false;
  if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) % kEsz) != 0) return false;
  // Rows on the 16-byte grid longer than kFlGridRowBytes run faster in the
  // grouped kernel, which reads them straight into registers (GB300, 2^28
  // elements: fp32 rows of 256 elements at 0.96 of the copy peak there
  // against 0.85 here, bf16 rows of 512 at 0.88 against 0.87). So do shorter
  // fp32 rows on the grid that fill at least 80% of the grouped kernel's
  // chunk slots (a power of two, at least 8, per row): 32, 64 and 128
  // elements ran at 0.91-0.93 there against 0.85-0.87 here, while 16 (0.51
  // there, 0.79 here) and 100 (0.77, 0.86) come here. 16-bit rows on the
  // grid came out ahead here at every length up to 512 bytes (bf16 at 128
  // elements 0.84 against 0.72), and rows off the grid at every length taken.
  const bool grid_rows = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                         (cols * kEsz) % 16 == 0 && (ld_y * kEsz) % 16 == 0;
  if (grid_rows && cols * kEsz > kFlGridRowBytes) return false;
  if (kKind == 0 && grid_rows) {
    const int64_t chunks = cols * kEsz / 16;
    int64_t slots = 8;
    while (slots < chunks) slots *= 2;
    if (5 * chunks >= 4 * slots) return false;
  }
  // 16-bit rows on the grid of 16 or 32 chunks: groups of 2 or 4 threads of
  // eight chunks, no chunk slot left over (GB300, 2^28 elements: bf16 rows
  // of 128 elements 0.83 -> 0.94 of the copy peak, 256 0.82 -> 0.86; rows of
  // 64, one thread a row, fell to 0.62, and rows that leave slots over, such
  // as 200, lost 3%)
  if constexpr (kKind != 0) {
    if (grid_rows && same_phase(x, y, cols, ld_y, kEsz) && (cols * kEsz == 256 || cols * kEsz == 512)) {
      if (cols * kEsz == 256)
        launch_flat<kKind, 2, kFlNvC, true, false>(x, y, m, l, rows, cols, ld_y, k, err, fault, stream);
      else
        launch_flat<kKind, 4, kFlNvC, true, false>(x, y, m, l, rows, cols, ld_y, k, err, fault, stream);
      return true;
    }
  }
  // the most chunks a row spans: rows 16-byte multiples long all have x's
  // offset, others may lie at any
  const int s0 = static_cast<int>((reinterpret_cast<uintptr_t>(x) & 15u) / kEsz);
  const int smax = ((cols * kEsz) % 16 == 0 || rows == 1) ? s0 : kEpc - 1;
  const int64_t chunks = (cols + smax + kEpc - 1) / kEpc;
  // y laid out like x, rows back to back: tiles of y leave by bulk copies
  // when its rows are off the 16-byte grid (on the grid every chunk is whole
  // and goes out as one 16-byte store already)
  const bool y_like_x = ld_y == cols && ((reinterpret_cast<uintptr_t>(x) ^ reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
  if (y_like_x && !grid_rows)
    launch_flat_g<kKind, true, true>(chunks, grid_rows, x, y, m, l, rows, cols, ld_y, k, err, fault, stream);
  else if (same_phase(x, y, cols, ld_y, kEsz))
    launch_flat_g<kKind, true, false>(chunks, grid_rows, x, y, m, l, rows, cols, ld_y, k, err, fault, stream);
  else
    launch_flat_g<kKind, false, false>(chunks, grid_rows, x, y, m, l, rows, cols, ld_y, k, err, fault, stream);
  return true;
}

}  // namespace

bool flat_rows(int kind, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
               int64_t ld_x, int64_t ld_y, const ScaleConsts& k, unsigned int* err,
               const RowsFault& fault, cudaStream_t stream) {
  if (kind == 0) return flat_rows_as<0>(x, y, m, l, rows, cols, ld_x, ld_y, k, err, fault, stream);
  if (kind == 1) return flat_rows_as<1>(x, y, m, l, rows, cols, ld_x, ld_y, k, err, fault, stream);
  return flat_rows_as<2>(x, y, m, l, rows, cols, ld_x, ld_y, k, err, fault, stream);
}

}  // namespace oss
