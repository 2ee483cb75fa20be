// Rows too long for a thread-block cluster's shared memory (over 1.6 MB):
// the whole GPU works on a few rows at a time.
//
// The online normaliser of the curionode page ("One pass, exactly") gives
// each slice of a row its own (max, sum) state, and the pairwise merge
// identity combines slice states in any order. A cooperative launch (every
// CTA resident at once) takes the rows in groups small enough to stay in L2:
// each CTA streams one slice of one row of the group from HBM and forms its
// state; the states of a row meet in a small workspace at a grid-wide
// barrier; every CTA of the row merges them, in slice order, and reads its
// slice again -- from L2 -- to write y. HBM sees one read and one write per
// element, where the streaming kernel it replaces reads x twice from HBM.
//
// The barrier is a counter in the workspace (zeroed before each launch), on
// which each CTA arrives once per group and then waits, with a time limit:
// a CTA that gives up records the error word (kernel 2, site 2) and goes on
// without waiting again, so a failed launch ends after about one limit.

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "softmax_common.cuh"

namespace oss {
namespace {

constexpr int64_t kWideL2Budget = int64_t(64) << 20;        // bytes of x a group may hold
constexpr unsigned long long kWideTimeoutNs = 2000000000ull;  // wait at the grid barrier
constexpr int kWideCtasPerSm = 8;
constexpr int kWideUnroll = 4;  // 16-byte chunks each thread has in flight

struct WideArgs {
  float2* states;        // [2][grid]: (raw max, base-2 sum) of each CTA's slice, by group parity
  unsigned int* arrive;  // grid barrier: arrivals so far (zero at launch)
  unsigned int* err;
  int rows_per_group;    // R; the grid is R * slices CTAs
  int slices;
  int64_t slice_chunks;  // chunks (of the vector width) per slice
};

// Element e of a row as fp32 (kind 0 fp32, 1 bf16, 2 fp16).
template <int kKind>
__device__ __forceinline__ float load_elem(const void* row, int64_t e) {
  if constexpr (kKind == 0) return static_cast<const float*>(row)[e];
  else return h16_one<kKind>(static_cast<const uint16_t*>(row)[e]);
}
template <int kKind>
__device__ __forceinline__ void store_elem(void* row, int64_t e, float v) {
  if constexpr (kKind == 0) static_cast<float*>(row)[e] = v;
  else static_cast<uint16_t*>(row)[e] = static_cast<uint16_t>(h16_pack<kKind>(v, 0.f) & 0xffffu);
}

// Elements per 16-byte chunk.
template <int kKind>
constexpr int chunk_elems() { return kKind == 0 ? 4 : 8; }

// Element e of a raw 16-byte chunk (E = 4 fp32 or 8 16-bit elements; for
// E = 1, element 0 is the low word as fp32 or the low half as 16-bit).
template <int kKind>
__device__ __forceinline__ float chunk_elem(const uint4& w, int e) {
  const uint32_t word = (e >> (kKind == 0 ? 0 : 1)) == 0 ? w.x
                      : (e >> (kKind == 0 ? 0 : 1)) == 1 ? w.y
                      : (e >> (kKind == 0 ? 0 : 1)) == 2 ? w.z : w.w;
  if constexpr (kKind == 0) return __uint_as_float(word);
  else return (e & 1) ? h16_hi<kKind>(word) : h16_lo<kKind>(word);
}

// fp32 values back into a raw chunk, the inverse of chunk_elem (values are
// widened elements or -inf, which every type represents exactly).
template <int kKind, int E>
__device__ __forceinline__ uint4 pack_chunk(const float (&t)[8]) {
  if constexpr (kKind == 0) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    w.x = __float_as_uint(t[0]);
    if (E > 1) { w.y = __float_as_uint(t[1]); w.z = __float_as_uint(t[2]); w.w = __float_as_uint(t[3]); }
    return w;
  } else {
    if (E == 1) return make_uint4(h16_pack<kKind>(t[0], t[0]), 0u, 0u, 0u);
    return make_uint4(h16_pack<kKind>(t[0], t[1]), h16_pack<kKind>(t[2], t[3]),
                      h16_pack<kKind>(t[4], t[5]), h16_pack<kKind>(t[6], t[7]));
  }
}

template <int kKind>
__device__ __forceinline__ void store_chunk16(void* row, int64_t c, const float (&v)[8]) {
  uint4 u;
  if constexpr (kKind == 0) {
    u = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                   __float_as_uint(v[3]));
  } else {
    u = make_uint4(h16_pack<kKind>(v[0], v[1]), h16_pack<kKind>(v[2], v[3]),
                   h16_pack<kKind>(v[4], v[5]), h16_pack<kKind>(v[6], v[7]));
  }
  __stcs(reinterpret_cast<uint4*>(row) + c, u);
}

// The grid barrier of group q: arrive, then wait until every CTA of the
// launch has arrived q + 1 times. Returns false after a give-up (and from
// then on, without waiting: `gave_up` is sticky).
__device__ __forceinline__ bool grid_barrier(unsigned int* arrive, unsigned int target,
                                             unsigned int* err, bool& gave_up) {
  __syncthreads();
  __shared__ int ok_s;
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(arrive, 1u);
    int ok = 1;
    if (!gave_up) {
      const uint64_t t0 = timer_ns();
      for (uint32_t n = 0;; ++n) {
        unsigned int seen;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(arrive) : "memory");
        if (seen >= target) break;
        if ((n & 15u) == 15u) {
          __nanosleep(256);
          if (timer_ns() - t0 > kWideTimeoutNs) {
            report_error(err, kKernelSoftmaxRows | (2u << 8));
            ok = 0;
            break;
          }
        }
      }
    } else {
      ok = 0;
    }
    __threadfence();
    ok_s = ok;
  }
  __syncthreads();
  const bool ok = ok_s != 0;
  if (!ok) gave_up = true;
  return ok;
}

template <int kKind, bool kVec>
__global__ void __launch_bounds__(kThreads)
softmax_rows_wide_kernel(const void* __restrict__ x, void* __restrict__ y, float* __restrict__ m_out,
                         float* __restrict__ l_out, int64_t rows, int64_t cols, int64_t ld_x,
                         int64_t ld_y, ScaleConsts k, WideArgs a) {
  __shared__ float2 sh[kWarps];
  __shared__ float2 row_state;
  constexpr int E = kVec ? chunk_elems<kKind>() : 1;
  constexpr int esize = kKind == 0 ? 4 : 2;
  const int64_t nchunks = (cols + E - 1) / E;
  const int tid = threadIdx.x;
  const int G = static_cast<int>(gridDim.x);
  const int r = static_cast<int>(blockIdx.x) / a.slices;  // row within a group
  const int s = static_cast<int>(blockIdx.x) - r * a.slices;
  const int64_t c_lo = static_cast<int64_t>(s) * a.slice_chunks;
  const int64_t c_hi = (c_lo + a.slice_chunks < nchunks) ? c_lo + a.slice_chunks : nchunks;
  const int64_t groups = (rows + a.rows_per_group - 1) / a.rows_per_group;
  bool gave_up = false;
  for (int64_t q = 0; q < groups; ++q) {
    const int64_t row = q * a.rows_per_group + r;
    const bool live = row < rows;
    const char* xr = static_cast<const char*>(x) + (live ? row : 0) * ld_x * esize;
    char* yr = static_cast<char*>(y) + (live ? row : 0) * ld_y * esize;
    // pass 1: this slice's (max, sum), the recurrence per thread over its
    // chunks, kWideUnroll chunks in flight at a time (one rescale each batch)
    float xm = neg_inf(), ls = 0.f;
    if (live) {
      for (int64_t c0 = c_lo + tid; c0 < c_hi; c0 += kWideUnroll * kThreads) {
        // raw 16-byte chunks; elements past the slice or the row read as
        // -inf (a word of -inf patterns), whose weight is exactly 0
        uint4 w[kWideUnroll];
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u) {
          const int64_t c = c0 + static_cast<int64_t>(u) * kThreads;
          if (kVec && c < c_hi && (c + 1) * E <= cols) {
            w[u] = __ldcg(reinterpret_cast<const uint4*>(xr) + c);
          } else {
            float t[8];
#pragma unroll
            for (int e = 0; e < E; ++e)
              t[e] = (c < c_hi && c * E + e < cols) ? load_elem<kKind>(xr, c * E + e) : neg_inf();
            w[u] = pack_chunk<kKind, E>(t);
          }
        }
        float bm = neg_inf();
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u)
#pragma unroll
          for (int e = 0; e < E; ++e) bm = fmaxf(bm, chunk_elem<kKind>(w[u], e));
        const float xn = fmaxf(xm, bm);
        if (xn == neg_inf()) continue;  // nothing visible yet: no -inf - -inf
        const float Mn = base2_of(xn, k);
        const float corr = (xm == neg_inf()) ? 0.f : ex2(base2_of(xm, k) - Mn);
        float add = 0.f;
#pragma unroll
        for (int u = 0; u < kWideUnroll; ++u)
#pragma unroll
          for (int e = 0; e < E; ++e) add += weight(chunk_elem<kKind>(w[u], e), Mn, k);
        ls = ls * corr + add;
        xm = xn;
      }
    }
    cta_merge(xm, ls, k, sh);
    float2* st = a.states + (q & 1) * G;
    if (tid == 0) st[blockIdx.x] = make_float2(xm, ls);
    // every slice state of the group is in the workspace after this
    grid_barrier(a.arrive, static_cast<unsigned int>((q + 1) * G), a.err, gave_up);
    // the row's state: the slices' states merged in slice order by warp 0
    if (tid < 32) {
      const float2* rs = st + r * a.slices;
      float x2 = neg_inf(), l2 = 0.f;
      for (int i = tid; i < a.slices; i += 32) {  // lane-wise, in slice order
        const float2 e = __ldcg(rs + i);
        const float xn = fmaxf(x2, e.x);
        if (xn == neg_inf()) continue;
        const float Mn = base2_of(xn, k);
        l2 = ((x2 == neg_inf()) ? 0.f : l2 * ex2(base2_of(x2, k) - Mn)) +
             ((e.x == neg_inf()) ? 0.f : e.y * ex2(base2_of(e.x, k) - Mn));
        x2 = xn;
      }
      // then across the lanes, the same fixed tree in every CTA of the row
      float xw = x2;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) xw = fmaxf(xw, __shfl_xor_sync(0xffffffffu, xw, off));
      float lw = (x2 == neg_inf()) ? 0.f : l2 * ex2(base2_of(x2, k) - base2_of(xw, k));
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
      if (tid == 0) row_state = make_float2(xw, lw);
    }
    __syncthreads();
    const float2 rsx = row_state;
    // pass 2: y = 2^(x c - M) / l over this slice, x read again (from L2),
    // kWideUnroll chunks in flight at a time
    if (live) {
      const float M = (rsx.x == neg_inf()) ? 0.f : base2_of(rsx.x, k);
      const float inv = (rsx.y > 0.f) ? 1.0f / rsx.y : 0.f;
      for (int64_t c0 = c_lo + tid; c0 < c_hi; c0 += kWideUnroll * kThreads) {
        if constexpr (kVec) {
          uint4 w[kWideUnroll];
#pragma unroll
          for (int u = 0; u < kWideUnroll; ++u) {
            const int64_t c = c0 + static_cast<int64_t>(u) * kThreads;
            if (c < c_hi && (c + 1) * E <= cols) w[u] = __ldcs(reinterpret_cast<const uint4*>(xr) + c);
          }
#pragma unroll
          for (int u = 0; u < kWideUnroll; ++u) {
            const int64_t c = c0 + static_cast<int64_t>(u) * kThreads;
            if (c >= c_hi) continue;
            if ((c + 1) * E <= cols) {
              float v[8];
#pragma unroll
              for (int e = 0; e < E; ++e) v[e] = weight(chunk_elem<kKind>(w[u], e), M, k) * inv;
              store_chunk16<kKind>(yr, c, v);
            } else {
              for (int64_t e = c * E; e < cols; ++e)
                store_elem<kKind>(yr, e, weight(load_elem<kKind>(xr, e), M, k) * inv);
            }
          }
        } else {
          float v[kWideUnroll];
#pragma unroll
          for (int u = 0; u < kWideUnroll; ++u) {
            const int64_t c = c0 + static_cast<int64_t>(u) * kThreads;
            v[u] = (c < c_hi) ? load_elem<kKind>(xr, c) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < kWideUnroll; ++u) {
            const int64_t c = c0 + static_cast<int64_t>(u) * kThreads;
            if (c < c_hi) store_elem<kKind>(yr, c, weight(v[u], M, k) * inv);
          }
        }
      }
      if (s == 0 && tid == 0) write_ml(rsx.x, rsx.y, k, row, m_out, l_out);
    }
    __syncthreads();  // sh and row_state are reused by the next group
  }
}

// CTAs of the wide kernel that can be resident at once on this device (per
// instance), computed once per device.
int wide_resident(const void* kernel, int kidx) {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices][6];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev][kidx].load(std::memory_order_acquire);
    if (c > 0) return c;
  }
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (per_sm > kWideCtasPerSm) per_sm = kWideCtasPerSm;
  const int n = per_sm * sms;
  if (dev >= 0 && dev < kMaxDevices) cache[dev][kidx].store(n, std::memory_order_release);
  return n;
}

template <int kKind, bool kVec>
bool launch_wide(const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
                 int64_t ld_x, int64_t ld_y, const ScaleConsts& k, void* ws, int64_t ws_bytes,
                 unsigned int* err, cudaStream_t stream) {
  const void* kernel = reinterpret_cast<const void*>(softmax_rows_wide_kernel<kKind, kVec>);
  const int G = wide_resident(kernel, kKind * 2 + (kVec ? 1 : 0));
  if (G < 2) return false;
  const int64_t esize = kKind == 0 ? 4 : 2;
  const int64_t row_bytes = cols * esize;
  int64_t R = kWideL2Budget / (row_bytes > 0 ? row_bytes : 1);
  if (R < 1) R = 1;
  if (R > rows) R = rows;
  if (R > G) R = G;
  const int slices = static_cast<int>(G / R);
  const int grid = static_cast<int>(R) * slices;
  const int64_t E = kVec ? chunk_elems<kKind>() : 1;
  const int64_t nchunks = (cols + E - 1) / E;
  const size_t need = static_cast<size_t>(2 * grid) * sizeof(float2) + 16;
  if (!ws || static_cast<uint64_t>(ws_bytes) < need) return false;
  WideArgs a;
  a.states = static_cast<float2*>(ws);
  a.arrive = reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + 2 * grid * sizeof(float2));
  a.err = err;
  a.rows_per_group = static_cast<int>(R);
  a.slices = slices;
  a.slice_chunks = (nchunks + slices - 1) / slices;
  if (cudaMemsetAsync(a.arrive, 0, sizeof(unsigned int), stream) != cudaSuccess) return false;
  void* args[] = {const_cast<void**>(&x), &y, &m, &l, &rows, &cols, &ld_x, &ld_y,
                  const_cast<ScaleConsts*>(&k), &a};
  if (cudaLaunchCooperativeKernel(kernel, dim3(grid), dim3(kThreads), args, 0, stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

}  // namespace

int64_t softmax_workspace_bytes(int64_t row_bytes) {
  // the cluster path holds rows of up to kClMaxCtas * kClSingleCap bytes
  // (one chunk less off the 16-byte grid); longer ones take the wide kernel
  if (row_bytes <= static_cast<int64_t>(kClMaxCtas) * kClSingleCap - 32) return 0;
  return wide_workspace_bytes();
}

int64_t wide_workspace_bytes() {
  // the largest grid any instance can have: kWideCtasPerSm CTAs on every SM
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  return static_cast<int64_t>(2 * kWideCtasPerSm * sms) * sizeof(float2) + 16;
}

bool wide_rows(int kind, const void* x, void* y, float* m, float* l, int64_t rows, int64_t cols,
               int64_t ld_x, int64_t ld_y, const ScaleConsts& k, bool on_grid, void* ws,
               int64_t ws_bytes, unsigned int* err, cudaStream_t stream) {
  switch (kind * 2 + (on_grid ? 1 : 0)) {
    case 0: return launch_wide<0, false>(x, y, m, l, rows, cols, ld_x, ld_y, k, ws, ws_bytes, err, stream);
    case 1: return launch_wide<0, true>(x, y, m, l, rows, cols, ld_x, ld_y, k, ws, ws_bytes, err, stream);
    case 2: return launch_wide<1, false>(x, y, m, l, rows, cols, ld_x, ld_y, k, ws, ws_bytes, err, stream);
    case 3: return launch_wide<1, true>(x, y, m, l, rows, cols, ld_x, ld_y, k, ws, ws_bytes, err, stream);
    case 4: return launch_wide<2, false>(x, y, m, l, rows, cols, ld_x, ld_y, k, ws, ws_bytes, err, stream);
    case 5: return launch_wide<2, true>(x, y, m, l, rows, cols, ld_x, ld_y, k, ws, ws_bytes, err, stream);
  }
  return false;
}

}  // namespace oss
