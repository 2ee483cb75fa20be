// G2: fused attention forward on the tcgen05 tensor cores (sm_103a).
//
// Per tile of scores S the running state of each query row is updated as the
// metalworking page's five-line recurrence states it ("Online Softmax"):
//   m_new = max(m, rowmax S);  c = 2^(m - m_new);  P = 2^(S - m_new);
//   l = l*c + rowsum P;        O = O*c + P V;      m = m_new;
// and after the last tile O /= l. Scores are kept in base 2 with
// scale * log2(e) folded in once, and every exponential is exp2, the rescale
// factor included (roadmapper "Online softmax", "Things that break"). The
// state starts at m = -inf, l = 0; a row whose keys are all masked so far
// subtracts 0 instead of -inf, so P = 0 and no NaN appears (roadmapper,
// "Initialise honestly"). No score row is ever written to memory (curionode
// "The Online Softmax.", "One pass, exactly").
//
// The rescale is conditional, in the spirit of the metal-flash-attention
// guard the metalworking page quotes (correction 1 unless the maximum rose):
// a warp moves its rows' reference maximum only when one of them rose by
// more than 2^8, so the O round trip through tensor memory is rare; any
// reference gives the same O / l in exact arithmetic, and weights stay
// below 256.
//
// Launches are persistent: one CTA of 352 threads per SM walks a share of the
// 128-row query tiles, and loads and QK^T of the next query tile start while
// the current one finishes. Non-causal tiles follow a round rule (work_tile);
// causal tiles, whose costs differ, follow a greedy schedule built on the
// host (tile_of). CTA layout:
//   * warps 0..7 -- softmax: warp w owns 16 query rows, tensor-memory lanes
//                   32 (w % 4) + 16 (w / 4) .. + 15; each row's scores are
//                   spread over four threads (the 16x256b access shape), so
//                   two softmax warps share each SM sub-partition and a row
//                   maximum takes two shuffles.
//   * warp 8     -- TMA producer: the Q tile of each query tile, then K and V
//                   tiles (128 keys) into two 3-stage rings, K two steps
//                   ahead of V.
//   * warp 9     -- one thread issues S_b = Q K_j^T (A, B from shared memory);
//                   the warp owns the tensor-memory allocation.
//   * warp 10    -- one thread issues O += P_j V_j (A = P from tensor memory,
//                   B from shared memory).
//   Issuing a tcgen05.mma costs its thread tens of cycles, so the two MMA
//   streams have a thread each.
// Tensor memory (512 fp32 columns x 128 lanes): S_0 | S_1 | S_2 | O. KV steps
// are counted across the CTA's query tiles; step g uses score buffer g % 3
// (and ring stage g % 3); the softmax writes P_g as bf16 pairs over the first
// 64 columns of S_{g % 3}. With three score buffers QK^T runs up to two steps
// ahead of the softmax. The epilogue of a query tile reads O out of tensor
// memory before the first P V of the next one overwrites it.
//
// Causal: query i sees keys 0..i (Sq == Sk). Query tiles start 64 rows before
// a KV-tile boundary; KV tiles wholly above the diagonal are skipped and the
// two diagonal tiles are visited first, from the last one down, so the first
// KV tile a causal CTA sees is masked for all of its first 64 rows -- the
// case the -inf guard exists for.
//
// Every wait on an mbarrier is bounded: on timeout the thread raises a
// CTA-wide abort flag and writes the device error word (tagged with the
// launch, so the launch's other CTAs stop too); all roles then drain their
// own in-flight copies and MMAs (again with a bound), and tensor memory is
// released before the CTA exits.

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "device_common.cuh"
#include "oss_internal.h"

namespace oss {
namespace {

constexpr int kD = 128;           // head dimension
constexpr int kBM = 128;          // query rows per CTA (= tensor-memory lanes)
constexpr int kBN = 128;          // keys per KV tile
constexpr int kStages = 3;        // depth of the K ring and of the V ring (= score buffers)
constexpr int kKLead = 2;         // K loads run this many steps ahead of V loads
constexpr int kSoftWarps = 8;     // warps 0..7: softmax, 16 query rows each
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kProducerWarp = 8;  // warp 8: TMA producer
constexpr int kQkWarp = 9;        // warp 9: issues S = Q K^T, owns tensor memory
constexpr int kPvWarp = 10;       // warp 10: issues O += P V
constexpr int kThreads = (kPvWarp + 1) * 32;
constexpr int kCausalShift = 64;  // causal query tiles start 64 rows before a KV tile
constexpr int kCausalGroup = 4;   // heads per causal scheduling group (K/V of 4 heads fit L2)

// shared memory (bytes from the 1024-aligned base); every operand is stored
// as two halves of 64 head dims (128-byte rows, 128-byte swizzle)
constexpr int kHalf = 128 * 128;                   // 128 rows x 64 bf16 = 16 KB
constexpr int kTile = 2 * kHalf;                   // 32 KB
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTile;
constexpr int kOffV = kOffK + kStages * kTile;
constexpr int kOffEnd = kOffV + kStages * kTile;   // 224 KB
constexpr int kSmemBytes = kOffEnd + 1024;         // + alignment slack

// tensor-memory columns (512 fp32 x 128 lanes): S_0 | S_1 | S_2 | O. KV step g
// (counted across the CTA's query tiles) uses score buffer g % 3; P_g (bf16
// pairs) is written over its first half.
constexpr int kSBuf = 3;
static_assert(kSBuf == kStages, "K/V ring stage and score buffer share one index");
constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t col_s(int b) { return 128u * b; }
constexpr uint32_t kColO = 384;

// When the rows' maxima are moved and O rescaled (the policy is a template
// parameter; the metalworking page, "Recognition guide", sets two real
// kernels side by side here: MLX multiplies O by the correction on every
// tile, metal-flash-attention only when the maximum rose). O lives in tensor
// memory, so a rescale costs the softmax warp a wait for the previous P V and
// a round trip of its rows of O; the decision is per warp (tensor-memory
// access is warp-wide):
//   kRescaleThreshold -- move a warp's reference maxima only when one of its
//                        rows rose by more than kRescaleSlack (base 2); weights
//                        stay below 2^kRescaleSlack. The default.
//   kRescaleOnRise    -- move them whenever one of its rows rose at all.
//   kRescaleAlways    -- move them (and rescale O) on every tile.
// Any reference below the true maximum gives the same O / l in exact
// arithmetic (it cancels), so all three compute the same result.
enum RescalePolicy : int { kRescaleThreshold = 0, kRescaleOnRise = 1, kRescaleAlways = 2 };
constexpr float kRescaleSlack = 8.0f;

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kDrainNs = 200000000ull;     // 0.2 s to drain own copies

// wait sites (error word bits 8..15)
enum Site : unsigned int {
  kSiteQFull = 1, kSiteKFull, kSiteVFull, kSiteKEmpty, kSiteVEmpty,
  kSiteSFull, kSitePReady, kSiteODone, kSiteDrain, kSiteQEmpty, kSiteOFree
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Non-blocking test of a phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait, slow path: polls until the phase completes, another thread
// aborts, or the time limit passes (then it raises the abort flag and
// records the site). Kept out of line; the fast path below is inlined
// because every wait sits on the pipeline's critical path (measured: an
// out-of-line call costs the caller a few hundred cycles).
// A give-up is recorded in the device error word together with the launch's
// tag (bits 16..31); the other CTAs of the same launch see the tag on their
// next slow-path poll and give up too, so a failed launch ends after one
// timeout instead of one per wave of CTAs.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned int* err, unsigned int site,
                                           uint64_t timeout_ns, unsigned int tag) {
  const uint64_t t0 = global_timer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((n & 63u) == 0) {
      const unsigned int e = *reinterpret_cast<volatile unsigned int*>(err);
      if (e != 0 && (e >> 16) == tag) {
        *abort_flag = 1;
        return false;
      }
      if (global_timer() - t0 > timeout_ns) {
        *abort_flag = 1;
        report_error(err, kKernelAttnFwd | (site << 8) | (tag << 16));
        return false;
      }
    }
  }
}

// Bounded wait. Returns false on timeout or when another thread has aborted.
// The limit is the kernel's timeout_ns (kTimeoutNs unless a test shortens it).
#define wait_bar(bar, parity, abort_flag, err, site) \
  (mbar_test_wait((bar), (parity)) ||                 \
   wait_bar_slow((bar), (parity), (abort_flag), (err), (site), p.timeout_ns, p.tag))

// Bounded wait used while draining: ignores the abort flag.
__device__ __noinline__ bool drain_bar(uint32_t bar, uint32_t parity, unsigned int* err) {
  const uint64_t t0 = global_timer();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0 && global_timer() - t0 > kDrainNs) {
      report_error(err, kKernelAttnFwd | (kSiteDrain << 8));
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

#define OSS_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define OSS_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                  "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
#define OSS_RW8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                   "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])

// Completes outstanding tcgen05.ld of this thread; the register operands tie
// the loaded values to the wait so no use is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  asm volatile("" : OSS_RW8(0), OSS_RW8(8), OSS_RW8(16), OSS_RW8(24));
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16 lanes x 64 columns (shape 16x256b, 8 repetitions). Thread t holds, for
// repetition k, columns 8k + 2(t%4) and 8k + 2(t%4) + 1 of lane t/4 in
// r[4k], r[4k+1] and of lane 8 + t/4 in r[4k+2], r[4k+3].
__device__ __forceinline__ void tmem_ld16x256_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : OSS_R8(0), OSS_R8(8), OSS_R8(16), OSS_R8(24)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16x256_x8(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      OSS_W8(0), OSS_W8(8), OSS_W8(16), OSS_W8(24)
      : "memory");
}

// 16 lanes x 32 columns (shape 16x128b, 8 repetitions). Thread t writes,
// for repetition k, column 4k + t%4 of lane t/4 from r[2k] and of lane
// 8 + t/4 from r[2k+1].
__device__ __forceinline__ void tmem_st16x128_x8(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      OSS_W8(0), OSS_W8(8)
      : "memory");
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 4 x 4 transpose of 32-bit words among the four lanes 4q .. 4q + 3 of a
// warp (j = lane % 4): lane j gives a[i] = element (j, i) and gets back
// a[i] = element (i, j). Two exchange rounds, at lane distance 1 and 2.
__device__ __forceinline__ void lane_transpose4(uint32_t (&a)[4], int j) {
  const bool o1 = (j & 1) != 0;
  uint32_t x = o1 ? a[0] : a[1];
  uint32_t y = o1 ? a[2] : a[3];
  x = __shfl_xor_sync(0xffffffffu, x, 1);
  y = __shfl_xor_sync(0xffffffffu, y, 1);
  if (o1) { a[0] = x; a[2] = y; } else { a[1] = x; a[3] = y; }
  const bool o2 = (j & 2) != 0;
  x = o2 ? a[0] : a[2];
  y = o2 ? a[1] : a[3];
  x = __shfl_xor_sync(0xffffffffu, x, 2);
  y = __shfl_xor_sync(0xffffffffu, y, 2);
  if (o2) { a[0] = x; a[1] = y; } else { a[2] = x; a[3] = y; }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
  return w;
}

// ---------------------------------------------------------------------------
// Descriptors
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (16-byte units), the fixed 0b001 field at bit 46,
// swizzle mode 2 at bits 61..63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
         (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B
// bf16 (bits 7-9 = 1, 10-12 = 1), A K-major, B K-major (bit 16 = 0) or
// N-major (bit 16 = 1), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t make_idesc(uint32_t M, uint32_t N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((N >> 3) << 17) | ((M >> 4) << 24);
}
constexpr uint32_t kIdescQK = make_idesc(kBM, kBN, false);  // S = Q K^T (N = 128 keys)
constexpr uint32_t kIdescPV = make_idesc(kBM, kD, true);    // O += P V (N = 128 dims)

// A 16-element step along K of a K-major operand moves 32 bytes inside the
// 128-byte swizzled row (the first four steps), then to the second half.
__device__ __forceinline__ uint64_t kstep_kmajor(int kk, int half_bytes) {
  return static_cast<uint64_t>((kk >> 2) * (half_bytes >> 4) + (kk & 3) * 2);
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

struct AttnParams {
  uint16_t* o;
  float* lse;
  unsigned int* err;
  int Sq, Sk, BH, n_qblocks, n_tiles;
  float C;  // scale * log2(e)
  int causal;
  uint64_t timeout_ns;  // limit of every bounded wait
  unsigned int tag;     // launch tag, 1..65535, in bits 16..31 of a reported error
  int skip_v_step;      // test hook: the producer skips the V load of this step (-1: none)
  // partial-state output (sequence-sharded attention): when part_o != null the
  // epilogue writes (m, l, O unnormalised) of row r to slot part_index of a
  // [rows, part_stride] partial array instead of O / l and lse
  float* part_m;
  float* part_l;
  float* part_o;
  int part_stride, part_index;
  // Split tail (non-causal, with a workspace): after full_rounds rounds of
  // whole query tiles, the remaining tiles from split_first on are cut along
  // the keys into split_f parts, one part per CTA; each part writes its
  // (m, l, O) to the workspace and the last part of a tile to finish merges
  // them. split_f < 2: no split.
  int full_rounds, split_first, split_f, split_items;
  float* ws_o;            // [split tiles][split_f][16][softmax threads][4]: unnormalised O
  float* ws_ml;           // [split tiles][split_f][softmax threads][4]: base-2 m, l of rows a, b
  unsigned int* ws_cnt;   // [split tiles][softmax warps]: (launch tag << 8) | parts done
};

struct Barriers {
  uint64_t q_full;   // Q tile landed
  uint64_t q_free;   // every QK^T of the tile in the Q buffer is done
  uint64_t k_full[kStages], v_full[kStages];
  uint64_t s_full[kSBuf];
  uint64_t p_ready[2][kSBuf];  // P of keys 0..63 / 64..127 written (the two halves of P V)
  uint64_t o_done[kSBuf];  // P V done, for the steps of each buffer (keeps parity waits exact)
  uint64_t o_free;   // the epilogue has read O out of tensor memory
  uint64_t drain[2];  // one per issuing thread
};

// A unit of work: query tile `lin`, whole (part < 0) or part `part` of a tile
// split along the keys.
struct Work {
  int lin, part;
};

// A query tile: (b, h), first query row, number of KV tiles and how many of
// them (the diagonal ones, causal only) are visited first; the work unit
// visits n_steps of them, from position kv_lo of that order.
struct TileInfo {
  int bh, q0, n_kv, n_diag;
  int kv_lo, n_steps, part, tail;
};

// Query tile number lin of the launch. Causal tiles start kCausalShift rows
// before a KV tile boundary (the first tile hangs over row 0; the TMA fills
// the rows above with zeros). Numbering: the tiles processed at the same time
// should share (b, h), so that K and V are read from HBM once and then from
// L2. Non-causal: (b, h)-major. Causal: groups of kCausalGroup heads,
// heaviest query tiles first within each group.
__host__ __device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int imax(int a, int b) { return a > b ? a : b; }

__host__ __device__ __forceinline__ TileInfo tile_info(const AttnParams& p, Work w) {
  const int lin = w.lin;
  int bh, qb;
  if (!p.causal) {
    bh = lin / p.n_qblocks;
    qb = lin - bh * p.n_qblocks;
  } else {
    const int per_group = kCausalGroup * p.n_qblocks;
    const int g = lin / per_group;
    const int gsize = imin(kCausalGroup, p.BH - g * kCausalGroup);
    const int r = lin - g * per_group;
    const int qb_lin = r / gsize;
    bh = g * kCausalGroup + (r - qb_lin * gsize);
    qb = p.n_qblocks - 1 - qb_lin;
  }
  TileInfo t;
  t.bh = bh;
  t.q0 = qb * kBM - (p.causal ? kCausalShift : 0);
  const int kv_end = p.causal ? imin(p.Sk, t.q0 + kBM) : p.Sk;
  t.n_kv = (kv_end + kBN - 1) / kBN;
  // KV tiles that reach past the tile's first row touch the diagonal; they
  // are visited first, from the last one down: for a shifted causal tile the
  // first one is masked for all of the tile's first kCausalShift rows.
  const int diag_first = p.causal ? imax(0, t.q0) / kBN : t.n_kv;
  t.n_diag = t.n_kv - diag_first;
  t.part = w.part;
  if (w.part < 0) {
    t.kv_lo = 0;
    t.n_steps = t.n_kv;
    t.tail = -1;
  } else {  // keys of part i: KV tiles [i n / f, (i + 1) n / f)
    t.kv_lo = w.part * t.n_kv / p.split_f;
    t.n_steps = (w.part + 1) * t.n_kv / p.split_f - t.kv_lo;
    t.tail = lin - p.split_first;
  }
  return t;
}

// KV tile visited at step j of a work unit.
__device__ __forceinline__ int kv_tile(const TileInfo& t, int j) {
  const int v = t.kv_lo + j;
  return v < t.n_diag ? (t.n_kv - 1 - v) : (v - t.n_diag);
}

// The k-th query tile of this CTA, or -1. With G CTAs, round k hands tiles
// k*G .. k*G + G - 1 to them, in reverse CTA order on odd rounds (a CTA that
// drew a heavier tile in one round draws a lighter one in the next). With
// one CTA per tile (G = number of tiles) CTA i takes tile i only.
__device__ __forceinline__ int work_tile(int k, int n_tiles) {
  const int G = static_cast<int>(gridDim.x);
  const int idx = (k & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const long long lin = static_cast<long long>(k) * G + idx;
  return lin < n_tiles ? static_cast<int>(lin) : -1;
}

// Per-CTA lists of query tiles, for causal launches: computed on the host
// (greedy, heaviest first: the tiles in their launch order, each to the CTA
// with the least work so far) and passed as a kernel parameter.
constexpr int kSchedMaxCtas = 160;
constexpr int kSchedMaxTiles = 15000;
template <bool kSched>
struct TileSched {
  unsigned char unused;
};
template <>
struct TileSched<true> {
  uint16_t off[kSchedMaxCtas + 1];  // CTA c walks list[off[c] .. off[c + 1])
  uint16_t list[kSchedMaxTiles];
};

// The k-th work unit of this CTA (lin < 0: none left): from the host's lists,
// or by the round rule of work_tile, then, with a split tail, one part of a
// split tile per CTA.
template <bool kSched>
__device__ __forceinline__ Work tile_of(int k, const AttnParams& p, const TileSched<kSched>& sc) {
  if constexpr (kSched) {
    const int b = sc.off[blockIdx.x];
    return {(b + k < static_cast<int>(sc.off[blockIdx.x + 1])) ? static_cast<int>(sc.list[b + k]) : -1,
            -1};
  } else {
    if (p.split_f < 2) return {work_tile(k, p.n_tiles), -1};
    if (k < p.full_rounds) return {work_tile(k, p.n_tiles), -1};
    const int seg = static_cast<int>(blockIdx.x);
    if (k == p.full_rounds && seg < p.split_items)
      return {p.split_first + seg / p.split_f, seg % p.split_f};
    return {-1, -1};
  }
}

constexpr int kMaxSplit = 8;  // parts a split tile is cut into at most

// Counts one finished part of a split tile on its counter and returns how
// many of the tile's parts are done, this one included. The counter holds
// (launch tag << 8) | parts done; a value left by another launch (one that
// gave up on a wait, say) carries another tag and counts as zero. The
// compare-and-swap has acquire-release semantics at GPU scope: it publishes
// the part this warp has written (its lanes' stores are ordered before it
// by the warp barrier the caller takes) and, for the last part, makes every
// other part's stores visible. At most kMaxSplit threads contend for a
// counter, so the loop ends within that many rounds; the bound only guards
// against the impossible.
__device__ __forceinline__ unsigned int count_part(unsigned int* c, unsigned int tag) {
  unsigned int cur;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(cur) : "l"(c) : "memory");
  for (int round = 0; round < 4 * kMaxSplit; ++round) {
    const unsigned int n = ((cur >> 8) == tag) ? (cur & 0xffu) + 1u : 1u;
    unsigned int seen;
    asm volatile("atom.acq_rel.gpu.global.cas.b32 %0, [%1], %2, %3;"
                 : "=r"(seen)
                 : "l"(c), "r"(cur), "r"((tag << 8) | n)
                 : "memory");
    if (seen == cur) return n;
    cur = seen;
  }
  return 0;
}

// Stores half h (head dims 64 h .. 64 h + 63) of two rows of O in bf16:
// va[2 k + e], vb[2 k + e] hold dims 64 h + 8 k + cq + e of rows a and b,
// scaled by inv_a, inv_b. Each 8-dim chunk of a row is spread over the row's
// four threads (2 dims each); a 4 x 4 transpose among them hands every
// thread whole chunks, written with 16-byte stores.
__device__ __forceinline__ void store_o_half(uint4* oa, uint4* ob, const float (&va)[16],
                                             const float (&vb)[16], float inv_a, float inv_b,
                                             int h, int jj, bool live_a, bool live_b) {
#pragma unroll
  for (int mb = 0; mb < 2; ++mb) {
    uint32_t wa[4], wb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = 4 * mb + i;  // chunk 8 h + k of the row
      wa[i] = pack_bf16x2(va[2 * k] * inv_a, va[2 * k + 1] * inv_a);
      wb[i] = pack_bf16x2(vb[2 * k] * inv_b, vb[2 * k + 1] * inv_b);
    }
    lane_transpose4(wa, jj);
    lane_transpose4(wb, jj);
    const int chunk = 8 * h + 4 * mb + jj;
    if (live_a) oa[chunk] = make_uint4(wa[0], wa[1], wa[2], wa[3]);
    if (live_b) ob[chunk] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
  }
}

template <bool kSched, int kPolicy>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q,
                const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const AttnParams p,
                const __grid_constant__ TileSched<kSched> sched) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bars.q_full), 1);
    mbar_init(smem_addr(&bars.q_free), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&bars.k_full[s]), 1);
      mbar_init(smem_addr(&bars.v_full[s]), 1);
    }
    for (int b = 0; b < kSBuf; ++b) {
      mbar_init(smem_addr(&bars.s_full[b]), 1);
      mbar_init(smem_addr(&bars.p_ready[0][b]), kSoftThreads);
      mbar_init(smem_addr(&bars.p_ready[1][b]), kSoftThreads);
      mbar_init(smem_addr(&bars.o_done[b]), 1);
    }
    mbar_init(smem_addr(&bars.o_free), kSoftThreads);
    mbar_init(smem_addr(&bars.drain[0]), 1);
    mbar_init(smem_addr(&bars.drain[1]), 1);
    abort_flag_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == kQkWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_slot;

  // Every role walks the same sequence of query tiles (work_tile) and counts
  // KV steps g across them: step g uses ring stage and score buffer g % 3, in
  // round g / 3, so the pipeline runs on from one query tile into the next.
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_q)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_v)) : "memory");
      const uint32_t qbar = smem_addr(&bars.q_full);
      // K_g is consumed by QK_g, which runs up to two steps ahead of P_g V,
      // the consumer of V_g; so K loads run kKLead steps ahead of V loads,
      // and each ring is refilled as soon as its own consumer is done: K stage
      // g % 3 when QK_g has completed (s_full), V stage g % 3 when P_g V has
      // (o_done) -- ring stage and score buffer coincide. The KV tile and
      // (b, h) of each K load are kept for the V load of the same step.
      int k_issued = 0, v_issued = 0, q_loads = 0, skipped_v = -1;
      int key_row[kStages] = {0, 0, 0}, key_bh[kStages] = {0, 0, 0};
      int kt = 0, j = 0;  // K stream: tile ordinal, step within the tile
      Work wk = tile_of(0, p, sched);
      TileInfo t{};
      if (wk.lin >= 0) t = tile_info(p, wk);
      for (int g = 0;; ++g) {
        // V of step g - kKLead first: it is the load the P V thread waits on
        // soonest, and the Q wait below may block until this tile's QK^T end
        const int gv = g - kKLead;
        if (gv >= 0 && gv < k_issued) {
          if (gv == p.skip_v_step) {
            skipped_v = gv;  // test hook: this V tile never arrives
          } else {
            const int s = gv % kStages;
            const int round = gv / kStages;
            if (round > 0 && !wait_bar(smem_addr(&bars.o_done[s]), (round - 1) & 1, abort_flag,
                                       p.err, kSiteVEmpty))
              break;
            const uint32_t vb = smem_addr(&bars.v_full[s]);
            mbar_expect_tx(vb, kTile);
            for (int h = 0; h < 2; ++h)
              tma_load_3d(sbase + kOffV + s * kTile + h * kHalf, &tmap_v, vb, h * 64, key_row[s],
                          key_bh[s]);
            v_issued = gv + 1;
          }
        }
        if (wk.lin < 0) {
          if (gv + 1 >= k_issued) break;  // the last V load has been issued
          continue;
        }
        if (j == 0) {
          // the single Q buffer is free once every QK^T of the previous tile is done
          if (kt > 0 && !wait_bar(smem_addr(&bars.q_free), (kt - 1) & 1, abort_flag, p.err,
                                  kSiteQEmpty))
            break;
          mbar_expect_tx(qbar, kTile);
          for (int h = 0; h < 2; ++h)
            tma_load_3d(sbase + kOffQ + h * kHalf, &tmap_q, qbar, h * 64, t.q0, t.bh);
          ++q_loads;
        }
        const int s = g % kStages;
        const int round = g / kStages;
        if (round > 0 && !wait_bar(smem_addr(&bars.s_full[s]), (round - 1) & 1, abort_flag,
                                   p.err, kSiteKEmpty))
          break;
        const uint32_t kb = smem_addr(&bars.k_full[s]);
        mbar_expect_tx(kb, kTile);
        key_row[s] = kv_tile(t, j) * kBN;
        key_bh[s] = t.bh;
        for (int h = 0; h < 2; ++h)
          tma_load_3d(sbase + kOffK + s * kTile + h * kHalf, &tmap_k, kb, h * 64, key_row[s],
                      key_bh[s]);
        k_issued = g + 1;
        if (++j == t.n_steps) {
          j = 0;
          wk = tile_of(++kt, p, sched);
          if (wk.lin >= 0) t = tile_info(p, wk);
        }
      }
      // drain: every issued copy must land before the CTA may exit
      if (q_loads > 0) drain_bar(qbar, (q_loads - 1) & 1, p.err);
      for (int i = k_issued - 1; i >= 0 && i >= k_issued - kStages; --i)
        drain_bar(smem_addr(&bars.k_full[i % kStages]), (i / kStages) & 1, p.err);
      for (int i = v_issued - 1; i >= 0 && i >= v_issued - kStages; --i)
        if (i != skipped_v) drain_bar(smem_addr(&bars.v_full[i % kStages]), (i / kStages) & 1, p.err);
    }
  } else if (warp == kQkWarp) {
    // ------------------------------------------------------------ QK issuer
    // S_{g % 3} = Q K_g^T: the buffer last held P_{g-3}, so P_{g-3} V must be
    // done with it. Issuing a tcgen05.mma costs its thread tens of cycles, so
    // QK^T and P V are issued by two threads.
    if (lane == 0) {
      bool ok = true;
      // operand descriptors built once; a 16-element K step only adds a
      // constant to the start-address field (16-byte units)
      const uint64_t dq = smem_desc(sbase + kOffQ, 16, 1024);
      int g = 0;
      for (int kt = 0; ok; ++kt) {
        const Work wk = tile_of(kt, p, sched);
        if (wk.lin < 0) break;
        const TileInfo t = tile_info(p, wk);
        if (!(ok = wait_bar(smem_addr(&bars.q_full), kt & 1, abort_flag, p.err, kSiteQFull)))
          break;
        // The previous tile's last P V goes through the tensor pipe before this
        // tile's first QK^T: its epilogue waits on it, while the softmax has
        // nothing to do with the new scores until that epilogue is over. (The
        // wait is exact: the next phase of that o_done needs a QK^T this thread
        // has not issued.)
        if (kt > 0 && !(ok = wait_bar(smem_addr(&bars.o_done[(g - 1) % kStages]),
                                      ((g - 1) / kStages) & 1, abort_flag, p.err, kSiteODone)))
          break;
        for (int j = 0; j < t.n_steps; ++j, ++g) {
          const int s = g % kStages;  // K stage = score buffer
          if (!(ok = wait_bar(smem_addr(&bars.k_full[s]), (g / kStages) & 1, abort_flag, p.err,
                              kSiteKFull)))
            break;
          if (g >= kStages && !(ok = wait_bar(smem_addr(&bars.o_done[s]), (g / kStages - 1) & 1,
                                              abort_flag, p.err, kSiteODone)))
            break;
          tc_fence_after();
          const uint64_t dk = smem_desc(sbase + kOffK + s * kTile, 16, 1024);
          const uint32_t d_s = tbase + col_s(s);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_ss(d_s, dq + kstep_kmajor(kk, kHalf), dk + kstep_kmajor(kk, kHalf), kIdescQK,
                   kk > 0 ? 1u : 0u);
          tc_commit(smem_addr(&bars.s_full[s]));  // scores ready; K stage s free
        }
        if (ok) tc_commit(smem_addr(&bars.q_free));  // Q buffer free once these MMAs are done
      }
      // drain: no MMA of this thread may still write tensor memory when it is freed
      tc_commit(smem_addr(&bars.drain[0]));
      drain_bar(smem_addr(&bars.drain[0]), 0, p.err);
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    // O += P_g V_g once the softmax has written P_g over S_{g % 3}. The first
    // step of a query tile overwrites O, so it also waits until the epilogue
    // of the previous tile has read O out.
    if (lane == 0) {
      bool ok = true;
      const uint32_t d_o = tbase + kColO;
      int g = 0;
      for (int kt = 0; ok; ++kt) {
        const Work wk = tile_of(kt, p, sched);
        if (wk.lin < 0) break;
        const TileInfo t = tile_info(p, wk);
        for (int j = 0; j < t.n_steps; ++j, ++g) {
          const int s = g % kStages;
          if (!(ok = wait_bar(smem_addr(&bars.v_full[s]), (g / kStages) & 1, abort_flag, p.err,
                              kSiteVFull)))
            break;
          if (j == 0 && kt > 0 &&
              !(ok = wait_bar(smem_addr(&bars.o_free), (kt - 1) & 1, abort_flag, p.err,
                              kSiteOFree)))
            break;
          // the two halves of P V (keys 0..63, 64..127) start as soon as the
          // softmax has written the matching half of P
          const uint64_t dv = smem_desc(sbase + kOffV + s * kTile, kHalf, 1024);
          const uint32_t a_p = tbase + col_s(s);
#pragma unroll
          for (int hp = 0; hp < 2; ++hp) {
            if (!(ok = wait_bar(smem_addr(&bars.p_ready[hp][s]), (g / kStages) & 1, abort_flag,
                                p.err, kSitePReady)))
              break;
            tc_fence_after();
#pragma unroll
            for (int kk = 4 * hp; kk < 4 * hp + 4; ++kk)
              mma_ts(d_o, a_p + kk * 8, dv + static_cast<uint64_t>(kk * (2048 >> 4)), kIdescPV,
                     (j > 0 || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          tc_commit(smem_addr(&bars.o_done[s]));  // buffer s and V stage s free
        }
      }
      tc_commit(smem_addr(&bars.drain[1]));
      drain_bar(smem_addr(&bars.drain[1]), 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w owns 16 query rows: lanes 32 (w % 4) + 16 (w / 4) .. + 15 of
    // tensor memory (a warp reaches only its quadrant 32 (w % 4) .. + 31).
    // In the 16x256b access shape each row's 128 scores are spread over four
    // consecutive threads, 32 each; thread t holds rows ra = t/4 and rb =
    // 8 + t/4 of the warp's 16, columns 8k + cq + {0, 1} (cq = 2 (t % 4)).
    // Row maxima are finished with two shuffles; the row sums stay per
    // thread (the four threads of a row share its reference maximum) and are
    // added up once, after the last KV tile.
    const int lane0 = (warp & 3) * 32 + (warp >> 2) * 16;  // first lane of this warp
    const int ra = lane0 + (lane >> 2);
    const int rb = ra + 8;
    const int cq = 2 * (lane & 3);
    const uint32_t tl = tbase + (static_cast<uint32_t>(lane0) << 16);
    const float C = p.C;
    bool ok = true;
    int g = 0;
    for (int kt = 0; ok; ++kt) {
      const Work wk = tile_of(kt, p, sched);
      if (wk.lin < 0) break;
      const TileInfo t = tile_info(p, wk);
      const int row_a = t.q0 + ra, row_b = t.q0 + rb;  // query indices (may be < 0: padding)
      float m_a = neg_inf(), m_b = neg_inf();       // reference maxima, base 2
      float mt_a = neg_inf(), mt_b = neg_inf();     // true row maxima, base 2 (partial states)
      float l_a = 0.f, l_b = 0.f;                   // this thread's share of the row sums
      for (int j = 0; j < t.n_steps; ++j, ++g) {
        const int b = g % kSBuf;
        const uint32_t colS = col_s(b);
        ok = __all_sync(0xffffffffu, wait_bar(smem_addr(&bars.s_full[b]), (g / kSBuf) & 1,
                                              abort_flag, p.err, kSiteSFull));
        if (!ok) break;
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld16x256_x8(tl + colS, r0);        // columns 0..63
        tmem_ld16x256_x8(tl + colS + 64, r1);   // columns 64..127
        tmem_ld_wait(r0);
        tmem_ld_wait(r1);
        // sa[16 h + 2 k + e], sb[...]: column 64 h + 8 k + cq + e of rows ra, rb
        float sa[32], sb[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            sa[2 * k + e] = __uint_as_float(r0[4 * k + e]);
            sb[2 * k + e] = __uint_as_float(r0[4 * k + 2 + e]);
            sa[16 + 2 * k + e] = __uint_as_float(r1[4 * k + e]);
            sb[16 + 2 * k + e] = __uint_as_float(r1[4 * k + 2 + e]);
          }
        }
        const int key0 = kv_tile(t, j) * kBN;
        const bool ragged = key0 + kBN > p.Sk;
        const bool diag = p.causal && key0 + kBN - 1 > t.q0;
        if (ragged || diag) {
          // visible keys of a row: column < lim
          const int lim_a = min(p.Sk, p.causal ? row_a + 1 : p.Sk) - key0;
          const int lim_b = min(p.Sk, p.causal ? row_b + 1 : p.Sk) - key0;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int col = (i >> 4) * 64 + ((i >> 1) & 7) * 8 + cq + (i & 1);
            if (col >= lim_a) sa[i] = neg_inf();
            if (col >= lim_b) sb[i] = neg_inf();
          }
        }
        // row maxima: this thread's 32 columns, then the row's four threads
        float xa0 = neg_inf(), xa1 = neg_inf(), xb0 = neg_inf(), xb1 = neg_inf();
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          xa0 = fmax3(xa0, sa[i], sa[i + 1]);
          xa1 = fmax3(xa1, sa[i + 2], sa[i + 3]);
          xb0 = fmax3(xb0, sb[i], sb[i + 1]);
          xb1 = fmax3(xb1, sb[i + 2], sb[i + 3]);
        }
        float xa = fmaxf(xa0, xa1), xb = fmaxf(xb0, xb1);
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 1));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 1));
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 2));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 2));
        const float mtile_a = xa * C, mtile_b = xb * C;
        const float mnew_a = fmaxf(m_a, mtile_a), mnew_b = fmaxf(m_b, mtile_b);
        mt_a = fmaxf(mt_a, mtile_a);
        mt_b = fmaxf(mt_b, mtile_b);
        // Move the reference maxima (and rescale O) as the policy says;
        // between moves the weights are taken relative to a reference at most
        // kRescaleSlack below the true maximum (threshold policy).
        bool rescale;
        if constexpr (kPolicy == kRescaleAlways)
          rescale = true;
        else if constexpr (kPolicy == kRescaleOnRise)
          rescale = __any_sync(0xffffffffu, (mnew_a > m_a) || (mnew_b > m_b));
        else
          rescale = __any_sync(0xffffffffu, (mnew_a > m_a + kRescaleSlack) ||
                                                (mnew_b > m_b + kRescaleSlack));
        float corr_a = 1.f, corr_b = 1.f;
        if (rescale) {
          corr_a = ex2(m_a - ((mnew_a == neg_inf()) ? 0.f : mnew_a));  // 0 while m = -inf
          corr_b = ex2(m_b - ((mnew_b == neg_inf()) ? 0.f : mnew_b));
          m_a = mnew_a;
          m_b = mnew_b;
        }
        if (rescale && j > 0) {
          // O still holds the previous tiles' sum: wait for P_{j-1} V (whose
          // completion implies every earlier one), then rescale this warp's rows
          ok = __all_sync(0xffffffffu, wait_bar(smem_addr(&bars.o_done[(g - 1) % kSBuf]),
                                                ((g - 1) / kSBuf) & 1, abort_flag, p.err, kSiteODone));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            uint32_t ov[32];
            tmem_ld16x256_x8(tl + kColO + 64 * h, ov);
            tmem_ld_wait(ov);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float2 oa = __fmul2_rn(make_float2(__uint_as_float(ov[4 * k]), __uint_as_float(ov[4 * k + 1])),
                                           make_float2(corr_a, corr_a));
              const float2 ob = __fmul2_rn(make_float2(__uint_as_float(ov[4 * k + 2]), __uint_as_float(ov[4 * k + 3])),
                                           make_float2(corr_b, corr_b));
              ov[4 * k] = __float_as_uint(oa.x);
              ov[4 * k + 1] = __float_as_uint(oa.y);
              ov[4 * k + 2] = __float_as_uint(ob.x);
              ov[4 * k + 3] = __float_as_uint(ob.y);
            }
            tmem_st16x256_x8(tl + kColO + 64 * h, ov);
          }
        }
        // P = 2^(S C - m), the -inf guard subtracting 0 for an empty row, in two
        // halves of 64 keys; each half is released to P V as soon as it is in
        // tensor memory (the O rescale above is complete by then: the first
        // tcgen05.wait::st covers it). bf16 pairs (keys c, c + 1) go to packed
        // column c / 2 = 32 h + 4 k + t % 4, where the 16x128b shape puts
        // repetition k of thread t when it writes packed columns 32 h .. + 31.
        const float2 Cv = make_float2(C, C);
        const float2 mva = make_float2(-((m_a == neg_inf()) ? 0.f : m_a), -((m_a == neg_inf()) ? 0.f : m_a));
        const float2 mvb = make_float2(-((m_b == neg_inf()) ? 0.f : m_b), -((m_b == neg_inf()) ? 0.f : m_b));
        float2 acc_a = make_float2(0.f, 0.f), acc_b = acc_a;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int kk = 8 * h + k;
            const float2 ta = __ffma2_rn(make_float2(sa[2 * kk], sa[2 * kk + 1]), Cv, mva);
            const float2 tb = __ffma2_rn(make_float2(sb[2 * kk], sb[2 * kk + 1]), Cv, mvb);
            const float2 ea = make_float2(ex2(ta.x), ex2(ta.y));
            const float2 eb = make_float2(ex2(tb.x), ex2(tb.y));
            acc_a = __fadd2_rn(acc_a, ea);
            acc_b = __fadd2_rn(acc_b, eb);
            pk[2 * k] = pack_bf16x2(ea.x, ea.y);
            pk[2 * k + 1] = pack_bf16x2(eb.x, eb.y);
          }
          tmem_st16x128_x8(tl + colS + 32 * h, pk);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(smem_addr(&bars.p_ready[h][b]));
        }
        l_a = fmaf(l_a, corr_a, acc_a.x + acc_a.y);
        l_b = fmaf(l_b, corr_b, acc_b.x + acc_b.y);
      }
      // the row sums: the four threads of a row add their shares
      l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
      l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
      // epilogue: O / l and lse for these rows, once the tile's last P V is
      // done (its completion implies every earlier one)
      if (ok)
        ok = __all_sync(0xffffffffu, wait_bar(smem_addr(&bars.o_done[(g - 1) % kSBuf]),
                                              ((g - 1) / kSBuf) & 1, abort_flag, p.err, kSiteODone));
      const bool live_a = row_a >= 0 && row_a < p.Sq;
      const bool live_b = row_b >= 0 && row_b < p.Sq;
      const bool writes_row = (lane & 3) == 0;  // one thread per row writes m, l, lse
      if (ok && p.part_o) {
        // partial state relative to the true row maximum: rescale the sums
        // taken against the reference by 2^(m_ref - m_true) <= 1
        tc_fence_after();
        const bool empty_a = (mt_a == neg_inf()) || !(l_a > 0.f);
        const bool empty_b = (mt_b == neg_inf()) || !(l_b > 0.f);
        const float f_a = empty_a ? 0.f : ex2(m_a - mt_a);
        const float f_b = empty_b ? 0.f : ex2(m_b - mt_b);
        const size_t slot_a = (static_cast<size_t>(t.bh) * p.Sq + row_a) * p.part_stride + p.part_index;
        const size_t slot_b = (static_cast<size_t>(t.bh) * p.Sq + row_b) * p.part_stride + p.part_index;
        float2* oa = reinterpret_cast<float2*>(p.part_o + slot_a * kD);
        float2* ob = reinterpret_cast<float2*>(p.part_o + slot_b * kD);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t ov[32];
          tmem_ld16x256_x8(tl + kColO + 64 * h, ov);
          tmem_ld_wait(ov);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int col = 64 * h + 8 * k + cq;
            if (live_a)
              oa[col >> 1] = make_float2(__uint_as_float(ov[4 * k]) * f_a, __uint_as_float(ov[4 * k + 1]) * f_a);
            if (live_b)
              ob[col >> 1] = make_float2(__uint_as_float(ov[4 * k + 2]) * f_b, __uint_as_float(ov[4 * k + 3]) * f_b);
          }
        }
        if (writes_row) {
          const float kLn2 = 0.69314718055994530942f;
          if (live_a) {
            p.part_m[slot_a] = empty_a ? neg_inf() : mt_a * kLn2;
            p.part_l[slot_a] = empty_a ? 0.f : l_a * f_a;
          }
          if (live_b) {
            p.part_m[slot_b] = empty_b ? neg_inf() : mt_b * kLn2;
            p.part_l[slot_b] = empty_b ? 0.f : l_b * f_b;
          }
        }
      } else if (ok && t.part >= 0) {
        // A part of a split tile: its (m, l, O) go to the workspace; the last
        // part of the tile to finish merges every part, in part order, so the
        // result does not depend on which CTA merges. A thread's 64 values of
        // O (rows a, b; the 16x256b layout) are 16 vectors of 4; vector e of
        // the CTA's 256 threads lies contiguous, so every warp access is 512
        // contiguous bytes, and the part that merges reads the same thread's
        // vectors of the other parts.
        tc_fence_after();
        const int f = p.split_f;
        const int me = warp * 32 + lane;                       // this thread's slot in a part
        const size_t part0 = static_cast<size_t>(t.tail) * f;  // part 0 of this tile
        {
          // O of this part, [h][k][a0 a1 b0 b1]: 16 float4 per thread
          float4* wo = reinterpret_cast<float4*>(p.ws_o) + (part0 + t.part) * 16 * kSoftThreads + me;
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            uint32_t ov[32];
            tmem_ld16x256_x8(tl + kColO + 64 * h, ov);
            tmem_ld_wait(ov);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              wo[(8 * h + e) * kSoftThreads] = make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                                          __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3]));
          }
          reinterpret_cast<float4*>(p.ws_ml)[(part0 + t.part) * kSoftThreads + me] =
              make_float4(m_a, l_a, m_b, l_b);
        }
        __syncwarp();
        unsigned int* cnt = p.ws_cnt + static_cast<size_t>(t.tail) * kSoftWarps + warp;
        unsigned int done = 0;
        if (lane == 0) done = count_part(cnt, p.tag);
        done = __shfl_sync(0xffffffffu, done, 0);
        __syncwarp();  // the lanes' reads below come after lane 0's acquire
        if (done == static_cast<unsigned int>(f)) {
          // the merge identity over the parts: M = max m_i, weights 2^(m_i - M)
          float4 st[kMaxSplit];
#pragma unroll
          for (int i = 0; i < kMaxSplit; ++i)
            st[i] = (i < f) ? __ldcg(reinterpret_cast<const float4*>(p.ws_ml) + (part0 + i) * kSoftThreads + me)
                            : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
          float Ma = neg_inf(), Mb = neg_inf();
#pragma unroll
          for (int i = 0; i < kMaxSplit; ++i) {
            Ma = fmaxf(Ma, st[i].x);
            Mb = fmaxf(Mb, st[i].z);
          }
          float La = 0.f, Lb = 0.f;
          float wpa[kMaxSplit], wpb[kMaxSplit];
#pragma unroll
          for (int i = 0; i < kMaxSplit; ++i) {
            wpa[i] = (st[i].x == neg_inf()) ? 0.f : ex2(st[i].x - Ma);
            wpb[i] = (st[i].z == neg_inf()) ? 0.f : ex2(st[i].z - Mb);
            La = fmaf(wpa[i], st[i].y, La);
            Lb = fmaf(wpb[i], st[i].w, Lb);
          }
          // acc = sum_i w_i O_i in part order, so every CTA that merges
          // rounds the same way
          float acc[64];
#pragma unroll
          for (int e = 0; e < 64; ++e) acc[e] = 0.f;
#pragma unroll 1
          for (int i = 0; i < f; ++i) {
            float xa = 0.f, xb = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxSplit; ++q)
              if (q == i) { xa = wpa[q]; xb = wpb[q]; }
            float4 v4[16];
            const float4* po = reinterpret_cast<const float4*>(p.ws_o) + (part0 + i) * 16 * kSoftThreads + me;
#pragma unroll
            for (int e = 0; e < 16; ++e) v4[e] = __ldcg(po + e * kSoftThreads);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              acc[4 * e] = fmaf(xa, v4[e].x, acc[4 * e]);
              acc[4 * e + 1] = fmaf(xa, v4[e].y, acc[4 * e + 1]);
              acc[4 * e + 2] = fmaf(xb, v4[e].z, acc[4 * e + 2]);
              acc[4 * e + 3] = fmaf(xb, v4[e].w, acc[4 * e + 3]);
            }
          }
          const float inv_a = (La > 0.f) ? 1.0f / La : 0.f;
          const float inv_b = (Lb > 0.f) ? 1.0f / Lb : 0.f;
          uint4* oa = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(t.bh) * p.Sq + row_a) * kD);
          uint4* ob = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(t.bh) * p.Sq + row_b) * kD);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float va[16], vb[16];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              va[2 * k] = acc[32 * h + 4 * k];
              va[2 * k + 1] = acc[32 * h + 4 * k + 1];
              vb[2 * k] = acc[32 * h + 4 * k + 2];
              vb[2 * k + 1] = acc[32 * h + 4 * k + 3];
            }
            store_o_half(oa, ob, va, vb, inv_a, inv_b, h, lane & 3, live_a, live_b);
          }
          if (writes_row && p.lse) {
            const float kLn2 = 0.69314718055994530942f;
            if (live_a)
              p.lse[static_cast<size_t>(t.bh) * p.Sq + row_a] = (La > 0.f) ? (Ma + __log2f(La)) * kLn2 : neg_inf();
            if (live_b)
              p.lse[static_cast<size_t>(t.bh) * p.Sq + row_b] = (Lb > 0.f) ? (Mb + __log2f(Lb)) * kLn2 : neg_inf();
          }
          __syncwarp();
          if (lane == 0) *cnt = 0u;  // ready for the next launch
        }
      } else if (ok) {
        tc_fence_after();
        const float inv_a = (l_a > 0.f) ? 1.0f / l_a : 0.f;
        const float inv_b = (l_b > 0.f) ? 1.0f / l_b : 0.f;
        uint4* oa = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(t.bh) * p.Sq + row_a) * kD);
        uint4* ob = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(t.bh) * p.Sq + row_b) * kD);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t ov[32];
          tmem_ld16x256_x8(tl + kColO + 64 * h, ov);
          tmem_ld_wait(ov);
          float va[16], vb[16];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            va[2 * k] = __uint_as_float(ov[4 * k]);
            va[2 * k + 1] = __uint_as_float(ov[4 * k + 1]);
            vb[2 * k] = __uint_as_float(ov[4 * k + 2]);
            vb[2 * k + 1] = __uint_as_float(ov[4 * k + 3]);
          }
          store_o_half(oa, ob, va, vb, inv_a, inv_b, h, lane & 3, live_a, live_b);
        }
        if (writes_row && p.lse) {
          const float kLn2 = 0.69314718055994530942f;
          if (live_a)
            p.lse[static_cast<size_t>(t.bh) * p.Sq + row_a] = (l_a > 0.f) ? (m_a + __log2f(l_a)) * kLn2 : neg_inf();
          if (live_b)
            p.lse[static_cast<size_t>(t.bh) * p.Sq + row_b] = (l_b > 0.f) ? (m_b + __log2f(l_b)) * kLn2 : neg_inf();
        }
      }
      // O has been read: the next tile's first P V may overwrite it
      tc_fence_before();
      mbar_arrive(smem_addr(&bars.o_free));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kQkWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [BH][S][128] bf16 viewed as a 3-D tensor; boxes of 64 dims x box_rows rows, 128B swizzle.
bool make_map(CUtensorMap* map, const uint16_t* base, int S, int BH, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                           static_cast<cuuint64_t>(S) * kD * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estride[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), dims, strides,
             box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Greedy schedule of the causal query tiles over G CTAs: tiles are taken in
// launch order (groups of heads, heaviest first within a group) and each
// goes to the CTA with the least work so far, a tile's work being its KV
// steps plus a fixed fill / drain overhead. Each CTA's list keeps launch
// order, so the CTAs move through the head groups together (L2 reuse).
constexpr int kTileOverheadSteps = 3;

bool build_schedule(const AttnParams& prm, int G, TileSched<true>* sc) {
  const int T = prm.n_tiles;
  if (T > kSchedMaxTiles || G > kSchedMaxCtas || G < 1) return false;
  std::vector<int> owner(T);
  std::vector<int> count(G, 0);
  using Load = std::pair<long long, int>;  // (work so far, CTA)
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int c = 0; c < G; ++c) heap.push({0, c});
  for (int lin = 0; lin < T; ++lin) {
    const Load l = heap.top();
    heap.pop();
    owner[lin] = l.second;
    ++count[l.second];
    heap.push({l.first + tile_info(prm, Work{lin, -1}).n_kv + kTileOverheadSteps, l.second});
  }
  sc->off[0] = 0;
  for (int c = 0; c < G; ++c) sc->off[c + 1] = static_cast<uint16_t>(sc->off[c] + count[c]);
  for (int c = G; c < kSchedMaxCtas; ++c) sc->off[c + 1] = sc->off[G];
  std::vector<int> pos(sc->off, sc->off + G);
  for (int lin = 0; lin < T; ++lin) sc->list[pos[owner[lin]]++] = static_cast<uint16_t>(lin);
  return true;
}

// Launch of the kernel instance for a rescale policy (grid of `grid` CTAs).
template <bool kSched>
void launch_policy(int policy, int grid, cudaStream_t stream, const CUtensorMap& mq,
                   const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& prm,
                   const TileSched<kSched>& sched) {
  const dim3 g(static_cast<unsigned>(grid));
  if (policy == kRescaleOnRise)
    attn_fwd_kernel<kSched, kRescaleOnRise><<<g, kThreads, kSmemBytes, stream>>>(mq, mk, mv, prm, sched);
  else if (policy == kRescaleAlways)
    attn_fwd_kernel<kSched, kRescaleAlways><<<g, kThreads, kSmemBytes, stream>>>(mq, mk, mv, prm, sched);
  else
    attn_fwd_kernel<kSched, kRescaleThreshold><<<g, kThreads, kSmemBytes, stream>>>(mq, mk, mv, prm,
                                                                                    sched);
}

// The split tail of a non-causal launch on `sms` SMs: whole query tiles in
// full rounds of one tile per CTA, then the remaining tiles cut along the keys
// into f parts so that every CTA gets one part (f = sms / remaining, at most
// kMaxSplit and at most the tile's KV tiles). No split when the tiles fill
// the rounds exactly or f < 2.
struct SplitPlan {
  int full_rounds = 0, split_first = 0, split_f = 0, split_items = 0;
  long long tail = 0;
};

SplitPlan split_plan(long long tiles, int n_kv, int sms) {
  SplitPlan sp;
  if (tiles <= 0 || sms <= 0) return sp;
  const long long rounds = tiles / sms;
  const long long tail = tiles - rounds * sms;
  if (tail == 0) return sp;
  long long f = sms / tail;
  if (f > kMaxSplit) f = kMaxSplit;
  if (f > n_kv) f = n_kv;
  if (f < 2) return sp;
  sp.full_rounds = static_cast<int>(rounds);
  sp.split_first = static_cast<int>(rounds * sms);
  sp.split_f = static_cast<int>(f);
  sp.split_items = static_cast<int>(f * tail);
  sp.tail = tail;
  return sp;
}

// Workspace of a split tail: O, then (m, l), then the counters.
size_t split_bytes_o(const SplitPlan& sp) {
  return static_cast<size_t>(sp.tail) * sp.split_f * kBM * kD * sizeof(float);
}
size_t split_bytes_ml(const SplitPlan& sp) {
  return static_cast<size_t>(sp.tail) * sp.split_f * kSoftThreads * 4 * sizeof(float);
}
size_t split_bytes(const SplitPlan& sp) {
  if (sp.split_f < 2) return 0;
  return split_bytes_o(sp) + split_bytes_ml(sp) +
         static_cast<size_t>(sp.tail) * kSoftWarps * sizeof(unsigned int);
}

// The last schedule built by this host thread, reused while the shape stays.
struct SchedCache {
  int bh = -1, n_qblocks = -1, sk = -1, grid = -1;
  TileSched<true> sched;
};

}  // namespace

cudaError_t launch_attention_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 uint16_t* o, float* lse, int B, int H, int Sq, int Sk, int D,
                                 float scale, bool causal, unsigned int* err_word,
                                 const AttnFault& fault, const AttnPartialOut* partial,
                                 int rescale_policy, void* workspace, int64_t workspace_bytes,
                                 cudaStream_t stream) {
  if (rescale_policy < kRescaleThreshold || rescale_policy > kRescaleAlways)
    return cudaErrorInvalidValue;
  if (D != kD) return cudaErrorNotSupported;
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, Sq, BH, kBM) || !make_map(&mk, k, Sk, BH, kBN) ||
      !make_map(&mv, v, Sk, BH, kBN))
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // the kernels' shared-memory limit, raised once per device
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> smem_set[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices || !smem_set[dev].load(std::memory_order_acquire)) {
    const void* kernels[] = {
        reinterpret_cast<const void*>(attn_fwd_kernel<false, kRescaleThreshold>),
        reinterpret_cast<const void*>(attn_fwd_kernel<true, kRescaleThreshold>),
        reinterpret_cast<const void*>(attn_fwd_kernel<false, kRescaleOnRise>),
        reinterpret_cast<const void*>(attn_fwd_kernel<true, kRescaleOnRise>),
        reinterpret_cast<const void*>(attn_fwd_kernel<false, kRescaleAlways>),
        reinterpret_cast<const void*>(attn_fwd_kernel<true, kRescaleAlways>)};
    for (const void* kf : kernels) {
      e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
    }
    if (dev >= 0 && dev < kMaxDevices) smem_set[dev].store(true, std::memory_order_release);
  }
  AttnParams prm;
  prm.o = o;
  prm.lse = lse;
  prm.err = err_word;
  prm.Sq = Sq;
  prm.Sk = Sk;
  prm.BH = BH;
  prm.n_qblocks = (Sq + (causal ? kCausalShift : 0) + kBM - 1) / kBM;
  prm.C = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  prm.causal = causal ? 1 : 0;
  prm.timeout_ns = fault.timeout_ns > 0 ? static_cast<uint64_t>(fault.timeout_ns) : kTimeoutNs;
  static std::atomic<unsigned int> launches{0};
  prm.tag = launches.fetch_add(1, std::memory_order_relaxed) % 65535u + 1u;
  prm.skip_v_step = fault.skip_v_step;
  prm.part_m = partial ? partial->m : nullptr;
  prm.part_l = partial ? partial->l : nullptr;
  prm.part_o = partial ? partial->o : nullptr;
  prm.part_stride = partial ? partial->stride : 1;
  prm.part_index = partial ? partial->index : 0;
  prm.full_rounds = prm.split_first = prm.split_f = prm.split_items = 0;
  prm.ws_o = prm.ws_ml = nullptr;
  prm.ws_cnt = nullptr;
  const long long tiles = static_cast<long long>(prm.n_qblocks) * BH;
  if (tiles > 0x7fffffffLL) return cudaErrorNotSupported;
  prm.n_tiles = static_cast<int>(tiles);
  // Persistent: one CTA per SM walking its share of the query tiles.
  // Non-causal tiles all cost the same and follow the round rule; causal
  // tiles range from 1 to Sk / 128 KV steps and follow a greedy schedule
  // built here. A causal launch with more tiles than the schedule holds
  // uses one CTA per tile, and the block scheduler balances them.
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int G = static_cast<int>(tiles < sms ? tiles : sms);
  if (causal) {
    thread_local SchedCache cache;
    const bool hit = cache.bh == BH && cache.n_qblocks == prm.n_qblocks && cache.sk == Sk &&
                     cache.grid == G;
    if (hit || build_schedule(prm, G, &cache.sched)) {
      cache.bh = BH;
      cache.n_qblocks = prm.n_qblocks;
      cache.sk = Sk;
      cache.grid = G;
      launch_policy<true>(rescale_policy, G, stream, mq, mk, mv, prm, cache.sched);
      return cudaGetLastError();
    }
    cache.bh = -1;  // not schedulable: one CTA per tile
    TileSched<false> none{};
    launch_policy<false>(rescale_policy, static_cast<int>(tiles), stream, mq, mk, mv, prm, none);
    return cudaGetLastError();
  }
  TileSched<false> none{};
  int grid = G;
  if (workspace && !partial) {
    const SplitPlan sp = split_plan(tiles, (Sk + kBN - 1) / kBN, sms);
    const size_t need = split_bytes(sp);
    if (need > 0 && static_cast<uint64_t>(workspace_bytes) >= need) {
      uint8_t* w = static_cast<uint8_t*>(workspace);
      prm.full_rounds = sp.full_rounds;
      prm.split_first = sp.split_first;
      prm.split_f = sp.split_f;
      prm.split_items = sp.split_items;
      prm.ws_o = reinterpret_cast<float*>(w);
      prm.ws_ml = reinterpret_cast<float*>(w + split_bytes_o(sp));
      prm.ws_cnt = reinterpret_cast<unsigned int*>(w + split_bytes_o(sp) + split_bytes_ml(sp));
      grid = sms;  // one part of a split tile for every CTA
    }
  }
  launch_policy<false>(rescale_policy, grid, stream, mq, mk, mv, prm, none);
  return cudaGetLastError();
}

int64_t attention_workspace_counters(int B, int H, int Sq, int Sk, bool causal, int64_t* bytes) {
  *bytes = 0;
  if (causal || B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  const long long tiles = static_cast<long long>((Sq + kBM - 1) / kBM) * B * H;
  const SplitPlan sp = split_plan(tiles, (Sk + kBN - 1) / kBN, sms);
  if (sp.split_f >= 2) *bytes = static_cast<int64_t>(sp.tail) * kSoftWarps * sizeof(unsigned int);
  return 0;
}

int64_t attention_workspace_bytes(int B, int H, int Sq, int Sk, bool causal) {
  if (causal || B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  const long long tiles = static_cast<long long>((Sq + kBM - 1) / kBM) * B * H;
  return static_cast<int64_t>(split_bytes(split_plan(tiles, (Sk + kBN - 1) / kBN, sms)));
}

}  // namespace oss
