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
// CTA layout (224 threads, one CTA per SM, one 128-row query tile):
//   * warps 0..3 -- softmax: warp w reaches tensor-memory lanes 32 w .. +31;
//                   each thread owns one query row.
//   * warp 4     -- TMA producer: Q once, then K and V tiles (128 keys) into
//                   two 3-stage rings, K two steps ahead of V.
//   * warp 5     -- one thread issues S_b = Q K_j^T (A, B from shared memory);
//                   the warp owns the tensor-memory allocation.
//   * warp 6     -- one thread issues O += P_j V_j (A = P from tensor memory,
//                   B from shared memory).
//   Issuing a tcgen05.mma costs its thread tens of cycles, so the two MMA
//   streams have a thread each.
// Tensor memory (512 fp32 columns x 128 lanes): S_0 | S_1 | S_2 | O. KV step
// j uses score buffer b = j % 3 (and ring stage j % 3); the softmax writes P_j
// as bf16 pairs over the first 64 columns of S_b. With three score buffers
// QK^T runs up to two steps ahead of the softmax.
//
// Causal: query i sees keys 0..i (Sq == Sk). Query tiles start 64 rows before
// a KV-tile boundary; KV tiles wholly above the diagonal are skipped and the
// two diagonal tiles are visited first, from the last one down, so the first
// KV tile a causal CTA sees is masked for all of its first 64 rows -- the
// case the -inf guard exists for.
//
// Every wait on an mbarrier is bounded: on timeout the thread raises a
// CTA-wide abort flag and writes the device error word; all roles then drain
// their own in-flight copies and MMAs (again with a bound), and tensor memory
// is released before the CTA exits.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "oss_internal.h"

namespace oss {
namespace {

constexpr int kD = 128;           // head dimension
constexpr int kBM = 128;          // query rows per CTA (= tensor-memory lanes)
constexpr int kBN = 128;          // keys per KV tile
constexpr int kStages = 3;        // depth of the K ring and of the V ring (= score buffers)
constexpr int kKLead = 2;         // K loads run this many steps ahead of V loads
constexpr int kThreads = 224;
constexpr int kProducerWarp = 4;  // warps 0..3: softmax, one thread per query row
constexpr int kQkWarp = 5;        // warp 5: issues S = Q K^T, owns tensor memory
constexpr int kPvWarp = 6;        // warp 6: issues O += P V
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

// tensor-memory columns (512 fp32 x 128 lanes): S_0 | S_1 | S_2 | O. KV step j
// uses score buffer j % 3; P_j (bf16 pairs) is written over its first half.
constexpr int kSBuf = 3;
static_assert(kSBuf == kStages, "K/V ring stage and score buffer share one index");
constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t col_s(int b) { return 128u * b; }
constexpr uint32_t kColO = 384;

// The reference maximum of a warp's rows moves only when one of them rises
// by more than this (base-2 units): weights stay below 2^8 = 256.
constexpr float kRescaleSlack = 8.0f;

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kDrainNs = 200000000ull;     // 0.2 s to drain own copies

// wait sites (error word bits 8..15)
enum Site : unsigned int {
  kSiteQFull = 1, kSiteKFull, kSiteVFull, kSiteKEmpty, kSiteVEmpty,
  kSiteSFull, kSitePReady, kSiteODone, kSiteDrain
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
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned int* err, unsigned int site,
                                           uint64_t timeout_ns) {
  const uint64_t t0 = global_timer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((n & 63u) == 0 && global_timer() - t0 > timeout_ns) {
      *abort_flag = 1;
      report_error(err, kKernelAttnFwd | (site << 8));
      return false;
    }
  }
}

// Bounded wait. Returns false on timeout or when another thread has aborted.
// The limit is the kernel's timeout_ns (kTimeoutNs unless a test shortens it).
#define wait_bar(bar, parity, abort_flag, err, site) \
  (mbar_test_wait((bar), (parity)) ||                 \
   wait_bar_slow((bar), (parity), (abort_flag), (err), (site), p.timeout_ns))

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

// 32 consecutive columns of this warp's 32 lanes: thread i gets lane i.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : OSS_R8(0), OSS_R8(8), OSS_R8(16), OSS_R8(24)
      : "r"(taddr));
}

// Completes outstanding tcgen05.ld of this thread; the register operands tie
// the loaded values to the wait so no use is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  asm volatile("" : OSS_RW8(0), OSS_RW8(8), OSS_RW8(16), OSS_RW8(24));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      OSS_W8(0), OSS_W8(8), OSS_W8(16), OSS_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      OSS_W8(0), OSS_W8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
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
  int Sq, Sk, BH, n_qblocks;
  float C;  // scale * log2(e)
  int causal;
  uint64_t timeout_ns;  // limit of every bounded wait
  int skip_v_step;      // test hook: the producer skips the V load of this step (-1: none)
  // partial-state output (sequence-sharded attention): when part_o != null the
  // epilogue writes (m, l, O unnormalised) of row r to slot part_index of a
  // [rows, part_stride] partial array instead of O / l and lse
  float* part_m;
  float* part_l;
  float* part_o;
  int part_stride, part_index;
};

struct Barriers {
  uint64_t q_full;
  uint64_t k_full[kStages], v_full[kStages];
  uint64_t s_full[kSBuf], p_ready[kSBuf];
  uint64_t o_done[kSBuf];  // P_j V done, for steps j of each buffer (keeps parity waits exact)
  uint64_t drain[2];  // one per issuing thread
};

__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q,
                const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Query tile of this CTA. Causal tiles start kCausalShift rows before a KV
  // tile boundary (the first tile hangs over row 0; the TMA fills the rows
  // above with zeros), and the heaviest tiles are launched first.
  // CTA order: the ~150 CTAs resident at a time should share (b, h), so
  // that K and V are read from HBM once and then from L2. Non-causal:
  // (b, h)-major. Causal: groups of kCausalGroup heads, heaviest query tiles
  // first within each group.
  const int lin = blockIdx.x;
  int bh, qb;
  if (!p.causal) {
    bh = lin / p.n_qblocks;
    qb = lin - bh * p.n_qblocks;
  } else {
    const int per_group = kCausalGroup * p.n_qblocks;
    const int g = lin / per_group;
    const int gsize = min(kCausalGroup, p.BH - g * kCausalGroup);
    const int r = lin - g * per_group;
    const int qb_lin = r / gsize;
    bh = g * kCausalGroup + (r - qb_lin * gsize);
    qb = p.n_qblocks - 1 - qb_lin;
  }
  const int q0 = qb * kBM - (p.causal ? kCausalShift : 0);
  const int kv_end = p.causal ? min(p.Sk, q0 + kBM) : p.Sk;
  const int n_kv = (kv_end + kBN - 1) / kBN;
  // KV tiles that reach past the tile's first row touch the diagonal; they
  // are visited first, from the last one down: for a shifted causal tile the
  // first one is masked for all of the tile's first kCausalShift rows.
  const int diag_first = p.causal ? max(0, q0) / kBN : n_kv;
  const int n_diag = n_kv - diag_first;
  auto kv_tile = [&](int j) { return j < n_diag ? (n_kv - 1 - j) : (j - n_diag); };

  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bars.q_full), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&bars.k_full[s]), 1);
      mbar_init(smem_addr(&bars.v_full[s]), 1);
    }
    for (int b = 0; b < kSBuf; ++b) {
      mbar_init(smem_addr(&bars.s_full[b]), 1);
      mbar_init(smem_addr(&bars.p_ready[b]), kBM);
      mbar_init(smem_addr(&bars.o_done[b]), 1);
    }
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

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_v)) : "memory");
      const uint32_t qbar = smem_addr(&bars.q_full);
      mbar_expect_tx(qbar, kTile);
      for (int h = 0; h < 2; ++h)
        tma_load_3d(sbase + kOffQ + h * kHalf, &tmap_q, qbar, h * 64, q0, bh);
      // K_j is consumed by QK_j, which runs up to two steps ahead of P_j V,
      // the consumer of V_j; so K loads run kKLead steps ahead of V loads,
      // and each ring is refilled as soon as its own consumer is done: K stage
      // j % 3 when QK_j has completed (s_full[j % 3]), V stage j % 3 when
      // P_j V has (o_done[j % 3]) -- ring stage and score buffer coincide.
      int k_issued = 0, v_issued = 0, skipped_v = -1;
      for (int i = 0; i < n_kv + kKLead; ++i) {
        if (i < n_kv) {
          const int s = i % kStages;
          const int round = i / kStages;
          if (round > 0 && !wait_bar(smem_addr(&bars.s_full[s]), (round - 1) & 1, abort_flag,
                                     p.err, kSiteKEmpty))
            break;
          const uint32_t kb = smem_addr(&bars.k_full[s]);
          mbar_expect_tx(kb, kTile);
          for (int h = 0; h < 2; ++h)
            tma_load_3d(sbase + kOffK + s * kTile + h * kHalf, &tmap_k, kb, h * 64,
                        kv_tile(i) * kBN, bh);
          k_issued = i + 1;
        }
        const int j = i - kKLead;
        if (j >= 0 && j < n_kv && j == p.skip_v_step) {
          skipped_v = j;  // test hook: this V tile never arrives
        } else if (j >= 0 && j < n_kv) {
          const int s = j % kStages;
          const int round = j / kStages;
          if (round > 0 && !wait_bar(smem_addr(&bars.o_done[s]), (round - 1) & 1, abort_flag,
                                     p.err, kSiteVEmpty))
            break;
          const uint32_t vb = smem_addr(&bars.v_full[s]);
          mbar_expect_tx(vb, kTile);
          for (int h = 0; h < 2; ++h)
            tma_load_3d(sbase + kOffV + s * kTile + h * kHalf, &tmap_v, vb, h * 64,
                        kv_tile(j) * kBN, bh);
          v_issued = j + 1;
        }
      }
      // drain: every issued copy must land before the CTA may exit
      drain_bar(qbar, 0, p.err);
      for (int j = k_issued - 1; j >= 0 && j >= k_issued - kStages; --j)
        drain_bar(smem_addr(&bars.k_full[j % kStages]), (j / kStages) & 1, p.err);
      for (int j = v_issued - 1; j >= 0 && j >= v_issued - kStages; --j)
        if (j != skipped_v) drain_bar(smem_addr(&bars.v_full[j % kStages]), (j / kStages) & 1, p.err);
    }
  } else if (warp == kQkWarp) {
    // ------------------------------------------------------------ QK issuer
    // S_{j % 3} = Q K_j^T for j = 0, 1, ...: the buffer last held P_{j-3},
    // so P_{j-3} V must be done with it. Issuing a tcgen05.mma costs its
    // thread tens of cycles, so QK^T and P V are issued by two threads.
    if (lane == 0) {
      bool ok = wait_bar(smem_addr(&bars.q_full), 0, abort_flag, p.err, kSiteQFull);
      // operand descriptors built once; a 16-element K step only adds a
      // constant to the start-address field (16-byte units)
      const uint64_t dq = smem_desc(sbase + kOffQ, 16, 1024);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % kStages;  // K stage = score buffer
        if (!(ok = wait_bar(smem_addr(&bars.k_full[s]), (j / kStages) & 1, abort_flag, p.err,
                            kSiteKFull)))
          break;
        if (j >= kStages && !(ok = wait_bar(smem_addr(&bars.o_done[s]), (j / kStages - 1) & 1,
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
      // drain: no MMA of this thread may still write tensor memory when it is freed
      tc_commit(smem_addr(&bars.drain[0]));
      drain_bar(smem_addr(&bars.drain[0]), 0, p.err);
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    // O += P_j V_j once the softmax has written P_j over S_{j % 3}.
    if (lane == 0) {
      bool ok = true;
      const uint32_t d_o = tbase + kColO;
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % kStages;
        if (!(ok = wait_bar(smem_addr(&bars.v_full[s]), (j / kStages) & 1, abort_flag, p.err,
                            kSiteVFull)))
          break;
        if (!(ok = wait_bar(smem_addr(&bars.p_ready[s]), (j / kStages) & 1, abort_flag, p.err,
                            kSitePReady)))
          break;
        tc_fence_after();
        const uint64_t dv = smem_desc(sbase + kOffV + s * kTile, kHalf, 1024);
        const uint32_t a_p = tbase + col_s(s);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(d_o, a_p + kk * 8, dv + static_cast<uint64_t>(kk * (2048 >> 4)), kIdescPV,
                 (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(smem_addr(&bars.o_done[s]));  // buffer s and V stage s free
      }
      tc_commit(smem_addr(&bars.drain[1]));
      drain_bar(smem_addr(&bars.drain[1]), 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp;                         // tensor-memory lane quadrant
    const int r_in_tile = quad * 32 + lane;
    const int row = q0 + r_in_tile;                // query index (may be < 0: padding)
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    const float C = p.C;
    float m = neg_inf();       // reference maximum, base 2
    float m_true = neg_inf();  // true row maximum, base 2 (for partial states)
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j % kSBuf;
      const uint32_t colS = col_s(b);
      ok = __all_sync(0xffffffffu, wait_bar(smem_addr(&bars.s_full[b]), (j / kSBuf) & 1,
                                            abort_flag, p.err, kSiteSFull));
      if (!ok) break;
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32(tl + colS + 0, r0);
      tmem_ld32(tl + colS + 32, r1);
      tmem_ld32(tl + colS + 64, r2);
      tmem_ld32(tl + colS + 96, r3);
      tmem_ld_wait(r0);
      tmem_ld_wait(r1);
      tmem_ld_wait(r2);
      tmem_ld_wait(r3);
      float s[kBN];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s[c] = __uint_as_float(r0[c]);
        s[32 + c] = __uint_as_float(r1[c]);
        s[64 + c] = __uint_as_float(r2[c]);
        s[96 + c] = __uint_as_float(r3[c]);
      }
      const int key0 = kv_tile(j) * kBN;
      const bool ragged = key0 + kBN > p.Sk;
      const bool diag = p.causal && key0 + kBN - 1 > q0;
      if (ragged || diag) {
        const int lim = min(p.Sk, p.causal ? row + 1 : p.Sk) - key0;  // visible keys: c < lim
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c >= lim) s[c] = neg_inf();
      }
      // row maximum of this tile: four independent chains of 3-input max
      float mx0 = neg_inf(), mx1 = neg_inf(), mx2 = neg_inf(), mx3 = neg_inf();
#pragma unroll
      for (int c = 0; c < kBN; c += 8) {
        mx0 = fmax3(mx0, s[c + 0], s[c + 1]);
        mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
        mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
        mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
      }
      const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * C;
      const float m_new = fmaxf(m, m_tile);
      m_true = fmaxf(m_true, m_tile);
      // Move the reference maximum only when some row of this warp has risen
      // by more than kRescaleSlack (base 2). Otherwise keep it: exactly the
      // same result in exact arithmetic (the reference cancels in O / l),
      // weights stay <= 2^kRescaleSlack, and the O round trip is skipped.
      const bool rescale = __any_sync(0xffffffffu, m_new > m + kRescaleSlack);
      float corr = 1.f;
      if (rescale) {
        const float m_use_new = (m_new == neg_inf()) ? 0.f : m_new;
        corr = ex2(m - m_use_new);  // 0 while m = -inf
        m = m_new;
      }
      const float m_use = (m == neg_inf()) ? 0.f : m;  // the -inf guard
      const float2 Cv = make_float2(C, C);
      const float2 mv = make_float2(-m_use, -m_use);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
#pragma unroll
      for (int ch = 0; ch < kBN / 32; ++ch) {
        // 32 weights -> 16 bf16 pairs, stored over the first columns of S_b
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const int cc = ch * 32 + c;
          const float2 t0 = __ffma2_rn(make_float2(s[cc], s[cc + 1]), Cv, mv);
          const float2 t1 = __ffma2_rn(make_float2(s[cc + 2], s[cc + 3]), Cv, mv);
          const float2 e0 = make_float2(ex2(t0.x), ex2(t0.y));
          const float2 e1 = make_float2(ex2(t1.x), ex2(t1.y));
          acc0 = __fadd2_rn(acc0, e0);
          acc1 = __fadd2_rn(acc1, e1);
          pk[(c >> 1) + 0] = pack_bf16x2(e0.x, e0.y);
          pk[(c >> 1) + 1] = pack_bf16x2(e1.x, e1.y);
        }
        tmem_st16(tl + colS + ch * 16, pk);
      }
      const float2 acc = __fadd2_rn(acc0, acc1);
      l = fmaf(l, corr, acc.x + acc.y);
      if (rescale && j > 0) {
        // O still holds the previous tiles' sum: wait for P_{j-1} V (whose
        // completion implies every earlier one), then rescale
        ok = __all_sync(0xffffffffu, wait_bar(smem_addr(&bars.o_done[(j - 1) % kSBuf]),
                                              ((j - 1) / kSBuf) & 1, abort_flag, p.err, kSiteODone));
        if (!ok) break;
        tc_fence_after();
        const float2 cv = make_float2(corr, corr);
#pragma unroll 1
        for (int cc = 0; cc < kD; cc += 32) {
          uint32_t ov[32];
          tmem_ld32(tl + kColO + cc, ov);
          tmem_ld_wait(ov);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(ov[c]), __uint_as_float(ov[c + 1])), cv);
            ov[c] = __float_as_uint(o2.x);
            ov[c + 1] = __float_as_uint(o2.y);
          }
          tmem_st32(tl + kColO + cc, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_addr(&bars.p_ready[b]));
    }
    // epilogue: O / l and lse for this row, once P_{n-1} V is done (its
    // completion implies every earlier one)
    if (ok)
      ok = __all_sync(0xffffffffu, wait_bar(smem_addr(&bars.o_done[(n_kv - 1) % kSBuf]),
                                            ((n_kv - 1) / kSBuf) & 1, abort_flag, p.err, kSiteODone));
    if (ok && p.part_o) {
      // partial state relative to the true row maximum: rescale the sums
      // taken against the reference by 2^(m_ref - m_true) <= 1
      tc_fence_after();
      const bool empty = (m_true == neg_inf()) || !(l > 0.f);
      const float f = empty ? 0.f : ex2(m - m_true);
      const bool live = row >= 0 && row < p.Sq;
      const size_t slot = (static_cast<size_t>(bh) * p.Sq + row) * p.part_stride + p.part_index;
      float4* orow = reinterpret_cast<float4*>(p.part_o + slot * kD);
#pragma unroll 1
      for (int cc = 0; cc < kD; cc += 32) {
        uint32_t ov[32];
        tmem_ld32(tl + kColO + cc, ov);
        tmem_ld_wait(ov);
        if (live) {
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            orow[(cc + c) >> 2] = make_float4(__uint_as_float(ov[c]) * f, __uint_as_float(ov[c + 1]) * f,
                                              __uint_as_float(ov[c + 2]) * f, __uint_as_float(ov[c + 3]) * f);
        }
      }
      if (live) {
        const float kLn2 = 0.69314718055994530942f;
        p.part_m[slot] = empty ? neg_inf() : m_true * kLn2;
        p.part_l[slot] = empty ? 0.f : l * f;
      }
    } else if (ok) {
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.0f / l : 0.f;
      const bool live = row >= 0 && row < p.Sq;
      uint4* orow = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(bh) * p.Sq + row) * kD);
#pragma unroll 1
      for (int cc = 0; cc < kD; cc += 32) {
        uint32_t ov[32];
        tmem_ld32(tl + kColO + cc, ov);
        tmem_ld_wait(ov);
        if (live) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(ov[c + 0]) * inv, __uint_as_float(ov[c + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv);
            orow[(cc + c) >> 3] = w;
          }
        }
      }
      if (live && p.lse) {
        const float kLn2 = 0.69314718055994530942f;
        p.lse[static_cast<size_t>(bh) * p.Sq + row] =
            (l > 0.f) ? (m + __log2f(l)) * kLn2 : neg_inf();
      }
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

}  // namespace

cudaError_t launch_attention_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 uint16_t* o, float* lse, int B, int H, int Sq, int Sk, int D,
                                 float scale, bool causal, unsigned int* err_word,
                                 const AttnFault& fault, const AttnPartialOut* partial,
                                 cudaStream_t stream) {
  if (D != kD) return cudaErrorNotSupported;
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, Sq, BH, kBM) || !make_map(&mk, k, Sk, BH, kBN) ||
      !make_map(&mv, v, Sk, BH, kBN))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
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
  prm.skip_v_step = fault.skip_v_step;
  prm.part_m = partial ? partial->m : nullptr;
  prm.part_l = partial ? partial->l : nullptr;
  prm.part_o = partial ? partial->o : nullptr;
  prm.part_stride = partial ? partial->stride : 1;
  prm.part_index = partial ? partial->index : 0;
  const long long grid = static_cast<long long>(prm.n_qblocks) * BH;
  if (grid > 0x7fffffffLL) return cudaErrorNotSupported;
  attn_fwd_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(mq, mk, mv, prm);
  return cudaGetLastError();
}

}  // namespace oss
