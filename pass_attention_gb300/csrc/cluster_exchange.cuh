// Exchange of (max, sum) states between the CTAs of a thread-block cluster
// on mbarriers: each CTA's thread 0 sends its state to every CTA of the
// cluster by asynchronous stores into distributed shared memory
// (st.async ... mbarrier::complete_tx), which complete 8 bytes of
// transaction each on the receiver's barrier; the receiver's threads wait on
// their own barrier for all C states. No cluster-wide barrier and no fence
// per row: the receipt of the states is what orders the reads after them.
//
// Protocol, per exchange e (e = 0, 1, 2, ...): slot set and barrier e & 1,
// phase parity (e >> 1) & 1. Thread 0 arms its barrier for C * 8 bytes
// (mbarrier.arrive.expect_tx) and sends; a peer's store for exchange e + 2
// into the same set can only come after that peer received this CTA's state
// for e + 1, which thread 0 sends only after its wait for e completed and
// after a CTA barrier that every reader of e's slots has passed. A CTA ends
// with a cluster barrier, so none leaves while a peer may still store into it.
#pragma once

#include "softmax_common.cuh"

namespace oss {
namespace {

constexpr uint32_t kSiteStates = 2;  // wait site: the cluster's states for a row

// (a, b) into the same shared-memory slot of CTA `rank` of the cluster, by an
// asynchronous store that completes 8 bytes of transaction on that CTA's
// mbarrier at the address of `bar`
__device__ __forceinline__ void st_async_peer_f2(const void* slot, const void* bar, uint32_t rank, float a,
                                                 float b) {
  uint32_t rs, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rs) : "r"(smem_u32(slot)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(rs),
               "f"(a), "f"(b), "r"(rb)
               : "memory");
}

// Thread 0: arm this CTA's barrier for the C states (plus `extra` bytes, 0
// but in the test hook) and send state (a, b) into slot `rank` of every CTA.
__device__ __forceinline__ void send_state(float2* slots, uint64_t* bar, uint32_t C, uint32_t rank, float a,
                                           float b, uint32_t extra) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(C * 8u + extra)
               : "memory");
  for (uint32_t r = 0; r < C; ++r) st_async_peer_f2(&slots[rank], bar, r, a, b);
}

// Wait for the phase of `bar` with `parity`, at most `timeout_ns`; a give-up
// records kernel 2, site 2 in the error word and returns false.
__device__ __forceinline__ bool wait_states_bounded(uint32_t bar, uint32_t parity, unsigned int* err,
                                                    uint64_t timeout_ns) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try(bar, parity)) return true;
    if ((n & 63u) == 0 && timer_ns() - t0 > timeout_ns) {
      report_error(err, kKernelSoftmaxRows | (kSiteStates << 8));
      return false;
    }
  }
}

}  // namespace
}  // namespace oss
