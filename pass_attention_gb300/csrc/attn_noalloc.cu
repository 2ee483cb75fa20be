// os_attention_fwd_noalloc: the attention forward for callers that cannot
// allocate device memory.
//
// os_attention_fwd_ws wants a caller-owned workspace for the split tail of a
// non-causal launch (the last round's query tiles cut along the keys, their
// partial states merged on the device). Some callers have no way to give it
// one: a plugin or callback that a host framework hands only its input and
// output buffers, while the framework's own pool owns the rest of device
// memory; or a latency-critical thread that must not call cudaMalloc, which
// can block on the driver and synchronise the device. This entry point gives
// them the same kernel with the workspace taken from a fixed array in device
// memory that the library declares statically (every GPU that loads the
// library holds it until the process exits), and it allocates nothing.
//
// Every call on a device shares that one array. Two calls whose kernels
// overlap on the GPU (on two streams, or from two threads) race on it and
// give wrong results: order them on one stream or by events.

#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/oss.h"
#include "oss_internal.h"

namespace {

// The fixed workspace: 16 MiB. The split tail needs at most one part per SM
// (64 KB of O and 4 KB of (m, l) each) plus its counters: 10.4 MB on a
// 152-SM GB300.
constexpr int64_t kNoAllocBytes = int64_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// The device address of g_noalloc_scratch on the current device. In host
// code the array's name is only a host-side stand-in, not a device address,
// so the address is looked up once per device, with that device current,
// by cudaGetSymbolAddress; the first call on each device does this set-up,
// and that first call should come before any stream capture.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return nullptr;
  }
  g_scratch_addr[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace

extern "C" os_status os_attention_fwd_noalloc(const os_bf16* q, const os_bf16* k,
                                              const os_bf16* v, os_bf16* o, float* lse, int32_t B,
                                              int32_t H, int32_t Sq, int32_t Sk, int32_t D,
                                              float scale, int causal, void* stream) {
  const int64_t need = os_attention_fwd_workspace_bytes(B, H, Sq, Sk, D, causal);
  if (need < 0) return OS_ERR_CUDA;
  if (need > kNoAllocBytes) return OS_ERR_UNSUPPORTED;  // beyond the fixed workspace
  if (need == 0)  // no split tail for this shape: no workspace at all
    return os_attention_fwd_ws(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, nullptr, 0, stream);
  void* ws = scratch_address();
  if (!ws) return OS_ERR_CUDA;
  // The array keeps the last call's contents; only the per-tile counters at
  // the end of the used region must start at zero. Completed calls leave
  // them at zero, but a call that gave up on a wait may not: clear them.
  int64_t counter_bytes = 0;
  if (oss::attention_workspace_counters(B, H, Sq, Sk, causal != 0, &counter_bytes) < 0)
    return OS_ERR_CUDA;
  unsigned char* w = static_cast<unsigned char*>(ws);
  if (cudaMemsetAsync(w + need - counter_bytes, 0, static_cast<size_t>(counter_bytes),
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return OS_ERR_CUDA;
  return os_attention_fwd_ws(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, ws, need, stream);
}
