// Device helpers shared by the liboss kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace oss {

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero form).
// Exact at 0 (2^0 = 1), returns +0 for -inf.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Reciprocal on the special-function unit (PTX rcp.approx, flush-to-zero form).
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Streaming (evict-first) 16-byte global load / store.
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, float4 v) { __stcs(p, v); }

// bf16 raw bits -> fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// fp32 -> bf16 bits, round to nearest even (inputs are finite here).
__device__ __forceinline__ uint32_t f32_to_bf16_rn(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

// Record a give-up on a bounded wait; the first code wins.
__device__ __forceinline__ void report_error(unsigned int* err, unsigned int code) {
  if (err) atomicCAS(err, 0u, code);
}

}  // namespace oss
