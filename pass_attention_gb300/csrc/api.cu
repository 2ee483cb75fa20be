// The C ABI of liboss (include/oss.h): host-side validation, then launch.
// Nothing here synchronises, allocates device memory or prints.
// os_softmax_rows_from_host creates four CUDA events per call (released at
// its end) and, once per device, two copy streams.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/oss.h"
#include "oss_internal.h"

// One error word per device, written by kernels that give up on a bounded
// wait (first code wins) and read back by os_check_device_error.
__device__ unsigned int g_oss_error_word;

namespace {

constexpr int kMaxDevices = 64;
// Device address of g_oss_error_word, per device, filled on first use. Host
// threads may race to fill a slot; they store the same address, and the
// atomic makes that race well defined.
std::atomic<unsigned int*> g_err_ptr[kMaxDevices];

unsigned int* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned int* cached = g_err_ptr[dev].load(std::memory_order_acquire);
  if (!cached) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_oss_error_word) != cudaSuccess) return nullptr;
    cached = static_cast<unsigned int*>(p);
    g_err_ptr[dev].store(cached, std::memory_order_release);
  }
  return cached;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

os_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return OS_OK;
  if (e == cudaErrorNotSupported) return OS_ERR_UNSUPPORTED;
  return OS_ERR_CUDA;
}

bool valid_scale(float s) { return std::isfinite(s) && s > 0.f; }

// Armed by os_debug_inject_fault, consumed by the next os_attention_fwd on
// the same host thread.
thread_local oss::AttnFault t_fault;
// Armed by os_debug_inject_fault (kind 2), consumed by the next
// os_softmax_rows or os_softmax_rows_16bit on the same host thread.
thread_local oss::RowsFault t_rows_fault;
// Set by os_attention_set_rescale_policy; kept for the host thread's later
// attention calls.
thread_local int t_rescale_policy = OS_RESCALE_THRESHOLD;

// The two copy streams of os_softmax_rows_from_host on the current device
// (non-blocking, made on first use and kept for the process).
cudaError_t copy_streams(cudaStream_t* up, cudaStream_t* down) {
  static std::mutex mu;
  static cudaStream_t streams[kMaxDevices][2];
  static bool made[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!made[dev]) {
    if ((e = cudaStreamCreateWithFlags(&streams[dev][0], cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&streams[dev][1], cudaStreamNonBlocking)) != cudaSuccess) {
      cudaStreamDestroy(streams[dev][0]);
      return e;
    }
    made[dev] = true;
  }
  *up = streams[dev][0];
  *down = streams[dev][1];
  return cudaSuccess;
}

// The pipeline of os_softmax_rows_from_host over blocks of chunk_rows rows:
// a block's upload on `up`, its kernel on `main` once the upload landed, its
// downloads on `down` once the kernel ended. `up` and `down` start after the
// work already on `main`, and `main` ends after the last download. A wait
// enqueued on an event keeps the record it saw, so each event is recorded
// again for the next block.
cudaError_t from_host_pipeline(const float* x_host, float* y_host, float* m_host, float* l_host,
                               float* x_dev, float* y_dev, float* m_dev, float* l_dev, int64_t rows,
                               int64_t cols, float scale, int64_t chunk_rows, cudaStream_t main,
                               cudaStream_t up, cudaStream_t down, const cudaEvent_t* ev) {
  cudaError_t e;
  if ((e = cudaEventRecord(ev[0], main)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(up, ev[0], 0)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(down, ev[0], 0)) != cudaSuccess) return e;
  for (int64_t r0 = 0; r0 < rows; r0 += chunk_rows) {
    const int64_t n = (rows - r0 < chunk_rows) ? rows - r0 : chunk_rows;
    const int64_t off = r0 * cols;
    const size_t bytes = static_cast<size_t>(n * cols) * sizeof(float);
    const size_t vb = static_cast<size_t>(n) * sizeof(float);
    if ((e = cudaMemcpyAsync(x_dev + off, x_host + off, bytes, cudaMemcpyHostToDevice, up)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(ev[1], up)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(main, ev[1], 0)) != cudaSuccess) return e;
    if ((e = oss::launch_softmax_rows(x_dev + off, y_dev + off, m_dev ? m_dev + r0 : nullptr,
                                      l_dev ? l_dev + r0 : nullptr, n, cols, cols, cols, scale,
                                      error_word(), oss::RowsFault(), nullptr, 0, main)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(ev[2], main)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(down, ev[2], 0)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(y_host + off, y_dev + off, bytes, cudaMemcpyDeviceToHost, down)) != cudaSuccess)
      return e;
    if (m_host && (e = cudaMemcpyAsync(m_host + r0, m_dev + r0, vb, cudaMemcpyDeviceToHost, down)) != cudaSuccess)
      return e;
    if (l_host && (e = cudaMemcpyAsync(l_host + r0, l_dev + r0, vb, cudaMemcpyDeviceToHost, down)) != cudaSuccess)
      return e;
  }
  if ((e = cudaEventRecord(ev[3], down)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(main, ev[3], 0);
}

}  // namespace

extern "C" {

int32_t os_abi_version(void) { return OSS_ABI_VERSION; }

const char* os_status_string(os_status status) {
  switch (status) {
    case OS_OK: return "OS_OK";
    case OS_ERR_INVALID_ARGUMENT: return "OS_ERR_INVALID_ARGUMENT";
    case OS_ERR_MISALIGNED: return "OS_ERR_MISALIGNED";
    case OS_ERR_UNSUPPORTED: return "OS_ERR_UNSUPPORTED";
    case OS_ERR_CUDA: return "OS_ERR_CUDA";
    case OS_ERR_TIMEOUT: return "OS_ERR_TIMEOUT";
  }
  return "OS_ERR_UNKNOWN";
}

os_status os_softmax_rows_ws(const float* x, float* y, float* m, float* l, int64_t rows,
                             int64_t cols, int64_t ld_x, int64_t ld_y, float scale, void* workspace,
                             int64_t workspace_bytes, void* stream) {
  if (!x || !y) return OS_ERR_INVALID_ARGUMENT;
  if (rows <= 0 || cols <= 0 || ld_x < cols || ld_y < cols) return OS_ERR_INVALID_ARGUMENT;
  if (cols > (int64_t(1) << 30) || rows > (int64_t(1) << 40)) return OS_ERR_INVALID_ARGUMENT;
  if (!valid_scale(scale)) return OS_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < 0 || (!workspace && workspace_bytes != 0)) return OS_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
       reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(l)) & 3u)
    return OS_ERR_MISALIGNED;
  if (!aligned16(workspace)) return OS_ERR_MISALIGNED;
  const oss::RowsFault fault = t_rows_fault;
  t_rows_fault = oss::RowsFault();
  return from_cuda(oss::launch_softmax_rows(x, y, m, l, rows, cols, ld_x, ld_y, scale,
                                            error_word(), fault, workspace, workspace_bytes,
                                            static_cast<cudaStream_t>(stream)));
}

os_status os_softmax_rows(const float* x, float* y, float* m, float* l, int64_t rows,
                          int64_t cols, int64_t ld_x, int64_t ld_y, float scale, void* stream) {
  return os_softmax_rows_ws(x, y, m, l, rows, cols, ld_x, ld_y, scale, nullptr, 0, stream);
}

os_status os_softmax_rows_16bit_ws(const void* x, void* y, float* m, float* l, int64_t rows,
                                   int64_t cols, int64_t ld_x, int64_t ld_y, float scale,
                                   int32_t dtype, void* workspace, int64_t workspace_bytes,
                                   void* stream) {
  if (!x || !y) return OS_ERR_INVALID_ARGUMENT;
  if (rows <= 0 || cols <= 0 || ld_x < cols || ld_y < cols) return OS_ERR_INVALID_ARGUMENT;
  if (cols > (int64_t(1) << 30) || rows > (int64_t(1) << 40)) return OS_ERR_INVALID_ARGUMENT;
  if (!valid_scale(scale) || (dtype != OS_DTYPE_BF16 && dtype != OS_DTYPE_F16))
    return OS_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < 0 || (!workspace && workspace_bytes != 0)) return OS_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 1u) return OS_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(l)) & 3u) return OS_ERR_MISALIGNED;
  if (!aligned16(workspace)) return OS_ERR_MISALIGNED;
  const oss::RowsFault fault = t_rows_fault;
  t_rows_fault = oss::RowsFault();
  return from_cuda(oss::launch_softmax_rows16(static_cast<const uint16_t*>(x),
                                              static_cast<uint16_t*>(y), m, l, rows, cols, ld_x,
                                              ld_y, scale, dtype, error_word(), fault, workspace,
                                              workspace_bytes, static_cast<cudaStream_t>(stream)));
}

os_status os_softmax_rows_16bit(const void* x, void* y, float* m, float* l, int64_t rows,
                                int64_t cols, int64_t ld_x, int64_t ld_y, float scale,
                                int32_t dtype, void* stream) {
  return os_softmax_rows_16bit_ws(x, y, m, l, rows, cols, ld_x, ld_y, scale, dtype, nullptr, 0,
                                  stream);
}

int64_t os_softmax_rows_workspace_bytes(int64_t rows, int64_t cols, int32_t dtype) {
  if (rows <= 0 || cols <= 0) return 0;
  if (dtype != 0 && dtype != OS_DTYPE_BF16 && dtype != OS_DTYPE_F16) return 0;
  return oss::softmax_workspace_bytes(cols * (dtype == 0 ? 4 : 2));
}

os_status os_softmax_rows_from_host(const float* x_host, float* y_host, float* m_host, float* l_host,
                                    float* x_dev, float* y_dev, float* m_dev, float* l_dev,
                                    int64_t rows, int64_t cols, float scale, int64_t chunk_rows,
                                    void* stream) {
  if (!x_host || !y_host || !x_dev || !y_dev) return OS_ERR_INVALID_ARGUMENT;
  if ((m_host && !m_dev) || (l_host && !l_dev)) return OS_ERR_INVALID_ARGUMENT;
  if (rows <= 0 || cols <= 0 || chunk_rows < 0) return OS_ERR_INVALID_ARGUMENT;
  if (cols > (int64_t(1) << 30) || rows > (int64_t(1) << 40)) return OS_ERR_INVALID_ARGUMENT;
  if (!valid_scale(scale)) return OS_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(x_dev) | reinterpret_cast<uintptr_t>(y_dev) |
       reinterpret_cast<uintptr_t>(m_dev) | reinterpret_cast<uintptr_t>(l_dev)) & 3u)
    return OS_ERR_MISALIGNED;
  if (chunk_rows == 0) {  // about 64 MiB of x a block
    chunk_rows = (int64_t(64) << 20) / (cols * 4);
    if (chunk_rows < 1) chunk_rows = 1;
  }
  cudaStream_t up = nullptr, down = nullptr;
  cudaError_t e = copy_streams(&up, &down);
  if (e != cudaSuccess) return from_cuda(e);
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  for (int i = 0; i < 4 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
  if (e == cudaSuccess)
    e = from_host_pipeline(x_host, y_host, m_host, l_host, x_dev, y_dev, m_dev, l_dev, rows, cols, scale,
                           chunk_rows, static_cast<cudaStream_t>(stream), up, down, ev);
  // an event destroyed while work it was recorded on is pending is released
  // once that work completes: this does not wait
  for (int i = 0; i < 4; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  return from_cuda(e);
}

os_status os_softmax_rows_multipass(const float* x, float* y, float* m, float* l, int64_t rows,
                                    int64_t cols, int64_t ld_x, int64_t ld_y, float scale,
                                    int32_t passes, void* stream) {
  if (!x || !y || !m || !l) return OS_ERR_INVALID_ARGUMENT;
  if (rows <= 0 || cols <= 0 || ld_x < cols || ld_y < cols) return OS_ERR_INVALID_ARGUMENT;
  if (cols > (int64_t(1) << 30) || rows > (int64_t(1) << 40)) return OS_ERR_INVALID_ARGUMENT;
  if (!valid_scale(scale) || (passes != 2 && passes != 3)) return OS_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
       reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(l)) & 3u)
    return OS_ERR_MISALIGNED;
  return from_cuda(oss::launch_softmax_rows_multipass(x, y, m, l, rows, cols, ld_x, ld_y, scale,
                                                      passes, static_cast<cudaStream_t>(stream)));
}

os_status os_attention_fwd(const os_bf16* q, const os_bf16* k, const os_bf16* v, os_bf16* o,
                           float* lse, int32_t B, int32_t H, int32_t Sq, int32_t Sk, int32_t D,
                           float scale, int causal, void* stream) {
  if (!q || !k || !v || !o) return OS_ERR_INVALID_ARGUMENT;
  if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return OS_ERR_INVALID_ARGUMENT;
  if (!valid_scale(scale)) return OS_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return OS_ERR_MISALIGNED;
  if (D != 128) return OS_ERR_UNSUPPORTED;
  if (causal && Sq != Sk) return OS_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * H > 65535 * 64) return OS_ERR_UNSUPPORTED;
  unsigned int* err = error_word();
  if (!err) return OS_ERR_CUDA;
  const oss::AttnFault fault = t_fault;
  t_fault = oss::AttnFault();
  return from_cuda(oss::launch_attention_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale,
                                             causal != 0, err, fault, nullptr, t_rescale_policy,
                                             nullptr, 0, static_cast<cudaStream_t>(stream)));
}

int64_t os_attention_fwd_workspace_bytes(int32_t B, int32_t H, int32_t Sq, int32_t Sk, int32_t D,
                                         int causal) {
  if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || D != 128) return 0;
  if (static_cast<int64_t>(B) * H > 65535 * 64) return 0;
  return oss::attention_workspace_bytes(B, H, Sq, Sk, causal != 0);
}

os_status os_attention_fwd_ws(const os_bf16* q, const os_bf16* k, const os_bf16* v, os_bf16* o,
                              float* lse, int32_t B, int32_t H, int32_t Sq, int32_t Sk, int32_t D,
                              float scale, int causal, void* workspace, int64_t workspace_bytes,
                              void* stream) {
  if (!q || !k || !v || !o) return OS_ERR_INVALID_ARGUMENT;
  if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return OS_ERR_INVALID_ARGUMENT;
  if (!valid_scale(scale)) return OS_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < 0 || (!workspace && workspace_bytes != 0)) return OS_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace))
    return OS_ERR_MISALIGNED;
  if (D != 128) return OS_ERR_UNSUPPORTED;
  if (causal && Sq != Sk) return OS_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * H > 65535 * 64) return OS_ERR_UNSUPPORTED;
  const int64_t need = oss::attention_workspace_bytes(B, H, Sq, Sk, causal != 0);
  if (need < 0) return OS_ERR_CUDA;
  if (need > 0 && workspace && workspace_bytes < need) return OS_ERR_INVALID_ARGUMENT;
  unsigned int* err = error_word();
  if (!err) return OS_ERR_CUDA;
  const oss::AttnFault fault = t_fault;
  t_fault = oss::AttnFault();
  return from_cuda(oss::launch_attention_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale,
                                             causal != 0, err, fault, nullptr, t_rescale_policy,
                                             workspace, workspace_bytes,
                                             static_cast<cudaStream_t>(stream)));
}

os_status os_attention_fwd_partial(const os_bf16* q, const os_bf16* k, const os_bf16* v,
                                   int32_t B, int32_t H, int32_t Sq, int32_t Sk, int32_t D,
                                   float scale, int causal, float* part_m, float* part_l,
                                   float* part_o, int32_t part_stride, int32_t part_index,
                                   void* stream) {
  if (!q || !k || !v || !part_m || !part_l || !part_o) return OS_ERR_INVALID_ARGUMENT;
  if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return OS_ERR_INVALID_ARGUMENT;
  if (part_stride <= 0 || part_index < 0 || part_index >= part_stride) return OS_ERR_INVALID_ARGUMENT;
  if (!valid_scale(scale)) return OS_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(part_o)) return OS_ERR_MISALIGNED;
  if (D != 128) return OS_ERR_UNSUPPORTED;
  if (causal && Sq != Sk) return OS_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * H > 65535 * 64) return OS_ERR_UNSUPPORTED;
  unsigned int* err = error_word();
  if (!err) return OS_ERR_CUDA;
  const oss::AttnFault fault = t_fault;
  t_fault = oss::AttnFault();
  const oss::AttnPartialOut out{part_m, part_l, part_o, part_stride, part_index};
  return from_cuda(oss::launch_attention_fwd(q, k, v, nullptr, nullptr, B, H, Sq, Sk, D, scale,
                                             causal != 0, err, fault, &out, t_rescale_policy,
                                             nullptr, 0, static_cast<cudaStream_t>(stream)));
}

os_status os_attention_decode_splitkv(const os_bf16* q, const os_bf16* k, const os_bf16* v,
                                      const int32_t* kv_len, int32_t B, int32_t H, int32_t Lmax,
                                      int32_t D, int32_t num_splits, float scale, float* part_m,
                                      float* part_l, float* part_o, void* stream) {
  if (!q || !k || !v || !kv_len || !part_m || !part_l || !part_o) return OS_ERR_INVALID_ARGUMENT;
  if (B <= 0 || H <= 0 || Lmax <= 0 || D <= 0 || num_splits <= 0) return OS_ERR_INVALID_ARGUMENT;
  if (!valid_scale(scale)) return OS_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(part_o))
    return OS_ERR_MISALIGNED;
  if (D != 128 || num_splits > 64 || B > 65535 || H > 65535) return OS_ERR_UNSUPPORTED;
  return from_cuda(oss::launch_decode_splitkv(q, k, v, kv_len, B, H, Lmax, D, num_splits, scale,
                                              part_m, part_l, part_o,
                                              static_cast<cudaStream_t>(stream)));
}

os_status os_merge_partials(const float* part_m, const float* part_l, const float* part_o,
                            int64_t groups, int32_t num_splits, int32_t D, int finalize,
                            void* o_out, float* m_out, float* l_out, float* lse_out,
                            void* stream) {
  if (!part_m || !part_l || !part_o || !o_out) return OS_ERR_INVALID_ARGUMENT;
  if (groups <= 0 || num_splits <= 0 || D <= 0) return OS_ERR_INVALID_ARGUMENT;
  if (!aligned16(part_o) || !aligned16(o_out)) return OS_ERR_MISALIGNED;
  if (num_splits > 64 || D > 256 || (D & 3)) return OS_ERR_UNSUPPORTED;
  return from_cuda(oss::launch_merge_partials(part_m, part_l, part_o, groups, num_splits, D,
                                              finalize, o_out, m_out, l_out, lse_out,
                                              static_cast<cudaStream_t>(stream)));
}

os_status os_attention_set_rescale_policy(int32_t policy) {
  if (policy != OS_RESCALE_THRESHOLD && policy != OS_RESCALE_ON_RISE && policy != OS_RESCALE_ALWAYS)
    return OS_ERR_INVALID_ARGUMENT;
  t_rescale_policy = policy;
  return OS_OK;
}

int32_t os_attention_rescale_policy(void) { return t_rescale_policy; }

os_status os_debug_inject_fault(int32_t kind, int32_t step, int64_t timeout_ns) {
  if (kind < 0 || kind > 2 || step < 0 || timeout_ns < 0) return OS_ERR_INVALID_ARGUMENT;
  t_fault = oss::AttnFault();
  t_rows_fault = oss::RowsFault();
  if (kind == 1) {
    t_fault.skip_v_step = step;
    t_fault.timeout_ns = timeout_ns;
  } else if (kind == 2) {
    t_rows_fault.extra_tx = 16;
    t_rows_fault.timeout_ns = timeout_ns;
  }
  return OS_OK;
}

os_status os_check_device_error(void* stream, int32_t* code) {
  if (code) *code = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return OS_ERR_CUDA;
  unsigned int* err = error_word();
  if (!err) return OS_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyAsync(&word, err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return OS_ERR_CUDA;
  if (cudaMemsetAsync(err, 0, sizeof(word), s) != cudaSuccess) return OS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return OS_ERR_CUDA;
  if (code) *code = static_cast<int32_t>(word);
  return word ? OS_ERR_TIMEOUT : OS_OK;
}

}  // extern "C"
