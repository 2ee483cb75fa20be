// Host-side launchers behind the C ABI in include/oss.h. Arguments are
// already validated by api.cu when these run.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace oss {

// Kernel ids stored in bits 0..7 of the device error word.
enum KernelId : unsigned int { kKernelAttnFwd = 1, kKernelSoftmaxRows = 2 };

// Test hook for the bounded wait of the cluster-resident row kernel (see
// os_debug_inject_fault): extra_tx > 0 makes each CTA expect that many bytes
// more than its first row's copies deliver; timeout_ns > 0 replaces the
// default wait limit.
struct RowsFault {
  uint32_t extra_tx = 0;
  int64_t timeout_ns = 0;
};

// err_word: the device error word (the cluster-resident kernel records a
// give-up on its bounded wait there); may be null.
// ws (may be null, ws_bytes 0): a workspace of softmax_workspace_bytes()
// bytes; with it, rows beyond the cluster path's 1.6 MB are read once from
// HBM instead of twice.
cudaError_t launch_softmax_rows(const float* x, float* y, float* m, float* l,
                                int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                                float scale, unsigned int* err_word, const RowsFault& fault,
                                void* ws, int64_t ws_bytes, cudaStream_t stream);

// 16-bit rows: dtype 1 = bf16, 2 = fp16 (x and y); m, l fp32 or null.
cudaError_t launch_softmax_rows16(const uint16_t* x, uint16_t* y, float* m, float* l,
                                  int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                                  float scale, int dtype, unsigned int* err_word,
                                  const RowsFault& fault, void* ws, int64_t ws_bytes,
                                  cudaStream_t stream);

// Workspace the row softmax of rows of `row_bytes` bytes uses on the current
// device (0: none; -1: the device could not be queried).
int64_t softmax_workspace_bytes(int64_t row_bytes);

// Comparators: passes = 2 (online (m, l) pass, then a write pass) or 3 (max
// pass, sum pass, write pass); each pass re-reads x from HBM. m, l required.
cudaError_t launch_softmax_rows_multipass(const float* x, float* y, float* m, float* l,
                                          int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                                          float scale, int passes, cudaStream_t stream);

cudaError_t launch_decode_splitkv(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  const int32_t* kv_len, int B, int H, int Lmax, int D,
                                  int num_splits, float scale, float* part_m, float* part_l,
                                  float* part_o, cudaStream_t stream);

cudaError_t launch_merge_partials(const float* part_m, const float* part_l, const float* part_o,
                                  int64_t groups, int num_splits, int D, int finalize,
                                  void* o_out, float* m_out, float* l_out, float* lse_out,
                                  cudaStream_t stream);

// Test hook for the bounded waits of the attention kernel (see
// os_debug_inject_fault): skip_v_step >= 0 makes the producer skip that V
// load; timeout_ns > 0 replaces the default wait limit.
struct AttnFault {
  int skip_v_step = -1;
  int64_t timeout_ns = 0;
};

// Partial-state output of the attention forward: row r's (m, l, O) go to
// slot r * stride + index of m, l [rows * stride] and o [rows * stride, D].
struct AttnPartialOut {
  float* m;
  float* l;
  float* o;
  int stride;
  int index;
};

// Returns cudaErrorNotSupported for shapes the kernel does not cover. With
// partial != nullptr the kernel writes partial states instead of o and lse.
// rescale_policy: an os_rescale_policy value (0 threshold, 1 on rise, 2
// every tile). workspace (may be null): at least attention_workspace_bytes
// bytes, counters zero; with it, a non-causal launch whose query tiles do not
// fill the last round splits that round's tiles along the keys.
cudaError_t launch_attention_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 uint16_t* o, float* lse, int B, int H, int Sq, int Sk, int D,
                                 float scale, bool causal, unsigned int* err_word,
                                 const AttnFault& fault, const AttnPartialOut* partial,
                                 int rescale_policy, void* workspace, int64_t workspace_bytes,
                                 cudaStream_t stream);

// Workspace the attention forward of this shape uses on the current device
// (0: none; -1: the device could not be queried).
int64_t attention_workspace_bytes(int B, int H, int Sq, int Sk, bool causal);

// Bytes of per-tile counters at the end of that workspace (*bytes; 0 when it
// uses none). Returns -1 when the device could not be queried, else 0.
int64_t attention_workspace_counters(int B, int H, int Sq, int Sk, bool causal, int64_t* bytes);

// log2(e) split into a float and the float nearest to the remainder, so that
// hi + lo carries about 48 bits of it.
void split_constant(double c, float* hi, float* lo);

}  // namespace oss
