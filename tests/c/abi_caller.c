/* A plain C caller of liboss, built by tests/test_c_caller.py against
 * include/oss.h and the in-tree liboss.so. It makes only the calls that
 * return before touching a device (version, status names, argument
 * checks), so it runs on a machine without a GPU; it prints one line per
 * check and exits 1 on the first mismatch. */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "oss.h"

static int failures = 0;

static void expect(const char* what, int got, int want) {
  printf("%s: %d (want %d)\n", what, got, want);
  if (got != want) failures++;
}

int main(void) {
  /* a 16-byte aligned address that no call below dereferences */
  void* a = (void*)(uintptr_t)4096;
  float* f = (float*)a;
  float nan_scale = nanf("");

  expect("abi version", os_abi_version(), OSS_ABI_VERSION);
  expect("OS_OK name", strcmp(os_status_string(OS_OK), "OS_OK"), 0);
  expect("timeout name", strcmp(os_status_string(OS_ERR_TIMEOUT), "OS_ERR_TIMEOUT"), 0);

  expect("rows: null x", os_softmax_rows(NULL, f, NULL, NULL, 4, 8, 8, 8, 1.0f, NULL),
         OS_ERR_INVALID_ARGUMENT);
  expect("rows: ld_x < cols", os_softmax_rows(f, f, NULL, NULL, 4, 8, 7, 8, 1.0f, NULL),
         OS_ERR_INVALID_ARGUMENT);
  expect("rows: NaN scale", os_softmax_rows(f, f, NULL, NULL, 4, 8, 8, 8, nan_scale, NULL),
         OS_ERR_INVALID_ARGUMENT);
  expect("rows16: bad dtype", os_softmax_rows_16bit(a, a, NULL, NULL, 4, 8, 8, 8, 1.0f, 7, NULL),
         OS_ERR_INVALID_ARGUMENT);
  expect("from_host: m without device m",
         os_softmax_rows_from_host(f, f, f, NULL, f, f, NULL, NULL, 4, 8, 1.0f, 0, NULL),
         OS_ERR_INVALID_ARGUMENT);
  expect("attention: D = 64", os_attention_fwd((const os_bf16*)a, (const os_bf16*)a,
                                               (const os_bf16*)a, (os_bf16*)a, NULL, 1, 1, 128,
                                               128, 64, 1.0f, 0, NULL),
         OS_ERR_UNSUPPORTED);
  expect("decode: zero splits",
         os_attention_decode_splitkv((const os_bf16*)a, (const os_bf16*)a, (const os_bf16*)a,
                                     (const int32_t*)a, 1, 1, 128, 128, 0, 1.0f, f, f, f, NULL),
         OS_ERR_INVALID_ARGUMENT);
  expect("merge: zero groups", os_merge_partials(f, f, f, 0, 2, 128, 1, a, NULL, NULL, NULL, NULL),
         OS_ERR_INVALID_ARGUMENT);
  expect("rescale policy 3", os_attention_set_rescale_policy(3), OS_ERR_INVALID_ARGUMENT);
  expect("fault kind 3", os_debug_inject_fault(3, 0, 0), OS_ERR_INVALID_ARGUMENT);
  return failures ? 1 : 0;
}
