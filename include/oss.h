/*
 * liboss -- online softmax, fused attention forward, split-KV decode and the
 * (m, l, O) merge on one NVIDIA GB300 (sm_103a).
 *
 * The method: a row's softmax is computed block by block while carrying a
 * running maximum m and a running sum l of exp(x - m); when a block raises
 * the maximum, l (and, for attention, the output accumulator O) is multiplied
 * by exp(m_old - m_new) before the block is added. After the last block
 * O /= l. Sources: roadmapper "Online softmax" ("The recurrence",
 * "Initialise honestly"), curionode "The Online Softmax." (introduction,
 * "One pass, exactly"), metalworking "Online Softmax" (the five-line
 * recurrence and its closing note on split-KV decode).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Tensors are DEVICE pointers allocated and owned by the caller (besides
 *   them, os_softmax_rows_from_host takes host pointers). The library never
 *   allocates, frees or keeps them.
 * - Layouts are row-major; the attention tensors are dense [B, H, S, D].
 * - Each call validates its arguments on the host, then enqueues its kernels
 *   on `stream` (a cudaStream_t passed as void*; NULL = the legacy default
 *   stream) and returns without synchronising. A non-OK status means nothing
 *   was enqueued (except OS_ERR_CUDA, which reports a failed launch).
 * - Outputs must not overlap inputs or each other.
 * - m is reported in natural units: m = max of scale * x. l is the sum of
 *   exp(scale * x - m), i.e. the normaliser relative to the maximum
 *   (curionode "The Online Softmax.", "Workshop"); lse = m + ln(l).
 * - A fully masked or empty row reports m = -inf, l = 0, lse = -inf and a
 *   zero output instead of NaN (roadmapper "Online softmax", "Initialise
 *   honestly", describes the NaN an unguarded empty block produces).
 * - bf16 tensors are passed as `os_bf16` (the raw 16-bit patterns).
 * - The library keeps one device error word per device; kernels that wait
 *   on an mbarrier give up after a bounded number of polls and set it.
 *   os_check_device_error reads and clears it.
 */
#ifndef OSS_H
#define OSS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OSS_ABI_VERSION 1

#if defined(__GNUC__)
#define OSS_API __attribute__((visibility("default")))
#else
#define OSS_API
#endif

typedef uint16_t os_bf16; /* IEEE-754 binary32 truncated to its top 16 bits (bfloat16) */

typedef enum os_status {
  OS_OK = 0,
  OS_ERR_INVALID_ARGUMENT = 1, /* null pointer, non-positive size, ld < cols, bad scale */
  OS_ERR_MISALIGNED = 2,       /* a base address or leading dimension is not 16-byte aligned */
  OS_ERR_UNSUPPORTED = 3,      /* a valid request this version does not implement */
  OS_ERR_CUDA = 4,             /* a CUDA runtime or driver call failed (launch, attribute, ...) */
  OS_ERR_TIMEOUT = 5           /* a kernel gave up on a bounded wait (os_check_device_error) */
} os_status;

/*
 * os_softmax_rows -- one-pass safe softmax of each row of a row-major matrix.
 *
 * Defines (curionode "The Online Softmax.", introduction and "One pass,
 * exactly"; the running pair (m, l) of roadmapper "Online softmax", "The
 * recurrence"):
 *     m[r] = max_j fl32(scale * x[r, j])
 *     l[r] = sum_j exp(scale * x[r, j] - m[r])
 *     y[r, j] = exp(scale * x[r, j] - m[r]) / l[r]
 * computed with exp2 and log2(e) folded into the scale once. Each element of
 * x is read from HBM once and each element of y written once.
 *
 *   x     [rows, ld_x] fp32, device. Entries may be -inf (masked); +inf / NaN
 *         inputs, and finite ones with |scale * x * log2(e)| beyond the fp32
 *         range, are undefined.
 *   y     [rows, ld_y] fp32, device, written for j < cols.
 *   m, l  [rows] fp32, device, or NULL to skip.
 *   rows  >= 1; cols >= 1; ld_x >= cols, ld_y >= cols (elements).
 *   scale finite and > 0.
 * Alignment: x, y, m and l 4-byte aligned. When each row of x starts at the
 * same offset from a 16-byte boundary as the same row of y (x and y 16-byte
 * aligned with ld_x, ld_y multiples of 4; or, say, y laid out like x), the
 * kernel moves the row in 16-byte chunks on that grid and reads each element
 * once and writes it once: rows of up to 16384 elements are held in
 * registers (several rows per CTA up to 2048 elements); longer rows of up to
 * 1.6 MB by a thread-block cluster of up to eight CTAs, whose slices' (max,
 * sum) states are merged through distributed shared memory: in the cluster's
 * registers for rows on the 16-byte grid of 20481..65536 elements, in its
 * shared memory otherwise. For a row off the 16-byte grid, the loads of its first and last
 * chunks may read (never write) bytes of the same 16-byte granules outside
 * the row. Short rows of a matrix whose x rows lie back to back (ld_x ==
 * cols; rows of up to 512 bytes, or 1 KB off the 16-byte grid) are taken a
 * tile of whole rows at a time, copied into shared memory by bulk
 * asynchronous copies whatever their offsets, with y at any offset and
 * leading dimension; the 16-byte granules holding x's first and last
 * elements may be read (never written) whole. Other rows whose x and y
 * offsets differ, and rows longer than 1.6 MB, are streamed twice (two reads,
 * one write; os_softmax_rows_ws reads them once).
 * Errors: OS_ERR_INVALID_ARGUMENT, OS_ERR_MISALIGNED, OS_ERR_CUDA.
 */
OSS_API os_status os_softmax_rows(const float* x, float* y, float* m, float* l,
                          int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                          float scale, void* stream);

/*
 * os_softmax_rows_workspace_bytes -- bytes of workspace os_softmax_rows_ws /
 * os_softmax_rows_16bit_ws use for rows of `cols` elements of type `dtype`
 * (0 = fp32, OS_DTYPE_BF16, OS_DTYPE_F16) on the current device: a few tens
 * of KB for rows longer than the 1.6 MB a thread-block cluster holds, 0 for
 * shorter rows (they never use it); -1 when the device cannot be queried.
 */
OSS_API int64_t os_softmax_rows_workspace_bytes(int64_t rows, int64_t cols, int32_t dtype);

/*
 * os_softmax_rows_ws -- os_softmax_rows with a caller-owned device
 * workspace. Rows longer than a cluster's shared memory holds (over 1.6 MB)
 * then take the whole GPU a few rows at a time (as many as fit in L2):
 * every CTA streams one slice of a row once, forming the slice's (max, sum)
 * state of the online normaliser; the slices' states meet in the workspace
 * at a grid-wide barrier of a cooperative launch and are merged in slice
 * order with the pairwise identity (curionode "The Online Softmax.", "One
 * pass, exactly"); each CTA then reads its slice again, from L2, to write y.
 * HBM sees one read and one write per element; without a workspace such rows
 * are read twice from HBM. Results are those of os_softmax_rows, within its
 * tolerance; shorter rows ignore the workspace.
 *
 *   workspace        device memory of at least os_softmax_rows_workspace_bytes
 *                    bytes, 16-byte aligned (contents need no initialising:
 *                    the call zeroes what it needs, with an asynchronous
 *                    memset on `stream`), or NULL with workspace_bytes 0.
 *   workspace_bytes  its size; too small: the rows are streamed twice.
 * Calls that may run at the same time (other streams) need workspaces of
 * their own. Other arguments and errors as os_softmax_rows; a grid barrier
 * that waits longer than 2 s gives up and os_check_device_error then reports
 * OS_ERR_TIMEOUT with code 2 | (2 << 8).
 */
OSS_API os_status os_softmax_rows_ws(const float* x, float* y, float* m, float* l,
                                     int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                                     float scale, void* workspace, int64_t workspace_bytes,
                                     void* stream);

/* Element type of a 16-bit row (os_softmax_rows_16bit). */
typedef enum os_dtype {
  OS_DTYPE_BF16 = 1, /* bfloat16: the top 16 bits of an IEEE binary32 */
  OS_DTYPE_F16 = 2   /* IEEE-754 binary16 */
} os_dtype;

/*
 * os_softmax_rows_16bit -- os_softmax_rows for rows stored in bf16 or fp16,
 * the same definition with the same one-pass recurrence (curionode "The
 * Online Softmax.", "One pass, exactly"). Each element is widened to fp32
 * exactly; weights, m and l are formed in fp32 as in os_softmax_rows; y is
 * rounded once to the row's type (round to nearest even), so it carries that
 * type's rounding error (2^-8 relative for bf16, 2^-11 for fp16, whose
 * results below 2^-14 are subnormal).
 *
 *   x     [rows, ld_x] 16-bit elements of type `dtype`, device. -inf entries
 *         are masked; +inf / NaN inputs are undefined.
 *   y     [rows, ld_y] same type, device, written for j < cols.
 *   m, l  [rows] fp32, device, or NULL to skip (natural units, as
 *         os_softmax_rows).
 *   rows >= 1; cols >= 1; ld_x >= cols, ld_y >= cols (elements); scale
 *   finite and > 0; dtype an os_dtype.
 * Alignment: x and y 2-byte aligned, m and l 4-byte aligned. When x's and
 * y's rows start at the same offsets from a 16-byte boundary, rows of up to
 * 16384 elements are held in registers and longer rows of up to 1.6 MB by a
 * cluster, as for os_softmax_rows (in its registers for rows on the 16-byte
 * grid of 18433..131072 elements; one read, one write per
 * element, the same granule reads at the ends of a row off the grid). Short
 * rows of a matrix whose x rows lie back to back are staged in shared memory
 * by tiles as for os_softmax_rows, with y at any layout; other rows are
 * streamed twice.
 * Errors: OS_ERR_INVALID_ARGUMENT, OS_ERR_MISALIGNED, OS_ERR_CUDA.
 */
OSS_API os_status os_softmax_rows_16bit(const void* x, void* y, float* m, float* l,
                                        int64_t rows, int64_t cols, int64_t ld_x, int64_t ld_y,
                                        float scale, int32_t dtype, void* stream);

/*
 * os_softmax_rows_16bit_ws -- os_softmax_rows_16bit with a workspace, as
 * os_softmax_rows_ws (the same single read from HBM for rows over 1.6 MB).
 */
OSS_API os_status os_softmax_rows_16bit_ws(const void* x, void* y, float* m, float* l,
                                           int64_t rows, int64_t cols, int64_t ld_x,
                                           int64_t ld_y, float scale, int32_t dtype,
                                           void* workspace, int64_t workspace_bytes, void* stream);

/*
 * os_softmax_rows_from_host -- os_softmax_rows on rows that sit in host
 * memory: the library copies x up, runs the row softmax and copies y (and m,
 * l) back. The pages define no host-side call; this is the end-to-end form
 * of the row softmax (the curionode page's "one pass, exactly": the row is
 * read once), for a caller whose rows live on the host.
 *   x_host [rows, cols] fp32, host, dense (leading dimension cols); read.
 *   y_host [rows, cols] fp32, host, dense; written.
 *   m_host, l_host [rows] fp32, host, or NULL to skip (natural units, as
 *         os_softmax_rows).
 *   x_dev, y_dev [rows, cols] fp32, device, dense, owned by the caller: the
 *         staging copies (x_dev ends up holding x, y_dev holding y).
 *   m_dev, l_dev [rows] fp32, device, owned by the caller; required when
 *         m_host (l_host) is given, else may be NULL.
 *   rows >= 1; cols >= 1; scale finite and > 0; chunk_rows >= 0 (rows per
 *   block; 0: about 64 MiB of x a block).
 * The rows go in blocks of chunk_rows: block b's upload, kernel and
 * download run on three streams (two copy streams the library makes once
 * per device, and `stream` for the kernels), so block b + 1 uploads while
 * block b computes and block b - 1 downloads. The copies start after the
 * work already enqueued on `stream`, and `stream` waits for the last
 * download: the call returns at once, and the host outputs are complete when
 * `stream` is (synchronise it before reading them or freeing any buffer).
 * Host buffers must be page-locked (cudaHostAlloc, or pinned by the caller)
 * for the copies to overlap; pageable memory gives the same results, with
 * copies that do not overlap. Every row gets the kernel os_softmax_rows gives
 * it, so the results equal those of os_softmax_rows on x_dev. Creates and
 * releases four CUDA events per call; allocates no memory.
 * Errors: OS_ERR_INVALID_ARGUMENT (null x_host, y_host, x_dev or y_dev; a
 *         host m or l without its device buffer; a bad size or scale),
 *         OS_ERR_MISALIGNED (a device buffer not 4-byte aligned),
 *         OS_ERR_CUDA (a copy, an event or a launch failed; outputs undefined).
 */
OSS_API os_status os_softmax_rows_from_host(const float* x_host, float* y_host, float* m_host,
                                            float* l_host, float* x_dev, float* y_dev, float* m_dev,
                                            float* l_dev, int64_t rows, int64_t cols, float scale,
                                            int64_t chunk_rows, void* stream);

/*
 * os_softmax_rows_multipass -- the same outputs as os_softmax_rows, computed
 * the way the curionode page describes the methods the online form replaces
 * (introduction): passes = 3 is the safe softmax -- a maximum pass, a sum pass
 * and a normalising pass -- and passes = 2 runs the online normaliser over
 * the row and then a normalising pass. Each pass is a separate sweep over
 * the whole matrix, so x is read from HBM `passes` times (os_softmax_rows
 * reads it once). Provided to measure that saving; m and l are required (they
 * carry the state between passes).
 *   Arguments and alignment as os_softmax_rows, plus passes in {2, 3}.
 * Errors: OS_ERR_INVALID_ARGUMENT (also for other passes, null m or l),
 * OS_ERR_MISALIGNED, OS_ERR_CUDA.
 */
OSS_API os_status os_softmax_rows_multipass(const float* x, float* y, float* m, float* l,
                                            int64_t rows, int64_t cols, int64_t ld_x,
                                            int64_t ld_y, float scale, int32_t passes,
                                            void* stream);

/*
 * os_attention_fwd -- fused attention forward that never stores a score row.
 *
 * Defines (metalworking "Online Softmax", the five-line recurrence;
 * curionode "The Online Softmax.", "One pass, exactly", on tiling attention
 * without storing a row of scores):
 *     S_ij = scale * q_i . k_j            (j <= i only, when causal)
 *     o_i  = sum_j exp(S_ij - m_i) v_j / l_i,   lse_i = m_i + ln(l_i)
 * Keys stream through in tiles; per tile the running (m, l, O) is rescaled
 * by exp2(m_old - m_new) and the tile added (S = Q K^T and O += P V run on
 * the tcgen05 tensor cores with fp32 accumulation in tensor memory; P is
 * rounded to bf16 for the P V product, l sums the fp32 P).
 *
 *   q    [B, H, Sq, D] bf16, device.   k, v [B, H, Sk, D] bf16, device.
 *   o    [B, H, Sq, D] bf16, device (round to nearest even).
 *   lse  [B, H, Sq] fp32, device (natural log), or NULL to skip.
 *   B, H, Sq, Sk >= 1.  D == 128 (other head sizes: OS_ERR_UNSUPPORTED).
 *   scale finite and > 0.
 *   causal != 0: query i attends to keys 0..i; requires Sq == Sk
 *   (OS_ERR_UNSUPPORTED otherwise).
 * Alignment: q, k, v, o 16-byte aligned.
 * Errors: OS_ERR_INVALID_ARGUMENT, OS_ERR_MISALIGNED, OS_ERR_UNSUPPORTED,
 * OS_ERR_CUDA; a timed-out internal wait is reported by os_check_device_error.
 */
OSS_API os_status os_attention_fwd(const os_bf16* q, const os_bf16* k, const os_bf16* v,
                           os_bf16* o, float* lse,
                           int32_t B, int32_t H, int32_t Sq, int32_t Sk, int32_t D,
                           float scale, int causal, void* stream);

/*
 * os_attention_fwd_workspace_bytes -- bytes of workspace os_attention_fwd_ws
 * uses for this shape on the current device; 0 when it uses none (causal
 * launches, and launches whose query tiles fill whole rounds of the GPU's
 * SMs), -1 when the device cannot be queried.
 */
OSS_API int64_t os_attention_fwd_workspace_bytes(int32_t B, int32_t H, int32_t Sq, int32_t Sk,
                                                 int32_t D, int causal);

/*
 * os_attention_fwd_ws -- os_attention_fwd with a caller-owned device
 * workspace, which lets a non-causal launch keep every SM busy to the end:
 * the kernel walks the 128-row query tiles in rounds of one tile per SM;
 * when the last round would leave SMs idle, its tiles are cut along the keys
 * into 2..8 parts, one per SM, each part's partial state (m, l, O) goes to
 * the workspace, and the last part of a tile to finish combines them with
 * the pairwise merge identity of the curionode page ("One pass, exactly"),
 * always in part order, so results do not depend on which SM finishes last.
 * The outputs are those of os_attention_fwd, within its tolerance.
 *
 *   workspace        device memory of at least os_attention_fwd_workspace_bytes
 *                    bytes, 16-byte aligned, or NULL with workspace_bytes 0
 *                    (then the call is os_attention_fwd). It must be all
 *                    zeros the first time it is used (fill it with zeros
 *                    once): it holds the per-tile counters of finished parts,
 *                    which every call that completes leaves at zero again.
 *                    After a call that reported OS_ERR_TIMEOUT, zero it again
 *                    before reuse.
 *   workspace_bytes  its size; smaller than required: OS_ERR_INVALID_ARGUMENT.
 * Calls that may run at the same time (other streams) need workspaces of
 * their own. Other arguments and errors as os_attention_fwd.
 */
OSS_API os_status os_attention_fwd_ws(const os_bf16* q, const os_bf16* k, const os_bf16* v,
                                      os_bf16* o, float* lse, int32_t B, int32_t H, int32_t Sq,
                                      int32_t Sk, int32_t D, float scale, int causal,
                                      void* workspace, int64_t workspace_bytes, void* stream);

/*
 * os_attention_fwd_noalloc -- os_attention_fwd_ws for callers that cannot
 * allocate device memory. The online-softmax pages this library follows have
 * no counterpart to this call: it exists because some callers cannot hand
 * over a workspace, such as a plugin that its host framework gives only the
 * input and output buffers while the framework's own pool owns the rest of
 * device memory, or a latency-critical thread that must not call cudaMalloc
 * (which can block and synchronise the device).
 *
 * The split tail's workspace comes from a fixed 16 MiB array in device
 * memory that the library declares statically; every GPU that loads the
 * library holds those 16 MiB until the process exits. The call itself
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine). The first call on a device looks up the array's device address
 * on that device (cudaGetSymbolAddress, once per device); make that first
 * call before any stream capture.
 *
 * Arguments, layout, outputs and tolerance are os_attention_fwd's; the
 * caller still owns and passes q, k, v, o and lse. Every call clears the
 * counters it needs at zero (an asynchronous memset on `stream`), so the
 * array's leftover contents from an earlier call, even one that timed out,
 * do no harm. All calls on a device share the one array: calls whose work
 * overlaps on the GPU (other streams, other threads) race on it and give
 * wrong results, so order them on one stream or with events.
 *
 * Errors: those of os_attention_fwd; OS_ERR_UNSUPPORTED also when the shape
 * needs more than the 16 MiB array holds (the split tail takes about 68 KB
 * per SM, 10.4 MB on a GPU with 152 SMs); OS_ERR_CUDA when the device or the
 * array's address cannot be queried.
 */
OSS_API os_status os_attention_fwd_noalloc(const os_bf16* q, const os_bf16* k, const os_bf16* v,
                                           os_bf16* o, float* lse, int32_t B, int32_t H,
                                           int32_t Sq, int32_t Sk, int32_t D, float scale,
                                           int causal, void* stream);

/*
 * Rescale policies of the attention forward: when a tile raises a row's
 * maximum, the running sum l and the accumulator O are multiplied by
 * exp(m_old - m_new) (metalworking "Online Softmax", the five-line
 * recurrence). The same page's "Recognition guide" sets two kernels side by
 * side that disagree on when to do it: MLX multiplies on every tile,
 * metal-flash-attention only when the maximum rose. Here O lives in tensor
 * memory, so each rescale costs a wait for the previous P V and a round trip
 * of O; the decision is taken per warp of 16 rows. All three policies compute
 * the same O and lse in exact arithmetic (the reference maximum cancels in
 * O / l); their rounding differs within the documented tolerance.
 */
typedef enum os_rescale_policy {
  OS_RESCALE_THRESHOLD = 0, /* default: move the reference maximum only when a
                               row of the warp rose by more than 8 (base 2), so
                               the weights stay below 2^8; rarely rescales */
  OS_RESCALE_ON_RISE = 1,   /* metal-flash-attention's guard: whenever a row of
                               the warp rose at all */
  OS_RESCALE_ALWAYS = 2     /* MLX's form: on every tile */
} os_rescale_policy;

/*
 * os_attention_set_rescale_policy -- choose the rescale policy of the
 * os_attention_fwd and os_attention_fwd_partial calls the calling host
 * thread makes from now on (other threads keep theirs; a new thread starts
 * with OS_RESCALE_THRESHOLD, the fastest measured). Provided to measure the
 * trade named above; results agree within the attention tolerance.
 * Errors: OS_ERR_INVALID_ARGUMENT for another value (the setting is kept).
 */
OSS_API os_status os_attention_set_rescale_policy(int32_t policy);

/* The calling host thread's current os_rescale_policy. */
OSS_API int32_t os_attention_rescale_policy(void);

/*
 * os_attention_fwd_partial -- the attention forward over one shard of the
 * keys, written as partial softmax states instead of O / l, so that shards of
 * a long sequence (processed one after another, or on different devices) can
 * be combined with os_merge_partials -- the use of the pairwise identity the
 * curionode page names for ring attention ("One pass, exactly").
 *
 * For query row r = (b, h, i) over the keys of this call:
 *     part_m[s] = max_j scale * q_i . k_j              (natural units)
 *     part_l[s] = sum_j exp(scale * q_i . k_j - part_m[s])
 *     part_o[s] = sum_j exp(scale * q_i . k_j - part_m[s]) v_j   (fp32, not divided by l)
 * at slot s = r * part_stride + part_index: part_m, part_l are
 * [B*H*Sq, part_stride] fp32 and part_o [B*H*Sq, part_stride, D] fp32, the
 * layout os_merge_partials reads with groups = B*H*Sq, num_splits =
 * part_stride. A row with no visible key writes (-inf, 0, 0).
 *
 *   q [B, H, Sq, D], k, v [B, H, Sk, D] bf16 (the shard's keys), device.
 *   causal != 0 (Sq == Sk): query i sees keys 0..i of this shard -- the
 *   diagonal shard of a causally masked sequence; earlier shards use 0.
 *   B, H, Sq, Sk >= 1; D == 128; 0 <= part_index < part_stride; scale > 0.
 * Alignment: q, k, v, part_o 16-byte aligned.
 * Errors: as os_attention_fwd.
 */
OSS_API os_status os_attention_fwd_partial(const os_bf16* q, const os_bf16* k, const os_bf16* v,
                                           int32_t B, int32_t H, int32_t Sq, int32_t Sk,
                                           int32_t D, float scale, int causal,
                                           float* part_m, float* part_l, float* part_o,
                                           int32_t part_stride, int32_t part_index,
                                           void* stream);

/*
 * os_attention_decode_splitkv -- one query token per (batch, head) against a
 * padded KV cache, cut into num_splits chunks, each chunk written as a
 * partial softmax state (metalworking "Online Softmax", closing note: split-KV
 * decode merges partial softmaxes with the same correction identity instead
 * of float atomics).
 *
 * For batch b with L = kv_len[b] and chunk = ceil(L / num_splits), split j
 * covers keys [j*chunk, min(L, (j+1)*chunk)). Its partial is
 *     part_m = max_t scale * q . k_t                     (natural units)
 *     part_l = sum_t exp(scale * q . k_t - part_m)
 *     part_o = sum_t exp(scale * q . k_t - part_m) v_t   (NOT divided by l)
 * An empty split writes (-inf, 0, 0).
 *
 *   q       [B, H, D] bf16, device.
 *   k, v    [B, H, Lmax, D] bf16, device; only rows t < kv_len[b] are read.
 *   kv_len  [B] int32, DEVICE; each value in 1..Lmax (values outside are
 *           clamped to [0, Lmax] on the device; 0 gives all-empty splits).
 *   part_m, part_l  [B, H, num_splits] fp32, device.
 *   part_o  [B, H, num_splits, D] fp32, device.
 *   B, H, Lmax >= 1.  D == 128.  1 <= num_splits <= 64.  scale finite, > 0.
 * Alignment: q, k, v, part_o 16-byte aligned.
 * Errors: OS_ERR_INVALID_ARGUMENT, OS_ERR_MISALIGNED, OS_ERR_UNSUPPORTED,
 * OS_ERR_CUDA.
 */
OSS_API os_status os_attention_decode_splitkv(const os_bf16* q, const os_bf16* k, const os_bf16* v,
                                      const int32_t* kv_len,
                                      int32_t B, int32_t H, int32_t Lmax, int32_t D,
                                      int32_t num_splits, float scale,
                                      float* part_m, float* part_l, float* part_o,
                                      void* stream);

/*
 * os_merge_partials -- merge num_splits partial states (m, l, O) per group
 * with the pairwise identity (curionode "The Online Softmax.", "One pass,
 * exactly": the identity for pairs of partial results is associative, so
 * they can be merged in any order or tree):
 *     m = max(m1, m2);  l = l1 e^(m1-m) + l2 e^(m2-m);  O = O1 e^(m1-m) + O2 e^(m2-m)
 * in a fixed pairwise tree ((0,1),(2,3),...; an odd element is carried up),
 * with no atomics, so the result is the same on every run. Two empty sides
 * merge to (-inf, 0, 0).
 *
 *   part_m, part_l  [groups, num_splits] fp32, device.
 *   part_o          [groups, num_splits, D] fp32, device (unnormalised).
 *   finalize != 0: o_out is bf16 [groups, D] = O / l (0 for an empty group).
 *   finalize == 0: o_out is fp32 [groups, D] = the merged unnormalised O, so
 *                  merges can nest (hierarchical or across shards).
 *   m_out, l_out, lse_out  [groups] fp32, device, each may be NULL.
 *   groups >= 1.  1 <= num_splits <= 64.  1 <= D <= 256, D % 4 == 0.
 * Alignment: part_o and o_out 16-byte aligned.
 * Errors: OS_ERR_INVALID_ARGUMENT, OS_ERR_MISALIGNED, OS_ERR_UNSUPPORTED,
 * OS_ERR_CUDA.
 */
OSS_API os_status os_merge_partials(const float* part_m, const float* part_l, const float* part_o,
                            int64_t groups, int32_t num_splits, int32_t D, int finalize,
                            void* o_out, float* m_out, float* l_out, float* lse_out,
                            void* stream);

/*
 * os_check_device_error -- synchronise `stream`, then read and clear the
 * current device's error word. *code receives 0 when no kernel gave up on a
 * wait since the last check, otherwise an OS_ERR_TIMEOUT detail code
 * (bits 0..7 = kernel id, bits 8..15 = wait site): kernel 1 is the attention
 * forward (see os_debug_inject_fault); 2 | (1 << 8) is a row softmax whose
 * wait for its row's bulk copies into shared memory gave up, 2 | (2 << 8) one
 * whose wait for the (max, sum) states of the other CTAs of its cluster gave
 * up. Returns
 * OS_ERR_TIMEOUT when the word was set, OS_ERR_CUDA when a CUDA call failed,
 * OS_OK otherwise.
 * `code` may be NULL.
 * The word keeps the FIRST error written since it was last cleared. Call
 * this after any launch that may have failed, before the next launch: while
 * an old error sits in the word, a new failing attention launch cannot
 * publish its own tag there, so its other CTAs no longer stop early and each
 * waits out its own time limit (the launch still ends; it only ends later).
 */
OSS_API os_status os_check_device_error(void* stream, int32_t* code);

/*
 * os_debug_inject_fault -- test hook for the bounded waits. Arms a fault for
 * the next call of the kind's entry point made by the calling host thread
 * (that call disarms it):
 *   kind 0: disarm.
 *   kind 1: the kernel's load warp skips the V tile of KV step `step` (counted
 *           in the order each CTA visits its KV tiles), so the thread that
 *           issues P V waits on a phase that never completes. After
 *           `timeout_ns` (0: the default of 2 s) it raises the CTA's abort
 *           flag; every role drains its own copies and MMAs, tensor memory is
 *           freed, and the kernel exits (the other CTAs of the launch see
 *           the recorded error and stop too). os_check_device_error then
 *           returns OS_ERR_TIMEOUT with code & 0xFFFF = 1 | (3 << 8) (kernel
 *           1, wait site 3: V tile full); bits 16..31 hold the launch's tag.
 *           The CUDA context stays usable; the outputs of that call are
 *           undefined.
 *   kind 2: the next os_softmax_rows or os_softmax_rows_16bit call. If it
 *           holds its rows in a cluster's shared memory (rows longer than
 *           16384 elements and at most 1.6 MB that the register path below
 *           does not take) or stages short rows of a dense matrix in shared
 *           memory, every CTA's barrier for the bulk copies of its first row
 *           (or tile) is told to expect 16 bytes more than are copied; the
 *           code is then 2 | (1 << 8). If it holds its rows in a cluster's
 *           registers (rows on the 16-byte grid of 18433..131072 16-bit or
 *           20481..65536 fp32 elements), every CTA's barrier for the
 *           cluster's states of its first row expects 16 bytes more than
 *           the states; the code is then 2 | (2 << 8). The wait gives up
 *           after `timeout_ns` (0: 2 s); from then on each CTA waits (and
 *           copies or sends) no more but still meets its barriers, so the
 *           launch ends. os_check_device_error then returns OS_ERR_TIMEOUT
 *           with that code. The outputs of that call are undefined; other
 *           paths ignore the hook. `step` is unused.
 * No GPU fault, trap or endless wait is involved.
 * Errors: OS_ERR_INVALID_ARGUMENT (kind not 0/1/2, step < 0, timeout_ns < 0).
 */
OSS_API os_status os_debug_inject_fault(int32_t kind, int32_t step, int64_t timeout_ns);

/* Human-readable name of a status (static storage; never NULL). */
OSS_API const char* os_status_string(os_status status);

/* OSS_ABI_VERSION of the loaded library. */
OSS_API int32_t os_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OSS_H */
