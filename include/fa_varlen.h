/*
 * fa_varlen.h -- C ABI of the GB300 (sm_103a) varlen attention library.
 *
 * Operation.  Packed variable-length scaled-dot-product attention in TND
 * layout, as defined by the web page "CANN/ops-transformer FlashAttention梯度V2"
 * (aclnnFlashAttentionUnpaddingScoreGradV2), section 功能说明 / 计算公式
 * (function description / formulas):
 *
 *     S  = Mask(scale * Q K^T)            P = Dropout(Softmax(S), keep_prob)
 *     Y  = P V
 *     dV = P^T dY      dQ = scale * dS K      dK = scale * dS^T Q
 *
 * with dS = P * (dP * Z / keep_prob - D), dP = dY V^T, D_i = sum_d dY_id Y_id.
 * fa_varlen_bwd is the product; fa_varlen_fwd produces the Y and softmax
 * statistics it consumes.
 *
 * Layout (parameter table + constraint section of that page).
 *   q, dy, y, dq : [total_q,  head_num,    head_dim], contiguous, row-major
 *   k, v, dk, dv : [total_kv, head_num_kv, head_dim], contiguous
 *   Sequence b owns rows [sum_{b'<b} L_b', sum_{b'<=b} L_b') of T ("T is B and
 *   S merged, packed tightly").  Element (t, n, d) sits at (t*N + n)*D + d.
 *   softmax_max, softmax_sum : float32 [total_q, head_num, 8] (the
 *   constraint section's TND statistics shape); lane 0 is read, the forward
 *   writes all 8 lanes.  max = row maximum of the scaled, masked logits;
 *   sum = sum_j exp(S_ij - max).  A row with no allowed key: max = -inf,
 *   sum = 0.
 *   seq_lens_q / seq_lens_kv : HOST arrays of `batch` int64 per-sequence
 *   actual lengths (actualSeqQLen / actualSeqKvLen), zero allowed.
 *   drop_mask : optional device bit mask, one bit per (b, n, i, j) at index
 *   O_b + (n*Lq_b + i)*Lk_b + j with O_b = N * sum_{b'<b} Lq_b'*Lk_b',
 *   least significant bit first, 1 = keep.  Read only when keep_prob < 1.
 *   Mask: key j is allowed for query i (0-based inside the sequence) iff
 *   i - pre_tokens <= j <= i + next_tokens (preTokens / nextTokens rows of
 *   the parameter table).  Causal = next_tokens 0, pre_tokens >= max length.
 *   sparse_mode (parameter table row sparseMode; the page defers the
 *   per-mode details to a document it does not include; these are the
 *   readings): 0 and 4 = that window (and the optional explicit mask of
 *   the options structs); 1 = the explicit mask alone; 2 = lower triangle
 *   aligned at the top-left corner, j <= i; 3 = lower triangle aligned at
 *   the bottom-right corner, j <= i + Lk - Lq.  Modes 1, 2 and 3 ignore
 *   pre_tokens / next_tokens (constraint section).  The outer-split starts of the options structs
 *   move the chosen window onto global positions.
 *   Grouped heads: query head n uses key/value head n / (head_num/head_num_kv)
 *   (constraint section: Nq/Nkv must be an integer).
 *
 * Ownership.  The caller owns every buffer, including the workspace, which
 * is sized by the *_workspace_size call first (the page's two-phase
 * GetWorkspaceSize / execute interface).  The library keeps no state
 * between calls except per-device kernel attributes.
 *
 * Asynchrony.  Compute calls only enqueue work on `stream` and return; the
 * only host-visible effects before the stream completes are argument
 * checks.  Schedules derived from the host length arrays are copied into
 * the workspace with one cudaMemcpyAsync per call.
 *
 * Errors (the page's return-code table: ACLNN_ERR_PARAM_NULLPTR for a null
 * required pointer, ACLNN_ERR_PARAM_INVALID for out-of-range arguments):
 *   FA_ERR_NULLPTR     a required pointer is NULL
 *   FA_ERR_INVALID     layout != "TND", head_num not in [1, 256], head_dim
 *                      not in [1, 768], keep_prob not in (0, 1], batch not
 *                      in [1, 2048], a negative length, lengths not summing
 *                      to total_q / total_kv, total_q > 1M, head_num not a
 *                      multiple of head_num_kv, unknown dtype, non-finite
 *                      scale, drop_mask_bytes too small
 *   FA_ERR_UNSUPPORTED a valid request this library does not implement:
 *                      head_dim not in {32, 64, 96, 128, 192} (the
 *                      tensor-core backward takes 64 and 128 in 16-bit
 *                      types; the rest run on the CUDA-core kernels),
 *                      sparse_mode 6, 7, 8
 *                      (sparse_mode 5 or outside 0..8: FA_ERR_INVALID)
 *   FA_ERR_WORKSPACE   workspace_bytes below the size the size call gave
 *   FA_ERR_CUDA        a CUDA launch or copy failed
 *   FA_ERR_TIMEOUT     (fa_varlen_read_error only) a kernel's bounded wait
 *                      expired; its outputs are invalid
 * Empty input: total_q == total_kv == 0 returns FA_OK without launching
 * anything; with total_q == 0 alone the backward writes zero dk / dv.
 */
#ifndef FA_VARLEN_H
#define FA_VARLEN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_NULLPTR = 1,
  FA_ERR_INVALID = 2,
  FA_ERR_UNSUPPORTED = 3,
  FA_ERR_WORKSPACE = 4,
  FA_ERR_CUDA = 5,
  FA_ERR_TIMEOUT = 6
} fa_status;

/* Storage type of q, k, v, dy, y, dq, dk, dv (parameter table: FLOAT16,
 * BFLOAT16, FLOAT32; all of them share one type). */
typedef enum { FA_DTYPE_FP32 = 0, FA_DTYPE_FP16 = 1, FA_DTYPE_BF16 = 2 } fa_dtype;

/* Backward kernel choice (fa_varlen_bwd_ex).  AUTO picks the tcgen05
 * tensor-core kernel for 16-bit types at head dims 32, 64, 96 and 128 (32
 * and 96 run zero-padded to 64 and 128) and the CUDA-core kernel otherwise
 * (FLOAT32, head dim 192); SIMT forces the CUDA-core kernel for any type;
 * TCGEN05 on a case it does not cover is FA_ERR_UNSUPPORTED. */
typedef enum { FA_BWD_AUTO = 0, FA_BWD_SIMT = 1, FA_BWD_TCGEN05 = 2 } fa_bwd_impl;

typedef struct {
  int32_t impl;            /* fa_bwd_impl */
  /* Nonzero: bitwise-reproducible dq.  Each CTA takes its work item from a
   * ticket counter in the workspace header, the items of one (sequence,
   * head) unit run in descending key-tile order, and the dq partial of every
   * (query head, 64-row query tile) is added in descending key-tile order,
   * each adder waiting (bounded by wait_timeout_ns) on a per-tile counter
   * for the one before it.  A CTA waits only on items taken before its own,
   * so the waits always end.  dk and dv are deterministic in either mode.
   * This follows the page's remark that the default (atomic) dq summation is
   * non-deterministic (constraints section).  On the tensor-core kernel the
   * ordered adds cost about 1.5x the default main-kernel time. */
  int32_t deterministic;
  int64_t wait_timeout_ns; /* bound on every in-kernel wait; <= 0: 2 s */
  /* Optional cudaEvent_t[4] (caller-created, may be NULL): recorded on
   * `stream` before the preprocess kernel, before the main kernel, after the
   * main kernel and after the dQ convert kernel, for per-kernel timing. */
  void *const *events;
  /* Outer split (the parameter table's qStartIdxOptional / kvStartIdxOptional):
   * host arrays of `batch` global start indices (>= 0) of each sequence's
   * query / key-value chunk, or NULL for 0.  The window is then evaluated on
   * global positions: key j of the chunk is allowed for query i iff
   * (qs + i) - pre_tokens <= ks + j <= (qs + i) + next_tokens.  Dropout bits
   * stay indexed by the chunk-local (i, j).  A negative start is
   * FA_ERR_INVALID.  The forward must be given the same starts. */
  const int64_t *q_start_idx;
  const int64_t *kv_start_idx;
  /* Explicit attention mask (parameter table row attenMaskOptional; 1 = the
   * position is excluded, 0 = it takes part): DEVICE uint8 matrix of
   * atten_mask_rows x atten_mask_cols, row-major, shared by every sequence
   * and head and indexed by each sequence's chunk-local (i, j).  Read in
   * sparse_mode 1 (alone) and 0 / 4 (together with the window); modes 2 and
   * 3 ignore it.  The compute calls with sparse_mode 1 require it
   * (FA_ERR_NULLPTR otherwise), the size calls do not; a mask with
   * rows < max Lq or cols < max Lk is FA_ERR_INVALID.  The forward must be
   * given the same mask. */
  const uint8_t *atten_mask;
  int64_t atten_mask_rows;
  int64_t atten_mask_cols;
} fa_bwd_options;

/* Options of fa_varlen_fwd_ex (fields as in fa_bwd_options; NULL / 0 for
 * none). */
typedef struct {
  const int64_t *q_start_idx;
  const int64_t *kv_start_idx;
  const uint8_t *atten_mask;
  int64_t atten_mask_rows;
  int64_t atten_mask_cols;
} fa_fwd_options;

/* Forward workspace size in bytes (same scalar arguments as fa_varlen_fwd). */
fa_status fa_varlen_fwd_workspace_size(
    const int64_t *seq_lens_q, const int64_t *seq_lens_kv, int64_t batch,
    int64_t total_q, int64_t total_kv, int64_t head_num, int64_t head_num_kv,
    int64_t head_dim, fa_dtype dtype, const char *layout, double keep_prob,
    int64_t pre_tokens, int64_t next_tokens, int64_t sparse_mode,
    size_t *workspace_bytes);

/* Forward: y (attentionIn of the backward) and the [T, N, 8] statistics. */
fa_status fa_varlen_fwd(
    const void *q, const void *k, const void *v,
    const uint8_t *drop_mask, int64_t drop_mask_bytes,
    const int64_t *seq_lens_q, const int64_t *seq_lens_kv, int64_t batch,
    int64_t total_q, int64_t total_kv, int64_t head_num, int64_t head_num_kv,
    int64_t head_dim, fa_dtype dtype, const char *layout, double scale,
    double keep_prob, int64_t pre_tokens, int64_t next_tokens,
    int64_t sparse_mode,
    void *y, float *softmax_max, float *softmax_sum,
    void *workspace, size_t workspace_bytes, fa_stream_t stream);

/* fa_varlen_fwd with options (NULL = defaults); same workspace size. */
fa_status fa_varlen_fwd_ex(
    const void *q, const void *k, const void *v,
    const uint8_t *drop_mask, int64_t drop_mask_bytes,
    const int64_t *seq_lens_q, const int64_t *seq_lens_kv, int64_t batch,
    int64_t total_q, int64_t total_kv, int64_t head_num, int64_t head_num_kv,
    int64_t head_dim, fa_dtype dtype, const char *layout, double scale,
    double keep_prob, int64_t pre_tokens, int64_t next_tokens,
    int64_t sparse_mode,
    void *y, float *softmax_max, float *softmax_sum,
    void *workspace, size_t workspace_bytes, fa_stream_t stream,
    const fa_fwd_options *options);

/* Backward workspace size in bytes.  Depends on the lengths, head counts,
 * head_dim and the kernel AUTO would choose for `dtype`. */
fa_status fa_varlen_bwd_workspace_size(
    const int64_t *seq_lens_q, const int64_t *seq_lens_kv, int64_t batch,
    int64_t total_q, int64_t total_kv, int64_t head_num, int64_t head_num_kv,
    int64_t head_dim, fa_dtype dtype, const char *layout, double keep_prob,
    int64_t pre_tokens, int64_t next_tokens, int64_t sparse_mode,
    size_t *workspace_bytes);

/* Backward: dq, dk, dv from q, k, v, dy, y (attentionIn) and the forward
 * statistics.  dq, dk, dv are fully overwritten (rows of keys that no query
 * attends to get zeros).  Non-deterministic: dq is summed with fp32 atomics
 * (the constraint section: non-deterministic by default); the options'
 * deterministic flag of fa_varlen_bwd_ex makes it reproducible. */
fa_status fa_varlen_bwd(
    const void *q, const void *k, const void *v, const void *dy,
    const uint8_t *drop_mask, int64_t drop_mask_bytes,
    const float *softmax_max, const float *softmax_sum, const void *y,
    const int64_t *seq_lens_q, const int64_t *seq_lens_kv, int64_t batch,
    int64_t total_q, int64_t total_kv, int64_t head_num, int64_t head_num_kv,
    int64_t head_dim, fa_dtype dtype, const char *layout, double scale,
    double keep_prob, int64_t pre_tokens, int64_t next_tokens,
    int64_t sparse_mode,
    void *dq, void *dk, void *dv,
    void *workspace, size_t workspace_bytes, fa_stream_t stream);

/* fa_varlen_bwd with options (NULL = defaults).  Its workspace is sized by
 * fa_varlen_bwd_workspace_size_ex with the same options. */
fa_status fa_varlen_bwd_workspace_size_ex(
    const int64_t *seq_lens_q, const int64_t *seq_lens_kv, int64_t batch,
    int64_t total_q, int64_t total_kv, int64_t head_num, int64_t head_num_kv,
    int64_t head_dim, fa_dtype dtype, const char *layout, double keep_prob,
    int64_t pre_tokens, int64_t next_tokens, int64_t sparse_mode,
    const fa_bwd_options *options, size_t *workspace_bytes);

fa_status fa_varlen_bwd_ex(
    const void *q, const void *k, const void *v, const void *dy,
    const uint8_t *drop_mask, int64_t drop_mask_bytes,
    const float *softmax_max, const float *softmax_sum, const void *y,
    const int64_t *seq_lens_q, const int64_t *seq_lens_kv, int64_t batch,
    int64_t total_q, int64_t total_kv, int64_t head_num, int64_t head_num_kv,
    int64_t head_dim, fa_dtype dtype, const char *layout, double scale,
    double keep_prob, int64_t pre_tokens, int64_t next_tokens,
    int64_t sparse_mode,
    void *dq, void *dk, void *dv,
    void *workspace, size_t workspace_bytes, fa_stream_t stream,
    const fa_bwd_options *options);

/* fa_varlen_bwd for callers that cannot allocate device memory (no
 * counterpart on the FAG-V2 page; an addition of this library).  Code that
 * runs inside a custom allocator or a memory-pool callback, or a runtime
 * that owns all device memory, may be unable to call cudaMalloc for a
 * workspace.  This entry point takes none: its scratch is a 64 MiB array
 * reserved by the library's CUDA module on every device that loads the
 * library, held until the process exits.  It allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine).
 *   - Arguments, layout and results are those of fa_varlen_bwd.
 *   - Problems whose workspace (fa_varlen_bwd_workspace_size) exceeds
 *     64 MiB are rejected with FA_ERR_WORKSPACE before any launch.  Example:
 *     the fp32 dQ accumulator alone takes total_q * head_num * head_dim * 4
 *     bytes.
 *   - The array exists once per CUDA context: in the device's primary
 *     context (the one the runtime and PyTorch use) and in any other
 *     context, made through the driver API, that calls this entry point.
 *   - The first call in a context looks up the array's device address
 *     there (cudaGetSymbolAddress, with that context current) and caches
 *     it under the context's unique id; make that first call before any
 *     stream capture in the context.  cudaDeviceReset destroys the primary
 *     context and the array with it; the next call, in the new primary
 *     context, looks the address up again.
 *   - Every call in a context shares the one array and leaves its contents
 *     behind; each call re-initialises what it needs.  Calls whose GPU work
 *     overlaps (other streams, other host threads) race on the array and
 *     give wrong results: serialise them.
 *   - A bounded in-kernel wait that expires leaves its code in the array's
 *     error word; fa_varlen_bwd_static_scratch_read_error reads it. */
fa_status fa_varlen_bwd_static_scratch(
    const void *q, const void *k, const void *v, const void *dy,
    const uint8_t *drop_mask, int64_t drop_mask_bytes,
    const float *softmax_max, const float *softmax_sum, const void *y,
    const int64_t *seq_lens_q, const int64_t *seq_lens_kv, int64_t batch,
    int64_t total_q, int64_t total_kv, int64_t head_num, int64_t head_num_kv,
    int64_t head_dim, fa_dtype dtype, const char *layout, double scale,
    double keep_prob, int64_t pre_tokens, int64_t next_tokens,
    int64_t sparse_mode,
    void *dq, void *dk, void *dv, fa_stream_t stream);

/* The error word of the last fa_varlen_bwd_static_scratch call in the
 * current context, read after synchronising `stream` (the stream that call
 * ran on): FA_OK, or FA_ERR_TIMEOUT when a bounded in-kernel wait expired
 * and that call's dq / dk / dv are invalid.  *code receives the raw word
 * (0 = no error).  It allocates nothing.  Errors: FA_ERR_NULLPTR (code),
 * FA_ERR_CUDA. */
fa_status fa_varlen_bwd_static_scratch_read_error(fa_stream_t stream, int32_t *code);

/* Reads the error word that the last call on `workspace` left in it, after
 * synchronising `stream`: FA_OK, or FA_ERR_TIMEOUT when a bounded in-kernel
 * wait expired.  *code receives the raw word (0 = no error). */
fa_status fa_varlen_read_error(const void *workspace, size_t workspace_bytes,
                               fa_stream_t stream, int32_t *code);

/* Self-test of the in-kernel failure detection, with no GPU fault involved.
 * Launches one small kernel whose threads wait, through the same bounded
 * wait the backward kernel uses, on an mbarrier phase that nothing ever
 * completes.  The wait gives up after wait_timeout_ns, records its timeout
 * code in the error word at the start of `workspace` (device memory, at
 * least 256 bytes; the word is cleared first) as a stalled backward would,
 * and the kernel returns normally, so the context stays usable.  Read the
 * outcome with fa_varlen_read_error, which then returns FA_ERR_TIMEOUT.
 * Errors: FA_ERR_NULLPTR (workspace), FA_ERR_WORKSPACE (< 256 bytes),
 * FA_ERR_INVALID (wait_timeout_ns outside [1000, 10^10]), FA_ERR_CUDA. */
fa_status fa_varlen_selftest_wait_timeout(void *workspace, size_t workspace_bytes,
                                          int64_t wait_timeout_ns, fa_stream_t stream);

/* Human-readable name of a status. */
const char *fa_status_string(fa_status status);

/* Synthetic-input utility (no part of the attention arithmetic): fills
 * mask[0, ceil(nbits/8)) with SplitMix64 keep bits, bit g = 1 iff
 * splitmix64(seed, g) < floor(keep_prob * 2^64), LSB first; bits past nbits
 * in the last byte are 0.  Asynchronous on `stream`. */
fa_status fa_gen_keep_mask(uint8_t *mask, int64_t nbits, uint64_t seed,
                           double keep_prob, fa_stream_t stream);

/* Host-only introspection of the backward tile scheduler (no GPU needed).
 * Writes the work list the backward would run, as 4 int32 per item:
 * {sequence, key/value head, key tile, lo | count << 16}, in unit order:
 * the items of each (sequence, head) unit together, longest first, units
 * ordered by their longest item.  The backward launches the same items in
 * this order, except that it sorts the last two waves (2 x SM count items)
 * longest first, or the whole list when Q, dY, K, V and the fp32 dQ
 * accumulator together fit in 85% of the device's L2; at head dims 64 and
 * below the tensor-core kernel also pairs adjacent kv heads.  An item means
 * key rows [tile*kv_tile, tile*kv_tile + kv_tile) of that sequence and head
 * visit query tiles of 64 rows [lo, lo + count) of every query head of the
 * group.  kv_tile is 64 (CUDA-core kernel) or 128 (tcgen05 kernel).
 * *n_items receives the item count; at most `capacity` items are written.
 * Errors: FA_ERR_NULLPTR, FA_ERR_INVALID (batch, lengths, head count,
 * kv_tile out of range). */
fa_status fa_varlen_bwd_schedule(const int64_t *seq_lens_q, const int64_t *seq_lens_kv,
                                 int64_t batch, int64_t head_num_kv, int64_t pre_tokens,
                                 int64_t next_tokens, int32_t kv_tile, int32_t *items,
                                 int64_t capacity, int64_t *n_items);

/* fa_varlen_bwd_schedule with the launch-time ordering made explicit, as
 * the backward applies it: head_num, head_dim and dtype size the working
 * set (Q, dY, K, V and the fp32 dQ accumulator); when it fits in 85% of
 * l2_bytes the whole list is sorted longest first, else the last
 * tail_items items are (the backward passes the device's L2 size and twice
 * its SM count; 0 turns either off).  head_pairs != 0 groups two adjacent
 * kv heads per item (WorkItem head field: first | (count - 1) << 16), as
 * the tensor-core kernel does at head_dim 64.  An item's "length" for the
 * sorts is its query-tile count times its head count.  Errors as for
 * fa_varlen_bwd_schedule, plus FA_ERR_INVALID for head_num, head_dim or
 * dtype out of range and negative l2_bytes / tail_items. */
fa_status fa_varlen_bwd_schedule_ex(const int64_t *seq_lens_q, const int64_t *seq_lens_kv,
                                    int64_t batch, int64_t head_num, int64_t head_num_kv,
                                    int64_t head_dim, fa_dtype dtype, int64_t pre_tokens,
                                    int64_t next_tokens, int32_t kv_tile, int64_t l2_bytes,
                                    int64_t tail_items, int32_t head_pairs, int32_t *items,
                                    int64_t capacity, int64_t *n_items);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t fa_varlen_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_VARLEN_H */
