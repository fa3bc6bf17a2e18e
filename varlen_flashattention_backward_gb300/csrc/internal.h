// Internal declarations shared by the host side (abi.cpp) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_varlen.h"

namespace fav {

constexpr int kQTile = 64;        // query rows per tile, every kernel
constexpr int kSimtKvTile = 64;   // key rows per work item, CUDA-core kernels
constexpr int kTcKvTile = 128;    // key rows per work item, tcgen05 kernel
constexpr int kMaxBatch = 2048;

// One per sequence, uploaded into the workspace (40 bytes).
struct SeqInfo {
  int32_t cu_q;      // first row of the sequence in q / dy / y / dq
  int32_t cu_k;      // first row in k / v / dk / dv
  int32_t len_q;
  int32_t len_k;
  int32_t qpad;      // first row in the 64-row-padded statistics index space
  // Window of this sequence on chunk-local indices: key j is allowed for
  // query i iff i - pre <= j <= i + next.  preTokens / nextTokens shifted by
  // the chunk starts (pre - (qs - ks), next + (qs - ks)), clamped to +-2^28,
  // which keeps every sum with an index inside int32.
  int32_t pre;
  int64_t mask_off;  // dropout bit of (head 0, i 0, j 0): N * sum_{b'<b} Lq*Lk
  int32_t next;
  int32_t pad_;
};
static_assert(sizeof(SeqInfo) == 40, "SeqInfo layout");

// One unit of work.  Backward: key tile `tile` of sequence `seq` for key/value
// head `head`, covering query tiles [lo, lo + count) of every query head of
// the group.  Forward: query tile `tile` of query head `head`, covering key
// tiles [lo, lo + count).
struct WorkItem {
  int32_t seq;
  int32_t head;
  int32_t tile;
  int32_t range;     // lo | (count << 16)
};

__host__ __device__ inline int item_lo(const WorkItem &w) { return w.range & 0xFFFF; }
__host__ __device__ inline int item_count(const WorkItem &w) { return (w.range >> 16) & 0xFFFF; }

// Error word codes written by kernels into the workspace header.
enum : int32_t {
  kErrNone = 0,
  kErrTimeoutBase = 0x100,   // + role id of the wait that expired
  kRoleSimtDq = 8,           // the CUDA-core backward's ordered dQ wait
};

// Workspace header (kHeaderBytes): the error word at byte 0 and, in the
// deterministic mode, the work-item ticket counter at byte kTicketOffset.
constexpr size_t kTicketOffset = 64;

struct BwdParams {
  const void *q, *k, *v, *dy, *y;
  const float *smax, *ssum;
  const uint8_t *mask;
  int64_t mask_bytes;
  void *dq, *dk, *dv;
  const SeqInfo *seqs;
  const WorkItem *items;
  float *lse2;      // [N][Tp]  (max + ln sum) * log2(e) + lse2_shift; +inf for padding rows
  float *dsum;      // [N][Tp]  dsum_scale * sum_d dY * Y;  0 for padding rows
  float *dq_acc;    // [Tq][N][D] fp32 accumulator of dS K (unscaled)
  int32_t *err;
  // Deterministic mode: CTAs take items in ticket order (*ticket counts up
  // from 0) and add their dQ partials of (query head n, padded query tile g)
  // in descending key-tile order.  sem[n * (tp / 64) + g] (zeroed by the
  // preprocess) counts the partials already added; qfirst[g] is the first
  // key tile in that order (the highest that visits tile g).
  int deterministic;
  int32_t *ticket;
  int32_t *sem;
  const int32_t *qfirst;
  // Dropout with every 128-key tile of every keep-mask row starting on a
  // 16-byte boundary (all key lengths multiples of 128, mask 16-byte
  // aligned): the tensor-core kernel copies each stage's keep bits into
  // shared memory beside Q and dY.
  int drop_rows16;
  int n_items, batch, n, n_kv, d, tp, total_q, total_kv;
  int prefetch_ahead;   // tcgen05 kernel: item distance of the K/V L2 prefetch (the SM count)
  float scale, scale_log2, inv_keep;
  // Folded into lse2 and dsum by the preprocess: 0 and 1, except for the
  // tensor-core kernel with dropout, which takes log2(keep_prob) and
  // keep_prob (its exponentials then give P / keep_prob directly).
  float lse2_shift, dsum_scale;
  int use_dropout;
  long long timeout_ns;
  // Explicit attention mask (uint8 [am_rows][am_cols], 1 = excluded) at
  // each sequence's chunk-local (i, j), or null.
  const uint8_t *atten_mask;
  int64_t am_cols;
  int64_t am_rows;
  int am_tma;   // tcgen05 kernel: the mask tiles come in by TMA (set at launch)
};

struct FwdParams {
  const void *q, *k, *v;
  const uint8_t *mask;
  int64_t mask_bytes;
  void *y;
  float *smax, *ssum;
  const SeqInfo *seqs;
  const WorkItem *items;
  int n_items, batch, n, n_kv, d;
  float scale, inv_keep;
  int use_dropout;
  const uint8_t *atten_mask;   // as BwdParams::atten_mask
  int64_t am_cols;
};

// Kernel launchers (return the launch error).
cudaError_t launch_bwd_preprocess(const BwdParams &p, fa_dtype dt, cudaStream_t s);
cudaError_t launch_bwd_simt(const BwdParams &p, fa_dtype dt, cudaStream_t s);
cudaError_t launch_bwd_tcgen05(const BwdParams &p, fa_dtype dt, cudaStream_t s);
// Head dims below the tensor-core kernel's compute width (32, 96).
cudaError_t launch_bwd_tcgen05_pad(const BwdParams &p, fa_dtype dt, cudaStream_t s);
cudaError_t launch_dq_convert(const BwdParams &p, fa_dtype dt, cudaStream_t s);
cudaError_t launch_fwd_simt(const FwdParams &p, fa_dtype dt, cudaStream_t s);
cudaError_t launch_gen_keep_mask(uint8_t *mask, int64_t nbits, uint64_t seed,
                                 uint64_t threshold, int keep_all, cudaStream_t s);
bool tcgen05_supported(fa_dtype dt, int head_dim);
cudaError_t launch_wait_timeout_selftest(int32_t *err, long long timeout_ns, cudaStream_t s);

}  // namespace fav
