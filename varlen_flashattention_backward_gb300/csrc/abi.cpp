// Host side of the C ABI: argument checks, the tile scheduler, the workspace
// layout and the kernel launch sequence.
//
// The argument rules follow the FAG-V2 page (aclnnFlashAttentionUnpaddingScoreGradV2):
// its return-code table (null required pointer -> ACLNN_ERR_PARAM_NULLPTR;
// out-of-range type/format -> ACLNN_ERR_PARAM_INVALID), its constraint
// section (TND only; T in [1, 1M]; N in [1, 256]; D in [1, 768]; keepProb in
// (0, 1]; Nq/Nkv integer; at most 2K sequences; zero-length sequences
// allowed) and its two-phase GetWorkspaceSize / execute interface.

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "internal.h"

namespace fav {
namespace {

constexpr size_t kAlign = 256;
constexpr size_t kHeaderBytes = 256;
constexpr int64_t kMaxTotal = int64_t(1) << 20;   // T: 1 ~ 1M
constexpr long long kDefaultTimeoutNs = 2000000000LL;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
// Window bounds beyond +-2^28 act like unbounded ones (lengths are below
// 2^20), and keep index arithmetic inside int32 on the device.
int64_t clamp_window(int64_t x) {
  const int64_t lim = int64_t(1) << 28;
  return std::max(-lim, std::min(lim, x));
}

struct Problem {
  const int64_t *lens_q, *lens_kv;
  int64_t batch, total_q, total_kv, n, n_kv, d;
  fa_dtype dtype;
  double keep_prob;
  int64_t pre, next, sparse_mode;
  int64_t tp;         // padded statistics rows
  int64_t mask_bits;
  // Outer split: per-sequence global start of the query / key-value chunk
  // (host arrays of length batch), or null for 0.
  const int64_t *q_start = nullptr, *kv_start = nullptr;
  // Explicit attention mask (device, rows x cols), or null.
  const uint8_t *atten_mask = nullptr;
  int64_t am_rows = 0, am_cols = 0;

  // Window of sequence b on chunk-local indices (see SeqInfo::pre).  The
  // sparse mode picks the window on global positions (modes 0 and 4: the
  // preTokens / nextTokens band; 2: lower triangle aligned at the top-left
  // corner; 3: lower triangle aligned at the bottom-right corner, j <= i +
  // Lk - Lq; modes 1-3 ignore preTokens / nextTokens), then the chunk starts
  // shift it onto chunk-local indices.
  int64_t shift(int64_t b) const {
    return (q_start ? q_start[b] : 0) - (kv_start ? kv_start[b] : 0);
  }
  int64_t mode_pre(int64_t) const {
    return (sparse_mode >= 1 && sparse_mode <= 3) ? (int64_t(1) << 28) : clamp_window(pre);
  }
  int64_t mode_next(int64_t b) const {
    if (sparse_mode == 1) return int64_t(1) << 28;
    if (sparse_mode == 2) return 0;
    if (sparse_mode == 3) return lens_kv[b] - lens_q[b];
    return clamp_window(next);
  }
  // The mask the kernels read: modes 0, 1 and 4 only.
  const uint8_t *mask_used() const {
    return (sparse_mode == 0 || sparse_mode == 1 || sparse_mode == 4) ? atten_mask : nullptr;
  }
  int64_t pre_of(int64_t b) const { return clamp_window(mode_pre(b) - shift(b)); }
  int64_t next_of(int64_t b) const { return clamp_window(mode_next(b) + shift(b)); }
};

// Checks shared by every entry point.  `need_ptrs` lists pointers that must
// be non-null.
fa_status check_problem(Problem &pr, const char *layout,
                        std::initializer_list<const void *> need_ptrs) {
  for (const void *ptr : need_ptrs)
    if (ptr == nullptr) return FA_ERR_NULLPTR;
  if (pr.lens_q == nullptr || pr.lens_kv == nullptr || layout == nullptr) return FA_ERR_NULLPTR;
  if (std::strcmp(layout, "TND") != 0) return FA_ERR_INVALID;
  if (pr.dtype != FA_DTYPE_FP32 && pr.dtype != FA_DTYPE_FP16 && pr.dtype != FA_DTYPE_BF16)
    return FA_ERR_INVALID;
  if (pr.n < 1 || pr.n > 256) return FA_ERR_INVALID;
  if (pr.n_kv < 1 || pr.n_kv > pr.n || pr.n % pr.n_kv != 0) return FA_ERR_INVALID;
  if (pr.d < 1 || pr.d > 768) return FA_ERR_INVALID;
  if (!(pr.keep_prob > 0.0 && pr.keep_prob <= 1.0)) return FA_ERR_INVALID;
  if (pr.batch < 1 || pr.batch > kMaxBatch) return FA_ERR_INVALID;
  if (pr.total_q < 0 || pr.total_q > kMaxTotal || pr.total_kv < 0 || pr.total_kv > kMaxTotal)
    return FA_ERR_INVALID;
  int64_t sq = 0, sk = 0, tp = 0, bits = 0;
  for (int64_t b = 0; b < pr.batch; ++b) {
    const int64_t lq = pr.lens_q[b], lk = pr.lens_kv[b];
    if (lq < 0 || lk < 0) return FA_ERR_INVALID;
    sq += lq;
    sk += lk;
    tp += ceil_div(lq, kQTile) * kQTile;
    bits += pr.n * lq * lk;
  }
  if (sq != pr.total_q || sk != pr.total_kv) return FA_ERR_INVALID;
  for (int64_t b = 0; b < pr.batch; ++b)
    if ((pr.q_start && pr.q_start[b] < 0) || (pr.kv_start && pr.kv_start[b] < 0))
      return FA_ERR_INVALID;
  // sparseMode: 0..8, 5 not supported (parameter table); this library
  // implements modes 0-4 (the window modes and the explicit mask).
  if (pr.sparse_mode < 0 || pr.sparse_mode > 8 || pr.sparse_mode == 5) return FA_ERR_INVALID;
  if (pr.sparse_mode > 4) return FA_ERR_UNSUPPORTED;
  if (pr.atten_mask != nullptr) {
    int64_t mq = 0, mk = 0;
    for (int64_t b = 0; b < pr.batch; ++b) {
      mq = std::max(mq, pr.lens_q[b]);
      mk = std::max(mk, pr.lens_kv[b]);
    }
    if (pr.am_rows < mq || pr.am_cols < mk || pr.am_cols < 1) return FA_ERR_INVALID;
  }
  // Head dims with kernels: the CUDA-core kernels take every one of this
  // list; the tensor-core backward takes 64 and 128.
  if (pr.d != 32 && pr.d != 64 && pr.d != 96 && pr.d != 128 && pr.d != 192)
    return FA_ERR_UNSUPPORTED;
  pr.tp = tp;
  pr.mask_bits = bits;
  return FA_OK;
}

std::vector<SeqInfo> build_seqs(const Problem &pr) {
  std::vector<SeqInfo> s(size_t(pr.batch));
  int64_t cq = 0, ck = 0, qp = 0, mo = 0;
  for (int64_t b = 0; b < pr.batch; ++b) {
    const int64_t lq = pr.lens_q[b], lk = pr.lens_kv[b];
    s[b].cu_q = int32_t(cq);
    s[b].cu_k = int32_t(ck);
    s[b].len_q = int32_t(lq);
    s[b].len_k = int32_t(lk);
    s[b].qpad = int32_t(qp);
    s[b].pre = int32_t(pr.pre_of(b));
    s[b].next = int32_t(pr.next_of(b));
    s[b].pad_ = 0;
    s[b].mask_off = mo;
    cq += lq;
    ck += lk;
    qp += ceil_div(lq, kQTile) * kQTile;
    mo += pr.n * lq * lk;
  }
  return s;
}

// Backward work list: one item per (sequence, key/value head, key tile).  A
// key tile [k0, k1) sees queries i with k0 - next <= i <= k1 - 1 + pre; only
// the query tiles meeting that range are visited, so fully masked causal or
// band tiles cost nothing.
//
// Order: the items of one (sequence, head) unit are contiguous, longest
// first, and units are ordered by their longest item, longest first.  The
// hardware dispatches CTAs in this order as SMs free up (greedy list
// scheduling), so the tail of the grid holds short items, while the units
// in flight at any moment stay few: their Q, dY and dQ accumulator rows
// (about 1 MB each per 2048 tokens) stay resident in L2 across the key
// tiles that re-read them.
//
// In the deterministic mode the items of a unit stay in ascending key-tile
// order instead, so that a CTA only ever waits for items taken before its own
// (see BwdParams::deterministic).
// Backward work list.  Items of one (sequence, kv head) unit read the same
// Q and dY tiles, so by default a unit's items are kept together (longest
// first) and units are ordered by their longest item: the Q/dY of the units
// in flight then stay in L2.  When the whole working set (Q, dY, K, V and
// the fp32 dQ accumulator) fits in `l2_bytes` there is no locality to keep,
// and the list is ordered longest item first across units, which balances
// the SMs better (measured: -7% on 4 sequences of 512-2048 tokens x 16
// heads; unit order kept workloads of 0.4-1.1 GB 2-50% faster).
// In unit order the last `tail_items` items (two waves of CTAs) are still
// sorted longest first, so that no long item starts last (-5% on 8 x 2048
// tokens x 16 heads).  `tile_order` keeps each unit's items in descending
// key-tile order (the deterministic mode).  With `head_pairs` a unit is two
// adjacent kv heads (the last may hold one): WorkItem::head is then
// first | (count - 1) << 16.
std::vector<WorkItem> build_bwd_items(const Problem &pr, int kv_tile, bool tile_order,
                                      size_t l2_bytes = 0, bool head_pairs = false,
                                      size_t tail_items = 0) {
  struct Unit {
    size_t first, count;
    int max_len;
  };
  std::vector<WorkItem> items;
  std::vector<Unit> units;
  for (int64_t b = 0; b < pr.batch; ++b) {
    const int64_t lq = pr.lens_q[b], lk = pr.lens_kv[b];
    const int64_t tiles = ceil_div(lk, kv_tile);
    const int64_t hstep = head_pairs ? 2 : 1;
    for (int64_t h = 0; h < pr.n_kv; h += hstep) {
      const int32_t head = int32_t(h) | int32_t(std::min(hstep, pr.n_kv - h) - 1) << 16;
      Unit u{items.size(), size_t(tiles), 0};
      for (int64_t t = 0; t < tiles; ++t) {
        const int64_t k0 = t * kv_tile, k1 = std::min(lk, k0 + kv_tile);
        const int64_t lo = std::max<int64_t>(0, k0 - pr.next_of(b));
        const int64_t hi = std::min<int64_t>(lq - 1, k1 - 1 + pr.pre_of(b));
        int64_t qlo = 0, cnt = 0;
        if (lq > 0 && lo <= hi) {
          qlo = lo / kQTile;
          cnt = hi / kQTile - qlo + 1;
        }
        items.push_back({int32_t(b), head, int32_t(t), int32_t(qlo | (cnt << 16))});
        u.max_len = std::max(u.max_len, int(cnt) * int(1 + (head >> 16)));
      }
      if (!tile_order)
        std::stable_sort(items.begin() + u.first, items.end(),
                         [](const WorkItem &a, const WorkItem &c) {
                           return item_count(a) > item_count(c);
                         });
      else   // deterministic mode: descending key tiles (see build_qtables)
        std::reverse(items.begin() + u.first, items.end());
      if (tiles > 0) units.push_back(u);
    }
  }
  std::stable_sort(units.begin(), units.end(),
                   [](const Unit &a, const Unit &c) { return a.max_len > c.max_len; });
  std::vector<WorkItem> out;
  out.reserve(items.size());
  for (const Unit &u : units)
    out.insert(out.end(), items.begin() + u.first, items.begin() + u.first + u.count);
  const double elem = pr.dtype == FA_DTYPE_FP32 ? 4.0 : 2.0;
  const double working = double(pr.total_q) * pr.n * pr.d * (2.0 * elem + 4.0) +
                         double(pr.total_kv) * pr.n_kv * pr.d * 2.0 * elem;
  const auto longer = [](const WorkItem &a, const WorkItem &c) {
    return item_count(a) * (1 + (a.head >> 16)) > item_count(c) * (1 + (c.head >> 16));
  };
  if (!tile_order && l2_bytes > 0 && working <= 0.85 * double(l2_bytes))
    std::stable_sort(out.begin(), out.end(), longer);
  else if (!tile_order && tail_items > 0 && out.size() > tail_items)
    std::stable_sort(out.end() - std::ptrdiff_t(tail_items), out.end(), longer);
  return out;
}

// An attribute of the current device, or 0 when it cannot be read.
size_t device_attr(cudaDeviceAttr attr) {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return size_t(v > 0 ? v : 0);
}

// Forward work list: one item per (sequence, query head, query tile) with the
// key tiles its window meets.
std::vector<WorkItem> build_fwd_items(const Problem &pr) {
  std::vector<WorkItem> items;
  for (int64_t b = 0; b < pr.batch; ++b) {
    const int64_t lq = pr.lens_q[b], lk = pr.lens_kv[b];
    const int64_t tiles = ceil_div(lq, kQTile);
    for (int64_t t = 0; t < tiles; ++t) {
      const int64_t q0 = t * kQTile, q1 = std::min(lq, q0 + kQTile);
      const int64_t lo = std::max<int64_t>(0, q0 - pr.pre_of(b));
      const int64_t hi = std::min<int64_t>(lk - 1, q1 - 1 + pr.next_of(b));
      int64_t klo = 0, cnt = 0;
      if (lk > 0 && lo <= hi) {
        klo = lo / kSimtKvTile;
        cnt = hi / kSimtKvTile - klo + 1;
      }
      for (int64_t h = 0; h < pr.n; ++h)
        items.push_back({int32_t(b), int32_t(h), int32_t(t), int32_t(klo | (cnt << 16))});
    }
  }
  std::stable_sort(items.begin(), items.end(), [](const WorkItem &a, const WorkItem &c) {
    return item_count(a) > item_count(c);
  });
  return items;
}

int64_t count_items(const Problem &pr, int tile, bool fwd) {
  int64_t c = 0;
  for (int64_t b = 0; b < pr.batch; ++b)
    c += fwd ? ceil_div(pr.lens_q[b], tile) * pr.n : ceil_div(pr.lens_kv[b], tile) * pr.n_kv;
  return c;
}

// Per padded query tile: the first key tile visiting it (the deterministic
// mode's order base) and the number of key tiles visiting it, stored as
// [qfirst | qcount].  The key tiles that visit
// one query tile form a contiguous range for every window, because both ends
// of a key tile's query range grow with the tile index; `contiguous` reports
// that property, which the deterministic mode relies on.
void build_qtables(const Problem &pr, const std::vector<SeqInfo> &seqs,
                   const std::vector<WorkItem> &items, std::vector<int32_t> &tab,
                   bool *contiguous) {
  const size_t g_tiles = size_t(pr.tp / kQTile);
  std::vector<int32_t> lo(g_tiles, INT32_MAX), hi(g_tiles, -1), cnt(g_tiles, 0);
  for (const WorkItem &w : items) {
    if ((w.head & 0xFFFF) != 0) continue;   // the items of (the pair starting at) kv head 0
    const size_t g0 = size_t(seqs[size_t(w.seq)].qpad / kQTile) + size_t(item_lo(w));
    for (int t = 0; t < item_count(w); ++t) {
      lo[g0 + t] = std::min(lo[g0 + t], w.tile);
      hi[g0 + t] = std::max(hi[g0 + t], w.tile);
      ++cnt[g0 + t];
    }
  }
  // The first half holds, per query tile, the highest key tile that visits
  // it: partials are added in descending key-tile order.  Each key tile
  // walks its query tiles upward from its diagonal, so under a causal or
  // banded window the next higher key tile reaches every query tile one
  // or two tiles earlier, and the adds seldom wait (ascending order made
  // every key tile wait for all lower ones at each query tile).
  tab.assign(2 * g_tiles, 0);
  *contiguous = true;
  for (size_t g = 0; g < g_tiles; ++g) {
    tab[g_tiles + g] = cnt[g];
    if (cnt[g] == 0) continue;
    if (hi[g] - lo[g] + 1 != cnt[g]) *contiguous = false;
    tab[g] = hi[g];
  }
}

struct BwdLayout {
  size_t seqs, items, qfirst, lse, dsum, sem, dqacc, total;
};

int choose_bwd_impl(const Problem &pr, const fa_bwd_options *opt) {
  int impl = opt ? opt->impl : FA_BWD_AUTO;
  if (impl == FA_BWD_AUTO)
    impl = tcgen05_supported(pr.dtype, int(pr.d)) ? FA_BWD_TCGEN05 : FA_BWD_SIMT;
  return impl;
}

BwdLayout bwd_layout(const Problem &pr, int impl) {
  // The item area is sized for the finer 64-key tiling so that a workspace
  // sized for one kernel also fits the other (see choose_bwd_impl's fallback).
  (void)impl;
  const int tile = kSimtKvTile;
  BwdLayout L;
  size_t off = kHeaderBytes;
  L.seqs = off;
  off = align_up(off + sizeof(SeqInfo) * size_t(pr.batch));
  L.items = off;
  off = align_up(off + sizeof(WorkItem) * size_t(count_items(pr, tile, false)));
  L.qfirst = off;   // [qfirst | qcount]
  off = align_up(off + 2 * sizeof(int32_t) * size_t(pr.tp / kQTile));
  L.lse = off;
  off = align_up(off + sizeof(float) * size_t(pr.n * pr.tp));
  L.dsum = off;
  off = align_up(off + sizeof(float) * size_t(pr.n * pr.tp));
  L.sem = off;
  off = align_up(off + sizeof(int32_t) * size_t(pr.n * (pr.tp / kQTile)));
  L.dqacc = off;
  off = align_up(off + sizeof(float) * size_t(pr.total_q * pr.n * pr.d));
  L.total = off;
  return L;
}

size_t fwd_layout_total(const Problem &pr, size_t *seqs_off, size_t *items_off) {
  size_t off = kHeaderBytes;
  *seqs_off = off;
  off = align_up(off + sizeof(SeqInfo) * size_t(pr.batch));
  *items_off = off;
  off = align_up(off + sizeof(WorkItem) * size_t(count_items(pr, kQTile, true)));
  return off;
}

// Copies from pageable memory of at most this size return without waiting
// for the stream; larger ones can make the host wait until the stream has
// drained, which would leave the GPU idle while the host builds the next
// call.  Larger plans therefore go up in pieces of this size.
constexpr size_t kPageableCopyPiece = size_t(64) << 10;

// Uploads [header | seqs | items | table]; the header's error word and
// ticket are 0.
// Copies host bytes to the device in pageable pieces of at most
// kPageableCopyPiece bytes.
fa_status copy_pieces(uint8_t *dst, const uint8_t *src, size_t bytes, cudaStream_t st) {
  for (size_t off = 0; off < bytes; off += kPageableCopyPiece) {
    const size_t n = std::min(kPageableCopyPiece, bytes - off);
    if (cudaMemcpyAsync(dst + off, src + off, n, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  return FA_OK;
}

// Uploads [header (zeroed) | sequences | work list] and, when given, the
// query-tile table at table_off (a separate copy: the work-list area is
// sized for the finer tiling and mostly unused by the coarser one).
fa_status upload_plan(void *ws, size_t seqs_off, size_t items_off,
                      const std::vector<SeqInfo> &seqs, const std::vector<WorkItem> &items,
                      cudaStream_t st, size_t table_off = 0,
                      const std::vector<int32_t> *table = nullptr) {
  const size_t bytes = items_off + sizeof(WorkItem) * items.size();
  std::vector<uint8_t> host(bytes, 0);
  std::memcpy(host.data() + seqs_off, seqs.data(), sizeof(SeqInfo) * seqs.size());
  if (!items.empty())
    std::memcpy(host.data() + items_off, items.data(), sizeof(WorkItem) * items.size());
  uint8_t *dst = static_cast<uint8_t *>(ws);
  fa_status r = copy_pieces(dst, host.data(), bytes, st);
  if (r != FA_OK || table == nullptr || table->empty()) return r;
  return copy_pieces(dst + table_off, reinterpret_cast<const uint8_t *>(table->data()),
                     sizeof(int32_t) * table->size(), st);
}

uint64_t keep_threshold(double keep_prob, int *keep_all) {
  *keep_all = keep_prob >= 1.0;
  if (*keep_all) return ~uint64_t(0);
  return uint64_t(keep_prob * 18446744073709551616.0);
}

}  // namespace
}  // namespace fav

using namespace fav;

extern "C" {

int32_t fa_varlen_version(void) { return 100; }

const char *fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_NULLPTR: return "FA_ERR_NULLPTR: a required pointer is null";
    case FA_ERR_INVALID: return "FA_ERR_INVALID: an argument is out of range";
    case FA_ERR_UNSUPPORTED:
      return "FA_ERR_UNSUPPORTED: valid request not implemented by this library";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace too small";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a bounded in-kernel wait expired";
  }
  return "unknown fa_status";
}

fa_status fa_varlen_fwd_workspace_size(const int64_t *seq_lens_q, const int64_t *seq_lens_kv,
                                       int64_t batch, int64_t total_q, int64_t total_kv,
                                       int64_t head_num, int64_t head_num_kv, int64_t head_dim,
                                       fa_dtype dtype, const char *layout, double keep_prob,
                                       int64_t pre_tokens, int64_t next_tokens,
                                       int64_t sparse_mode, size_t *workspace_bytes) {
  if (workspace_bytes == nullptr) return FA_ERR_NULLPTR;
  Problem pr{seq_lens_q, seq_lens_kv, batch, total_q, total_kv, head_num, head_num_kv,
             head_dim, dtype, keep_prob, pre_tokens, next_tokens, sparse_mode, 0, 0};
  fa_status st = check_problem(pr, layout, {});
  if (st != FA_OK) return st;
  size_t a, b;
  *workspace_bytes = fwd_layout_total(pr, &a, &b);
  return FA_OK;
}

fa_status fa_varlen_fwd_ex(const void *q, const void *k, const void *v,
                           const uint8_t *drop_mask, int64_t drop_mask_bytes,
                           const int64_t *seq_lens_q, const int64_t *seq_lens_kv,
                           int64_t batch, int64_t total_q, int64_t total_kv, int64_t head_num,
                           int64_t head_num_kv, int64_t head_dim, fa_dtype dtype,
                           const char *layout, double scale, double keep_prob,
                           int64_t pre_tokens, int64_t next_tokens, int64_t sparse_mode,
                           void *y, float *softmax_max, float *softmax_sum, void *workspace,
                           size_t workspace_bytes, fa_stream_t stream,
                           const fa_fwd_options *options) {
  Problem pr{seq_lens_q, seq_lens_kv, batch, total_q, total_kv, head_num, head_num_kv,
             head_dim, dtype, keep_prob, pre_tokens, next_tokens, sparse_mode, 0, 0};
  if (options) {
    pr.q_start = options->q_start_idx;
    pr.kv_start = options->kv_start_idx;
    pr.atten_mask = options->atten_mask;
    pr.am_rows = options->atten_mask_rows;
    pr.am_cols = options->atten_mask_cols;
  }
  // Pointers of an empty side (no query rows / no key rows) may be null.
  const bool hq = total_q > 0, hk = total_kv > 0;
  const void *ok = &pr;
  auto req = [ok](bool need, const void *ptr) { return need ? ptr : ok; };
  fa_status st = check_problem(pr, layout,
                               {req(hq, q), req(hk, k), req(hk, v), req(hq, y),
                                req(hq, softmax_max), req(hq, softmax_sum)});
  if (st != FA_OK) return st;
  if (pr.sparse_mode == 1 && pr.atten_mask == nullptr) return FA_ERR_NULLPTR;
  const bool dropout = keep_prob < 1.0;
  if (dropout && drop_mask == nullptr) return FA_ERR_NULLPTR;
  if (!std::isfinite(scale)) return FA_ERR_INVALID;
  if (dropout && drop_mask_bytes < (pr.mask_bits + 7) / 8) return FA_ERR_INVALID;
  if (total_q == 0) return FA_OK;
  size_t seqs_off, items_off;
  const size_t need = fwd_layout_total(pr, &seqs_off, &items_off);
  if (workspace == nullptr) return FA_ERR_NULLPTR;
  if (workspace_bytes < need) return FA_ERR_WORKSPACE;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  auto seqs = build_seqs(pr);
  auto items = build_fwd_items(pr);
  st = upload_plan(workspace, seqs_off, items_off, seqs, items, cs);
  if (st != FA_OK) return st;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  FwdParams p{};
  p.q = q; p.k = k; p.v = v;
  p.mask = drop_mask; p.mask_bytes = drop_mask_bytes;
  p.y = y; p.smax = softmax_max; p.ssum = softmax_sum;
  p.seqs = reinterpret_cast<const SeqInfo *>(ws + seqs_off);
  p.items = reinterpret_cast<const WorkItem *>(ws + items_off);
  p.n_items = int(items.size());
  p.batch = int(batch); p.n = int(head_num); p.n_kv = int(head_num_kv); p.d = int(head_dim);
  p.scale = float(scale);
  p.inv_keep = float(1.0 / keep_prob);
  p.use_dropout = dropout;
  p.atten_mask = pr.mask_used();
  p.am_cols = pr.am_cols;
  if (launch_fwd_simt(p, dtype, cs) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

fa_status fa_varlen_fwd(const void *q, const void *k, const void *v, const uint8_t *drop_mask,
                        int64_t drop_mask_bytes, const int64_t *seq_lens_q,
                        const int64_t *seq_lens_kv, int64_t batch, int64_t total_q,
                        int64_t total_kv, int64_t head_num, int64_t head_num_kv,
                        int64_t head_dim, fa_dtype dtype, const char *layout, double scale,
                        double keep_prob, int64_t pre_tokens, int64_t next_tokens,
                        int64_t sparse_mode, void *y, float *softmax_max, float *softmax_sum,
                        void *workspace, size_t workspace_bytes, fa_stream_t stream) {
  return fa_varlen_fwd_ex(q, k, v, drop_mask, drop_mask_bytes, seq_lens_q, seq_lens_kv, batch,
                          total_q, total_kv, head_num, head_num_kv, head_dim, dtype, layout,
                          scale, keep_prob, pre_tokens, next_tokens, sparse_mode, y,
                          softmax_max, softmax_sum, workspace, workspace_bytes, stream, nullptr);
}

fa_status fa_varlen_bwd_workspace_size_ex(const int64_t *seq_lens_q, const int64_t *seq_lens_kv,
                                          int64_t batch, int64_t total_q, int64_t total_kv,
                                          int64_t head_num, int64_t head_num_kv,
                                          int64_t head_dim, fa_dtype dtype, const char *layout,
                                          double keep_prob, int64_t pre_tokens,
                                          int64_t next_tokens, int64_t sparse_mode,
                                          const fa_bwd_options *options,
                                          size_t *workspace_bytes) {
  if (workspace_bytes == nullptr) return FA_ERR_NULLPTR;
  Problem pr{seq_lens_q, seq_lens_kv, batch, total_q, total_kv, head_num, head_num_kv,
             head_dim, dtype, keep_prob, pre_tokens, next_tokens, sparse_mode, 0, 0};
  if (options) {
    pr.q_start = options->q_start_idx;
    pr.kv_start = options->kv_start_idx;
    pr.atten_mask = options->atten_mask;
    pr.am_rows = options->atten_mask_rows;
    pr.am_cols = options->atten_mask_cols;
  }
  fa_status st = check_problem(pr, layout, {});
  if (st != FA_OK) return st;
  if (options && (options->impl < FA_BWD_AUTO || options->impl > FA_BWD_TCGEN05))
    return FA_ERR_INVALID;
  const int impl = choose_bwd_impl(pr, options);
  if (impl == FA_BWD_TCGEN05 && !tcgen05_supported(dtype, int(head_dim)))
    return FA_ERR_UNSUPPORTED;
  *workspace_bytes = bwd_layout(pr, impl).total;
  return FA_OK;
}

fa_status fa_varlen_bwd_workspace_size(const int64_t *seq_lens_q, const int64_t *seq_lens_kv,
                                       int64_t batch, int64_t total_q, int64_t total_kv,
                                       int64_t head_num, int64_t head_num_kv, int64_t head_dim,
                                       fa_dtype dtype, const char *layout, double keep_prob,
                                       int64_t pre_tokens, int64_t next_tokens,
                                       int64_t sparse_mode, size_t *workspace_bytes) {
  return fa_varlen_bwd_workspace_size_ex(seq_lens_q, seq_lens_kv, batch, total_q, total_kv,
                                         head_num, head_num_kv, head_dim, dtype, layout,
                                         keep_prob, pre_tokens, next_tokens, sparse_mode,
                                         nullptr, workspace_bytes);
}

fa_status fa_varlen_bwd_ex(const void *q, const void *k, const void *v, const void *dy,
                           const uint8_t *drop_mask, int64_t drop_mask_bytes,
                           const float *softmax_max, const float *softmax_sum, const void *y,
                           const int64_t *seq_lens_q, const int64_t *seq_lens_kv,
                           int64_t batch, int64_t total_q, int64_t total_kv, int64_t head_num,
                           int64_t head_num_kv, int64_t head_dim, fa_dtype dtype,
                           const char *layout, double scale, double keep_prob,
                           int64_t pre_tokens, int64_t next_tokens, int64_t sparse_mode,
                           void *dq, void *dk, void *dv, void *workspace,
                           size_t workspace_bytes, fa_stream_t stream,
                           const fa_bwd_options *options) {
  Problem pr{seq_lens_q, seq_lens_kv, batch, total_q, total_kv, head_num, head_num_kv,
             head_dim, dtype, keep_prob, pre_tokens, next_tokens, sparse_mode, 0, 0};
  if (options) {
    pr.q_start = options->q_start_idx;
    pr.kv_start = options->kv_start_idx;
    pr.atten_mask = options->atten_mask;
    pr.am_rows = options->atten_mask_rows;
    pr.am_cols = options->atten_mask_cols;
  }
  // Pointers of an empty side (no query rows / no key rows) may be null.
  const bool hq = total_q > 0, hk = total_kv > 0;
  const void *ok = &pr;
  auto req = [ok](bool need, const void *ptr) { return need ? ptr : ok; };
  fa_status st = check_problem(
      pr, layout,
      {req(hq, q), req(hk, k), req(hk, v), req(hq, dy), req(hq, softmax_max),
       req(hq, softmax_sum), req(hq, y), req(hq, dq), req(hk, dk), req(hk, dv)});
  if (st != FA_OK) return st;
  if (pr.sparse_mode == 1 && pr.atten_mask == nullptr) return FA_ERR_NULLPTR;
  const bool dropout = keep_prob < 1.0;
  if (dropout && drop_mask == nullptr) return FA_ERR_NULLPTR;
  if (!std::isfinite(scale)) return FA_ERR_INVALID;
  if (dropout && drop_mask_bytes < (pr.mask_bits + 7) / 8) return FA_ERR_INVALID;
  if (options && (options->impl < FA_BWD_AUTO || options->impl > FA_BWD_TCGEN05))
    return FA_ERR_INVALID;
  int impl = choose_bwd_impl(pr, options);
  if (impl == FA_BWD_TCGEN05 && !tcgen05_supported(dtype, int(head_dim)))
    return FA_ERR_UNSUPPORTED;
  if (total_q == 0 && total_kv == 0) return FA_OK;
  // The tensor-core kernel reads q, k, v, dy and writes dk, dv through TMA,
  // which needs 16-byte aligned bases; with no query rows there is nothing
  // for it to do.
  const auto al16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  const bool tma_ok =
      total_q > 0 && al16(q) && al16(k) && al16(v) && al16(dy) && al16(dk) && al16(dv);
  if (impl == FA_BWD_TCGEN05 && !tma_ok) {
    if (options && options->impl == FA_BWD_TCGEN05 && total_q > 0) return FA_ERR_UNSUPPORTED;
    impl = FA_BWD_SIMT;
  }
  const BwdLayout L = bwd_layout(pr, impl);
  if (workspace == nullptr) return FA_ERR_NULLPTR;
  if (workspace_bytes < L.total) return FA_ERR_WORKSPACE;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int tile = impl == FA_BWD_TCGEN05 ? kTcKvTile : kSimtKvTile;
  const bool det = options && options->deterministic != 0;
  auto seqs = build_seqs(pr);
  // The tensor-core kernel takes two kv heads per item at head dim 64 and below.
  const bool pairs = impl == FA_BWD_TCGEN05 && head_dim <= 64;
  auto items = build_bwd_items(pr, tile, det, device_attr(cudaDevAttrL2CacheSize), pairs,
                               2 * device_attr(cudaDevAttrMultiProcessorCount));
  // The deterministic mode's add order of each query tile.
  std::vector<int32_t> qtab;
  if (det) {
    bool contiguous = true;
    build_qtables(pr, seqs, items, qtab, &contiguous);
    if (!contiguous) return FA_ERR_UNSUPPORTED;
  }
  st = upload_plan(workspace, L.seqs, L.items, seqs, items, cs, L.qfirst, &qtab);
  if (st != FA_OK) return st;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  BwdParams p{};
  p.q = q; p.k = k; p.v = v; p.dy = dy; p.y = y;
  p.smax = softmax_max; p.ssum = softmax_sum;
  p.mask = drop_mask; p.mask_bytes = drop_mask_bytes;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.seqs = reinterpret_cast<const SeqInfo *>(ws + L.seqs);
  p.items = reinterpret_cast<const WorkItem *>(ws + L.items);
  p.lse2 = reinterpret_cast<float *>(ws + L.lse);
  p.dsum = reinterpret_cast<float *>(ws + L.dsum);
  p.dq_acc = reinterpret_cast<float *>(ws + L.dqacc);
  p.err = reinterpret_cast<int32_t *>(ws);
  p.deterministic = det ? 1 : 0;
  p.ticket = reinterpret_cast<int32_t *>(ws + kTicketOffset);
  p.sem = reinterpret_cast<int32_t *>(ws + L.sem);
  p.qfirst = reinterpret_cast<const int32_t *>(ws + L.qfirst);
  // Dropout keep bits by 16-byte copies: every key tile of every mask row
  // starts on a 16-byte boundary when all key lengths are multiples of 128
  // (then so are the per-sequence bit offsets) and the mask is aligned.
  p.drop_rows16 = dropout && (reinterpret_cast<uintptr_t>(drop_mask) & 15u) == 0;
  for (int64_t b = 0; b < batch && p.drop_rows16; ++b)
    if (seq_lens_kv[b] % kTcKvTile != 0) p.drop_rows16 = 0;
  p.n_items = int(items.size());
  p.batch = int(batch); p.n = int(head_num); p.n_kv = int(head_num_kv); p.d = int(head_dim);
  p.tp = int(pr.tp); p.total_q = int(total_q); p.total_kv = int(total_kv);
  p.scale = float(scale);
  p.scale_log2 = float(scale * 1.4426950408889634);
  p.inv_keep = float(1.0 / keep_prob);
  const bool fold = dropout && impl == FA_BWD_TCGEN05;
  p.lse2_shift = fold ? float(std::log2(keep_prob)) : 0.f;
  p.dsum_scale = fold ? float(keep_prob) : 1.f;
  p.use_dropout = dropout;
  p.timeout_ns = (options && options->wait_timeout_ns > 0) ? options->wait_timeout_ns
                                                           : kDefaultTimeoutNs;
  p.atten_mask = pr.mask_used();
  p.am_cols = pr.am_cols;
  p.am_rows = pr.am_rows;

  void *const *ev = options ? options->events : nullptr;
  auto mark = [&](int i) {
    return ev == nullptr || ev[i] == nullptr ||
           cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), cs) == cudaSuccess;
  };
  if (!mark(0)) return FA_ERR_CUDA;
  if (pr.tp > 0 && launch_bwd_preprocess(p, dtype, cs) != cudaSuccess) return FA_ERR_CUDA;
  if (!mark(1)) return FA_ERR_CUDA;
  if (!items.empty()) {
    cudaError_t e = impl == FA_BWD_TCGEN05 ? launch_bwd_tcgen05(p, dtype, cs)
                                           : launch_bwd_simt(p, dtype, cs);
    if (e != cudaSuccess) return FA_ERR_CUDA;
  }
  if (!mark(2)) return FA_ERR_CUDA;
  if (total_q > 0 && launch_dq_convert(p, dtype, cs) != cudaSuccess) return FA_ERR_CUDA;
  if (!mark(3)) return FA_ERR_CUDA;
  return FA_OK;
}

fa_status fa_varlen_bwd(const void *q, const void *k, const void *v, const void *dy,
                        const uint8_t *drop_mask, int64_t drop_mask_bytes,
                        const float *softmax_max, const float *softmax_sum, const void *y,
                        const int64_t *seq_lens_q, const int64_t *seq_lens_kv, int64_t batch,
                        int64_t total_q, int64_t total_kv, int64_t head_num,
                        int64_t head_num_kv, int64_t head_dim, fa_dtype dtype,
                        const char *layout, double scale, double keep_prob,
                        int64_t pre_tokens, int64_t next_tokens, int64_t sparse_mode, void *dq,
                        void *dk, void *dv, void *workspace, size_t workspace_bytes,
                        fa_stream_t stream) {
  return fa_varlen_bwd_ex(q, k, v, dy, drop_mask, drop_mask_bytes, softmax_max, softmax_sum,
                          y, seq_lens_q, seq_lens_kv, batch, total_q, total_kv, head_num,
                          head_num_kv, head_dim, dtype, layout, scale, keep_prob, pre_tokens,
                          next_tokens, sparse_mode, dq, dk, dv, workspace, workspace_bytes,
                          stream, nullptr);
}

fa_status fa_varlen_read_error(const void *workspace, size_t workspace_bytes, fa_stream_t stream,
                               int32_t *code) {
  if (workspace == nullptr || code == nullptr) return FA_ERR_NULLPTR;
  if (workspace_bytes < sizeof(int32_t)) return FA_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
    return FA_ERR_CUDA;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return FA_ERR_CUDA;
  *code = word;
  return word == 0 ? FA_OK : FA_ERR_TIMEOUT;
}

fa_status fa_varlen_bwd_schedule_ex(const int64_t *seq_lens_q, const int64_t *seq_lens_kv,
                                    int64_t batch, int64_t head_num, int64_t head_num_kv,
                                    int64_t head_dim, fa_dtype dtype, int64_t pre_tokens,
                                    int64_t next_tokens, int32_t kv_tile, int64_t l2_bytes,
                                    int64_t tail_items, int32_t head_pairs, int32_t *items,
                                    int64_t capacity, int64_t *n_items) {
  if (seq_lens_q == nullptr || seq_lens_kv == nullptr || n_items == nullptr) return FA_ERR_NULLPTR;
  if (capacity > 0 && items == nullptr) return FA_ERR_NULLPTR;
  if (batch < 1 || batch > kMaxBatch || head_num_kv < 1 || head_num_kv > 256 || head_num < 1 ||
      head_num > 256 || head_num % head_num_kv != 0 || head_dim < 1 || head_dim > 768 ||
      l2_bytes < 0 || tail_items < 0)
    return FA_ERR_INVALID;
  if (dtype != FA_DTYPE_FP32 && dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16)
    return FA_ERR_INVALID;
  if (kv_tile != kSimtKvTile && kv_tile != kTcKvTile) return FA_ERR_INVALID;
  int64_t tq = 0, tk = 0;
  for (int64_t b = 0; b < batch; ++b) {
    if (seq_lens_q[b] < 0 || seq_lens_kv[b] < 0 || seq_lens_q[b] > (int64_t(1) << 20) ||
        seq_lens_kv[b] > (int64_t(1) << 20))
      return FA_ERR_INVALID;
    tq += seq_lens_q[b];
    tk += seq_lens_kv[b];
  }
  Problem pr{seq_lens_q, seq_lens_kv, batch, tq, tk, head_num, head_num_kv, head_dim,
             dtype, 1.0, pre_tokens, next_tokens, 0, 0, 0};
  auto list = build_bwd_items(pr, kv_tile, false, size_t(l2_bytes), head_pairs != 0,
                              size_t(tail_items));
  *n_items = int64_t(list.size());
  const int64_t m = std::min<int64_t>(capacity, int64_t(list.size()));
  if (m > 0) std::memcpy(items, list.data(), size_t(m) * sizeof(WorkItem));
  return FA_OK;
}

fa_status fa_varlen_bwd_schedule(const int64_t *seq_lens_q, const int64_t *seq_lens_kv,
                                 int64_t batch, int64_t head_num_kv, int64_t pre_tokens,
                                 int64_t next_tokens, int32_t kv_tile, int32_t *items,
                                 int64_t capacity, int64_t *n_items) {
  return fa_varlen_bwd_schedule_ex(seq_lens_q, seq_lens_kv, batch, head_num_kv, head_num_kv, 128,
                                   FA_DTYPE_BF16, pre_tokens, next_tokens, kv_tile, 0, 0, 0,
                                   items, capacity, n_items);
}

fa_status fa_varlen_selftest_wait_timeout(void *workspace, size_t workspace_bytes,
                                          int64_t wait_timeout_ns, fa_stream_t stream) {
  if (workspace == nullptr) return FA_ERR_NULLPTR;
  if (workspace_bytes < kHeaderBytes) return FA_ERR_WORKSPACE;
  if (wait_timeout_ns < 1000 || wait_timeout_ns > 10000000000LL) return FA_ERR_INVALID;
  if (launch_wait_timeout_selftest(static_cast<int32_t *>(workspace), wait_timeout_ns,
                                   reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

fa_status fa_gen_keep_mask(uint8_t *mask, int64_t nbits, uint64_t seed, double keep_prob,
                           fa_stream_t stream) {
  if (mask == nullptr) return FA_ERR_NULLPTR;
  if (nbits < 0 || !(keep_prob > 0.0 && keep_prob <= 1.0)) return FA_ERR_INVALID;
  if (nbits == 0) return FA_OK;
  int keep_all = 0;
  const uint64_t thr = keep_threshold(keep_prob, &keep_all);
  if (launch_gen_keep_mask(mask, nbits, seed, thr, keep_all,
                           reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"
