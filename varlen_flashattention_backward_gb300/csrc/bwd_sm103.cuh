#pragma once

// Backward of varlen attention on the sm_103a tensor cores (tcgen05 + TMEM +
// TMA), bf16 or fp16 storage, at a compute width of 128 columns per head
// (64 with kD64 below); head dims 32 and 96 run zero-padded to 64 and 128
// (kPad).  The kernel template and its launcher; bwd_sm103.cu and
// bwd_sm103_pad.cu instantiate it.
//
// It computes the FAG-V2 page's backward (aclnnFlashAttentionUnpaddingScoreGradV2,
// section 功能说明 / 计算公式: dV = P^T dY, dQ = dS K / sqrt(d),
// dK = dS^T Q / sqrt(d), with scaleValue in place of 1/sqrt(d)), recomputing
// P from the saved softmax statistics.
//
// One CTA per work item: 128 keys of one (sequence, key/value head), looping
// over the 64-row query tiles the window reaches, for every query head of the
// group.  Per query tile the five contractions run on the tensor core with
// fp32 accumulators in TMEM (keys on the M side, so P^T and dS^T are already
// in the A-operand layout):
//
//   S^T  = K Q^T          M=128 keys, N=64 queries, K=128 (A, B in smem, K-major)
//   dP^T = V dY^T         same shape
//   dV  += P^T dY         M=128 keys, N=128 d, K=64 (A = P^T in TMEM, B = dY MN-major)
//   dK  += dS^T Q         same, A = dS^T in TMEM, B = Q
//   dQ^T = K^T dS^T       M=128 d, N=64 queries, K=128 keys (A = K MN-major, B = dS^T)
//
// dQ^T is drained from TMEM and added into the fp32 dq_acc with 16-byte
// reductions (four 128-byte row segments per warp instruction); dK and dV
// stay in TMEM for the whole item and are written once at the end.
//
// Warp roles (16 warps):
//   0      TMA producer: K, V once; Q, dY, lse, D per query tile (3 stages)
//   1      MMA issuer for S^T and dP^T (k-steps interleaved); owns the TMEM
//          allocation
//   2      MMA issuer for dV, then dK interleaved with dQ^T
//   3      deterministic mode: publishes each tile's dQ counter once the
//          drain's reductions are visible GPU-wide; idle otherwise
//   4-11   softmax: TMEM lane quarter = warp % 4 (one key per thread), column
//          half = (warp - 4) / 4 (32 of the 64 queries); P, dropout, dS; then
//          the dV (first half) / dK (second half) epilogue
//   12-15  dQ drain: TMEM lane = d
//
// Every mbarrier wait is bounded (BwdParams::timeout_ns); a wait that gives up
// records kErrTimeoutBase + role in the workspace error word, and the CTA
// winds down without further waits except bounded ones for its own copies
// and MMAs in flight, then frees TMEM.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "sm103.cuh"

namespace fav {
namespace {

using namespace sm103;

constexpr int BN = kTcKvTile;   // 128 keys per item
constexpr int BM = kQTile;      // 64 queries per iteration
constexpr int HD = 128;         // head dim
constexpr int STAGES = 3;
constexpr int NTHREADS = 512;

// TMEM columns (512 allocated; 128 lanes x 32-bit cells).
constexpr uint32_t COL_DV = 0;     // 128: dV accumulator, lane = key
constexpr uint32_t COL_DK = 128;   // 128: dK accumulator, lane = key
constexpr uint32_t COL_S = 256;    //  64: S^T (fp32)
constexpr uint32_t COL_DP = 320;   //  64: dP^T (fp32)
constexpr uint32_t COL_DQ = 384;   //  64: dQ^T (fp32), lane = d
constexpr uint32_t COL_P = 448;    //  32: P^T (bf16 pairs), MMA A operand
constexpr uint32_t COL_DS = 480;   //  32: dS^T (bf16 pairs), MMA A operand

// Shared memory (offsets from a 1024-byte aligned base).  Every tile is
// stored as 64-column boxes of 128-byte rows in the TMA 128-byte swizzle.
constexpr uint32_t SM_K = 0;                          // 2 boxes [128 x 64]
constexpr uint32_t SM_V = SM_K + 32768;
constexpr uint32_t SM_Q = SM_V + 32768;               // STAGES x 2 boxes [64 x 64]
constexpr uint32_t SM_DY = SM_Q + STAGES * 16384;
constexpr uint32_t SM_DS = SM_DY + STAGES * 16384;    // [128 keys x 64 queries]
constexpr uint32_t SM_LSE = SM_DS + 16384;            // STAGES x 64 floats
constexpr uint32_t SM_DSUM = SM_LSE + STAGES * 256;
constexpr uint32_t SM_BAR = SM_DSUM + STAGES * 256;
// The dropout instantiations keep each stage's keep bits after the
// barriers when they come in by 16-byte copies (BwdParams::drop_rows16):
// 64 query rows x 128 keys, one 16-byte chunk per row, LSB first.  Other
// instantiations have no such area.
constexpr uint32_t SM_DROP = SM_BAR + 256;
constexpr uint32_t DROP_STAGE = 64 * 16;
__host__ __device__ constexpr uint32_t sm_end(bool drop) { return SM_DROP + (drop ? STAGES * DROP_STAGE : 0u); }
__host__ __device__ constexpr uint32_t smem_bytes(bool drop) { return sm_end(drop) + 1024; }
static_assert(smem_bytes(true) <= 232448, "shared memory per CTA");
// With an explicit attention mask: STAGES x [64 queries x 128 keys] bytes of
// it, loaded by TMA beside each Q/dY stage (only that instantiation asks
// for the extra shared memory).
constexpr uint32_t AM_STAGE = 64 * 128;
__host__ __device__ constexpr uint32_t smem_bytes_mask(bool drop) { return sm_end(drop) + STAGES * AM_STAGE + 1024; }
static_assert(smem_bytes_mask(true) <= 232448, "shared memory per CTA");

// mbarrier slots
enum : int {
  B_KV = 0, B_FULL = 1, B_EMPTY = B_FULL + STAGES, B_SDFULL = B_EMPTY + STAGES, B_SDFREE,
  B_PFULL, B_PFREE, B_DSFULL, B_DSFREE, B_DQFULL, B_DQFREE, B_ACC, B_FINAL, B_FINAL_A,
  B_EPI, B_DQPUB = B_EPI + 2, B_PUBFREE, B_COUNT   // B_DQPUB, B_PUBFREE: deterministic mode
};
static_assert(B_COUNT * 8 <= 256, "barrier area");

enum : int {
  ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_SOFTMAX = 3, ROLE_DQ = 4, ROLE_EPILOGUE = 5,
  ROLE_SELFTEST = 7
};

struct TcMaps {
  CUtensorMap q, dy, k, v;
  CUtensorMap dk, dv;   // same shape as k / v, for the epilogue's bulk stores
  CUtensorMap am;       // the explicit mask, when it is loaded by TMA
};

// Bits [bit, bit + 32) of the keep mask, read without leaving
// [mask, mask + nbytes).
__device__ __forceinline__ uint32_t fetch_bits32(const uint8_t *mask, int64_t nbytes,
                                                 int64_t bit) {
  const uintptr_t base = reinterpret_cast<uintptr_t>(mask);
  const uintptr_t addr = base + uintptr_t(bit >> 3);
  const uintptr_t al = addr & ~uintptr_t(3);
  const int sh = int((addr - al) * 8 + uintptr_t(bit & 7));
  const uintptr_t end = base + uintptr_t(nbytes);
  uint32_t lo, hi;
  if (al >= base && al + 8 <= end) {
    lo = __ldg(reinterpret_cast<const uint32_t *>(al));
    hi = __ldg(reinterpret_cast<const uint32_t *>(al + 4));
  } else {
    uint64_t w = 0;
    for (int k = 0; k < 8; ++k) {
      const uintptr_t a = al + k;
      if (a >= base && a < end)
        w |= uint64_t(__ldg(reinterpret_cast<const uint8_t *>(a))) << (8 * k);
    }
    lo = uint32_t(w);
    hi = uint32_t(w >> 32);
  }
  return __funnelshift_r(lo, hi, sh);
}

// 32 x 32 bit-matrix transpose across the warp: on return, bit c of lane j's
// word is bit j of lane c's input word (recursive block swap).
__device__ __forceinline__ uint32_t transpose_bits32(uint32_t w, int lane) {
  const uint32_t masks[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int k = 0, s = 16; k < 5; ++k, s >>= 1) {
    const uint32_t o = __shfl_xor_sync(0xffffffffu, w, s);
    w = (lane & s) ? ((w & ~masks[k]) | ((o & ~masks[k]) >> s))
                   : ((w & masks[k]) | ((o & masks[k]) << s));
  }
  return w;
}

// Mask of a packed pair: each 16-bit half all ones where its keep bit is set.
// Bits c and 16 + c of the keep word (the pair's two queries) are read from
// ks[s] = keep << s (s = 0..7): pair c < 8 has them at bits 7 and 23 of
// ks[7 - c], pair c >= 8 at bits 15 and 31 of ks[15 - c]; prmt then fills
// each half with the sign of its byte.
__device__ __forceinline__ uint32_t pair_mask8(const uint32_t (&ks)[8], int c) {
  uint32_t m;
  if (c < 8)
    asm("prmt.b32 %0, %1, 0, 0xAA88;" : "=r"(m) : "r"(ks[7 - c]));
  else
    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(m) : "r"(ks[15 - c]));
  return m;
}

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return kBF16 ? pack_bf16(lo, hi) : pack_f16(lo, hi);
}

__device__ __forceinline__ void red_add_v4_f32(float *addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void st_global_v4(void *ptr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// 16-byte asynchronous copy global -> shared (L2 only) by this thread.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}

// Makes `bar` wait for this thread's cp.async copies issued so far: the
// barrier's pending count goes up by one now and down by one when they
// complete, so it must be called before the arrival that would complete the
// phase.
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Keep bits of one stage (BwdParams::drop_rows16): rows q0 .. q0 + rows - 1
// of query head n, keys k0 .. k0 + 127, one 16-byte chunk per row (its bit
// index mask_off + (n Lq + i) Lk + k0 is a multiple of 128), two rows per
// lane, copied with cp.async and tracked by the stage barrier `full`.  The
// whole producer warp calls it before the stage's arrive.expect_tx.
__device__ __forceinline__ void load_keep_bits(uint32_t dst, const uint8_t *mask,
                                               const SeqInfo &sq, int n, int q0, int k0,
                                               int rows, uint32_t full, int lane) {
  const int64_t bit0 = sq.mask_off + (int64_t(n) * sq.len_q + q0) * sq.len_k + k0;
  for (int r = lane; r < rows; r += 32)
    cp_async_16(dst + r * 16, mask + ((bit0 + int64_t(r) * sq.len_k) >> 3));
  cp_async_mbar_arrive(full);
  __syncwarp();
}

// Adds the dQ partial of one drain thread into dq_acc: its 16 four-column
// segments (query rows 4j + c of the tile, c = lane % 4), rows < `rows`.
__device__ __forceinline__ void dq_add(float *ptr, int64_t row_stride, const float (&out)[64],
                                       int c, int rows) {
#pragma unroll
  for (int j = 0; j < 16; ++j, ptr += 4 * row_stride)
    if (4 * j + c < rows)
      red_add_v4_f32(ptr, out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
}

// Named barrier 1 joins the four dQ drain warps (warps 12-15).
__device__ __forceinline__ void drain_bar_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}


struct Ctl {
  int *abort;         // shared-memory flag: some wait of this CTA gave up
  int32_t *err;       // global error word
  long long timeout;
};

__device__ __forceinline__ bool wait_or_abort(const Ctl &c, uint32_t bar, uint32_t parity,
                                              int role) {
  if (mbar_wait(bar, parity, c.timeout, c.abort)) return true;
  if (!*reinterpret_cast<volatile int *>(c.abort)) {
    atomicExch(c.abort, 1);
    atomicCAS(c.err, 0, kErrTimeoutBase + role);
  }
  return false;
}

// kDet: the deterministic mode (ticket-ordered items, ordered dQ adds).
// kMask: an explicit attention mask is read.  Each is a separate
// instantiation so that the default kernel carries none of its code (the
// mask's untaken branch alone cost 5-10% of the default kernel's time).
// kD64: head dim 64.  An item may cover two adjacent kv heads (the upper
// half of WorkItem::head holds the extra head count): their K and V fill the
// two 64-column boxes of the tiles, their dV and dK the two halves of the
// accumulators, and the loop runs over the query heads of both.  Q and dY
// load one box; S^T and dP^T take 4 k-steps and dV, dK are N = 64
// products.  dQ^T keeps M = 128 (d) starting at the item's own K box, so
// its rows 64-127 (the other box, or zeros) are not reduced.
// kPad: a head dim below the compute width (32 -> 64, 96 -> 128).  Q, dY,
// K, V, dK and dV then go through [rows][heads][d] tensor maps whose boxes
// read zeros past d and store nothing there; dQ rows and the partial-tile
// epilogue are cut at d.  Head dims 64 and 128 keep the plainer
// [rows][heads * d] maps (the 3-D form measured 2-3.5% slower there).
template <bool kBF16, bool kDet, bool kMask, bool kD64, bool kDrop, bool kPad>
__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_tc_kernel(const BwdParams p, const __grid_constant__ TcMaps maps) {
  constexpr int DD = kD64 ? 64 : HD;   // head dim of the tensors
  constexpr uint32_t SM_AM = sm_end(kDrop);   // explicit-mask stages
  constexpr int NBOX = DD / 64;         // 64-column boxes per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_item;
  __shared__ int s_dq_ok;
  auto bar = [&](int i) { return sb + SM_BAR + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WorkItem item_by_grid{};
  if (!kDet) item_by_grid = p.items[blockIdx.x];
  Ctl ctl{&s_abort, p.err, p.timeout_ns};
  // Waits for this CTA's own copies and MMAs in flight (which finish without
  // help from any other role) are bounded by at least a second, whatever
  // the caller's timeout, so that no CTA exits while they still write.
  const long long drain_ns = p.timeout_ns > 1000000000LL ? p.timeout_ns : 1000000000LL;

  if (threadIdx.x == 0) {
    s_abort = 0;
    if (kDet) s_item = atomicAdd(p.ticket, 1);
    mbar_init(bar(B_KV), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    mbar_init(bar(B_SDFULL), 1);
    mbar_init(bar(B_SDFREE), 8);
    mbar_init(bar(B_PFULL), 8);
    mbar_init(bar(B_PFREE), 1);
    mbar_init(bar(B_DSFULL), 8);
    mbar_init(bar(B_DSFREE), 1);
    mbar_init(bar(B_DQFULL), 1);
    mbar_init(bar(B_DQFREE), 4);
    mbar_init(bar(B_ACC), 1);
    mbar_init(bar(B_FINAL), 1);
    mbar_init(bar(B_FINAL_A), 1);
    mbar_init(bar(B_EPI), 4);       // epilogue: the four warps of the dV half
    mbar_init(bar(B_EPI + 1), 4);   // ... and of the dK half
    mbar_init(bar(B_DQPUB), 128);
    mbar_init(bar(B_PUBFREE), 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  if constexpr (kD64) {
    // With one kv head the second K box (rows 64-127 of the M = 128 dQ^T
    // product) is not loaded: zero it.
    if (kDet || (item_by_grid.head >> 16) == 0) {
      for (uint32_t o = threadIdx.x * 16u; o < 16384u; o += NTHREADS * 16u)
        st_shared_v4(sb + SM_K + 16384u + o, 0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const WorkItem item = kDet ? p.items[s_item] : item_by_grid;
  const SeqInfo sq = p.seqs[item.seq];
  const int kvh = item.head & 0xFFFF;
  const int nh = kD64 ? 1 + (item.head >> 16) : 1;   // kv heads of this item
  const int group = p.n / p.n_kv;
  const int k0 = item.tile * BN;
  const int qlo = item_lo(item), qcnt = item_count(item);
  const int per_head = qcnt * group;   // iterations per kv head
  const int n_it = per_head * nh;

  // Registers by warpgroup (setmaxnreg): the producer / MMA-issuer group
  // gives up registers it does not use to the two softmax groups, whose
  // 32-column S, dP and P rows are the kernel's largest live set; the drain
  // group keeps the launch's 128.  The split stays within the 512 x 128
  // registers the block was launched with: 4 warps x 32 x 72 + 8 x 32 x 152
  // + 4 x 32 x 128 = 64512; at compute width 64 (whose issuers need fewer)
  // 4 x 32 x 56 + 8 x 32 x 160 + 4 x 32 x 128 = 64512.
  if (warp < 4) {
  if constexpr (kD64)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
  else
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;");
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs this loop; copies are issued by one elected lane.
    if (n_it > 0) {
      if (lane == 0) {
        tma_prefetch_map(&maps.q);
        tma_prefetch_map(&maps.dy);
        tma_prefetch_map(&maps.k);
        tma_prefetch_map(&maps.v);
      }
      __syncwarp();
      const int ky = sq.cu_k + k0, kx = kvh * DD;
      const int kvbox = kD64 ? nh : NBOX;
      mbar_arrive_expect_tx_w(bar(B_KV), 2 * kvbox * 16384);
      for (int bx = 0; bx < kvbox; ++bx) {
        if constexpr (kPad) {
          // box bx: columns 64 bx .. of head kvh, or at compute width 64 the
          // whole (zero-padded) row of head kvh + bx
          const int x = kD64 ? 0 : 64 * bx, h = kD64 ? kvh + bx : kvh;
          tma_load_3d_w(sb + SM_K + bx * 16384, &maps.k, bar(B_KV), x, h, ky);
          tma_load_3d_w(sb + SM_V + bx * 16384, &maps.v, bar(B_KV), x, h, ky);
        } else {
          tma_load_2d_w(sb + SM_K + bx * 16384, &maps.k, bar(B_KV), kx + 64 * bx, ky);
          tma_load_2d_w(sb + SM_V + bx * 16384, &maps.v, bar(B_KV), kx + 64 * bx, ky);
        }
      }
      // The item `prefetch_ahead` places further down the list starts on
      // some SM about when this one ends: bring its K and V into L2 now.
      if (lane == 0 && blockIdx.x + p.prefetch_ahead < p.n_items) {
        const WorkItem nx = p.items[blockIdx.x + p.prefetch_ahead];
        const int nky = p.seqs[nx.seq].cu_k + nx.tile * BN, nkx = (nx.head & 0xFFFF) * DD;
        for (int bx = 0; bx < (kD64 ? 1 + (nx.head >> 16) : NBOX); ++bx) {
          if constexpr (kPad) {
            const int x = kD64 ? 0 : 64 * bx, h = (nx.head & 0xFFFF) + (kD64 ? bx : 0);
            tma_prefetch_l2_3d(&maps.k, x, h, nky);
            tma_prefetch_l2_3d(&maps.v, x, h, nky);
          } else {
            tma_prefetch_l2_2d(&maps.k, nkx + 64 * bx, nky);
            tma_prefetch_l2_2d(&maps.v, nkx + 64 * bx, nky);
          }
        }
      }
      __syncwarp();
      int issued = 0;
      for (int L = 0; L < n_it; ++L) {
        const int st = L % STAGES;
        if (L >= STAGES && !wait_or_abort(ctl, bar(B_EMPTY + st), ((L / STAGES) - 1) & 1,
                                          ROLE_PRODUCER))
          break;
        const int n = kvh * group + L / qcnt;
        const int q0 = (qlo + L % qcnt) * BM;
        const int qy = sq.cu_q + q0, qx = n * DD;
        const uint32_t full = bar(B_FULL + st);
        const int64_t srow = int64_t(n) * p.tp + sq.qpad + q0;
        const bool am_tile = kMask && p.am_tma;
        const bool drop_tile = kDrop && p.drop_rows16;
        const int rows = min(BM, sq.len_q - q0);
        if (drop_tile)
          load_keep_bits(sb + SM_DROP + st * DROP_STAGE, p.mask, sq, n, q0, k0, rows, full,
                         lane);
        mbar_arrive_expect_tx_w(full, 2 * NBOX * 8192 + 2 * 256 + (am_tile ? AM_STAGE : 0u));
        if (am_tile)   // mask rows q0.., columns k0.. (chunk-local); out of range reads 0
          tma_load_2d_w(sb + SM_AM + st * AM_STAGE, &maps.am, full, k0, q0);
        for (int bx = 0; bx < NBOX; ++bx) {
          if constexpr (kPad) {
            tma_load_3d_w(sb + SM_Q + st * 16384 + bx * 8192, &maps.q, full, 64 * bx, n, qy);
            tma_load_3d_w(sb + SM_DY + st * 16384 + bx * 8192, &maps.dy, full, 64 * bx, n, qy);
          } else {
            tma_load_2d_w(sb + SM_Q + st * 16384 + bx * 8192, &maps.q, full, qx + 64 * bx, qy);
            tma_load_2d_w(sb + SM_DY + st * 16384 + bx * 8192, &maps.dy, full, qx + 64 * bx, qy);
          }
        }
        bulk_load_w(sb + SM_LSE + st * 256, p.lse2 + srow, 256, full);
        bulk_load_w(sb + SM_DSUM + st * 256, p.dsum + srow, 256, full);
        ++issued;
      }
      // No copy may still be writing shared memory when the CTA exits.
      const int never = 0;
      mbar_wait(bar(B_KV), 0, drain_ns, &never);
      for (int L = issued > STAGES ? issued - STAGES : 0; L < issued; ++L)
        mbar_wait(bar(B_FULL + L % STAGES), (L / STAGES) & 1, drain_ns, &never);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Two warps issue the tensor-core work, so that two independent chains
    // of dependent MMAs are in flight at once (one issuing warp cannot keep
    // the tensor core busy with 36 small MMAs per tile):
    //   warp 1:  S^T = K Q^T and dP^T = V dY^T of tile L, interleaved;
    //   warp 2:  dV += P^T dY, then dK += dS^T Q interleaved with dQ^T.
    // A commit tracks the MMAs of the thread that issues it, so each warp
    // signals only its own work.  Each warp issues from straight-line code,
    // one elected lane per MMA (see mma_ss_w).
    if (n_it > 0) {
      const uint32_t id_s = idesc_f16(128, BM, false, false, kBF16);   // S^T, dP^T
      const uint32_t id_g = idesc_f16(128, DD, false, true, kBF16);    // dV, dK
      const uint32_t id_q = idesc_f16(128, BM, true, true, kBF16);     // dQ^T
      // Descriptors are built once per operand; a k-step adds its byte offset
      // >> 4 to the 14-bit start-address field (shared addresses stay below
      // 256 KB, so the field never carries).
      const uint64_t dk_ = sdesc_sw128(sb + SM_K, 16, 1024);     // K, K-major
      const uint64_t dv_ = sdesc_sw128(sb + SM_V, 16, 1024);     // V, K-major
      const uint64_t dkt = sdesc_sw128(sb + SM_K, 16384, 1024);  // K, MN-major (K^T)
      const uint64_t dds = sdesc_sw128(sb + SM_DS, 16384, 1024); // dS^T, MN-major
      if (warp == 1) {
        bool ok = wait_or_abort(ctl, bar(B_KV), 0, ROLE_MMA);
        for (int L = 0; ok && L < n_it; ++L) {
          const int st = L % STAGES;
          ok = wait_or_abort(ctl, bar(B_FULL + st), (L / STAGES) & 1, ROLE_MMA) &&
               (L == 0 || wait_or_abort(ctl, bar(B_SDFREE), (L - 1) & 1, ROLE_MMA));
          if (!ok) break;
          tc_fence_after();
          // D[128 x 64] = A[128 x 128] B[64 x 128]^T, both K-major (2 boxes along K)
          const uint64_t bq = sdesc_sw128(sb + SM_Q + st * 16384, 16, 1024);
          const uint64_t by = sdesc_sw128(sb + SM_DY + st * 16384, 16, 1024);
          const uint32_t mo = kD64 ? uint32_t(((L / per_head) * 16384) >> 4) : 0u;  // kv head box
#pragma unroll
          for (int kk = 0; kk < DD / 16; ++kk) {
            const uint32_t ao = (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4) + mo;
            const uint32_t bo = (((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
            const uint32_t acc = kk > 0 ? 1u : 0u;
            mma_ss_w(tmem + COL_S, dk_ + ao, bq + bo, id_s, acc);
            mma_ss_w(tmem + COL_DP, dv_ + ao, by + bo, id_s, acc);
          }
          mma_commit_w(bar(B_SDFULL));
        }
        // Every MMA of this warp has finished before TMEM is freed.
        mma_commit_w(bar(B_FINAL_A));
        const int never = 0;
        mbar_wait(bar(B_FINAL_A), 0, drain_ns, &never);
      } else {
        bool ok = wait_or_abort(ctl, bar(B_KV), 0, ROLE_MMA);
        for (int L = 0; ok && L < n_it; ++L) {
          const int st = L % STAGES;
          const int m = kD64 ? L / per_head : 0;                  // kv head of the item
          const uint32_t acc0 = (kD64 ? L - m * per_head : L) > 0 ? 1u : 0u;
          const uint32_t mcol = uint32_t(m * 64);                  // its accumulator half
          const uint32_t mo = uint32_t((m * 16384) >> 4);          // its K box
          if (!(ok = wait_or_abort(ctl, bar(B_PFULL), L & 1, ROLE_MMA))) break;
          tc_fence_after();
          {
            // dV[128 x 128] += P^T[128 x 64] (TMEM) dY[64 x 128] (MN-major)
            const uint64_t b0 = sdesc_sw128(sb + SM_DY + st * 16384, 8192, 1024);
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk)
              mma_ts_w(tmem + COL_DV + mcol, tmem + COL_P + kk * 8, b0 + ((kk * 2048) >> 4), id_g,
                       kk > 0 ? 1u : acc0);
          }
          mma_commit_w(bar(B_PFREE));
          if (!(ok = wait_or_abort(ctl, bar(B_DSFULL), L & 1, ROLE_MMA))) break;
          if (L > 0 && !(ok = wait_or_abort(ctl, bar(B_DQFREE), (L - 1) & 1, ROLE_MMA))) break;
          tc_fence_after();
          {
            // dK[128 x 128] += dS^T[128 x 64] (TMEM) Q[64 x 128] (MN-major), and
            // dQ^T[128 d x 64 q] = K^T[128 d x 128 keys] dS^T[128 keys x 64 q]
            const uint64_t b0 = sdesc_sw128(sb + SM_Q + st * 16384, 8192, 1024);
#pragma unroll
            for (int kk = 0; kk < BM / 16; ++kk) {
              mma_ts_w(tmem + COL_DK + mcol, tmem + COL_DS + kk * 8, b0 + ((kk * 2048) >> 4), id_g,
                       kk > 0 ? 1u : acc0);
              mma_ss_w(tmem + COL_DQ, dkt + mo + (((2 * kk) * 2048) >> 4),
                       dds + (((2 * kk) * 2048) >> 4), id_q, kk > 0 ? 1u : 0u);
              mma_ss_w(tmem + COL_DQ, dkt + mo + (((2 * kk + 1) * 2048) >> 4),
                       dds + (((2 * kk + 1) * 2048) >> 4), id_q, 1u);
            }
          }
          mma_commit_w(bar(B_DQFULL));
          mma_commit_w(bar(B_DSFREE));
          mma_commit_w(bar(B_EMPTY + st));
        }
        if (ok) mma_commit_w(bar(B_ACC));
        // Every MMA of this warp has finished before TMEM is freed.
        mma_commit_w(bar(B_FINAL));
        const int never = 0;
        mbar_wait(bar(B_FINAL), 0, drain_ns, &never);
      }
    }
  } else if (kDet) {
    // ------------------------------------------------------------ dQ publisher
    // Deterministic mode: once the four drain warps have issued a tile's dQ
    // reductions and arrived on B_DQPUB (release at CTA scope), this warp's
    // GPU-scope fence makes them visible before the tile's counter moves on
    // (the fence is cumulative over what the mbarrier wait has observed),
    // so the next key tile in the add order cannot add first.  The drain
    // goes on to its next tile meanwhile; B_PUBFREE keeps it at most one
    // tile ahead of this warp.
    for (int L = 0; L < n_it; ++L) {
      const int n = kvh * group + L / qcnt;
      const int qt = qlo + L % qcnt;
      if (!wait_or_abort(ctl, bar(B_DQPUB), L & 1, ROLE_DQ)) break;
      if (lane == 0) {
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        st_release_gpu(dq_counter(p, sq, n, qt), dq_rank(p, sq, item.tile, qt) + 1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PUBFREE));
    }
  }
  } else if (warp < 12) {
    if constexpr (kD64)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 160;");
    else
      asm volatile("setmaxnreg.inc.sync.aligned.u32 152;");
    // ------------------------------------------------------------ softmax / dS
    const int half = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int jl = quarter * 32 + lane;
    const int jg = k0 + jl;
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    for (int L = 0; L < n_it; ++L) {
      const int st = L % STAGES;
      const int n = kvh * group + L / qcnt;
      const int q0 = (qlo + L % qcnt) * BM;
      const int i0 = q0 + 32 * half;
      uint32_t r[32], rdp[32];
      float pr[32];
      if (!wait_or_abort(ctl, bar(B_SDFULL), L & 1, ROLE_SOFTMAX)) break;
      tc_fence_after();
      tmem_ld32x2(tmem + lane_off + COL_S + 32 * half, r, tmem + lane_off + COL_DP + 32 * half,
                  rdp);
      tc_fence_before();
      if (lane == 0) mbar_arrive(bar(B_SDFREE));
      {
        const uint32_t lse_addr = sb + SM_LSE + st * 256 + 128 * half;
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 l4 = ld_shared_f4(lse_addr + 16 * c4);
          fma2(pr[4 * c4], pr[4 * c4 + 1], __uint_as_float(r[4 * c4]),
               __uint_as_float(r[4 * c4 + 1]), sl2, sl2, -l4.x, -l4.y);
          fma2(pr[4 * c4 + 2], pr[4 * c4 + 3], __uint_as_float(r[4 * c4 + 2]),
               __uint_as_float(r[4 * c4 + 3]), sl2, sl2, -l4.z, -l4.w);
          pr[4 * c4 + 0] = ex2(pr[4 * c4 + 0]);
          pr[4 * c4 + 1] = ex2(pr[4 * c4 + 1]);
          pr[4 * c4 + 2] = ex2(pr[4 * c4 + 2]);
          pr[4 * c4 + 3] = ex2(pr[4 * c4 + 3]);
        }
      }
      const bool full_tile = (k0 + BN - 1 <= q0 + sq.next) && (k0 >= q0 + BM - 1 - sq.pre) &&
                             (k0 + BN <= sq.len_k);
      if (!full_tile) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int i = i0 + c;
          if (!(jg <= i + sq.next && jg >= i - sq.pre && jg < sq.len_k)) pr[c] = 0.f;
        }
      }
      if (kMask && jg < sq.len_k) {
        if (p.am_tma) {
          // the stage's mask tile: row = query - q0, column = key - k0
          const uint8_t *am = sm + SM_AM + st * AM_STAGE + (32 * half) * 128 + jl;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (i0 + c < sq.len_q && am[c * 128] != 0) pr[c] = 0.f;
        } else {
          // Explicit mask from global memory: for each of its 32 queries a
          // warp reads 32 consecutive bytes (its 32 keys) of one mask row.
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int i = i0 + c;
            if (i < sq.len_q && atten_masked(p.atten_mask, p.am_cols, i, jg)) pr[c] = 0.f;
          }
        }
      }
      uint32_t keep = 0xFFFFFFFFu;
      if constexpr (kDrop) {
        // Lane l reads query 2l (l < 16) or 2(l - 16) + 1: after the transpose
        // bit c of keep is query 2c and bit 16 + c query 2c + 1.
        const int ql = lane < 16 ? 2 * lane : 2 * lane - 31;
        const int il = i0 + ql;
        uint32_t w = 0;
        if (il < sq.len_q) {
          if (p.drop_rows16) {
            w = ld_shared_u32(sb + SM_DROP + st * DROP_STAGE + (32 * half + ql) * 16 +
                              quarter * 4);
          } else {
            const int64_t bit = sq.mask_off + (int64_t(n) * sq.len_q + il) * sq.len_k + k0 +
                                quarter * 32;
            w = fetch_bits32(p.mask, p.mask_bytes, bit);
          }
        }
        keep = transpose_bits32(w, lane);
      }
      uint32_t pk[16];
      uint32_t ks[8];   // shifted copies of keep for pair_mask8
#pragma unroll
      for (int s = 0; s < 8; ++s) ks[s] = keep << s;
      if constexpr (kDrop) {
        // With dropout the preprocess has put log2(keep_prob) into lse2 and
        // keep_prob into dsum, so pr is P / keep_prob and dv below is
        // keep_prob D.  A dropped entry is zero in the P^T operand; its dS is
        // -(P / keep_prob)(keep_prob D) = -P D, a kept one's the dropout-free
        // expression (P / keep_prob)(dP - keep_prob D) = P (dP / keep_prob - D).
        // Both are packed and the pair mask picks per bf16 half.
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack2<kBF16>(pr[2 * c], pr[2 * c + 1]) & pair_mask8(ks, c);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack2<kBF16>(pr[2 * c], pr[2 * c + 1]);
      }
      if (L > 0 && !wait_or_abort(ctl, bar(B_PFREE), (L - 1) & 1, ROLE_SOFTMAX)) break;
      tc_fence_after();
      tmem_st16(tmem + lane_off + COL_P + 16 * half, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));

      {
        const uint32_t dsum_addr = sb + SM_DSUM + st * 256 + 128 * half;
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 d4 = ld_shared_f4(dsum_addr + 16 * c4);
          const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
          float ds[4];
          sub2(ds[0], ds[1], __uint_as_float(rdp[4 * c4]), __uint_as_float(rdp[4 * c4 + 1]),
               dv[0], dv[1]);
          sub2(ds[2], ds[3], __uint_as_float(rdp[4 * c4 + 2]), __uint_as_float(rdp[4 * c4 + 3]),
               dv[2], dv[3]);
          mul2(ds[0], ds[1], ds[0], ds[1], pr[4 * c4], pr[4 * c4 + 1]);
          mul2(ds[2], ds[3], ds[2], ds[3], pr[4 * c4 + 2], pr[4 * c4 + 3]);
          pk[2 * c4] = pack2<kBF16>(ds[0], ds[1]);
          pk[2 * c4 + 1] = pack2<kBF16>(ds[2], ds[3]);
          if constexpr (kDrop) {
            float e[4];
            mul2(e[0], e[1], pr[4 * c4], pr[4 * c4 + 1], -dv[0], -dv[1]);
            mul2(e[2], e[3], pr[4 * c4 + 2], pr[4 * c4 + 3], -dv[2], -dv[3]);
            const uint32_t m0 = pair_mask8(ks, 2 * c4), m1 = pair_mask8(ks, 2 * c4 + 1);
            pk[2 * c4] = (pk[2 * c4] & m0) | (pack2<kBF16>(e[0], e[1]) & ~m0);
            pk[2 * c4 + 1] = (pk[2 * c4 + 1] & m1) | (pack2<kBF16>(e[2], e[3]) & ~m1);
          }
        }
      }
      if (L > 0 && !wait_or_abort(ctl, bar(B_DSFREE), (L - 1) & 1, ROLE_SOFTMAX)) break;
      tc_fence_after();
      tmem_st16(tmem + lane_off + COL_DS + 16 * half, pk);
      const uint32_t row = sb + SM_DS + uint32_t(jl) * 128u;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const uint32_t chunk = uint32_t((4 * half + cc) ^ (jl & 7));
        st_shared_v4(row + chunk * 16u, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DSFULL));
    }
    // ------------------------------------------------------------ epilogue
    // dV is complete once the last dV product has run (the last PFREE
    // commit), while that tile's dK and dQ^T products may still run: the dV
    // half starts then; the dK half waits for all products (B_ACC).
    bool have = n_it > 0 && !*reinterpret_cast<volatile int *>(&s_abort);
    if (have)
      have = half == 0 ? wait_or_abort(ctl, bar(B_PFREE), (n_it - 1) & 1, ROLE_EPILOGUE)
                       : wait_or_abort(ctl, bar(B_ACC), 0, ROLE_EPILOGUE);
    tc_fence_after();
    // A full key tile goes out through shared memory and two bulk tensor
    // stores per tensor (dV staged in the dY stages, which no product reads
    // after the last dV; dK in the Q stages, idle once every product has
    // run; two [128 x 64] boxes each in the 128-byte swizzle); the last,
    // partial tile of a sequence is stored row by row, so that no row of
    // the next sequence is touched.
    const bool tile_full = k0 + BN <= sq.len_k;
    if (tile_full && (n_it == 0 || have)) {
      const float sc = half == 0 ? 1.f : p.scale;
      const uint32_t col = half == 0 ? COL_DV : COL_DK;
      const uint32_t stage = sb + (half == 0 ? SM_DY : SM_Q);
#pragma unroll 1
      for (int c0 = 0; c0 < DD * nh; c0 += 32) {
        uint32_t r[32];
        if (n_it > 0) {
          tmem_ld32(tmem + lane_off + col + c0, r);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = 0u;
        }
        // columns c0 .. c0 + 31 = 16-byte chunks (c0 % 64) / 8 .. + 3 of box c0 / 64
        const uint32_t rowa = stage + uint32_t(c0 / 64) * 16384u + uint32_t(jl) * 128u;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack2<kBF16>(__uint_as_float(r[8 * v + 2 * e]) * sc,
                                __uint_as_float(r[8 * v + 2 * e + 1]) * sc);
          const uint32_t chunk = uint32_t(((c0 % 64) / 8 + v) ^ (jl & 7));
          st_shared_v4(rowa + chunk * 16u, w[0], w[1], w[2], w[3]);
        }
      }
      // The four warps of this half report their rows (bounded wait, so that
      // a warp that gave up cannot hold the others), then one thread stores.
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_EPI + half));
      if (quarter == 0 && lane == 0 &&
          wait_or_abort(ctl, bar(B_EPI + half), 0, ROLE_EPILOGUE)) {
        const CUtensorMap *m = half == 0 ? &maps.dv : &maps.dk;
        const int y = sq.cu_k + k0, x = kvh * DD;
        for (int bx = 0; bx < (kD64 ? nh : NBOX); ++bx) {
          if constexpr (kPad)
            tma_store_3d(m, stage + bx * 16384, kD64 ? 0 : 64 * bx, kD64 ? kvh + bx : kvh, y);
          else
            tma_store_2d(m, stage + bx * 16384, x + 64 * bx, y);
        }
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    } else if (n_it == 0 || have) {
      using T = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;
      T *out = static_cast<T *>(half == 0 ? p.dv : p.dk);
      const float sc = half == 0 ? 1.f : p.scale;
      const uint32_t col = half == 0 ? COL_DV : COL_DK;
      const bool valid = jg < sq.len_k;
      // nh heads adjacent; accumulator column c0 is column c0 % DD of head
      // kvh + c0 / DD, of which the first dd exist.
      const int dd = kPad ? p.d : DD;
      T *rowp = out + ((int64_t(sq.cu_k) + jg) * p.n_kv + kvh) * dd;
#pragma unroll 1
      for (int c0 = 0; c0 < DD * nh; c0 += 32) {
        uint32_t r[32];
        if (n_it > 0) {
          tmem_ld32(tmem + lane_off + col + c0, r);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = 0u;
        }
        if (valid) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack2<kBF16>(__uint_as_float(r[8 * v + 2 * e]) * sc,
                                  __uint_as_float(r[8 * v + 2 * e + 1]) * sc);
            if constexpr (kPad) {
              const int cc = c0 % DD + 8 * v;
              if (cc < dd) st_global_v4(rowp + (c0 / DD) * dd + cc, w[0], w[1], w[2], w[3]);
            } else {
              st_global_v4(rowp + c0 + 8 * v, w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ drain
    const int quarter = warp & 3;
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const int dd = kPad ? p.d : DD;   // head dim of dq_acc
    const int64_t row_stride = int64_t(p.n) * dd;
    for (int L = 0; L < n_it; ++L) {
      const int n = kvh * group + L / qcnt;
      const int q0 = (qlo + L % qcnt) * BM;
      if (!wait_or_abort(ctl, bar(B_DQFULL), L & 1, ROLE_DQ)) break;
      tc_fence_after();
      uint32_t a[32], b[32];
      tmem_ld32(tmem + lane_off + COL_DQ, a);
      tmem_ld32(tmem + lane_off + COL_DQ + 32, b);
      tc_fence_before();
      if (lane == 0) mbar_arrive(bar(B_DQFREE));
      // Deterministic mode: wait until the key tiles before this one in the add
      // order (descending key tiles) have added their partials of this query tile
      // (the counter holds how many have), add; warp 3 then publishes count + 1.
      if constexpr (kDet) {
        const int qt = qlo + L % qcnt;
        int32_t *ctr = dq_counter(p, sq, n, qt);
        const int rank = dq_rank(p, sq, item.tile, qt);
        if (warp == 12 && lane == 0) {
          const bool got = wait_counter(ctr, rank, p.timeout_ns,
                                        reinterpret_cast<volatile int *>(&s_abort));
          if (!got && !*reinterpret_cast<volatile int *>(&s_abort)) {
            atomicExch(&s_abort, 1);
            atomicCAS(p.err, 0, kErrTimeoutBase + ROLE_DQ);
          }
          s_dq_ok = got ? 1 : 0;
        }
        drain_bar_sync();
        if (!*reinterpret_cast<volatile int *>(&s_dq_ok)) break;
      }
      // Thread (quad m, c) holds column d = quarter*32 + 4m + c for 64 queries.
      // A 4 x 4 transpose inside each quad (two xor-shuffle rounds) gives it
      // d = quarter*32 + 4m + 0..3 at query 4j + c, so that each reduction
      // adds 16 contiguous bytes (4x fewer reduction instructions).  All
      // transposes come first, so that the 16 reductions issue back to back.
      const int rows = min(BM, sq.len_q - q0);
      const int c = lane & 3;
      float out[BM];
#pragma unroll
      for (int j = 0; j < BM / 4; ++j) {
        const uint32_t *src = j < 8 ? a : b;
        const int o = 4 * (j & 7);
        const float x0 = __uint_as_float(src[o]), x1 = __uint_as_float(src[o + 1]);
        const float x2 = __uint_as_float(src[o + 2]), x3 = __uint_as_float(src[o + 3]);
        const bool hi2 = c & 2, hi1 = c & 1;
        const float t0 = __shfl_xor_sync(0xffffffffu, hi2 ? x0 : x2, 2);
        const float t1 = __shfl_xor_sync(0xffffffffu, hi2 ? x1 : x3, 2);
        const float r0 = hi2 ? t0 : x0, r1 = hi2 ? t1 : x1;
        const float r2 = hi2 ? x2 : t0, r3 = hi2 ? x3 : t1;
        const float u0 = __shfl_xor_sync(0xffffffffu, hi1 ? r0 : r1, 1);
        const float u1 = __shfl_xor_sync(0xffffffffu, hi1 ? r2 : r3, 1);
        out[4 * j] = hi1 ? u0 : r0;
        out[4 * j + 1] = hi1 ? r1 : u0;
        out[4 * j + 2] = hi1 ? u1 : r2;
        out[4 * j + 3] = hi1 ? r3 : u1;
      }
      float *ptr = p.dq_acc + (int64_t(sq.cu_q) + q0 + c) * row_stride + int64_t(n) * dd +
                   quarter * 32 + (lane & ~3);
      // Rows d >= dd of dQ^T hold padding (zero columns of K past the head
      // dim, or at compute width 64 the other K box).
      if (kPad ? quarter * 32 + (lane & ~3) < dd : quarter * 32 < DD) {
#pragma unroll
        for (int j = 0; j < BM / 4; ++j, ptr += 4 * row_stride)
          if (4 * j + c < rows)
            red_add_v4_f32(ptr, out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
      }
      if constexpr (kDet) {
        // warp 3 publishes this tile (after the previous one)
        if (L > 0 && !wait_or_abort(ctl, bar(B_PUBFREE), (L - 1) & 1, ROLE_DQ)) break;
        mbar_arrive(bar(B_DQPUB));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// [rows][heads][d] 16-bit tensor as a 3-D map with [box_rows][1][64] boxes
// (64 columns of one head).  Columns at and past d read as zeros and are
// not written.  Needs d * 2 bytes to be a multiple of 16.
bool make_map3(CUtensorMap *m, const void *base, int64_t rows, int heads, int d, int box_rows,
               bool bf16) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(heads), cuuint64_t(rows)};
  cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(heads) * d * 2};
  cuuint32_t box[3] = {64, 1, cuuint32_t(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
             const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, heads * d] 16-bit tensor as a 2-D map with 64-column x box_rows boxes.
bool make_map(CUtensorMap *m, const void *base, int64_t rows, int heads, int d, int box_rows,
              bool bf16) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {cuuint64_t(heads) * d, cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(heads) * d * 2};
  cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
             const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kBF16, bool kDet, bool kMask, bool kD64, bool kDrop, bool kPad>
cudaError_t launch_t(const BwdParams &p, cudaStream_t st) {
  const int d = p.d;
  auto mk = kPad ? make_map3 : make_map;
  TcMaps maps{};
  if (!mk(&maps.q, p.q, p.total_q, p.n, d, BM, kBF16) ||
      !mk(&maps.dy, p.dy, p.total_q, p.n, d, BM, kBF16) ||
      !mk(&maps.k, p.k, p.total_kv, p.n_kv, d, BN, kBF16) ||
      !mk(&maps.v, p.v, p.total_kv, p.n_kv, d, BN, kBF16) ||
      !mk(&maps.dk, p.dk, p.total_kv, p.n_kv, d, BN, kBF16) ||
      !mk(&maps.dv, p.dv, p.total_kv, p.n_kv, d, BN, kBF16))
    return cudaErrorInvalidValue;
  BwdParams q = p;
  q.am_tma = 0;
  if (kMask) {
    // TMA needs a 16-byte aligned base and row pitch; otherwise the softmax
    // warps read the mask from global memory.
    const bool al = (reinterpret_cast<uintptr_t>(p.atten_mask) & 15u) == 0 && p.am_cols % 16 == 0;
    if (al) {
      EncodeTiledFn enc = encode_fn();
      if (enc == nullptr) return cudaErrorInvalidValue;
      cuuint64_t dims[2] = {cuuint64_t(p.am_cols), cuuint64_t(p.am_rows)};
      cuuint64_t strides[1] = {cuuint64_t(p.am_cols)};
      cuuint32_t box[2] = {128, 64};
      cuuint32_t es[2] = {1, 1};
      if (enc(&maps.am, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(p.atten_mask),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
      q.am_tma = 1;
    }
  }
  const uint32_t smem = kMask ? smem_bytes_mask(kDrop) : smem_bytes(kDrop);
  cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel<kBF16, kDet, kMask, kD64, kDrop, kPad>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&q.prefetch_ahead, cudaDevAttrMultiProcessorCount, dev)) !=
      cudaSuccess)
    return e;
  bwd_tc_kernel<kBF16, kDet, kMask, kD64, kDrop, kPad><<<p.n_items, NTHREADS, smem, st>>>(q, maps);
  return cudaGetLastError();
}

}  // namespace
}  // namespace fav
