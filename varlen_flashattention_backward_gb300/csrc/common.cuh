// Small device helpers shared by the kernels (type conversion, mask reads).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "internal.h"

namespace fav {

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <> __device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

// Keep bit of one (sequence, head, i, j): the dropMask bit layout described in
// fa_varlen.h (bit index mask_off + (n * Lq + i) * Lk + j, LSB first).
__device__ __forceinline__ float keep_bit(const uint8_t *mask, int64_t mask_off, int n, int lq,
                                          int lk, int i, int j) {
  const int64_t idx = mask_off + (int64_t(n) * lq + i) * lk + j;
  return float((__ldg(mask + (idx >> 3)) >> (idx & 7)) & 1);
}

__device__ __forceinline__ bool window_ok(int i, int j, int lq, int lk, int pre, int next) {
  return i < lq && j < lk && j >= i - pre && j <= i + next;
}

// Explicit attention mask: true when (i, j) is excluded (mask byte != 0).
// Callers pass in-range (i, j).
__device__ __forceinline__ bool atten_masked(const uint8_t *mask, int64_t cols, int i, int j) {
  return mask != nullptr && __ldg(mask + int64_t(i) * cols + j) != 0;
}

// Sequence owning padded statistics row `row` (the last sequence whose qpad
// is <= row; zero-length sequences own no rows).
__device__ __forceinline__ int seq_of_padded_row(const SeqInfo *seqs, int batch, int row) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seqs[mid].qpad <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// Ordered dQ adds of the deterministic mode (BwdParams::deterministic).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t *ptr) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(int32_t *ptr, int32_t v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

__device__ __forceinline__ long long timer_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Spins until *ptr == want.  Gives up (false) once timeout_ns has passed or,
// when `abort` is non-null, once *abort is set.
__device__ __forceinline__ bool wait_counter(const int32_t *ptr, int32_t want, long long timeout_ns,
                                             const volatile int *abort) {
  if (ld_acquire_gpu(ptr) == want) return true;
  const long long t0 = timer_ns();
  while (true) {
    __nanosleep(100);
    if (ld_acquire_gpu(ptr) == want) return true;
    if (abort != nullptr && *abort) return false;
    if (timer_ns() - t0 > timeout_ns) return false;
  }
}

// Item index of this CTA: its grid index, or in the deterministic mode the
// next ticket, so that items are taken in list order by CTAs that are already
// running.  Call from one thread.
__device__ __forceinline__ int take_item(const BwdParams &p) {
  return p.deterministic ? atomicAdd(p.ticket, 1) : int(blockIdx.x);
}

// Counter and rank of the dQ partial that key tile `tile` adds to query tile
// `qt` (0-based inside the sequence) of query head n.
__device__ __forceinline__ int32_t *dq_counter(const BwdParams &p, const SeqInfo &s, int n,
                                               int qt) {
  return p.sem + int64_t(n) * (p.tp / kQTile) + s.qpad / kQTile + qt;
}
// Place of key tile `tile` in the add order of query tile qt (descending
// key tiles: the table holds the highest one that visits qt).
__device__ __forceinline__ int dq_rank(const BwdParams &p, const SeqInfo &s, int tile, int qt) {
  return p.qfirst[s.qpad / kQTile + qt] - tile;
}

}  // namespace fav
