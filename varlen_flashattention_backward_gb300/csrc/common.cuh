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

}  // namespace fav
