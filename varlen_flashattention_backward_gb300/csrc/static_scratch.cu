// fa_varlen_bwd_static_scratch: the backward for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc at the point where they run the
// backward: code inside a custom allocator or a memory-pool callback, a
// runtime that owns all device memory and hands out only fixed buffers,
// or a host thread that must not take the allocator's locks.  This entry
// point takes no workspace.  Its scratch (the work list, the padded
// statistics, the fp32 dQ accumulator and the error word) lives in the
// file-scope array below, which the CUDA module reserves on every device
// that loads this library and keeps until the process exits.

#include <cuda_runtime.h>

#include <array>
#include <mutex>

#include "fa_varlen.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;   // 64 MiB
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a host-side stand-in;
// the device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_bwd_scratch[kStaticScratchBytes];

std::mutex g_mu;
std::array<void *, kMaxDevices> g_ptr{};   // device address per device, once known

// Device address of g_bwd_scratch on the current device, looked up once per
// device (with that device current) and cached.  Null on failure.
void *scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess) return nullptr;
    g_ptr[dev] = ptr;
  }
  return g_ptr[dev];
}

}  // namespace

extern "C" fa_status fa_varlen_bwd_static_scratch(
    const void *q, const void *k, const void *v, const void *dy, const uint8_t *drop_mask,
    int64_t drop_mask_bytes, const float *softmax_max, const float *softmax_sum, const void *y,
    const int64_t *seq_lens_q, const int64_t *seq_lens_kv, int64_t batch, int64_t total_q,
    int64_t total_kv, int64_t head_num, int64_t head_num_kv, int64_t head_dim, fa_dtype dtype,
    const char *layout, double scale, double keep_prob, int64_t pre_tokens, int64_t next_tokens,
    int64_t sparse_mode, void *dq, void *dk, void *dv, fa_stream_t stream) {
  size_t need = 0;
  fa_status st = fa_varlen_bwd_workspace_size(seq_lens_q, seq_lens_kv, batch, total_q, total_kv,
                                              head_num, head_num_kv, head_dim, dtype, layout,
                                              keep_prob, pre_tokens, next_tokens, sparse_mode,
                                              &need);
  if (st != FA_OK) return st;
  if (need > kStaticScratchBytes) return FA_ERR_WORKSPACE;
  void *scratch = scratch_address();
  if (scratch == nullptr) return FA_ERR_CUDA;
  return fa_varlen_bwd(q, k, v, dy, drop_mask, drop_mask_bytes, softmax_max, softmax_sum, y,
                       seq_lens_q, seq_lens_kv, batch, total_q, total_kv, head_num, head_num_kv,
                       head_dim, dtype, layout, scale, keep_prob, pre_tokens, next_tokens,
                       sparse_mode, dq, dk, dv, scratch, kStaticScratchBytes, stream);
}
