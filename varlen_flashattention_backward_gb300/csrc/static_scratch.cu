// fa_varlen_bwd_static_scratch: the backward for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc at the point where they run the
// backward: code inside a custom allocator or a memory-pool callback, a
// runtime that owns all device memory and hands out only fixed buffers,
// or a host thread that must not take the allocator's locks.  This entry
// point takes no workspace.  Its scratch (the work list, the padded
// statistics, the fp32 dQ accumulator and the error word) lives in the
// file-scope array below, which the CUDA module reserves in every context
// that loads this library and keeps until that context is destroyed.

#include <cuda.h>
#include <cuda_runtime.h>

#include <array>
#include <mutex>

#include "fa_varlen.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;   // 64 MiB
constexpr int kMaxContexts = 64;

// The scratch itself.  In host code this name is only a host-side stand-in;
// the device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_bwd_scratch[kStaticScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns &driver_fns() {
  static DriverFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
    cudaGetLastError();
  });
  return fns;
}

// Address of g_bwd_scratch, one entry per CUDA context.  The key is the
// context's unique id (cuCtxGetId), which the driver never gives to another
// context of the process: a context that is destroyed and created again
// (cudaDeviceReset, then the next runtime call) or a second context on the
// same device (created through the driver API) gets a lookup of its own.
struct Entry {
  unsigned long long ctx_id;
  void *ptr;
};
std::mutex g_mu;
std::array<Entry, kMaxContexts> g_table{};
int g_used = 0;

// Unique id of the context current on this thread; the device's primary
// context is made current first when none is.  0 on failure.
unsigned long long current_context_id() {
  const DriverFns &f = driver_fns();
  if (f.get_current == nullptr || f.get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return 0;
  if (ctx == nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  }
  unsigned long long id = 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_bwd_scratch in the current context: looked up once
// per context (cudaGetSymbolAddress with that context current; the first
// lookup also loads this library's module into the context) and cached.
// Null on failure, with the runtime's last-error state cleared.
void *scratch_address() {
  const unsigned long long id = current_context_id();
  if (id == 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < g_used; ++i)
    if (g_table[i].ctx_id == id) return g_table[i].ptr;
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || ptr == nullptr) {
    cudaGetLastError();
    return nullptr;
  }
  // A full table (more than kMaxContexts contexts over the process's life)
  // recycles the oldest entry.
  const int slot = g_used < kMaxContexts ? g_used++ : int(id % kMaxContexts);
  g_table[slot] = Entry{id, ptr};
  return ptr;
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

extern "C" fa_status fa_varlen_bwd_static_scratch_read_error(fa_stream_t stream,
                                                             int32_t *code) {
  if (code == nullptr) return FA_ERR_NULLPTR;
  void *scratch = scratch_address();
  if (scratch == nullptr) return FA_ERR_CUDA;
  return fa_varlen_read_error(scratch, kStaticScratchBytes, stream, code);
}
