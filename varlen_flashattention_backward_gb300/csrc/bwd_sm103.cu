// The tcgen05 backward at head dims 64 and 128 (bwd_sm103.cuh), its
// dispatch, and the failure-detection self-test kernel.

#include "bwd_sm103.cuh"

namespace fav {
namespace {

// Failure-detection self-test: every thread waits, with the backward's
// bounded wait, for a phase of an mbarrier that nothing arrives on.  The
// wait expires, records kErrTimeoutBase + ROLE_SELFTEST in *err, and the
// kernel ends normally.
__global__ void wait_timeout_selftest_kernel(int32_t *err, long long timeout_ns) {
  __shared__ uint64_t bar_word;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar_word);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(b, 1);
    mbar_fence_init();
  }
  __syncthreads();
  Ctl ctl{&abort_flag, err, timeout_ns};
  wait_or_abort(ctl, b, 0, ROLE_SELFTEST);
  __syncthreads();
}

template <bool kBF16, bool kD64, bool kDrop>
cudaError_t launch_dd(const BwdParams &p, cudaStream_t s) {
  const bool mask = p.atten_mask != nullptr;
  if (p.deterministic)
    return mask ? launch_t<kBF16, true, true, kD64, kDrop, false>(p, s)
                : launch_t<kBF16, true, false, kD64, kDrop, false>(p, s);
  return mask ? launch_t<kBF16, false, true, kD64, kDrop, false>(p, s)
              : launch_t<kBF16, false, false, kD64, kDrop, false>(p, s);
}

template <bool kBF16>
cudaError_t launch_dt(const BwdParams &p, cudaStream_t s) {
  if (p.d == 64)
    return p.use_dropout ? launch_dd<kBF16, true, true>(p, s) : launch_dd<kBF16, true, false>(p, s);
  if (p.d == HD)
    return p.use_dropout ? launch_dd<kBF16, false, true>(p, s) : launch_dd<kBF16, false, false>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int32_t *err, long long timeout_ns, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
  return cudaGetLastError();
}

// Head dims 64 and 128 run as they are; 32 and 96 run zero-padded to 64 and
// 128 (bwd_sm103_pad.cu).
bool tcgen05_supported(fa_dtype dt, int head_dim) {
  return (head_dim == 32 || head_dim == 64 || head_dim == 96 || head_dim == HD) &&
         (dt == FA_DTYPE_BF16 || dt == FA_DTYPE_FP16);
}

cudaError_t launch_bwd_tcgen05(const BwdParams &p, fa_dtype dt, cudaStream_t s) {
  if (p.d != 64 && p.d != HD) return launch_bwd_tcgen05_pad(p, dt, s);
  if (dt == FA_DTYPE_BF16) return launch_dt<true>(p, s);
  if (dt == FA_DTYPE_FP16) return launch_dt<false>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fav
