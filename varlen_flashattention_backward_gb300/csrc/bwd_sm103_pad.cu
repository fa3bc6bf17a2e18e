// The tcgen05 backward at head dims below the compute width (32 runs as
// 64, 96 as 128; bwd_sm103.cuh, kPad): its own translation unit, so that
// these instantiations compile beside the others.

#include "bwd_sm103.cuh"

namespace fav {
namespace {

template <bool kBF16, bool kD64, bool kDrop>
cudaError_t launch_dd(const BwdParams &p, cudaStream_t s) {
  const bool mask = p.atten_mask != nullptr;
  if (p.deterministic)
    return mask ? launch_t<kBF16, true, true, kD64, kDrop, true>(p, s)
                : launch_t<kBF16, true, false, kD64, kDrop, true>(p, s);
  return mask ? launch_t<kBF16, false, true, kD64, kDrop, true>(p, s)
              : launch_t<kBF16, false, false, kD64, kDrop, true>(p, s);
}

template <bool kBF16>
cudaError_t launch_dt(const BwdParams &p, cudaStream_t s) {
  if (p.d < 64)
    return p.use_dropout ? launch_dd<kBF16, true, true>(p, s) : launch_dd<kBF16, true, false>(p, s);
  if (p.d < HD)
    return p.use_dropout ? launch_dd<kBF16, false, true>(p, s) : launch_dd<kBF16, false, false>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_bwd_tcgen05_pad(const BwdParams &p, fa_dtype dt, cudaStream_t s) {
  if (dt == FA_DTYPE_BF16) return launch_dt<true>(p, s);
  if (dt == FA_DTYPE_FP16) return launch_dt<false>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fav
