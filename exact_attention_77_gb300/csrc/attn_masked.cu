// Masked forward and backward instances (sliding window and block map;
// attn_mask.cuh): one query tile per forward CTA, the one-CTA backward.
#include "attn_bwd.cuh"
#include "attn_fwd.cuh"

namespace attn {

cudaError_t launch_fwd_masked(const FwdParams& p, int d, cudaStream_t s) {
  if (d == 64) return launch_fwd_instance<64, 64, 1, false, 0, false, true>(p, s);
  if (d == 128) return launch_fwd_instance<128, 128, 1, false, 0, false, true>(p, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_masked(const BwdParams& p, int d, bool deterministic, cudaStream_t s, const LaunchEvents* ev) {
  if (d == 64)
    return deterministic ? launch_bwd_instance<64, false, true, true>(p, s, ev)
                         : launch_bwd_instance<64, false, false, true>(p, s, ev);
  if (d == 128)
    return deterministic ? launch_bwd_instance<128, false, true, true>(p, s, ev)
                         : launch_bwd_instance<128, false, false, true>(p, s, ev);
  return cudaErrorInvalidValue;
}

}  // namespace attn
