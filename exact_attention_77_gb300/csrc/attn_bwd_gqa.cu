// Grouped-query backward instances (one-CTA kernel, attn_bwd.cuh): a CTA owns
// a key tile of one K/V head and walks the query tiles of every query head
// sharing it, so dK and dV are summed over the group in tensor memory.
#include "attn_bwd.cuh"

namespace attn {

cudaError_t launch_bwd_gqa(const BwdParams& p, int d, bool causal, bool deterministic, cudaStream_t s,
                           const LaunchEvents* ev) {
  if (d == 64) {
    if (causal)
      return deterministic ? launch_bwd_instance<64, true, true, false, true>(p, s, ev)
                           : launch_bwd_instance<64, true, false, false, true>(p, s, ev);
    return deterministic ? launch_bwd_instance<64, false, true, false, true>(p, s, ev)
                         : launch_bwd_instance<64, false, false, false, true>(p, s, ev);
  }
  if (d == 128) {
    if (causal)
      return deterministic ? launch_bwd_instance<128, true, true, false, true>(p, s, ev)
                           : launch_bwd_instance<128, true, false, false, true>(p, s, ev);
    return deterministic ? launch_bwd_instance<128, false, true, false, true>(p, s, ev)
                         : launch_bwd_instance<128, false, false, false, true>(p, s, ev);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
