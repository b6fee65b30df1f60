// Backward kernel instances for d_qk = d_v = 64.
#include "attn_bwd.cuh"
#include "attn_bwd_persist.cuh"

namespace attn {

cudaError_t launch_bwd_d64(const BwdParams& p, bool causal, bool deterministic, cudaStream_t s, const LaunchEvents* ev) {
  if (causal) return deterministic ? launch_bwd_instance<64, true, true>(p, s, ev) : launch_bwd_instance<64, true, false>(p, s, ev);
  return deterministic ? launch_bwd_instance<64, false, true>(p, s, ev) : launch_bwd_instance<64, false, false>(p, s, ev);
}

}  // namespace attn
