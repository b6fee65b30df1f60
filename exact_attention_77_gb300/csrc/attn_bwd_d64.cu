// Backward kernel instances for d_qk = d_v = 64.
#include "attn_bwd.cuh"

namespace attn {

cudaError_t launch_bwd_d64(const BwdParams& p, bool causal, bool deterministic, cudaStream_t s) {
  if (causal) return deterministic ? launch_bwd_instance<64, true, true>(p, s) : launch_bwd_instance<64, true, false>(p, s);
  return deterministic ? launch_bwd_instance<64, false, true>(p, s) : launch_bwd_instance<64, false, false>(p, s);
}

}  // namespace attn
