// Backward kernel instances for d_qk = 192, d_v = 128 (attn_bwd192.cuh),
// with one K/V head per query head or grouped-query heads.
#include "attn_bwd192.cuh"

namespace attn {

cudaError_t launch_bwd_d192(const BwdParams& p, bool causal, bool deterministic, bool gqa, cudaStream_t s,
                            const LaunchEvents* ev) {
  if (gqa) {
    if (causal)
      return deterministic ? launch_bwd192_instance<true, true, true>(p, s, ev)
                           : launch_bwd192_instance<true, false, true>(p, s, ev);
    return deterministic ? launch_bwd192_instance<false, true, true>(p, s, ev)
                         : launch_bwd192_instance<false, false, true>(p, s, ev);
  }
  if (causal)
    return deterministic ? launch_bwd192_instance<true, true, false>(p, s, ev)
                         : launch_bwd192_instance<true, false, false>(p, s, ev);
  return deterministic ? launch_bwd192_instance<false, true, false>(p, s, ev)
                       : launch_bwd192_instance<false, false, false>(p, s, ev);
}

}  // namespace attn

#ifdef ATTN_TRACE
// Debug builds only: the phase-trace stamps of this translation unit's kernels.
extern "C" int attn_debug_trace_read_d192(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, attn::g_attn_trace, bytes) == cudaSuccess ? 0 : 5;
}
#endif
