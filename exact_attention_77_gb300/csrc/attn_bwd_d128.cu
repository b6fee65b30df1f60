// Backward kernel instances for d_qk = d_v = 128.
#include "attn_bwd.cuh"

namespace attn {

cudaError_t launch_bwd_d128(const BwdParams& p, bool causal, bool deterministic, cudaStream_t s, const LaunchEvents* ev) {
  if (causal) return deterministic ? launch_bwd_instance<128, true, true>(p, s, ev) : launch_bwd_instance<128, true, false>(p, s, ev);
  return deterministic ? launch_bwd_instance<128, false, true>(p, s, ev) : launch_bwd_instance<128, false, false>(p, s, ev);
}

}  // namespace attn

#ifdef ATTN_TRACE
// Debug builds only: copy the phase-trace stamps to host memory.
extern "C" int attn_debug_trace_read(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, attn::g_attn_trace, bytes) == cudaSuccess ? 0 : 5;
}
#endif
