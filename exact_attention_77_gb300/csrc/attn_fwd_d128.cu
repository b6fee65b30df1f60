// Forward kernel instances for d_qk = d_v = 128.
#include "attn_fwd.cuh"

namespace attn {

cudaError_t launch_fwd_d128(const FwdParams& p, bool causal, int nqt, int poly, cudaStream_t s) {
  if (nqt == 1) {
    if (causal) return poly ? launch_fwd_instance<128, 128, 1, true, kPolyCols>(p, s) : launch_fwd_instance<128, 128, 1, true, 0>(p, s);
    return poly ? launch_fwd_instance<128, 128, 1, false, kPolyCols>(p, s) : launch_fwd_instance<128, 128, 1, false, 0>(p, s);
  }
  if (causal) return poly ? launch_fwd_instance<128, 128, 2, true, kPolyCols>(p, s) : launch_fwd_instance<128, 128, 2, true, 0>(p, s);
  return poly ? launch_fwd_instance<128, 128, 2, false, kPolyCols>(p, s) : launch_fwd_instance<128, 128, 2, false, 0>(p, s);
}

}  // namespace attn

#ifdef ATTN_TRACE
// Debug builds only: copy the forward's phase-trace stamps to host memory.
extern "C" int attn_debug_trace_read_fwd(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, attn::g_attn_trace, bytes) == cudaSuccess ? 0 : 5;
}
#endif
