// Backward kernel instances for d_qk = d_v = 128.
#include "attn_bwd2.cuh"
#include "attn_bwd_persist.cuh"

namespace attn {

template <bool CAUSAL, bool DET>
cudaError_t launch_bwd2_main(const BwdParams& p, cudaStream_t stream) {
  using L = Bwd2Layout;
  auto kernel = bwd2_kernel<CAUSAL, DET>;
  cudaError_t e = prepare_kernel((const void*)kernel, L::kSmemBytes, L::kLaunchRegs, nullptr);
  if (e != cudaSuccess) return e;
  const int n_pairs = (p.n_tiles + 1) / 2;
  kernel<<<p.BH * n_pairs * 2, L::kThreads, L::kSmemBytes, stream>>>(p);  // clusters of two (kernel attribute)
  return cudaGetLastError();
}

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
