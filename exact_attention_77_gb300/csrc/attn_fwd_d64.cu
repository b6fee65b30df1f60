// Forward kernel instances for d_qk = d_v = 64.
#include "attn_fwd.cuh"

namespace attn {

cudaError_t launch_fwd_d64(const FwdParams& p, bool causal, int nqt, int poly, cudaStream_t s) {
  if (nqt == 1) {
    if (causal) return poly ? launch_fwd_instance<64, 64, 1, true, kPolyCols>(p, s) : launch_fwd_instance<64, 64, 1, true, 0>(p, s);
    return poly ? launch_fwd_instance<64, 64, 1, false, kPolyCols>(p, s) : launch_fwd_instance<64, 64, 1, false, 0>(p, s);
  }
  if (causal) return poly ? launch_fwd_instance<64, 64, 2, true, kPolyCols>(p, s) : launch_fwd_instance<64, 64, 2, true, 0>(p, s);
  return poly ? launch_fwd_instance<64, 64, 2, false, kPolyCols>(p, s) : launch_fwd_instance<64, 64, 2, false, 0>(p, s);
}

}  // namespace attn
