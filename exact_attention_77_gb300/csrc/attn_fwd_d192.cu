// Forward kernel instances for d_qk = 192, d_v = 128 (two query tiles per CTA).
#include "attn_fwd.cuh"

namespace attn {

cudaError_t launch_fwd_d192(const FwdParams& p, bool causal, int /*nqt*/, int poly, cudaStream_t s) {
  if (causal) return poly ? launch_fwd_instance<192, 128, 2, true, kPolyCols>(p, s) : launch_fwd_instance<192, 128, 2, true, 0>(p, s);
  return poly ? launch_fwd_instance<192, 128, 2, false, kPolyCols>(p, s) : launch_fwd_instance<192, 128, 2, false, 0>(p, s);
}

}  // namespace attn
