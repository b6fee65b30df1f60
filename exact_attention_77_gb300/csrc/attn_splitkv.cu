// Split-KV forward and the merge of partial results.
//
// "Attention at Scale -- From FlashAttention to FlashAttention-4": the
// FlashInfer section splits attention over a key set into independent parts
// combined by an associative merge operator, and the "Sequence-Aware Split
// Heuristic" section splits the key sequence across thread blocks when too
// few (batch, head) pairs exist to occupy the GPU, paying one reduction pass.
// Each part s over keys K_s yields its normalised output O_s and its
// log-sum-exp LSE_s; the merge is
//     LSE = log sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
// The forward kernel (attn_fwd.cuh, SPLIT instance) computes the parts; the
// kernel below merges them, one warp per query row.
#include <cuda_bf16.h>
#include <math.h>

#include <type_traits>

#include "attn_fwd.cuh"

namespace attn {

// o_parts [n_parts, rows, DV], lse_parts [n_parts, rows] (rows = BH * N).
// W warps (1, 2, 4 or 8) share a row, warp `sub` taking parts sub, sub + W,
// ..., four at a time so that their loads are in flight together; each lane
// owns DV / 32 adjacent columns.  A part with LSE = -inf drops out; a row
// whose parts are all empty gets O = 0 and LSE = -inf.
template <int DV>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ o_parts,
                                                    const float* __restrict__ lse_parts, int n_parts,
                                                    __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                    long long rows, int W) {
  constexpr int C = DV / 32;
  using Vec = typename std::conditional<C == 4, float4, float2>::type;
  __shared__ float s_m[8], s_z[8];
  __shared__ __align__(16) float s_acc[8][DV];
  // launched as a programmatic dependent of the split forward: wait for its
  // completion and memory (returns at once for an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = warp & (W - 1);
  const long long row = (long long)blockIdx.x * (8 / W) + warp / W;
  const bool live = row < rows;
  float m = -INFINITY;
  if (live)
    for (int s = sub * 32 + lane; s < n_parts; s += 32 * W) m = fmaxf(m, lse_parts[(size_t)s * rows + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (W > 1) {
    if (lane == 0) s_m[warp] = m;
    __syncthreads();
    for (int i = 0; i < W; ++i) m = fmaxf(m, s_m[warp - sub + i]);
  }
  float acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.f;
  float z = 0.f;
  auto part = [&](int s) { return o_parts + ((size_t)s * rows + row) * DV + lane * C; };
  auto add = [&](float l, const Vec& x) {
    const float w = expf(l - m);
    z += w;
    const float* xf = reinterpret_cast<const float*>(&x);
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = fmaf(w, xf[c], acc[c]);
  };
  if (live && m != -INFINITY) {
    int s = sub;
    for (; s + 3 * W < n_parts; s += 4 * W) {
      float l[4];
      Vec x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        l[u] = lse_parts[(size_t)(s + u * W) * rows + row];
        x[u] = *reinterpret_cast<const Vec*>(part(s + u * W));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) add(l[u], x[u]);
    }
    for (; s < n_parts; s += W) add(lse_parts[(size_t)s * rows + row], *reinterpret_cast<const Vec*>(part(s)));
  }
  if (W > 1) {
#pragma unroll
    for (int c = 0; c < C; ++c) s_acc[warp][lane * C + c] = acc[c];
    if (lane == 0) s_z[warp] = z;
    __syncthreads();
    if (sub != 0) return;
    for (int i = 1; i < W; ++i) {
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c] += s_acc[warp + i][lane * C + c];
      z += s_z[warp + i];
    }
  }
  if (!live) return;
  const float inv = z > 0.f ? 1.f / z : 0.f;
  __nv_bfloat16* dst = o + (size_t)row * DV + lane * C;
  if constexpr (C == 4) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(dst) = u;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0) lse[row] = z > 0.f ? m + logf(z) : -INFINITY;
}

cudaError_t launch_merge(const float* o_parts, const float* lse_parts, int n_parts, void* o, float* lse, int BH,
                         int N, int d_v, cudaStream_t s, bool pdl) {
  const long long rows = (long long)BH * N;
  const int W = n_parts >= 8 ? 8 : n_parts >= 4 ? 4 : n_parts >= 2 ? 2 : 1;
  const long long blocks = (rows + 8 / W - 1) / (8 / W);
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  auto* out = static_cast<__nv_bfloat16*>(o);
  void (*kernel)(const float*, const float*, int, __nv_bfloat16*, float*, long long, int);
  if (d_v == 128)
    kernel = merge_kernel<128>;
  else if (d_v == 64)
    kernel = merge_kernel<64>;
  else
    return cudaErrorInvalidValue;
  if (pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, o_parts, lse_parts, n_parts, out, lse, rows, W) == cudaSuccess)
      return cudaSuccess;
    (void)cudaGetLastError();  // not available here: ordinary launch
  }
  kernel<<<(unsigned)blocks, 256, 0, s>>>(o_parts, lse_parts, n_parts, out, lse, rows, W);
  return cudaGetLastError();
}

cudaError_t launch_fwd_split(const FwdParams& p, int d_qk, int nqt, cudaStream_t s) {
  if (d_qk == 64) return nqt == 1 ? launch_fwd_split_instance<64, 64, 1>(p, s) : launch_fwd_split_instance<64, 64, 2>(p, s);
  if (d_qk == 128)
    return nqt == 1 ? launch_fwd_split_instance<128, 128, 1>(p, s) : launch_fwd_split_instance<128, 128, 2>(p, s);
  if (d_qk == 192 && nqt == 2) return launch_fwd_split_instance<192, 128, 2>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace attn
