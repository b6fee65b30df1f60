// Probes: element-wise accuracy of the exponential paths used by the forward
// kernel (to reproduce "FlashAttention-4 ...", Table 2, on this GPU),
// throughput of the hardware unit against the FMA-pipe polynomial, and a
// self-test of the bounded pipeline wait.
#include "kernels.h"
#include "sm103.cuh"

namespace attn {

// Degree-4 and degree-5 fits (p(0) = 1, minimax relative error on [0, 1)),
// printed by exp2_fit.py; the cubic lives in sm103.cuh with the forward kernel.
__device__ __forceinline__ float ex2_poly_deg(float x, int deg) {
  x = fmaxf(x, -127.0f);
  const float t = __fadd_rd(x, 12582912.0f);
  const float f = x - (t - 12582912.0f);
  float p;
  if (deg == 4) {
    p = fmaf(fmaf(fmaf(fmaf(0.0134266853f, f, 0.0522424725f), f, 0.241280206f), f, 0.693044845f), f, 1.0f);
  } else {
    p = fmaf(fmaf(fmaf(fmaf(fmaf(0.00186713019f, f, 0.00901703006f), f, 0.0557999133f), f, 0.24016445f), f,
                  0.693151312f),
             f, 1.0f);
  }
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

__device__ __forceinline__ float exp2_by(float x, int method) {
  if (method == 0) return ex2_mufu(x);
  if (method == 3) return ex2_poly3(x);
  return ex2_poly_deg(x, method);
}

__global__ void exp2_probe_kernel(const float* __restrict__ x, float* __restrict__ out, int n, int method) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = exp2_by(x[i], method);
}

template <int METHOD>
__global__ void __launch_bounds__(256) exp2_throughput_kernel(float* sink, int iters) {
  // eight independent chains per thread keep the unit busy; the argument is
  // kept in [-1, 0] so neither path saturates
  float v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = -0.001f * (threadIdx.x + k);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = exp2_by(v[k] - 1.0f, METHOD) - 1.0f;
  }
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) acc += v[k];
  sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

// One thread waits on an mbarrier that nothing arrives on, through the same
// bounded wait the attention kernels use; it must give up after timeout_ns,
// record ATTN_ERR_TIMEOUT (where = 900) and return.
__global__ void wait_selftest_kernel(DeviceStatus* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    const uint32_t bar = smem_u32(&bar_storage);
    mbar_init(bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    const WaitCtl ctl{&abort_flag, status, timeout_ns};
    mbar_wait(bar, 0, ctl, 900);
  }
}

cudaError_t launch_wait_selftest(DeviceStatus* status, unsigned long long timeout_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_exp2_probe(const float* x, float* out, int n, int method, cudaStream_t s) {
  const int blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
  exp2_probe_kernel<<<blocks, 256, 0, s>>>(x, out, n, method);
  return cudaGetLastError();
}

cudaError_t launch_exp2_throughput(float* sink, int blocks, int iters, int method, cudaStream_t s) {
  switch (method) {
    case 0: exp2_throughput_kernel<0><<<blocks, 256, 0, s>>>(sink, iters); break;
    case 3: exp2_throughput_kernel<3><<<blocks, 256, 0, s>>>(sink, iters); break;
    case 4: exp2_throughput_kernel<4><<<blocks, 256, 0, s>>>(sink, iters); break;
    default: exp2_throughput_kernel<5><<<blocks, 256, 0, s>>>(sink, iters); break;
  }
  return cudaGetLastError();
}

}  // namespace attn
