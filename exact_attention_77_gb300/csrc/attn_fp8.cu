// FP8 forward: the quantiser that turns bf16 Q, K, V into e4m3 codes with
// block scales, and the e4m3 instances of the forward kernel.
//
// "FlashAttention 3 and 4: When the Bottleneck Moves", section 2.2: each
// block of values gets its own scale, and Q and K are multiplied by the same
// fixed random rotation R before quantising, which spreads outlying
// coordinates while (QR)(KR)^T = Q K^T keeps every score.
//
// Here R = D H / sqrt(d) with H the Sylvester-Hadamard matrix and D a
// diagonal of caller-chosen signs.  The quantiser applies sqrt(d) R = D H
// (a sign flip, then the fast Walsh-Hadamard transform, exact in FP32 for
// bf16 inputs whose magnitudes span less than 2^16 within a row), and the
// forward divides the scores by d (a power of two).  Blocks: the 128-row
// tiles of Q and of K, and all of V of one (b, h).  A block's scale is the
// smallest power of two s with max|x| <= 448 s; values are stored as
// e4m3(x / s), rounded to nearest even.
#include <cuda_bf16.h>
#include <math.h>

#include "attn_fwd.cuh"

namespace attn {

namespace {

constexpr int kQuantRowsPerWarp = 16;  // 8 warps x 16 rows = one 128-row tile

// Smallest power-of-two exponent k with amax <= 448 * 2^k (0 for amax = 0):
// with amax = f 2^e, f in [0.5, 1), and 448 = 0.875 2^9.
__device__ __forceinline__ int pow2_scale_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  int e;
  const float f = frexpf(amax, &e);
  return f <= 0.875f ? e - 9 : e - 8;
}

// max |V| over one 128-row tile, folded into vmax[bh] (non-negative floats
// order like their bit patterns).
__global__ void __launch_bounds__(256) v_amax_kernel(const QuantParams p) {
  const int tile = blockIdx.x % p.n_tiles, bh = blockIdx.x / p.n_tiles;
  const int rows = min(kTile, p.N - tile * kTile);
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.v) +
                                                    ((size_t)bh * p.N + (size_t)tile * kTile) * 128);
  float amax = 0.f;
  for (int i = threadIdx.x; i < rows * 16; i += 256) {  // 16 chunks of 8 values per row
    const uint4 u = src[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    atomicMax(p.vmax + bh, __float_as_uint(amax));
  }
}

// One CTA per (bh, tile) and tensor (blockIdx.y): 0 = Q, 1 = K (rotated,
// per-tile scale), 2 = V (per-head scale from vmax).  Lane l of a warp holds
// coordinates 4l .. 4l+3 of its rows.
__global__ void __launch_bounds__(256) quantize_kernel(const QuantParams p) {
  const int tile = blockIdx.x % p.n_tiles, bh = blockIdx.x / p.n_tiles, which = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const void* src_base = which == 0 ? p.q : which == 1 ? p.k : p.v;
  uint8_t* dst_base = which == 0 ? p.q8 : which == 1 ? p.k8 : p.v8;
  const size_t row0 = (size_t)bh * p.N + (size_t)tile * kTile;
  const int rows = min(kTile, p.N - tile * kTile);
  float x[kQuantRowsPerWarp][4];
  float amax = 0.f;
  // (selected without indexing the parameter array, which would copy it to local memory)
  const uint32_t sword = lane < 8 ? p.signs[0] : lane < 16 ? p.signs[1] : lane < 24 ? p.signs[2] : p.signs[3];
  const uint32_t sbits = (sword >> ((lane & 7) * 4)) & 0xFu;
#pragma unroll
  for (int i = 0; i < kQuantRowsPerWarp; ++i) {
    const int r = warp * kQuantRowsPerWarp + i;
    uint2 u = make_uint2(0u, 0u);
    if (r < rows)
      u = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(src_base) + (row0 + r) * 128 + lane * 4);
    x[i][0] = __uint_as_float(u.x << 16);
    x[i][1] = __uint_as_float(u.x & 0xFFFF0000u);
    x[i][2] = __uint_as_float(u.y << 16);
    x[i][3] = __uint_as_float(u.y & 0xFFFF0000u);
    if (which < 2) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if ((sbits >> c) & 1u) x[i][c] = -x[i][c];
      // Walsh-Hadamard butterflies: index bits 0-1 inside the lane, bits
      // 2-6 across lanes (partner lane = lane ^ 2^t)
      float a0 = x[i][0] + x[i][1], a1 = x[i][0] - x[i][1];
      float a2 = x[i][2] + x[i][3], a3 = x[i][2] - x[i][3];
      x[i][0] = a0 + a2;
      x[i][2] = a0 - a2;
      x[i][1] = a1 + a3;
      x[i][3] = a1 - a3;
#pragma unroll
      for (int t = 1; t < 32; t <<= 1) {
        const bool upper = (lane & t) != 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float o = __shfl_xor_sync(0xffffffffu, x[i][c], t);
          x[i][c] = upper ? o - x[i][c] : x[i][c] + o;
        }
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) amax = fmaxf(amax, fabsf(x[i][c]));
  }
  __shared__ float red[8];
  if (which < 2) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  } else {
    amax = __uint_as_float(p.vmax[bh]);
  }
  const int k = pow2_scale_exp(amax);
  const float inv = ldexpf(1.f, -k);
  if (threadIdx.x == 0) {
    const float sc = ldexpf(1.f, k);
    if (which == 0) p.sq[(size_t)bh * p.n_tiles + tile] = sc;
    else if (which == 1) p.sk[(size_t)bh * p.n_tiles + tile] = sc;
    else if (tile == 0) p.sv[bh] = sc;
  }
#pragma unroll
  for (int i = 0; i < kQuantRowsPerWarp; ++i) {
    const int r = warp * kQuantRowsPerWarp + i;
    if (r < rows)
      *reinterpret_cast<uint32_t*>(dst_base + (row0 + r) * 128 + lane * 4) =
          pack_e4m3x4(x[i][0] * inv, x[i][1] * inv, x[i][2] * inv, x[i][3] * inv);
  }
}

}  // namespace

cudaError_t launch_fp8_quantize(const QuantParams& p, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(p.vmax, 0, (size_t)p.BH * sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)p.n_tiles * (unsigned)p.BH;
  v_amax_kernel<<<blocks, 256, 0, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  quantize_kernel<<<dim3(blocks, 3), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const FwdParams& p, bool causal, cudaStream_t s) {
  return causal ? launch_fwd_instance<128, 128, 2, true, 0, true>(p, s)
                : launch_fwd_instance<128, 128, 2, false, 0, true>(p, s);
}

}  // namespace attn
