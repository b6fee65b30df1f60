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

constexpr int kQuantWarps = 16;
constexpr int kQuantRowsPerWarp = kTile / kQuantWarps;  // 16 warps x 8 rows = one 128-row tile

// Smallest power-of-two exponent k with amax <= 448 * 2^k (0 for amax = 0):
// with amax = f 2^e, f in [0.5, 1), and 448 = 0.875 2^9.
__device__ __forceinline__ int pow2_scale_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  int e;
  const float f = frexpf(amax, &e);
  return f <= 0.875f ? e - 9 : e - 8;
}

// max |V| over one 128-row tile, folded into vmax[bh] (non-negative floats
// order like their bit patterns).  Each thread takes 8 of the tile's 2048
// 16-byte chunks, all loads in flight together.
__global__ void __launch_bounds__(256) v_amax_kernel(const QuantParams p) {
  const int tile = blockIdx.x % p.n_tiles, bh = blockIdx.x / p.n_tiles;
  const int rows = min(kTile, p.N - tile * kTile);
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.v) +
                                                    ((size_t)bh * p.N + (size_t)tile * kTile) * 128);
  uint4 u[8];
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int i = threadIdx.x + it * 256;  // 16 chunks of 8 values per row
    u[it] = i < rows * 16 ? src[i] : make_uint4(0u, 0u, 0u, 0u);
  }
  float amax = 0.f;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const uint32_t w[4] = {u[it].x, u[it].y, u[it].z, u[it].w};
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
// per-tile scale), 2 = V (per-head scale from vmax).  Four lanes share a row:
// lane l takes row 8 * warp + l / 4 and its coordinates 32 (l % 4) .. + 31.
// The Walsh-Hadamard butterflies over index bits 0-4 run in registers, those
// over bits 5 and 6 exchange with lanes l ^ 1 and l ^ 2.
__global__ void __launch_bounds__(kQuantWarps * 32, 2) quantize_kernel(const QuantParams p) {
  const int tile = blockIdx.x % p.n_tiles, bh = blockIdx.x / p.n_tiles, which = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = lane & 3;
  const int r = warp * 8 + (lane >> 2);
  const void* src_base = which == 0 ? p.q : which == 1 ? p.k : p.v;
  uint8_t* dst_base = which == 0 ? p.q8 : which == 1 ? p.k8 : p.v8;
  const size_t row0 = (size_t)bh * p.N + (size_t)tile * kTile;
  const int rows = min(kTile, p.N - tile * kTile);
  const bool live = r < rows;
  float x[32];
  {
    uint4 u[4] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u),
                  make_uint4(0u, 0u, 0u, 0u)};
    if (live) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src_base) +
                                                        (row0 + r) * 128 + quarter * 32);
#pragma unroll
      for (int c = 0; c < 4; ++c) u[c] = src[c];
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[8 * c + 2 * j] = __uint_as_float(w[j] << 16);
        x[8 * c + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
  if (which < 2) {
    // (selected without indexing the parameter array, which would copy it to local memory)
    const uint32_t sw = quarter == 0 ? p.signs[0] : quarter == 1 ? p.signs[1] : quarter == 2 ? p.signs[2] : p.signs[3];
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if ((sw >> e) & 1u) x[e] = -x[e];
#pragma unroll
    for (int h = 1; h < 32; h <<= 1)
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if ((e & h) == 0) {
          const float a = x[e], b = x[e + h];
          x[e] = a + b;
          x[e + h] = a - b;
        }
#pragma unroll
    for (int t = 1; t < 4; t <<= 1) {
      const bool upper = (lane & t) != 0;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, x[e], t);
        x[e] = upper ? o - x[e] : x[e] + o;
      }
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(x[e]));
  __shared__ float red[kQuantWarps];
  if (which < 2) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
    for (int i = 1; i < kQuantWarps; ++i) amax = fmaxf(amax, red[i]);
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
  if (live) {
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      w[j] = pack_e4m3x4(x[4 * j] * inv, x[4 * j + 1] * inv, x[4 * j + 2] * inv, x[4 * j + 3] * inv);
    uint4* dst = reinterpret_cast<uint4*>(dst_base + (row0 + r) * 128 + quarter * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
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
  quantize_kernel<<<dim3(blocks, 3), kQuantWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const FwdParams& p, bool causal, cudaStream_t s) {
  return causal ? launch_fwd_instance<128, 128, 2, true, 0, true>(p, s)
                : launch_fwd_instance<128, 128, 2, false, 0, true>(p, s);
}

}  // namespace attn
