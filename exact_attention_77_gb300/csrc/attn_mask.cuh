// Sliding-window and block masks ("Attention at Scale -- From FlashAttention
// to FlashAttention-4", FlexAttention section: a boolean mask over (query,
// key) pairs, and a precomputed block map that lets the kernel skip blocks
// holding no visible pair).  Query i sees key j when
// i - left <= j <= i + right (left / right < 0: unbounded), j < N, and the
// block map is non-zero for (i / 128, j / 128).
#pragma once

#include "kernels.h"

namespace attn {

// Tile pair (qt, kt) holds at least one visible pair: over the tiles'
// rectangle j - i takes every value in [k0 - q1, k1 - q0], which must meet
// [-left, right]; then the block map.
__device__ __forceinline__ bool mask_tile_visible(const MaskSpec& m, int qt, int kt) {
  const int q0 = qt * 128, q1 = min(q0 + 127, m.N - 1);
  const int k0 = kt * 128, k1 = min(k0 + 127, m.N - 1);
  if (m.left >= 0 && k1 - q0 < -m.left) return false;
  if (m.right >= 0 && k0 - q1 > m.right) return false;
  if (m.block != nullptr && m.block[(size_t)qt * m.n_tiles + kt] == 0) return false;
  return true;
}

// Every live query row of tile qt sees every key of tile kt (no per-pair
// mask needed; the block map is already known to be non-zero).
__device__ __forceinline__ bool mask_tile_full(const MaskSpec& m, int qt, int kt) {
  const int q0 = qt * 128, q1 = min(q0 + 127, m.N - 1);
  const int k0 = kt * 128, k1 = k0 + 127;
  if (k1 >= m.N) return false;
  if (m.left >= 0 && k0 - q1 < -m.left) return false;
  if (m.right >= 0 && k1 - q0 > m.right) return false;
  return true;
}

// Per pair (the block map is applied per tile by the callers).
__device__ __forceinline__ bool mask_pair_visible(const MaskSpec& m, int i, int j) {
  return j < m.N && (m.left < 0 || j >= i - m.left) && (m.right < 0 || j <= i + m.right);
}

// Next visible key tile of query tile qt after kt (n_tiles if none).
__device__ __forceinline__ int mask_next_key_tile(const MaskSpec& m, int qt, int kt) {
  for (int k = kt + 1; k < m.n_tiles; ++k)
    if (mask_tile_visible(m, qt, k)) return k;
  return m.n_tiles;
}

// Next visible query tile of key tile kt below qt (-1 if none).
__device__ __forceinline__ int mask_prev_query_tile(const MaskSpec& m, int kt, int qt) {
  for (int q = qt - 1; q >= 0; --q)
    if (mask_tile_visible(m, q, kt)) return q;
  return -1;
}

}  // namespace attn
