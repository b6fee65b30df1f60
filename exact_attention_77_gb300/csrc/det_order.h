// Order of the dQ additions in the deterministic backward ("FlashAttention-4:
// Algorithm and Kernel Pipelining Co-Design for Asymmetric Hardware Scaling",
// abstract and Figures 7-8: a fixed order of the key tiles' contributions to
// each dQ tile makes the FP32 sums, and so dQ, bit-identical from run to run).
//
// Host and device share this file: the kernels walk and wait by it, and the
// C ABI's attn_bwd_det_plan writes the same plan out for the host-side tests.
#pragma once

#ifdef __CUDACC__
#define ATTN_HD __host__ __device__ __forceinline__
#else
#define ATTN_HD inline
#endif

namespace attn {

// The (head, key tile) work units in order: key-tile-major inside groups of
// ``group`` heads (the heads of a group interleaved), key tiles ascending, or
// from the last down with ``desc``.  Unit u is the jj-th of its head; its key
// tile is j = jj (or n - 1 - jj).  Every dQ tile takes its key-tile
// contributions in an order derived from this one, so a unit waits only on
// units of its own head that come earlier: with CTAs launched (or persistent
// CTAs taking units) in increasing order, the waits always point backwards.
struct DetUnit {
  int j, bh;   // key tile and head
  int jj;      // position among its head's units
  int g;       // heads in its group
  int h0;      // first head of its group
};

ATTN_HD DetUnit det_unit_of(int u, int n_heads, int n, int group, int desc) {
  DetUnit d;
  const int grp = u / (group * n);
  d.h0 = grp * group;
  d.g = group < n_heads - d.h0 ? group : n_heads - d.h0;  // the last group may be smaller
  const int rem = u - d.h0 * n;
  d.jj = rem / d.g;
  d.bh = d.h0 + (rem - d.jj * d.g);
  d.j = desc ? n - 1 - d.jj : d.jj;
  return d;
}

// Position of key tile j among the contributions to query tile i when every
// unit walks the query tiles in the same order (the ticket value at which its
// addition may go ahead): ascending j, or descending with desc (causal: only
// the tiles i >= j contribute).
ATTN_HD int det_rank(int i, int j, int n, bool causal, int desc) { return desc ? (causal ? i : n - 1) - j : j; }

// Rotated walk (non-causal, persistent CTAs that are all resident at once).
// The CTAs hold units [r G, r G + G) in round r, so a head's units
// jj_lo .. jj_hi of one round run side by side.  If they all walked the query
// tiles in the same order, the additions to a tile would queue one behind the
// other at the same step and the last unit of the round would start its
// additions about (jj_hi - jj_lo) hand-overs late.  Instead unit jj starts at
// query tile (n - 1 - sigma jj) mod n and walks down, wrapping: at every step
// the round's units of a head are at different tiles, and a tile's previous
// addition in the round was made sigma steps earlier.  A tile takes the
// additions of earlier rounds first (ascending jj), then the round's in the
// order of their visiting step; sigma is the largest stride (at most 3) that
// keeps those steps distinct (sigma (L - 1) < n for L units of a head in a
// round), 0 when no round holds two units of one head (then this is the
// plain walk and order above).
struct DetRot {
  int jj, jj_lo, jj_hi, sigma;
};

ATTN_HD DetRot det_rot(int u, int n_ctas, int n_heads, int n, int group, int desc) {
  const DetUnit d = det_unit_of(u, n_heads, n, group, desc);
  DetRot r;
  r.jj = d.jj;
  // this head's units are u(k) = h0 n + k g + (bh - h0); round u / n_ctas holds
  // those with lo <= k g <= hi
  const int base = d.h0 * n + (d.bh - d.h0);
  const int rd = u / n_ctas;
  const int lo = rd * n_ctas - base;
  const int hi = rd * n_ctas + n_ctas - 1 - base;  // >= jj g >= 0
  r.jj_lo = lo <= 0 ? 0 : (lo + d.g - 1) / d.g;
  r.jj_hi = hi / d.g < n - 1 ? hi / d.g : n - 1;
  int lmax = (n_ctas + d.g - 1) / d.g;  // most units of one head in a round
  if (lmax > n) lmax = n;
  if (lmax <= 1) {
    r.sigma = 0;
  } else {
    const int s = (n - 1) / (lmax - 1);
    r.sigma = s < 3 ? s : 3;
  }
  return r;
}

// Step at which unit jj visits query tile i (0 .. n-1).
ATTN_HD int det_rot_step(int i, int jj, int n, int sigma) {
  const int s = (n - 1 - i - sigma * jj) % n;
  return s < 0 ? s + n : s;
}

// First query tile of unit jj's walk (its step 0); the walk then goes down by
// one, from 0 back to n - 1.
ATTN_HD int det_rot_first(int jj, int n, int sigma) {
  const int i = (n - 1 - sigma * jj) % n;
  return i < 0 ? i + n : i;
}

// Ticket value at which the unit's addition to query tile i may go ahead:
// jj_lo plus the round's units k that visit tile i before this unit's step s.
// Unit k visits it at step (s + sigma (jj - k)) mod n, which is below s for
// k = jj - d exactly when the sum wraps (d >= (n - s) / sigma) and for
// k = jj + e exactly when it does not (e <= s / sigma).
ATTN_HD int det_rot_rank(int i, const DetRot& r, int n) {
  if (r.sigma == 0) return r.jj_lo;  // one unit of the head in the round
  const int s = det_rot_step(i, r.jj, n, r.sigma);
  const int d_min = (n - s + r.sigma - 1) / r.sigma;  // >= 1
  const int below = r.jj - r.jj_lo - d_min + 1;
  const int above = s / r.sigma;
  return r.jj_lo + (below > 0 ? below : 0) + (above < r.jj_hi - r.jj ? above : r.jj_hi - r.jj);
}

}  // namespace attn

#undef ATTN_HD
