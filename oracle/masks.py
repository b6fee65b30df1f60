"""Attention under a sliding-window mask and a block mask, forward and backward.

Test infrastructure only (see the package docstring).

Source: "Attention at Scale -- From FlashAttention to FlashAttention-4",
FlexAttention section: attention variants such as sliding windows are
expressed as a boolean mask over (query, key) pairs, and a precomputed
block-level sparsity map lets the kernel skip blocks that are entirely
masked.  The masked attention itself is the definition of section "The
Problem" with hidden scores set to -inf before the softmax.

Readings taken where the page is silent (one line of DESIGN each):
* Window: query i sees key j when i - left <= j <= i + right; left or right
  = -1 means unbounded on that side (left = -1, right = 0 is the causal
  mask).
* Block mask: a 0/1 map over (128-row query tile, 128-key tile) pairs shared
  by every (b, h); 0 hides every pair of that tile pair.  The mask is the
  conjunction of the window and the block map.
* A query row with no visible key gets O = 0, LSE = -inf and zero gradients.
"""
from __future__ import annotations

import numpy as np

TILE = 128


def mask_matrix(n_q: int, n_k: int, left: int = -1, right: int = -1, block=None, tile: int = TILE) -> np.ndarray:
    """Boolean [n_q, n_k]: True where query i sees key j."""
    i = np.arange(n_q)[:, None]
    j = np.arange(n_k)[None, :]
    m = np.ones((n_q, n_k), dtype=bool)
    if left >= 0:
        m &= j >= i - left
    if right >= 0:
        m &= j <= i + right
    if block is not None:
        block = np.asarray(block, dtype=bool)
        m &= block[(i // tile), (j // tile)]
    return m


def forward_head(q, k, v, scale: float, mask):
    """O = softmax(scale q k^T with -inf where ~mask) v and LSE, by the plain
    two-pass definition; rows without a visible key: O = 0, LSE = -inf."""
    s = np.where(mask, scale * (q @ k.T), -np.inf)
    mx = s.max(axis=1)
    live = np.isfinite(mx)
    e = np.where(mask, np.exp(s - np.where(live, mx, 0.0)[:, None]), 0.0)
    l = e.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        p = np.where(live[:, None], e / np.where(live, l, 1.0)[:, None], 0.0)
        lse = np.where(live, mx + np.log(np.where(live, l, 1.0)), -np.inf)
    return p @ v, lse


def backward_head(q, k, v, do, scale: float, mask):
    """dQ, dK, dV of sum(O * dO) by the chain rule through the masked softmax:
    dV = P^T dO, dP = dO V^T, dS = P o (dP - rowsum(P o dP)), dQ = scale dS K,
    dK = scale dS^T Q, with P = 0 on hidden pairs and on empty rows."""
    s = np.where(mask, scale * (q @ k.T), -np.inf)
    mx = s.max(axis=1)
    live = np.isfinite(mx)
    e = np.where(mask, np.exp(s - np.where(live, mx, 0.0)[:, None]), 0.0)
    l = e.sum(axis=1)
    p = np.where(live[:, None], e / np.where(live, l, 1.0)[:, None], 0.0)
    dv = p.T @ do
    dp = do @ v.T
    ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    return scale * ds @ k, scale * ds.T @ q, dv


def forward(q, k, v, scale: float, mask):
    """forward_head over [B, H, N, d] arrays with one mask for every head."""
    B, H = q.shape[:2]
    o = np.empty(q.shape[:3] + (v.shape[-1],))
    lse = np.empty(q.shape[:3])
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = forward_head(q[b, h], k[b, h], v[b, h], scale, mask)
    return o, lse


def backward(q, k, v, do, scale: float, mask):
    """backward_head over [B, H, N, d] arrays."""
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = backward_head(q[b, h], k[b, h], v[b, h], do[b, h], scale, mask)
    return dq, dk, dv


def visible_tiles(n: int, left: int = -1, right: int = -1, block=None, tile: int = TILE) -> np.ndarray:
    """[n_tiles, n_tiles] bool: tile pairs holding at least one visible pair
    (the pairs a kernel must visit; the rest can be skipped)."""
    m = mask_matrix(n, n, left, right, block, tile)
    nt = -(-n // tile)
    out = np.zeros((nt, nt), dtype=bool)
    for a in range(nt):
        for b in range(nt):
            out[a, b] = m[a * tile:(a + 1) * tile, b * tile:(b + 1) * tile].any()
    return out
