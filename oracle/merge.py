"""Partial attention over a subset of keys, and the merge of such partials.

Test infrastructure only (see the package docstring).

Source: "Attention at Scale -- From FlashAttention to FlashAttention-4",
FlashInfer section ("Composable attention"): attention over a key set can be
split into sub-problems over disjoint key subsets, computed independently,
and combined with an associative merge operator; the same page's "Sequence-
Aware Split Heuristic" section splits a sequence across thread blocks for
decode and pays one reduction pass.  The operator is written out from the
definition: over keys K = K_1 u K_2 (disjoint), with per-part softmax
normalisers l_s = sum_{j in K_s} exp(s_j), LSE_s = log l_s and normalised
partial outputs O_s = sum_{j in K_s} exp(s_j - LSE_s) v_j,

    LSE = log(exp(LSE_1) + exp(LSE_2)),  O = exp(LSE_1 - LSE) O_1 + exp(LSE_2 - LSE) O_2.

A part with no key has LSE = -inf and O = 0 and drops out of the merge.
"""
from __future__ import annotations

import numpy as np

from .attention import forward_head


def partial_head(q, k, v, scale: float, key_lo: int, key_hi: int):
    """O and LSE of one head's non-causal attention restricted to keys [key_lo, key_hi)."""
    nq = q.shape[0]
    if key_hi <= key_lo:
        return np.zeros((nq, v.shape[-1])), np.full(nq, -np.inf)
    return forward_head(q, k[key_lo:key_hi], v[key_lo:key_hi], scale, False)


def merge(o_parts, lse_parts):
    """Merge partials: o_parts [S, ..., d_v], lse_parts [S, ...] (natural log) -> (O, LSE)."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse_parts - m_safe)  # exp(-inf) = 0 for empty parts
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot > 0, m_safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
        o = np.where(tot[..., None] > 0, (w[..., None] * o_parts).sum(axis=0) / np.where(tot > 0, tot, 1.0)[..., None], 0.0)
    return o, lse


def split_bounds(n_keys: int, n_splits: int, tile: int = 128):
    """Key-range boundaries of a split into n_splits parts of whole 128-key tiles
    (the last part ragged), the partition the library's split-KV forward uses."""
    n_tiles = -(-n_keys // tile)
    per = -(-n_tiles // n_splits)
    return [min(n_keys, s * per * tile) for s in range(n_splits)] + [n_keys]
