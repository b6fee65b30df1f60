"""Plain FP64 attention: definition, explicit backward, and the online algorithm.

Test infrastructure only (see the package docstring).

Sources
-------
* "Attention at Scale -- From FlashAttention to FlashAttention-4", section
  "The Problem": attention is the N x N score matrix Q K^T, a softmax, then a
  product with V.  The scale 1/sqrt(d) and the causal mask are the usual
  scaled-dot-product attention; the scale is a caller argument here.
* Same page, section "The Evolution" (FlashAttention paragraph): the softmax
  can be computed incrementally by keeping a running max and sum per row.
* "FlashAttention 3 and 4: When the Bottleneck Moves", section 3.2 (second
  change): the running max may drift by up to tau = 8 doublings before a
  rescale happens; the result is renormalised once at the end.

Readings taken where the pages are silent
-----------------------------------------
* Layout [B, H, N, d], row-major; N_q = N_k = N.
* Causal mask is top-left aligned: query i sees keys j <= i.
* LSE is the natural-log log-sum-exp of the scaled scores of the unmasked keys.
* A row with no unmasked key (impossible when N_q = N_k) gets O = 0 and
  LSE = -inf.
"""
from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) to exact FP64 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _causal_mask(nq: int, nk: int, rows=None) -> np.ndarray:
    """True where key j is hidden from query i (j > i)."""
    i = np.arange(nq)[:, None] if rows is None else np.asarray(rows)[:, None]
    j = np.arange(nk)[None, :]
    return j > i


def _scores(q: np.ndarray, k: np.ndarray, scale: float, causal: bool, rows=None) -> np.ndarray:
    """S = scale * q k^T for one head, with -inf where the causal mask hides a key."""
    s = scale * (q @ k.T)
    if causal:
        s = np.where(_causal_mask(s.shape[0], s.shape[1], rows), -np.inf, s)
    return s


def _softmax_rows(s: np.ndarray):
    """Two-pass softmax of each row: max, then exponentials and their sum."""
    m = s.max(axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe[:, None])
    l = e.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        p = np.where(l[:, None] > 0, e / np.where(l > 0, l, 1.0)[:, None], 0.0)
        lse = np.where(l > 0, m_safe + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return p, lse


def forward_head(q, k, v, scale: float, causal: bool, rows=None):
    """One head: O = softmax(scale q k^T + mask) v and the per-row LSE.

    ``q`` holds the query rows whose global indices are ``rows`` (all rows when
    ``rows`` is None); ``k`` and ``v`` hold every key of the head.
    """
    s = _scores(q, k, scale, causal, rows)
    p, lse = _softmax_rows(s)
    return p @ v, lse


def forward(q, k, v, scale: float, causal: bool):
    """Full forward over [B, H, N, d] FP64 arrays; returns O [B,H,N,d_v], LSE [B,H,N]."""
    B, H, N, _ = q.shape
    o = np.empty(q.shape[:3] + (v.shape[-1],), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = forward_head(q[b, h], k[b, h], v[b, h], scale, causal)
    return o, lse


def forward_rows(q, k, v, scale: float, causal: bool, heads, rows):
    """Sampled forward: for each (b, h) in ``heads`` the rows ``rows`` of O and LSE.

    Each sampled row is computed against every key of its head, exactly as in
    ``forward``; returns arrays [len(heads), len(rows), d_v] and [len(heads), len(rows)].
    """
    rows = np.asarray(rows)
    o = np.empty((len(heads), len(rows), v.shape[-1]))
    lse = np.empty((len(heads), len(rows)))
    for t, (b, h) in enumerate(heads):
        o[t], lse[t] = forward_head(q[b, h][rows], k[b, h], v[b, h], scale, causal, rows)
    return o, lse


def backward_head(q, k, v, do, scale: float, causal: bool):
    """One head: dQ, dK, dV of L = sum(O * dO) by the explicit chain rule.

    P is recomputed from the definition.  dS uses the full softmax Jacobian:
    dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik), with dP = dO v^T.  Then
    dQ = scale dS k, dK = scale dS^T q, dV = P^T dO.
    """
    s = _scores(q, k, scale, causal)
    p, _ = _softmax_rows(s)
    dv = p.T @ do
    dp = do @ v.T
    jac_row = (p * dp).sum(axis=1, keepdims=True)
    ds = p * (dp - jac_row)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


def backward(q, k, v, do, scale: float, causal: bool):
    """Full backward over [B, H, N, d] FP64 arrays; returns dQ, dK, dV."""
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = backward_head(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
    return dq, dk, dv


def online_forward_head(q, k, v, scale: float, causal: bool, tile: int = 128, tau: float = 8.0):
    """The tiled online-softmax algorithm for one head, in FP64.

    Keys are visited one tile of ``tile`` keys at a time; each query row keeps
    a running max ``m`` (log2 units of the scaled score), a running sum ``l``
    and an unnormalised output ``acc``.  For every tile:

    1. scores of the tile, times log2(e), masked to -inf where hidden;
    2. the candidate max ``m_new = max(m, rowmax(tile))``;
    3. conditional rescale: only where ``m_new - m > tau`` (or ``m`` is still
       -inf) are ``acc`` and ``l`` multiplied by 2^(m - m_new) and ``m`` moved
       to ``m_new``; elsewhere ``m`` stays stale.  ``tau = 0`` rescales on
       every rise, the classic online softmax;
    4. ``p = 2^(score - m)``, ``l += sum(p)``, ``acc += p v_tile``.

    At the end ``O = acc / l`` and ``LSE = (m + log2 l) ln 2``.  Returns
    (O, LSE, rescale_count) where rescale_count counts row rescales after the
    first visited tile.
    """
    nq, nk = q.shape[0], k.shape[0]
    c = scale * LOG2E
    m = np.full(nq, -np.inf)
    l = np.zeros(nq)
    acc = np.zeros((nq, v.shape[1]))
    rescales = 0
    for j0 in range(0, nk, tile):
        j1 = min(nk, j0 + tile)
        s = c * (q @ k[j0:j1].T)
        if causal:
            s = np.where(np.arange(j0, j1)[None, :] > np.arange(nq)[:, None], -np.inf, s)
        m_new = np.maximum(m, s.max(axis=1))
        first = ~np.isfinite(m)
        need = first | (m_new - m > tau)
        need &= np.isfinite(m_new)
        rescales += int(np.count_nonzero(need & ~first))
        alpha = np.where(need & ~first, np.exp2(m - np.where(need, m_new, m)), 1.0)
        alpha = np.where(first, 0.0, alpha)
        acc *= alpha[:, None]
        l *= alpha
        m = np.where(need, m_new, m)
        m_use = np.where(np.isfinite(m), m, 0.0)
        p = np.exp2(s - m_use[:, None])
        l += p.sum(axis=1)
        acc += p @ v[j0:j1]
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(l[:, None] > 0, acc / np.where(l > 0, l, 1.0)[:, None], 0.0)
        lse = np.where(l > 0, (m + np.log2(np.where(l > 0, l, 1.0))) / LOG2E, -np.inf)
    return o, lse, rescales


def flops_forward(B: int, H: int, N: int, d_qk: int, d_v: int, causal: bool) -> float:
    """Forward FLOPs: 2 B H N^2 (d_qk + d_v), halved for causal (4 B H N^2 d when d_qk = d_v)."""
    f = 2.0 * B * H * N * N * (d_qk + d_v)
    return f / 2.0 if causal else f


def flops_backward(B: int, H: int, N: int, d_qk: int, d_v: int, causal: bool) -> float:
    """Backward FLOPs: 2.5 times the forward count (five matrix products against two)."""
    return 2.5 * flops_forward(B, H, N, d_qk, d_v, causal)
