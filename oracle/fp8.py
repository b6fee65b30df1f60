"""FP8 (e4m3) forward with per-block scales and a random rotation of Q and K.

Test infrastructure only (see the package docstring).

Source: "FlashAttention 3 and 4: When the Bottleneck Moves", section 2.2
(dropping to eight bits): values are rounded to an 8-bit floating-point
format; each block of values gets its own scale so that one block's outliers
do not stretch the others' range; and before quantising, Q and K are both
multiplied by the same fixed random rotation R, which spreads an outlying
coordinate over all coordinates while leaving every score unchanged, since
(QR)(KR)^T = Q R R^T K^T = Q K^T.  The page credits the two measures together
with a 2.6x smaller quantisation error.  "Attention at Scale -- From
FlashAttention to FlashAttention-4", FlashAttention-3 section, names the
same block quantisation for the FP8 mode.

Readings taken where the pages are silent (each is one line of DESIGN):
* Format: e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
  subnormals, no infinities, largest finite 448), rounding to nearest with
  ties to even, saturating at +-448.
* Rotation: R = D H / sqrt(d), H the d x d Sylvester-Hadamard matrix and D a
  diagonal of signs drawn at random once (an input here).  The quantiser
  applies sqrt(d) R = D H, exact in binary arithmetic, and the factor 1/d
  goes into the softmax scale: (Q D H)(K D H)^T / d = Q K^T.
* Blocks: for Q and K, each 128-row tile of one (b, h) (the tiles the
  forward loads); for V, one block per (b, h), because P V sums over every
  key tile into one accumulator.  A block's scale is the power of two
  s = 2^k with the smallest k such that amax(block) <= 448 s (s = 1 for an
  all-zero block); a value x is stored as e4m3(x / s).
* P is quantised as well.  With the conditional rescale of section 3.2
  (threshold tau, log2 units) P taken against the stale max m is at most
  2^tau, so P' = 2^(x - m + 8 - tau) <= 2^8 is stored as e4m3(P'); the row sum
  uses P' before rounding.  The library uses tau = 4 (tau = 0: the max moves
  on every rise).  As in the kernels, the rescale decision is taken per group
  of 32 consecutive query rows: when any row of the group rose by more than
  tau, every row of the group moves to its current max.
"""
from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)
E4M3_MAX = 448.0
P_MAX_LOG2 = 8.0  # P' = 2^(8 - tau) P <= 2^8
TAU = 4.0  # the library's rescale threshold for the FP8 forward
ROW_GROUP = 32  # rows that take one rescale decision together


def e4m3_decode(code: int) -> float:
    """Value of an e4m3 bit pattern (NaN for S.1111.111)."""
    s, e, m = (code >> 7) & 1, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return math.nan
    v = math.ldexp(m / 8.0, -6) if e == 0 else math.ldexp(1.0 + m / 8.0, e - 7)
    return -v if s else v


def e4m3_positive_values() -> np.ndarray:
    """The 127 non-negative finite e4m3 values (codes 0x00 .. 0x7E), ascending."""
    return np.array([e4m3_decode(c) for c in range(0x7F)])


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest e4m3 value, ties to even, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # spacing of the grid around a: 2^-9 below the normal range (2^-6), else
    # 2^(e-3) for a in [2^e, 2^(e+1))
    _, e2 = np.frexp(np.where(a > 0, a, 1.0))  # a = f 2^e2, f in [0.5, 1)
    quantum = np.where(a < 2.0 ** -6, 2.0 ** -9, np.ldexp(1.0, e2 - 1 - 3))
    q = np.round(a / quantum) * quantum  # np.round: half to even, exact here
    return np.copysign(np.minimum(q, E4M3_MAX), x)


def hadamard(d: int) -> np.ndarray:
    """Sylvester-Hadamard matrix of order d (a power of two): H_ij = (-1)^popcount(i & j)."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotation(signs) -> np.ndarray:
    """The orthogonal R = D H / sqrt(d) for the sign vector ``signs`` (+-1)."""
    signs = np.asarray(signs, dtype=np.float64)
    return signs[:, None] * hadamard(signs.size) / math.sqrt(signs.size)


def rotate_unnormalised(x, signs) -> np.ndarray:
    """x (sqrt(d) R) = (x * signs) H along the last axis."""
    signs = np.asarray(signs, dtype=np.float64)
    return (np.asarray(x, dtype=np.float64) * signs) @ hadamard(signs.size)


def pow2_scale(amax: float) -> float:
    """The smallest power of two s with amax <= 448 s (1 for amax = 0)."""
    if amax == 0.0:
        return 1.0
    f, e = math.frexp(amax)  # amax = f 2^e, f in [0.5, 1); 448 = 0.875 2^9
    k = e - 9 if f <= 0.875 else e - 8
    return math.ldexp(1.0, k)


def quantize_rows(x, block_rows):
    """Block-quantise x [..., N, d]: blocks of ``block_rows`` rows of each
    leading index (None: the whole tensor is one block).  Returns (values on
    the e4m3 grid, scales [..., n_blocks] or a scalar)."""
    x = np.asarray(x, dtype=np.float64)
    if block_rows is None:
        s = pow2_scale(float(np.abs(x).max()))
        return e4m3_round(x / s), s
    lead, n, d = x.shape[:-2], x.shape[-2], x.shape[-1]
    nb = -(-n // block_rows)
    codes = np.empty_like(x)
    scales = np.empty(lead + (nb,))
    for idx in np.ndindex(*lead):
        for b in range(nb):
            blk = x[idx + (slice(b * block_rows, (b + 1) * block_rows),)]
            s = pow2_scale(float(np.abs(blk).max()))
            scales[idx + (b,)] = s
            codes[idx + (slice(b * block_rows, (b + 1) * block_rows),)] = e4m3_round(blk / s)
    return codes, scales


def quantize_qkv(q, k, v, signs, tile: int = 128):
    """The quantiser: rotate Q and K by sqrt(d) R, then e4m3 with per-tile
    scales for Q and K and one scale per (b, h) for V.

    q, k, v [B, H, N, d] FP64.  Returns dict q8, k8, v8 (values on the e4m3
    grid), sq, sk [B, H, n_tiles], sv [B, H]."""
    q8, sq = quantize_rows(rotate_unnormalised(q, signs), tile)
    k8, sk = quantize_rows(rotate_unnormalised(k, signs), tile)
    n = v.shape[-2]
    v8, sv = quantize_rows(v, n)
    return {"q8": q8, "k8": k8, "v8": v8, "sq": sq, "sk": sk, "sv": sv[..., 0]}


def forward_head(q8, k8, v8, sq, sk, sv: float, scale: float, causal: bool, d: int, tile: int = 128,
                 quantize_p: bool = True, rows=None, tau: float = TAU):
    """FP8 forward of one head from quantised inputs, in FP64.

    q8 [Nq, d], k8 [Nk, d], v8 [Nk, d_v] on the e4m3 grid; sq [ceil(Nq/tile)],
    sk [ceil(Nk/tile)] the per-tile scales, sv the head's V scale; ``scale``
    the caller's softmax scale; d the rotated dimension (the 1/d of the
    rotation goes into the scores).  Online softmax over key tiles: scores
    x = scale/d * sq_i sk_j (q8 k8^T) in log2 units; candidate max
    m_new = max(m, rowmax x); where any row of a 32-row group has
    m_new > m + tau (or m is still -inf) the whole group moves to m_new, acc
    and l scaled by 2^(m - m_new); P' = 2^(x - m + 8 - tau) stored as
    e4m3(P') (or kept exact when quantize_p is False), l += sum P',
    acc += P' v8.  O = sv acc / l, LSE = (m - (8 - tau) + log2 l) ln 2.
    ``rows`` (optional): the query indices of q8's rows within the head, when
    q8 holds a sample of them (they select the tile scale, the causal mask
    and the rescale group; a sample must hold whole 32-row groups).
    Returns (O, LSE)."""
    nq, nk = q8.shape[0], k8.shape[0]
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    _, group = np.unique(rows // ROW_GROUP, return_inverse=True)
    p_off = P_MAX_LOG2 - tau
    c_row = (scale / d) * LOG2E * np.asarray(sq, dtype=np.float64)[rows // tile]
    m = np.full(nq, -np.inf)
    l = np.zeros(nq)
    acc = np.zeros((nq, v8.shape[1]))
    for jt, j0 in enumerate(range(0, nk, tile)):
        j1 = min(nk, j0 + tile)
        x = (c_row * sk[jt])[:, None] * (q8 @ k8[j0:j1].T)
        if causal:
            x = np.where(np.arange(j0, j1)[None, :] > rows[:, None], -np.inf, x)
        m_new = np.maximum(m, x.max(axis=1))
        rose = np.isfinite(m_new) & (~np.isfinite(m) | (m_new > m + tau))
        need = np.bincount(group, weights=rose)[group] > 0  # any row of the group
        alpha = np.where(need & np.isfinite(m), np.exp2(m - np.where(np.isfinite(m_new), m_new, 0.0)), 1.0)
        alpha = np.where(need & ~np.isfinite(m), 0.0, alpha)
        acc *= alpha[:, None]
        l *= alpha
        m = np.where(need, m_new, m)
        m_use = np.where(np.isfinite(m), m, 0.0)
        p = np.exp2(x - m_use[:, None] + p_off)
        l += p.sum(axis=1)
        acc += (e4m3_round(p) if quantize_p else p) @ v8[j0:j1]
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(l[:, None] > 0, sv * acc / np.where(l > 0, l, 1.0)[:, None], 0.0)
        lse = np.where(l > 0, (m - p_off + np.log2(np.where(l > 0, l, 1.0))) / LOG2E, -np.inf)
    return o, lse


def forward(qz: dict, scale: float, causal: bool, quantize_p: bool = True, tau: float = TAU):
    """forward_head over every (b, h) of quantize_qkv's output."""
    q8 = qz["q8"]
    B, H, N, d = q8.shape
    o = np.empty((B, H, N, qz["v8"].shape[-1]))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = forward_head(q8[b, h], qz["k8"][b, h], qz["v8"][b, h], qz["sq"][b, h],
                                              qz["sk"][b, h], float(qz["sv"][b, h]), scale, causal, d,
                                              quantize_p=quantize_p, tau=tau)
    return o, lse


def forward_per_tensor_unrotated(q, k, v, scale: float, causal: bool):
    """The comparison point of the error claim: one scale per tensor for Q, K
    and V, no rotation, P quantised the same way."""
    q8, sq = quantize_rows(q, None)
    k8, sk = quantize_rows(k, None)
    v8, sv = quantize_rows(v, None)
    B, H, N, d = q.shape
    o = np.empty((B, H, N, v.shape[-1]))
    lse = np.empty((B, H, N))
    nt = -(-N // 128)
    for b in range(B):
        for h in range(H):
            # no rotation: the 1/d of the rotated path is not applied, so the
            # scores use d = 1
            o[b, h], lse[b, h] = forward_head(q8[b, h], k8[b, h], v8[b, h], np.full(nt, sq), np.full(nt, sk), sv,
                                              scale, causal, 1)
    return o, lse
