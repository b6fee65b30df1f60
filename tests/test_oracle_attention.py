"""CPU pins for the FP64 attention oracle.

Each test checks the oracle against something other than itself: an
independent pure-Python brute force, central finite differences, closed-form
special cases, or invariants that the pages fix.  The last group plants
plausible mistakes into copies of the oracle and shows that a pin catches each.
"""
import math

import numpy as np
import pytest

from oracle import attention as ora


def _rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


# ---------------------------------------------------------------- brute force
def _brute_forward(q, k, v, scale, causal):
    """Pure-Python loops with math.fsum: no numpy arithmetic."""
    nq, nk, dv = len(q), len(k), len(v[0])
    out, lses = [], []
    for i in range(nq):
        s = []
        for j in range(nk):
            if causal and j > i:
                continue
            s.append((j, scale * math.fsum(q[i][t] * k[j][t] for t in range(len(q[i])))))
        mx = max(x for _, x in s)
        e = [(j, math.exp(x - mx)) for j, x in s]
        den = math.fsum(x for _, x in e)
        out.append([math.fsum(w * v[j][c] for j, w in e) / den for c in range(dv)])
        lses.append(mx + math.log(den))
    return out, lses


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,dqk,dv", [(1, 2, 3), (5, 4, 4), (8, 3, 2), (7, 4, 1)])
def test_forward_matches_brute_force(n, dqk, dv, causal):
    q, k, v = _rand((1, 2, n, dqk), 1), _rand((1, 2, n, dqk), 2), _rand((1, 2, n, dv), 3)
    scale = 1.0 / math.sqrt(dqk)
    o, lse = ora.forward(q, k, v, scale, causal)
    for h in range(2):
        bo, bl = _brute_forward(q[0, h].tolist(), k[0, h].tolist(), v[0, h].tolist(), scale, causal)
        np.testing.assert_allclose(o[0, h], np.array(bo), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[0, h], np.array(bl), rtol=1e-12, atol=1e-14)


# ------------------------------------------------------- finite differences
@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    n, dqk, dv = 6, 3, 4
    q, k, v, do = (_rand((n, dqk), 11), _rand((n, dqk), 12), _rand((n, dv), 13), _rand((n, dv), 14))
    scale = 0.7

    def loss(qq, kk, vv):
        o, _ = ora.forward_head(qq, kk, vv, scale, causal)
        return float(np.sum(o * do))

    dq, dk, dv_ = ora.backward_head(q, k, v, do, scale, causal)
    h = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv_)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        rel = np.linalg.norm(num - g) / np.linalg.norm(g)
        assert rel < 1e-6, (name, rel)


def test_jacobian_row_term_equals_do_dot_o():
    """sum_k P_ik dP_ik == dO_i . O_i, the identity the GPU's D = rowsum(dO*O) uses."""
    n, d = 9, 5
    q, k, v, do = (_rand((n, d), s) for s in (21, 22, 23, 24))
    scale = 0.4
    s = ora._scores(q, k, scale, True)
    p, _ = ora._softmax_rows(s)
    o, _ = ora.forward_head(q, k, v, scale, True)
    lhs = (p * (do @ v.T)).sum(axis=1)
    np.testing.assert_allclose(lhs, (do * o).sum(axis=1), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------- softmax facts
def test_softmax_rows_sum_to_one():
    s = _rand((16, 33), 5) * 7
    s[3, 10:] = -np.inf
    p, _ = ora._softmax_rows(s)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    assert np.all(p[3, 10:] == 0)


@pytest.mark.parametrize("tau", [0.0, 8.0])
@pytest.mark.parametrize("tile", [1, 3, 16, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_online_softmax_equals_two_pass(tau, tile, causal):
    n, d = 40, 8
    q, k, v = _rand((n, d), 31) * 2.5, _rand((n, d), 32) * 2.5, _rand((n, d), 33)
    scale = 1.0 / math.sqrt(d)
    o2, l2 = ora.forward_head(q, k, v, scale, causal)
    o1, l1, _ = ora.online_forward_head(q, k, v, scale, causal, tile=tile, tau=tau)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-13)


def test_conditional_rescale_skips_small_rises():
    """With a slowly rising max, tau = 8 rescales far less than tau = 0, same answer."""
    n, d = 64, 4
    q = np.ones((n, d))
    k = np.outer(np.linspace(0.0, 10.0, n), np.ones(d)) / d
    v = _rand((n, d), 41)
    o0, l0, r0 = ora.online_forward_head(q, k, v, 1.0, False, tile=4, tau=0.0)
    o8, l8, r8 = ora.online_forward_head(q, k, v, 1.0, False, tile=4, tau=8.0)
    assert r0 == n * 15 and r8 < r0 // 5
    np.testing.assert_allclose(o8, o0, rtol=1e-12)
    np.testing.assert_allclose(l8, l0, rtol=1e-13)


# ------------------------------------------------------------- special cases
@pytest.mark.parametrize("causal", [False, True])
def test_v_ones_gives_o_ones(causal):
    q, k = _rand((1, 3, 12, 4), 51), _rand((1, 3, 12, 4), 52)
    o, _ = ora.forward(q, k, np.ones((1, 3, 12, 5)), 0.5, causal)
    np.testing.assert_allclose(o, 1.0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_prefix_mean(causal):
    n = 10
    v = _rand((n, 3), 61)
    o, lse = ora.forward_head(np.zeros((n, 4)), _rand((n, 4), 62), v, 0.3, causal)
    for i in range(n):
        upto = i + 1 if causal else n
        np.testing.assert_allclose(o[i], v[:upto].mean(axis=0), atol=1e-14)
        assert abs(lse[i] - math.log(upto)) < 1e-14


def test_causal_first_row_and_single_key():
    q, k, v = _rand((6, 4), 71), _rand((6, 4), 72), _rand((6, 2), 73)
    o, lse = ora.forward_head(q, k, v, 0.9, True)
    np.testing.assert_allclose(o[0], v[0], atol=0)
    assert abs(lse[0] - 0.9 * float(q[0] @ k[0])) < 1e-15
    o1, _ = ora.forward(q[None, None, :1], k[None, None, :1], v[None, None, :1], 0.9, False)
    np.testing.assert_allclose(o1[0, 0], v[:1], atol=0)


# ------------------------------------------------------------------ invariants
def test_key_value_permutation_invariance():
    n, d = 20, 6
    q, k, v = _rand((n, d), 81), _rand((n, d), 82), _rand((n, d), 83)
    perm = np.random.Generator(np.random.PCG64(84)).permutation(n)
    o1, l1 = ora.forward_head(q, k, v, 0.5, False)
    o2, l2 = ora.forward_head(q, k[perm], v[perm], 0.5, False)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_rotation_invariance(causal):
    """(QR)(KR)^T = QK^T for orthogonal R (FlashAttention 3 and 4, section 2.2)."""
    n, d = 16, 8
    q, k, v = _rand((n, d), 91), _rand((n, d), 92), _rand((n, d), 93)
    r, _ = np.linalg.qr(_rand((d, d), 94))
    o1, l1 = ora.forward_head(q, k, v, 0.35, causal)
    o2, l2 = ora.forward_head(q @ r, k @ r, v, 0.35, causal)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_moves_lse_only(causal):
    n, d = 12, 5
    q, k, v = _rand((n, d), 101), _rand((n, d), 102), _rand((n, d), 103)
    u = _rand(d, 104)
    scale = 0.6
    o1, l1 = ora.forward_head(q, k, v, scale, causal)
    o2, l2 = ora.forward_head(q, k + u[None, :], v, scale, causal)
    np.testing.assert_allclose(o2, o1, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, scale * (q @ u), rtol=1e-11, atol=1e-12)


def test_sampled_rows_match_full_forward():
    q, k, v = _rand((2, 2, 30, 4), 111), _rand((2, 2, 30, 4), 112), _rand((2, 2, 30, 3), 113)
    rows = np.array([0, 7, 29, 13])
    for causal in (False, True):
        o, lse = ora.forward(q, k, v, 0.5, causal)
        so, sl = ora.forward_rows(q, k, v, 0.5, causal, [(1, 0), (0, 1)], rows)
        np.testing.assert_allclose(so[0], o[1, 0][rows], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(sl[1], lse[0, 1][rows], rtol=1e-14, atol=1e-15)


def test_flop_convention():
    assert ora.flops_forward(1, 1, 10, 4, 4, False) == 4 * 100 * 4
    assert ora.flops_forward(2, 3, 8, 192, 128, True) == 2 * 2 * 3 * 64 * 320 / 2
    assert ora.flops_backward(1, 1, 10, 4, 4, False) == 2.5 * 1600


# ---------------------------------------------- planted mistakes are caught
def _fd_rel(backward_fn, causal=True):
    n, dqk, dv = 5, 3, 2
    q, k, v, do = (_rand((n, dqk), 121), _rand((n, dqk), 122), _rand((n, dv), 123), _rand((n, dv), 124))
    scale = 0.8

    def loss(qq, kk, vv):
        return float(np.sum(ora.forward_head(qq, kk, vv, scale, causal)[0] * do))

    g = backward_fn(q, k, v, do, scale, causal)
    worst = 0.0
    for pos, x in enumerate((q, k, v)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args = [q, k, v]
            xp, xm = x.copy(), x.copy()
            xp[idx] += 1e-5
            xm[idx] -= 1e-5
            args[pos] = xp
            lp = loss(*args)
            args[pos] = xm
            num[idx] = (lp - loss(*args)) / 2e-5
        worst = max(worst, np.linalg.norm(num - g[pos]) / np.linalg.norm(num))
    return worst


def test_planted_backward_mistakes_are_caught():
    def no_jacobian_term(q, k, v, do, scale, causal):
        p, _ = ora._softmax_rows(ora._scores(q, k, scale, causal))
        ds = p * (do @ v.T)
        return scale * ds @ k, scale * ds.T @ q, p.T @ do

    def swapped_dk(q, k, v, do, scale, causal):
        dq, dk, dv = ora.backward_head(q, k, v, do, scale, causal)
        p, _ = ora._softmax_rows(ora._scores(q, k, scale, causal))
        dp = do @ v.T
        ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        return dq, scale * ds @ q, dv

    def transposed_dv(q, k, v, do, scale, causal):
        dq, dk, _ = ora.backward_head(q, k, v, do, scale, causal)
        p, _ = ora._softmax_rows(ora._scores(q, k, scale, causal))
        return dq, dk, p @ do

    assert _fd_rel(ora.backward_head) < 1e-6
    for bad in (no_jacobian_term, swapped_dk, transposed_dv):
        assert _fd_rel(bad) > 1e-2, bad.__name__


def test_planted_forward_mistakes_are_caught(monkeypatch):
    n, d = 6, 3
    q, k, v = _rand((n, d), 131), _rand((n, d), 132), _rand((n, d), 133)
    ref_o, _ = _brute_forward(q.tolist(), k.tolist(), v.tolist(), 0.5, True)

    def off_by_one_mask(nq, nk, rows=None):
        i = np.arange(nq)[:, None]
        return np.arange(nk)[None, :] >= i

    monkeypatch.setattr(ora, "_causal_mask", off_by_one_mask)
    with np.errstate(all="ignore"):
        bad_o, _ = ora.forward_head(q, k, v, 0.5, True)
    assert not np.allclose(bad_o, np.array(ref_o), atol=1e-6)
