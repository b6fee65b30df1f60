"""CPU pins of the masked-attention oracle (oracle/masks.py)."""
import math

import numpy as np
import pytest

from oracle import attention as ora
from oracle import masks as om


def _head(n, d, seed, dv=None):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, d)), rng.standard_normal((n, d)), rng.standard_normal((n, dv or d)),
            rng.standard_normal((n, dv or d)))


def test_mask_matrix_small_cases():
    m = om.mask_matrix(8, 8, left=2, right=1)
    assert m[5].nonzero()[0].tolist() == [3, 4, 5, 6]
    assert m[0].nonzero()[0].tolist() == [0, 1]
    assert m[7].nonzero()[0].tolist() == [5, 6, 7]
    assert np.array_equal(om.mask_matrix(5, 5, -1, 0), np.tril(np.ones((5, 5), bool)))
    assert om.mask_matrix(5, 5).all()
    blk = np.array([[1, 0], [0, 1]])
    mb = om.mask_matrix(6, 6, block=blk, tile=3)
    assert mb[:3, :3].all() and not mb[:3, 3:].any() and not mb[3:, :3].any() and mb[3:, 3:].all()


@pytest.mark.parametrize("n", [1, 7, 130])
def test_causal_and_full_windows_reduce_to_the_plain_oracle(n):
    q, k, v, do = _head(n, 8, 1)
    for causal, (left, right) in ((True, (-1, 0)), (False, (-1, -1))):
        mask = om.mask_matrix(n, n, left, right)
        o, lse = om.forward_head(q, k, v, 0.4, mask)
        o_ref, lse_ref = ora.forward_head(q, k, v, 0.4, causal)
        np.testing.assert_allclose(o, o_ref, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref, atol=1e-13)
        for got, ref in zip(om.backward_head(q, k, v, do, 0.4, mask), ora.backward_head(q, k, v, do, 0.4, causal)):
            np.testing.assert_allclose(got, ref, atol=1e-12)


def test_diagonal_window_returns_own_value():
    q, k, v, _ = _head(20, 4, 2)
    o, lse = om.forward_head(q, k, v, 0.7, om.mask_matrix(20, 20, 0, 0))
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.7 * np.einsum("id,id->i", q, k), atol=1e-14)


def test_brute_force_tiny_window():
    q, k, v, _ = _head(5, 3, 3)
    left, right, scale = 1, 2, 0.9
    o, lse = om.forward_head(q, k, v, scale, om.mask_matrix(5, 5, left, right))
    for i in range(5):
        js = [j for j in range(5) if i - left <= j <= i + right]
        sc = [scale * math.fsum(q[i, t] * k[j, t] for t in range(3)) for j in js]
        mx = max(sc)
        w = [math.exp(x - mx) for x in sc]
        z = math.fsum(w)
        assert abs(lse[i] - (mx + math.log(z))) < 1e-13
        for t in range(3):
            assert abs(o[i, t] - math.fsum(w[a] * v[js[a], t] for a in range(len(js))) / z) < 1e-13


def test_empty_rows_and_unseen_keys():
    n, tile = 6, 3
    q, k, v, do = _head(n, 4, 4)
    blk = np.array([[0, 0], [1, 1]])  # query tile 0 sees nothing
    mask = om.mask_matrix(n, n, block=blk, tile=tile)
    o, lse = om.forward_head(q, k, v, 0.5, mask)
    assert np.all(o[:3] == 0) and np.all(np.isneginf(lse[:3])) and np.all(np.isfinite(lse[3:]))
    dq, dk, dv = om.backward_head(q, k, v, do, 0.5, mask)
    assert np.all(dq[:3] == 0)
    blk2 = np.array([[1, 0], [1, 0]])  # key tile 1 is seen by no query
    dq, dk, dv = om.backward_head(q, k, v, do, 0.5, om.mask_matrix(n, n, block=blk2, tile=tile))
    assert np.all(dk[3:] == 0) and np.all(dv[3:] == 0)


def test_masked_backward_against_finite_differences():
    n, d = 9, 4
    q, k, v, do = _head(n, d, 5)
    mask = om.mask_matrix(n, n, 2, 1, block=np.array([[1, 1, 0], [1, 1, 1], [0, 1, 1]]), tile=3)
    grads = om.backward_head(q, k, v, do, 0.6, mask)
    f = lambda q_, k_, v_: float((om.forward_head(q_, k_, v_, 0.6, mask)[0] * do).sum())
    h = 1e-6
    for which, g in enumerate(grads):
        args = [q.copy(), k.copy(), v.copy()]
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            a = [x.copy() for x in args]
            b = [x.copy() for x in args]
            a[which][idx] += h
            b[which][idx] -= h
            num[idx] = (f(*a) - f(*b)) / (2 * h)
        assert np.linalg.norm(num - g) <= 1e-6 * max(1.0, np.linalg.norm(g)), which


def test_visible_tiles_of_a_window():
    vis = om.visible_tiles(512, left=128, right=0)
    want = np.zeros((4, 4), bool)
    for a in range(4):
        want[a, a] = True
        if a > 0:
            want[a, a - 1] = True
    assert np.array_equal(vis, want)
    # left = 127: row 128a sees back to 128a - 127, still inside tile a - 1
    assert np.array_equal(om.visible_tiles(512, left=127, right=0), want)
    # left = 0, right = 0: only the diagonal tiles
    assert np.array_equal(om.visible_tiles(300, 0, 0), np.eye(3, dtype=bool))
