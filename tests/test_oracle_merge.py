"""CPU pins of the split-KV partials and the merge operator (oracle/merge.py)."""
import math

import numpy as np

from oracle import attention as ora
from oracle import merge as om


def _head(nq, nk, d, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((nq, d)), rng.standard_normal((nk, d)), rng.standard_normal((nk, d))


def test_merge_of_any_partition_is_the_full_attention():
    q, k, v = _head(7, 300, 16, 1)
    scale = 1 / math.sqrt(16)
    o_ref, l_ref = ora.forward_head(q, k, v, scale, False)
    rng = np.random.default_rng(2)
    for _ in range(5):
        cuts = np.sort(rng.choice(np.arange(1, 300), size=4, replace=False))
        bounds = [0, *cuts.tolist(), 300]
        parts = [om.partial_head(q, k, v, scale, a, b) for a, b in zip(bounds[:-1], bounds[1:])]
        o, l = om.merge([p[0] for p in parts], [p[1] for p in parts])
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, l_ref, rtol=0, atol=1e-12)


def test_merge_ignores_empty_parts_and_single_part_is_identity():
    q, k, v = _head(3, 50, 8, 3)
    o1, l1 = om.partial_head(q, k, v, 0.3, 0, 50)
    o0, l0 = om.partial_head(q, k, v, 0.3, 20, 20)
    assert np.all(o0 == 0) and np.all(np.isneginf(l0))
    o, l = om.merge([o0, o1, o0], [l0, l1, l0])
    np.testing.assert_allclose(o, o1, atol=1e-15)
    np.testing.assert_allclose(l, l1, atol=1e-15)
    o, l = om.merge([o0], [l0])
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_merge_is_associative_and_order_free():
    q, k, v = _head(5, 90, 8, 4)
    parts = [om.partial_head(q, k, v, 0.5, a, b) for a, b in ((0, 30), (30, 31), (31, 90))]
    o3, l3 = om.merge([p[0] for p in parts], [p[1] for p in parts])
    o12, l12 = om.merge([parts[0][0], parts[1][0]], [parts[0][1], parts[1][1]])
    o, l = om.merge([o12, parts[2][0]], [l12, parts[2][1]])
    np.testing.assert_allclose(o, o3, atol=1e-13)
    np.testing.assert_allclose(l, l3, atol=1e-13)
    o, l = om.merge([p[0] for p in parts[::-1]], [p[1] for p in parts[::-1]])
    np.testing.assert_allclose(o, o3, atol=1e-13)


def test_merge_two_parts_closed_form():
    # two single-key parts: O = softmax of the two scores over v_1, v_2
    s1, s2 = 0.7, -1.3
    v1, v2 = np.array([1.0, 2.0]), np.array([-3.0, 0.5])
    o, l = om.merge([v1[None], v2[None]], [np.array([s1]), np.array([s2])])
    w1 = math.exp(s1) / (math.exp(s1) + math.exp(s2))
    np.testing.assert_allclose(o[0], w1 * v1 + (1 - w1) * v2, atol=1e-15)
    assert abs(l[0] - math.log(math.exp(s1) + math.exp(s2))) < 1e-15


def test_split_bounds_whole_tiles():
    assert om.split_bounds(1000, 3) == [0, 384, 768, 1000]
    assert om.split_bounds(128, 4) == [0, 128, 128, 128, 128]
    b = om.split_bounds(16384, 8)
    assert b[1] - b[0] == 2048 and b[-1] == 16384
