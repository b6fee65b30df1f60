"""GPU parity tests of the masked forward and backward (attn_fwd_masked,
attn_bwd_masked) against the FP64 oracle (oracle/masks.py).

Masks: sliding windows (including the causal window, a zero-width window and
two-sided windows), block maps drawn from a seeded generator (with query
tiles that see nothing and key tiles no query sees), and both combined.
Inputs are the seeded bf16 workloads of synth.  Rows with no visible key must
come out as O = 0, LSE = -inf, dQ = 0; every other row within the forward and
gradient tolerances.
"""
import math

import numpy as np
import pytest

from oracle import masks as om
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_77_gb300 as A

    A.get_lib()
    yield A
    G.check_status(A)


def _block(n, seed, density=0.6, empty_row=True, empty_col=True):
    t = -(-n // 128)
    rng = np.random.Generator(np.random.PCG64(seed))
    b = (rng.random((t, t)) < density).astype(np.uint8)
    if t >= 3:
        if empty_row:
            b[1, :] = 0
        if empty_col:
            b[:, t - 1] = 0
    return b


def _dev_block(block):
    if block is None:
        return None
    torch = G.torch_mod()
    return torch.from_numpy(np.ascontiguousarray(block)).cuda()


def run_fwd_masked(A, t, left, right, block, scale=None):
    torch = G.torch_mod()
    q, k, v = t["q"], t["k"], t["v"]
    B, H, N, d = q.shape
    scale = 1 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(v)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    A.attn_fwd_masked(q, k, v, o, lse, B, H, N, d, d, left, right, _dev_block(block), scale)
    return o, lse


def run_bwd_masked(A, t, o, lse, left, right, block, det, scale=None):
    torch = G.torch_mod()
    q, k, v, do = t["q"], t["k"], t["v"], t["do"]
    B, H, N, d = q.shape
    scale = 1 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nb = A.attn_bwd_workspace_bytes(B, H, N, d, d, det)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    A.attn_bwd_masked(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, d, left, right, _dev_block(block), scale, det, ws,
                      nb)
    return dq, dk, dv


def _check_fwd(o, lse, o_ref, lse_ref, what):
    o, lse = G.f64(o), G.f64(lse)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), what
    assert np.all(o[np.broadcast_to(empty[..., None], o.shape)] == 0), what
    live = ~empty
    if live.any():
        G.assert_fwd_close(o[live], lse[live], o_ref[live], lse_ref[live], what)


WINDOWS = [(-1, 0), (128, 0), (200, 50), (0, 0), (17, 17), (-1, -1), (300, -1)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 100, 257, 640])
@pytest.mark.parametrize("left,right", WINDOWS)
def test_window_forward_backward(A, d, N, left, right):
    t = G.inputs(1, 2, N, d, d, seed=21)
    q, k, v, do = (G.f64(t[n]) for n in ("q", "k", "v", "do"))
    mask = om.mask_matrix(N, N, left, right)
    o, lse = run_fwd_masked(A, t, left, right, None)
    G.check_status(A)
    o_ref, lse_ref = om.forward(q, k, v, 1 / math.sqrt(d), mask)
    _check_fwd(o, lse, o_ref, lse_ref, f"d{d} N{N} window({left},{right})")
    refs = om.backward(q, k, v, do, 1 / math.sqrt(d), mask)
    for det in (0, 1):
        grads = run_bwd_masked(A, t, o, lse, left, right, None, det)
        G.check_status(A)
        for name, got, ref in zip(("dq", "dk", "dv"), grads, refs):
            G.assert_grad_close(name, G.f64(got), ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,left,right", [(640, -1, -1), (640, -1, 0), (1000, 256, 256), (384, 0, 0)])
def test_block_map_forward_backward(A, d, N, left, right):
    t = G.inputs(1, 2, N, d, d, seed=22)
    q, k, v, do = (G.f64(t[n]) for n in ("q", "k", "v", "do"))
    block = _block(N, seed=23)
    mask = om.mask_matrix(N, N, left, right, block)
    o, lse = run_fwd_masked(A, t, left, right, block)
    G.check_status(A)
    o_ref, lse_ref = om.forward(q, k, v, 1 / math.sqrt(d), mask)
    _check_fwd(o, lse, o_ref, lse_ref, f"block d{d} N{N} window({left},{right})")
    refs = om.backward(q, k, v, do, 1 / math.sqrt(d), mask)
    for det in (0, 1):
        grads = run_bwd_masked(A, t, o, lse, left, right, block, det)
        G.check_status(A)
        for name, got, ref in zip(("dq", "dk", "dv"), grads, refs):
            G.assert_grad_close(name, G.f64(got), ref)
        # rows with no visible key get no gradient at all
        empty = np.isneginf(lse_ref)
        assert np.all(G.f64(grads[0])[np.broadcast_to(empty[..., None], grads[0].shape)] == 0)


def test_masked_deterministic_backward_is_bit_identical(A):
    torch = G.torch_mod()
    N, d = 1500, 128
    t = G.inputs(2, 3, N, d, d, seed=24)
    block = _block(N, seed=25, density=0.7)
    o, lse = run_fwd_masked(A, t, 400, 0, block)
    runs = [run_bwd_masked(A, t, o, lse, 400, 0, block, 1) for _ in range(3)]
    G.check_status(A)
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_causal_window_equals_the_causal_kernels(A):
    """left = -1, right = 0 is the causal mask: the masked path agrees with
    attn_fwd / attn_bwd causal within rounding."""
    N, d = 1024, 128
    t = G.inputs(1, 4, N, d, d, seed=26)
    o1, l1 = run_fwd_masked(A, t, -1, 0, None)
    o2, l2 = G.run_fwd(A, t, 1)
    G.check_status(A)
    assert float((o1.float() - o2.float()).abs().max()) <= 8e-3
    assert float((l1 - l2).abs().max()) <= 1e-4
    g1 = run_bwd_masked(A, t, o2, l2, -1, 0, None, 0)
    g2 = G.run_bwd(A, t, o2, l2, 1, 0)
    for a, b in zip(g1, g2):
        assert G.rel_fro(G.f64(a), G.f64(b)) <= 5e-3


def test_sliding_window_4k_sampled(A):
    """B = 1, H = 8, N = 4096, window (511, 0): forward on sampled rows of two
    heads against the oracle, each row against all keys; backward of one
    head in full."""
    B, H, N, d = 1, 8, 4096, 128
    t = G.inputs(B, H, N, d, d, seed=27)
    o, lse = run_fwd_masked(A, t, 511, 0, None)
    G.check_status(A)
    rows = G.seeded_rows(N, 64, seed=28)
    mask = om.mask_matrix(N, N, 511, 0)
    for h in (0, 5):
        q, k, v = (G.f64(t[n][0, h]) for n in ("q", "k", "v"))
        o_ref, lse_ref = om.forward_head(q[rows], k, v, 1 / math.sqrt(d), mask[rows])
        G.assert_fwd_close(G.f64(o[0, h])[rows], G.f64(lse[0, h])[rows], o_ref, lse_ref, f"head {h}")
    grads = run_bwd_masked(A, t, o, lse, 511, 0, None, 0)
    G.check_status(A)
    q, k, v, do = (G.f64(t[n][0, 3]) for n in ("q", "k", "v", "do"))
    refs = om.backward_head(q, k, v, do, 1 / math.sqrt(d), mask)
    for name, got, ref in zip(("dq", "dk", "dv"), grads, refs):
        G.assert_grad_close(name, G.f64(got[0, 3]), ref)
