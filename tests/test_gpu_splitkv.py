"""GPU parity tests of the split-KV forward and the merge operator against the
FP64 oracle (oracle/attention.py for the full attention over all keys,
oracle/merge.py for the merge of given partials).

Inputs: seeded N(0,1) bfloat16 tensors from synth.decode_inputs_torch (Q of
N_q rows, K and V of N_k rows per head), the decode-shaped workloads of the
sequence-aware split: few heads, few query rows, long key sequences.
"""
import math

import numpy as np
import pytest

import synth
from oracle import attention as ora
from oracle import merge as om
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


def run_splitkv(A, t, n_splits, scale=None):
    torch = G.torch_mod()
    q, k, v = t["q"], t["k"], t["v"]
    B, H, Nq, dqk = q.shape
    Nk, dv = k.shape[2], v.shape[-1]
    scale = 1.0 / math.sqrt(dqk) if scale is None else scale
    o = torch.empty((B, H, Nq, dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    nbytes = A.attn_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, dv, n_splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    A.attn_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, dqk, dv, scale, n_splits, ws, nbytes)
    return o, lse


def oracle_full(t, scale):
    q, k, v = (G.f64(t[n]) for n in ("q", "k", "v"))
    B, H = q.shape[:2]
    o = np.empty(q.shape[:3] + (v.shape[-1],))
    lse = np.empty(q.shape[:3])
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = ora.forward_head(q[b, h], k[b, h], v[b, h], scale, False)
    return o, lse


def _check(A, B, H, Nq, Nk, dqk, dv, n_splits, seed=0):
    t = synth.decode_inputs_torch(synth.DecodeShape(B, H, Nq, Nk, dqk, dv), seed=seed)
    o, lse = run_splitkv(A, t, n_splits)
    G.check_status(A)
    o_ref, lse_ref = oracle_full(t, 1.0 / math.sqrt(dqk))
    return G.assert_fwd_close(G.f64(o), G.f64(lse), o_ref, lse_ref,
                              f"B{B} H{H} Nq{Nq} Nk{Nk} d{dqk}/{dv} splits{n_splits}")


@pytest.mark.parametrize("dqk,dv", [(64, 64), (128, 128), (192, 128)])
@pytest.mark.parametrize("nq,nk", [(1, 1), (1, 1000), (7, 300), (128, 129), (130, 2048), (300, 1000)])
@pytest.mark.parametrize("n_splits", [1, 3, 8])
def test_splitkv_matches_full_attention(A, dqk, dv, nq, nk, n_splits):
    _check(A, 2, 3, nq, nk, dqk, dv, n_splits)


@pytest.mark.parametrize("dqk", [64, 128])
def test_splitkv_long_keys_one_range_per_tile(A, dqk):
    """16384 keys, one query per head, as many ranges as key tiles (128)."""
    _check(A, 1, 4, 1, 16384, dqk, dqk, 128, seed=4)


def test_splitkv_heuristic_choice(A):
    torch = G.torch_mod()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, H, Nq, Nk = 1, 8, 1, 16384
    n = A.attn_splitkv_heuristic(B, H, Nq, Nk, 128, sms)
    assert n > 1
    _check(A, B, H, Nq, Nk, 128, 128, n, seed=5)


def test_splitkv_ranges_agree_with_the_oracle_partition(A):
    """The library's ranges are the oracle's split_bounds: merging the oracle's
    partials over those ranges reproduces the GPU result as closely as the
    full attention does."""
    B, H, Nq, Nk, d, ns = 1, 2, 5, 1000, 128, 3
    t = synth.decode_inputs_torch(synth.DecodeShape(B, H, Nq, Nk, d, d), seed=6)
    o, lse = run_splitkv(A, t, ns)
    q, k, v = (G.f64(t[n]) for n in ("q", "k", "v"))
    bounds = om.split_bounds(Nk, ns)
    assert len(bounds) == ns + 1 and all(b1 > b0 for b0, b1 in zip(bounds[:-1], bounds[1:]))
    for h in range(H):
        parts = [om.partial_head(q[0, h], k[0, h], v[0, h], 1 / math.sqrt(d), a, b)
                 for a, b in zip(bounds[:-1], bounds[1:])]
        o_ref, lse_ref = om.merge([p[0] for p in parts], [p[1] for p in parts])
        G.assert_fwd_close(G.f64(o)[0, h], G.f64(lse)[0, h], o_ref, lse_ref)


@pytest.mark.parametrize("dv", [64, 128])
def test_merge_matches_oracle(A, dv):
    torch = G.torch_mod()
    rng = np.random.Generator(np.random.PCG64(9))
    S, BH, N = 5, 3, 37
    o_parts = rng.standard_normal((S, BH * N, dv)).astype(np.float32)
    lse_parts = (rng.standard_normal((S, BH * N)) * 4).astype(np.float32)
    lse_parts[1, :10] = -np.inf  # empty parts drop out
    lse_parts[:, 20] = -np.inf  # a row with no key at all
    o_parts[:, 20] = 0.0
    o = torch.empty((BH * N, dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(BH * N, dtype=torch.float32, device="cuda")
    A.attn_merge(torch.from_numpy(o_parts).cuda(), torch.from_numpy(lse_parts).cuda(), S, o, lse, BH, N, dv)
    G.check_status(A)
    o_ref, lse_ref = om.merge(o_parts.astype(np.float64), lse_parts.astype(np.float64))
    og, lg = G.f64(o), G.f64(lse)
    assert np.all(og[20] == 0) and np.isneginf(lg[20])
    live = np.isfinite(lse_ref)
    # bf16 output: one rounding of values of magnitude <~ 4
    assert np.abs(og - o_ref).max() <= G.O_MAX
    assert np.abs(lg[live] - lse_ref[live]).max() <= 1e-5 * max(1.0, np.abs(lse_ref[live]).max())


def test_merge_of_gpu_partials_is_the_gpu_full_forward(A):
    """attn_merge over two attn_fwd_splitkv calls on disjoint key halves gives
    the attention over all keys (the operator is associative)."""
    torch = G.torch_mod()
    B, H, Nq, Nk, d = 1, 2, 9, 512, 64
    t = synth.decode_inputs_torch(synth.DecodeShape(B, H, Nq, Nk, d, d), seed=8)
    halves = []
    for sl in (slice(0, 256), slice(256, 512)):
        th = {"q": t["q"], "k": t["k"][:, :, sl].contiguous(), "v": t["v"][:, :, sl].contiguous()}
        halves.append(run_splitkv(A, th, 1))
    o_parts = torch.stack([h[0].float().reshape(B * H * Nq, d) for h in halves])
    lse_parts = torch.stack([h[1].reshape(B * H * Nq) for h in halves])
    o = torch.empty((B * H * Nq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B * H * Nq, dtype=torch.float32, device="cuda")
    A.attn_merge(o_parts, lse_parts, 2, o, lse, B * H, Nq, d)
    G.check_status(A)
    o_ref, lse_ref = oracle_full(t, 1.0 / math.sqrt(d))
    G.assert_fwd_close(G.f64(o).reshape(o_ref.shape), G.f64(lse).reshape(lse_ref.shape), o_ref, lse_ref)
