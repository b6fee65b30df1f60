"""GPU parity tests of grouped-query attention (attn_fwd_gqa,
attn_fwd_splitkv_gqa, attn_bwd_gqa) against the FP64 oracle.

Query head h of H reads K/V head h // (H / H_kv); the oracle is the plain
attention of each query head against its K/V head (oracle/attention.py,
non-causal or causal).  Inputs: seeded bf16 N(0,1) tensors (synth), K and V
with H_kv heads.
"""
import math

import numpy as np
import pytest

import synth
from oracle import attention as ora
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


def _inputs(B, H, H_kv, N_q, N_k, dqk, dv, seed):
    tq = synth.decode_inputs_torch(synth.DecodeShape(B, H, N_q, 1, dqk, dv), seed=seed)
    tk = synth.decode_inputs_torch(synth.DecodeShape(B, H_kv, 1, N_k, dqk, dv), seed=seed + 1)
    return tq["q"], tk["k"], tk["v"]


def _oracle(q, k, v, causal):
    B, H = q.shape[:2]
    g = H // k.shape[1]
    o = np.empty(q.shape[:3] + (v.shape[-1],))
    lse = np.empty(q.shape[:3])
    scale = 1 / math.sqrt(q.shape[-1])
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = ora.forward_head(q[b, h], k[b, h // g], v[b, h // g], scale, causal)
    return o, lse


@pytest.mark.parametrize("dqk,dv", [(64, 64), (128, 128), (192, 128)])
@pytest.mark.parametrize("H,H_kv", [(8, 2), (6, 1), (4, 4)])
@pytest.mark.parametrize("N", [1, 300, 640])
@pytest.mark.parametrize("causal", [0, 1])
def test_forward_gqa(A, dqk, dv, H, H_kv, N, causal):
    torch = G.torch_mod()
    B = 2
    q, k, v = _inputs(B, H, H_kv, N, N, dqk, dv, seed=31)
    o = torch.empty((B, H, N, dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    A.attn_fwd_gqa(q, k, v, o, lse, B, H, H_kv, N, dqk, dv, causal, 1 / math.sqrt(dqk))
    G.check_status(A)
    o_ref, lse_ref = _oracle(G.f64(q), G.f64(k), G.f64(v), bool(causal))
    G.assert_fwd_close(G.f64(o), G.f64(lse), o_ref, lse_ref, f"H{H}/{H_kv} N{N} d{dqk} causal{causal}")


@pytest.mark.parametrize("H,H_kv,N_q", [(8, 2, 1), (8, 2, 5), (16, 1, 1), (32, 4, 3)])
@pytest.mark.parametrize("N_k", [1000, 4096])
@pytest.mark.parametrize("n_splits", [1, 4, 0])
def test_splitkv_gqa(A, H, H_kv, N_q, N_k, n_splits):
    torch = G.torch_mod()
    B, d = 2, 128
    q, k, v = _inputs(B, H, H_kv, N_q, N_k, d, d, seed=32)
    rows = (H // H_kv) * N_q
    if n_splits == 0:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        n_splits = A.attn_splitkv_heuristic(B, H_kv, rows, N_k, d, sms)
    nb = A.attn_fwd_splitkv_workspace_bytes(B, H_kv, rows, N_k, d, n_splits)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    o = torch.empty((B, H, N_q, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N_q), dtype=torch.float32, device="cuda")
    A.attn_fwd_splitkv_gqa(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, d, 1 / math.sqrt(d), n_splits, ws, nb)
    G.check_status(A)
    o_ref, lse_ref = _oracle(G.f64(q), G.f64(k), G.f64(v), False)
    G.assert_fwd_close(G.f64(o), G.f64(lse), o_ref, lse_ref, f"H{H}/{H_kv} Nq{N_q} Nk{N_k} splits{n_splits}")


def _oracle_bwd(q, k, v, do, causal):
    """dQ per query head; dK, dV of a K/V head summed over its query heads."""
    B, H = q.shape[:2]
    H_kv = k.shape[1]
    g = H // H_kv
    scale = 1 / math.sqrt(q.shape[-1])
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            a, kb, c = ora.backward_head(q[b, h], k[b, h // g], v[b, h // g], do[b, h], scale, causal)
            dq[b, h] = a
            dk[b, h // g] += kb
            dv[b, h // g] += c
    return dq, dk, dv


def _run_bwd_gqa(A, q, k, v, do, causal, det):
    torch = G.torch_mod()
    B, H, N, dqk = q.shape
    H_kv, dv_ = k.shape[1], v.shape[-1]
    scale = 1 / math.sqrt(dqk)
    o = torch.empty((B, H, N, dv_), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    A.attn_fwd_gqa(q, k, v, o, lse, B, H, H_kv, N, dqk, dv_, causal, scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nb = A.attn_bwd_workspace_bytes(B, H, N, dqk, dv_, det)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    A.attn_bwd_gqa(q, k, v, o, do, lse, dq, dk, dv, B, H, H_kv, N, dqk, dv_, causal, scale, det, ws, nb)
    return dq, dk, dv


@pytest.mark.parametrize("dqk,dv", [(64, 64), (128, 128), (192, 128)])
@pytest.mark.parametrize("H,H_kv", [(8, 2), (6, 1), (4, 4)])
@pytest.mark.parametrize("N", [1, 257, 640])
@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("det", [0, 1])
def test_backward_gqa(A, dqk, dv, H, H_kv, N, causal, det):
    B = 2
    q, k, v = _inputs(B, H, H_kv, N, N, dqk, dv, seed=33)
    do = synth.decode_inputs_torch(synth.DecodeShape(B, H, N, 1, dv, dv), seed=34)["q"]
    grads = _run_bwd_gqa(A, q, k, v, do, causal, det)
    G.check_status(A)
    refs = _oracle_bwd(G.f64(q), G.f64(k), G.f64(v), G.f64(do), bool(causal))
    for name, got, ref in zip(("dq", "dk", "dv"), grads, refs):
        G.assert_grad_close(name, G.f64(got), ref)


def test_backward_gqa_deterministic_is_bit_identical(A):
    torch = G.torch_mod()
    B, H, H_kv, N, d = 2, 8, 2, 1000, 128
    q, k, v = _inputs(B, H, H_kv, N, N, d, d, seed=35)
    do = synth.decode_inputs_torch(synth.DecodeShape(B, H, N, 1, d, d), seed=36)["q"]
    for causal in (0, 1):
        runs = [_run_bwd_gqa(A, q, k, v, do, causal, 1) for _ in range(3)]
        G.check_status(A)
        for r in runs[1:]:
            for a, b in zip(runs[0], r):
                assert torch.equal(a.view(torch.int16), b.view(torch.int16))
