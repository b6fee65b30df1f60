"""Helpers shared by the GPU tests: run the CUDA path through the C ABI, move
results to FP64 numpy, and compare with the oracle under the stated tolerances.

Tolerances (FP64 oracle vs the BF16 GPU path on identical inputs):
  forward O:  max |err| <= 2e-2 and mean |err| <= 2e-3
  LSE:        max |err| <= 1e-3
  dQ, dK, dV: relative Frobenius error <= 1e-2
"""
from __future__ import annotations

import math

import numpy as np

import synth

O_MAX, O_MEAN, LSE_MAX, GRAD_REL = 2e-2, 2e-3, 1e-3, 1e-2


def torch_mod():
    import torch

    return torch


def f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def inputs(B, H, N, dqk, dv, seed=0, with_do=True):
    shape = synth.AttentionShape(B, H, N, dqk, dv)
    return synth.attention_inputs_torch(shape, seed=seed, with_do=with_do, device="cuda")


def run_fwd(A, t, causal, scale=None):
    torch = torch_mod()
    q, k, v = t["q"], t["k"], t["v"]
    B, H, N, dqk = q.shape
    dv = v.shape[-1]
    scale = 1.0 / math.sqrt(dqk) if scale is None else scale
    o = torch.empty((B, H, N, dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    A.attn_fwd(q, k, v, o, lse, B, H, N, dqk, dv, int(causal), scale)
    return o, lse


def run_bwd(A, t, o, lse, causal, deterministic, scale=None):
    torch = torch_mod()
    q, k, v, do = t["q"], t["k"], t["v"], t["do"]
    B, H, N, dqk = q.shape
    dv = v.shape[-1]
    scale = 1.0 / math.sqrt(dqk) if scale is None else scale
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dvt = torch.empty_like(v)
    nbytes = A.attn_bwd_workspace_bytes(B, H, N, dqk, dv, int(deterministic))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    A.attn_bwd(q, k, v, o, do, lse, dq, dk, dvt, B, H, N, dqk, dv, int(causal), scale, int(deterministic), ws, nbytes)
    return dq, dk, dvt


def check_status(A):
    st, where = A.attn_get_device_status()
    assert st == 0, (A.status_string(st), where)


def assert_fwd_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    err = np.abs(o_gpu - o_ref)
    lerr = np.abs(lse_gpu - lse_ref)
    assert err.max() <= O_MAX, f"{what} O max abs err {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what} O mean abs err {err.mean():.3e}"
    assert lerr.max() <= LSE_MAX, f"{what} LSE max abs err {lerr.max():.3e}"
    return float(err.max()), float(err.mean()), float(lerr.max())


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_grad_close(name, got, ref):
    """Relative Frobenius error <= 1e-2; where the exact gradient is zero (one
    key: the softmax is constant), the result must be zero up to rounding."""
    if np.linalg.norm(ref) == 0.0:
        assert np.abs(got).max() <= 1e-3, (name, float(np.abs(got).max()))
        return 0.0
    e = rel_fro(got, ref)
    assert e <= GRAD_REL, (name, e)
    return e


def seeded_rows(n, count, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = rng.choice(n, size=min(count, n), replace=False)
    # always include the first and the last rows (the causal extremes / ragged tail)
    return np.unique(np.concatenate([rows, [0, n - 1]]))
