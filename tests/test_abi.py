"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports every
symbol include/attn.h declares, and rejects bad arguments before touching CUDA.

No compute call is made here: every call below fails argument validation,
which happens on the host before any CUDA API is used.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    from exact_attention_77_gb300 import build

    build.build()
    import exact_attention_77_gb300 as A

    return A


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes", "attn_get_device_status",
                     "attn_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (attn_[a-z0-9_]+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    # the binding wraps each of them under the same name
    for n in _declared():
        assert hasattr(lib, n), n


def test_library_links_no_gpu_driver(lib):
    out = subprocess.run(["ldd", lib._LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_status_strings(lib):
    assert lib.status_string(0) == "ATTN_OK"
    assert lib.status_string(6) == "ATTN_ERR_TIMEOUT"
    assert lib.status_string(99) == "ATTN_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    # D and LSE2 rows padded to 128, the fp32 dQ accumulator, tickets in deterministic mode
    b, h, n, d = 1, 2, 300, 64
    npad = 384
    base = 2 * b * h * npad * 4 + b * h * npad * d * 4
    assert lib.attn_bwd_workspace_bytes(b, h, n, d, d, 0) == base
    assert lib.attn_bwd_workspace_bytes(b, h, n, d, d, 1) == base + 256
    assert lib.attn_bwd_workspace_bytes(1, 1, 128, 192, 128, 0) == 0
    assert lib.attn_bwd_workspace_bytes(0, 1, 128, 64, 64, 0) == 0


def _fwd(lib, q=0x1000, k=0x1000, v=0x1000, o=0x1000, lse=0x1000, B=1, H=2, N=256, dqk=64, dv=64, causal=0,
         scale=0.125):
    return lib.get_lib().attn_fwd(q, k, v, o, lse, B, H, N, dqk, dv, causal, scale, None)


def test_forward_argument_errors(lib):
    A = lib
    assert _fwd(lib, q=0) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, N=0) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, B=-1) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, N=1 << 24) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, causal=2) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("inf")) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, dqk=96, dv=96) == A.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, dqk=128, dv=64) == A.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, k=0x1008) == A.ATTN_ERR_MISALIGNED
    assert _fwd(lib, lse=0x1004) == A.ATTN_ERR_MISALIGNED


def test_backward_argument_errors(lib):
    A = lib
    f = lib.get_lib().attn_bwd
    p = 0x1000
    ok_ws = lib.attn_bwd_workspace_bytes(1, 2, 256, 64, 64, 0)
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 192, 128, 0, 0.1, 0, p, ok_ws, None) == A.ATTN_ERR_UNSUPPORTED
    assert f(p, p, p, p, 0, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 0, p, ok_ws, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 3, p, ok_ws, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 0, None, ok_ws, None) == A.ATTN_ERR_WORKSPACE
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 0, p, ok_ws - 1, None) == A.ATTN_ERR_WORKSPACE
    det_ws = lib.attn_bwd_workspace_bytes(1, 2, 256, 64, 64, 1)
    assert det_ws > ok_ws
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 1, p, ok_ws, None) == A.ATTN_ERR_WORKSPACE
    assert f(p, p, p, p, p, p, p, 0x1002, p, 1, 2, 256, 64, 64, 0, 0.1, 0, p, ok_ws, None) == A.ATTN_ERR_MISALIGNED
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 0, 0x1004, ok_ws, None) == A.ATTN_ERR_MISALIGNED


def test_tuning_setters(lib):
    A = lib
    assert lib.get_lib().attn_set_rescale_threshold(-1.0) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_set_rescale_threshold(float("nan")) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_set_rescale_threshold(8.0) == A.ATTN_OK
    assert lib.get_lib().attn_set_bwd_pair(2) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_set_bwd_pair(1) == A.ATTN_OK
    assert lib.get_lib().attn_set_bwd_pair(0) == A.ATTN_OK
    assert lib.get_lib().attn_selftest_wait_timeout(0, None) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_exp2_probe(None, None, 4, 0, None) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_exp2_probe(0x1000, 0x1000, 4, 7, None) == A.ATTN_ERR_INVALID_ARG
