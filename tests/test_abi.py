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
    # atomic mode at d <= 128 adds the persistent kernel's region for the
    # pieces of cut units: FP32 dV + dK, 128 rows each, for min(160, units - 1)
    # pieces
    pieces = min(160, b * h * 3 - 1)
    assert lib.attn_bwd_workspace_bytes(b, h, n, d, d, 0) == base + pieces * 2 * 128 * d * 4
    assert lib.attn_bwd_workspace_bytes(b, h, n, d, d, 1) == base + 256
    assert lib.attn_bwd_workspace_bytes(1, 1, 100, d, d, 0) == 2 * 128 * 4 + 128 * d * 4  # one unit: never cut
    assert lib.attn_bwd_workspace_bytes(4, 16, 1024, 128, 128, 0) == (
        2 * 64 * 1024 * 4 + 64 * 1024 * 128 * 4 + 160 * 2 * 128 * 128 * 4)
    # d_qk = 192: the accumulator is d_qk wide
    assert lib.attn_bwd_workspace_bytes(1, 1, 128, 192, 128, 0) == 2 * 128 * 4 + 128 * 192 * 4
    assert lib.attn_bwd_workspace_bytes(1, 1, 128, 192, 192, 0) == 0
    assert lib.attn_bwd_workspace_bytes(1, 1, 128, 128, 64, 0) == 0
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
    assert _fwd(lib, scale=-0.125) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=0.0) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, dqk=96, dv=96) == A.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, dqk=128, dv=64) == A.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, k=0x1008) == A.ATTN_ERR_MISALIGNED
    assert _fwd(lib, lse=0x1004) == A.ATTN_ERR_MISALIGNED


def test_backward_argument_errors(lib):
    A = lib
    f = lib.get_lib().attn_bwd
    p = 0x1000
    ok_ws = lib.attn_bwd_workspace_bytes(1, 2, 256, 64, 64, 0)
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 192, 192, 0, 0.1, 0, p, ok_ws, None) == A.ATTN_ERR_UNSUPPORTED
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 96, 96, 0, 0.1, 0, p, ok_ws, None) == A.ATTN_ERR_UNSUPPORTED
    # (192, 128) is supported; a workspace sized for d = 64 is too small for it
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 192, 128, 0, 0.1, 0, p, ok_ws, None) == A.ATTN_ERR_WORKSPACE
    assert f(p, p, p, p, 0, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 0, p, ok_ws, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 3, p, ok_ws, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 0, None, ok_ws, None) == A.ATTN_ERR_WORKSPACE
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 0, p, ok_ws - 1, None) == A.ATTN_ERR_WORKSPACE
    # deterministic mode: tickets, and no region for cut units (atomic only)
    det_ws = lib.attn_bwd_workspace_bytes(1, 2, 256, 64, 64, 1)
    assert det_ws != ok_ws
    assert f(p, p, p, p, p, p, p, p, p, 1, 2, 256, 64, 64, 0, 0.1, 1, p, det_ws - 1, None) == A.ATTN_ERR_WORKSPACE
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
    assert lib.get_lib().attn_set_bwd_persist(2) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_set_bwd_persist(-2) == A.ATTN_ERR_INVALID_ARG
    for m in (1, 0, -1):
        assert lib.get_lib().attn_set_bwd_persist(m) == A.ATTN_OK
    assert lib.get_lib().attn_set_fwd_persist(2) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_set_fwd_persist(-2) == A.ATTN_ERR_INVALID_ARG
    for m in (1, 0, -1):
        assert lib.get_lib().attn_set_fwd_persist(m) == A.ATTN_OK
    assert lib.get_lib().attn_set_exp_poly(2) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_set_exp_poly(-1) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_set_exp_poly(1) == A.ATTN_OK
    assert lib.get_lib().attn_set_exp_poly(0) == A.ATTN_OK
    assert lib.get_lib().attn_set_det_schedule(-1, 0) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_set_det_schedule(4, 2) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_set_det_schedule(4, 1) == A.ATTN_OK
    assert lib.get_lib().attn_set_det_schedule(0, 0) == A.ATTN_OK
    assert lib.get_lib().attn_selftest_wait_timeout(0, None) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_exp2_probe(None, None, 4, 0, None) == A.ATTN_ERR_INVALID_ARG
    assert lib.get_lib().attn_exp2_probe(0x1000, 0x1000, 4, 7, None) == A.ATTN_ERR_INVALID_ARG


def test_splitkv_geometry_and_workspace(lib):
    A = lib
    # 1000 keys = 8 tiles; 3 requested ranges -> 3 tiles each -> ranges of 3, 3, 2 tiles
    rows = 3 * 2 * 5  # ranges * B * H * N_q
    want = -(-(rows * 128 * 4) // 256) * 256 + rows * 4
    assert A.attn_fwd_splitkv_workspace_bytes(1, 2, 5, 1000, 128, 3) == -(-want // 256) * 256
    # more ranges requested than tiles: one range per tile
    assert A.attn_fwd_splitkv_workspace_bytes(1, 1, 1, 300, 64, 50) == A.attn_fwd_splitkv_workspace_bytes(1, 1, 1, 300, 64, 3)
    # 8 tiles, 5 requested -> 2 tiles each -> 4 ranges
    assert A.attn_fwd_splitkv_workspace_bytes(1, 1, 1, 1000, 64, 5) == A.attn_fwd_splitkv_workspace_bytes(1, 1, 1, 1000, 64, 4)
    assert A.attn_fwd_splitkv_workspace_bytes(1, 1, 1, 1000, 96, 2) == 0
    assert A.attn_fwd_splitkv_workspace_bytes(1, 1, 0, 1000, 64, 2) == 0
    assert A.attn_fwd_splitkv_workspace_bytes(1, 1, 1, 1000, 64, 0) == 0


def test_splitkv_heuristic(lib):
    A = lib
    h = A.attn_splitkv_heuristic
    # decode (N_q <= 128, d <= 128): one-tile units, two CTAs per SM -> 296
    # slots on 148 SMs.  8 units -> 32 ranges (256 <= 296 < 512)
    assert h(1, 8, 1, 16384, 128, 148) == 32
    assert h(1, 8, 1, 16384, 128, 152) == 32
    assert h(1, 16, 1, 16384, 64, 152) == 16
    # 160 units > 304 / 2: no split
    assert h(1, 160, 1, 16384, 128, 152) == 1
    # d = 192: two-tile units, one CTA per SM -> 8 units -> 16 ranges
    assert h(1, 8, 1, 16384, 192, 152) == 16
    # 200 queries: two-tile units (1 per head), one CTA per SM -> 128 ranges, capped
    # at two tiles each: 8192 keys = 64 tiles -> 32 ranges
    assert h(1, 1, 200, 8192, 128, 152) == 32
    # short key sequences: each range at least two tiles
    assert h(1, 1, 1, 1024, 128, 148) == 4
    assert h(1, 1, 1, 128, 128, 148) == 1
    assert h(1, 1, 1, 0, 128, 148) == 0
    assert h(1, 1, 1, 100, 128, 0) == 0
    assert h(1, 1, 1, 100, 96, 148) == 0


def test_splitkv_and_merge_argument_errors(lib):
    A = lib
    f = lib.get_lib().attn_fwd_splitkv
    p = 0x1000
    ws = A.attn_fwd_splitkv_workspace_bytes(1, 2, 1, 1000, 128, 4)
    args = dict(q=p, k=p, v=p, o=p, lse=p, B=1, H=2, Nq=1, Nk=1000, dqk=128, dv=128, scale=0.1, ns=4, w=p, wb=ws)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"], a["dqk"], a["dv"],
                 a["scale"], a["ns"], a["w"], a["wb"], None)

    assert call(q=0) == A.ATTN_ERR_INVALID_ARG
    assert call(Nk=0) == A.ATTN_ERR_INVALID_ARG
    assert call(ns=0) == A.ATTN_ERR_INVALID_ARG
    assert call(scale=float("nan")) == A.ATTN_ERR_INVALID_ARG
    assert call(dqk=96, dv=96) == A.ATTN_ERR_UNSUPPORTED
    assert call(v=0x1008) == A.ATTN_ERR_MISALIGNED
    assert call(w=None) == A.ATTN_ERR_WORKSPACE
    assert call(wb=ws - 1) == A.ATTN_ERR_WORKSPACE
    assert call(w=0x1004) == A.ATTN_ERR_MISALIGNED
    m = lib.get_lib().attn_merge
    assert m(p, p, 0, p, p, 1, 1, 128, None) == A.ATTN_ERR_INVALID_ARG
    assert m(p, None, 2, p, p, 1, 1, 128, None) == A.ATTN_ERR_INVALID_ARG
    assert m(p, p, 2, p, p, 1, 1, 192, None) == A.ATTN_ERR_UNSUPPORTED
    assert m(p, 0x1004, 2, p, p, 1, 1, 128, None) == A.ATTN_ERR_MISALIGNED


def test_fp8_argument_errors(lib):
    A = lib
    L = lib.get_lib()
    p = 0x1000
    ws = A.attn_fp8_quantize_workspace_bytes(1, 2)
    assert ws == 256 and A.attn_fp8_quantize_workspace_bytes(0, 2) == 0
    signs = [1, -1] * 64

    def quant(**kw):
        a = dict(q=p, k=p, v=p, signs=signs, q8=p, k8=p, v8=p, sq=p, sk=p, sv=p, B=1, H=2, N=300, d=128, w=p, wb=ws)
        a.update(kw)
        return A.attn_fp8_quantize(a["q"], a["k"], a["v"], a["signs"], a["q8"], a["k8"], a["v8"], a["sq"], a["sk"],
                                   a["sv"], a["B"], a["H"], a["N"], a["d"], a["w"], a["wb"], stream=0, check=False)

    assert quant(q=0) == A.ATTN_ERR_INVALID_ARG
    assert quant(signs=[1] * 127 + [0]) == A.ATTN_ERR_INVALID_ARG
    assert quant(d=64, signs=[1] * 64) == A.ATTN_ERR_UNSUPPORTED
    assert quant(sk=0x1004) == A.ATTN_ERR_MISALIGNED
    assert quant(w=None) == A.ATTN_ERR_WORKSPACE
    assert quant(wb=ws - 4) == A.ATTN_ERR_WORKSPACE
    f = L.attn_fwd_fp8
    assert f(p, p, p, p, p, p, p, p, 1, 2, 300, 128, 0, -1.0, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, 0, p, p, 1, 2, 300, 128, 0, 0.1, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, p, p, p, 1, 2, 300, 64, 0, 0.1, None) == A.ATTN_ERR_UNSUPPORTED
    assert f(p, 0x1001, p, p, p, p, p, p, 1, 2, 300, 128, 0, 0.1, None) == A.ATTN_ERR_MISALIGNED
    assert f(p, p, p, p, p, p, p, p, 1, 2, 300, 128, 2, 0.1, None) == A.ATTN_ERR_INVALID_ARG


def test_masked_argument_errors(lib):
    A = lib
    L = lib.get_lib()
    p = 0x1000
    f = L.attn_fwd_masked
    assert f(p, p, p, p, p, 1, 2, 300, 128, 128, -2, 0, None, 0.1, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, 1, 2, 300, 128, 128, 5, -3, None, 0.1, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, 1, 2, 300, 192, 128, -1, 0, None, 0.1, None) == A.ATTN_ERR_UNSUPPORTED
    assert f(p, p, p, p, p, 1, 2, 300, 128, 128, -1, 0, 0x1003, 0.1, None) == A.ATTN_ERR_MISALIGNED
    assert f(0, p, p, p, p, 1, 2, 300, 128, 128, -1, 0, None, 0.1, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, 1, 2, 300, 128, 128, -1, 0, None, -0.1, None) == A.ATTN_ERR_INVALID_ARG
    b = L.attn_bwd_masked
    ws = A.attn_bwd_workspace_bytes(1, 2, 300, 64, 64, 0)
    assert b(p, p, p, p, p, p, p, p, p, 1, 2, 300, 64, 64, -2, 0, None, 0.1, 0, p, ws, None) == A.ATTN_ERR_INVALID_ARG
    assert b(p, p, p, p, p, p, p, p, p, 1, 2, 300, 64, 64, 16, 0, None, 0.1, 0, p, ws - 1, None) == A.ATTN_ERR_WORKSPACE
    assert b(p, p, p, p, p, p, p, p, p, 1, 2, 300, 64, 64, 16, 0, 0x1001, 0.1, 0, p, ws, None) == A.ATTN_ERR_MISALIGNED
    assert b(p, p, p, p, p, p, p, p, p, 1, 2, 300, 64, 64, 16, 0, None, 0.1, 2, p, ws, None) == A.ATTN_ERR_INVALID_ARG
    ws192 = A.attn_bwd_workspace_bytes(1, 2, 300, 192, 128, 0)
    assert ws192 > 0
    assert b(p, p, p, p, p, p, p, p, p, 1, 2, 300, 192, 128, 16, 0, None, 0.1, 0, p, ws192, None) == A.ATTN_ERR_UNSUPPORTED


def test_gqa_argument_errors(lib):
    A = lib
    L = lib.get_lib()
    p = 0x1000
    assert L.attn_fwd_gqa(p, p, p, p, p, 1, 8, 3, 256, 128, 128, 0, 0.1, None) == A.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_gqa(p, p, p, p, p, 1, 8, 0, 256, 128, 128, 0, 0.1, None) == A.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_gqa(p, p, p, p, p, 1, 8, 2, 256, 96, 96, 0, 0.1, None) == A.ATTN_ERR_UNSUPPORTED
    f = L.attn_fwd_splitkv_gqa
    ws = A.attn_fwd_splitkv_workspace_bytes(1, 2, 4, 1000, 128, 2)
    assert f(p, p, p, p, p, 1, 8, 3, 1, 1000, 128, 128, 0.1, 2, p, ws, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, 1, 8, 2, 0, 1000, 128, 128, 0.1, 2, p, ws, None) == A.ATTN_ERR_INVALID_ARG
    assert f(p, p, p, p, p, 1, 8, 2, 1, 1000, 128, 128, 0.1, 2, p, ws - 1, None) == A.ATTN_ERR_WORKSPACE
    ws2 = A.attn_bwd_workspace_bytes(1, 8, 256, 128, 128, 0)
    g = L.attn_bwd_gqa
    assert g(p, p, p, p, p, p, p, p, p, 1, 8, 3, 256, 128, 128, 0, 0.1, 0, p, ws2, None) == A.ATTN_ERR_INVALID_ARG
    assert g(p, p, p, p, p, p, p, p, p, 1, 8, 16, 256, 128, 128, 0, 0.1, 0, p, ws2, None) == A.ATTN_ERR_INVALID_ARG
    assert g(p, p, p, p, p, p, p, p, p, 1, 8, 2, 256, 128, 128, 0, 0.1, 0, p, ws2 - 1, None) == A.ATTN_ERR_WORKSPACE
