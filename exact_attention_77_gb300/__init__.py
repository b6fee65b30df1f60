"""Python binding of libattn.so (the GB300 exact-attention library).

Argument marshalling only: every function forwards to the C entry point of
the same name declared in include/attn.h.  Pointer arguments accept torch
tensors (their ``data_ptr()``) or plain integers; ``stream`` defaults to the
current torch CUDA stream.  Non-zero status codes raise ``AttnError``.

The library must have been built (``python -m exact_attention_77_gb300.build``);
the first call without it raises ImportError: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_WORKSPACE = 4
ATTN_ERR_CUDA = 5
ATTN_ERR_TIMEOUT = 6
ATTN_ERR_BOUNDS = 7

# name -> (restype, argtypes), mirroring include/attn.h
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SIGS = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, ctypes.c_size_t, _P]),
    "attn_get_device_status": (_I, [_P, ctypes.POINTER(_I)]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_exp2_probe": (_I, [_P, _P, _I, _I, _P]),
    "attn_exp2_throughput": (_I, [_P, _I, _I, _I, _P]),
    "attn_set_rescale_counter": (_I, [_P]),
    "attn_set_rescale_threshold": (_I, [_F]),
    "attn_set_bwd_pair": (_I, [_I]),
    "attn_set_fwd_persist": (_I, [_I]),
    "attn_set_bwd_persist": (_I, [_I]),
    "attn_set_exp_poly": (_I, [_I]),
    "attn_set_det_schedule": (_I, [_I, _I]),
    "attn_bwd_det_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "attn_selftest_wait_timeout": (_I, [ctypes.c_uint, _P]),
    "attn_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_fwd_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, ctypes.c_size_t, _P]),
    "attn_fwd_splitkv_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "attn_splitkv_heuristic": (_I, [_I, _I, _I, _I, _I, _I]),
    "attn_merge": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _P]),
    "attn_fp8_quantize_workspace_bytes": (ctypes.c_size_t, [_I, _I]),
    "attn_fp8_quantize": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, ctypes.c_size_t, _P]),
    "attn_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_masked": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _F, _P]),
    "attn_bwd_masked": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _F, _I, _P,
                             ctypes.c_size_t, _P]),
    "attn_fwd_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_splitkv_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, ctypes.c_size_t, _P]),
    "attn_bwd_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, ctypes.c_size_t,
                          _P]),
    "attn_profile_start": (_I, []),
    "attn_profile_stop": (_I, [_P]),
}


class attn_kernel_times_t(ctypes.Structure):
    _fields_ = [("launches_fwd", _I), ("launches_bwd_pre", _I), ("launches_bwd_main", _I),
                ("launches_bwd_convert", _I), ("ms_fwd", _F), ("ms_bwd_pre", _F), ("ms_bwd_main", _F),
                ("ms_bwd_convert", _F), ("launches_fwd_split", _I), ("launches_merge", _I), ("ms_fwd_split", _F),
                ("ms_merge", _F)]


class AttnError(RuntimeError):
    def __init__(self, status: int, where: int = 0):
        self.status = status
        self.where = where
        super().__init__(f"{status_string(status)} (status {status}, where {where})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is not built; run `python -m exact_attention_77_gb300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_LIB = None


def get_lib() -> ctypes.CDLL:
    """The loaded libattn.so (loaded on first use; ImportError if not built)."""
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != ATTN_OK:
        raise AttnError(status)


def status_string(status: int) -> str:
    return get_lib().attn_status_string(status).decode()


attn_status_string = status_string


def attn_fwd(q, k, v, o, lse, B, H, N, d_qk, d_v, causal, scale, stream=None, check=True) -> int:
    st = get_lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d_qk, d_v, int(causal), float(scale),
                      _stream(stream))
    if check:
        _check(st)
    return st


def attn_bwd_workspace_bytes(B, H, N, d_qk, d_v, deterministic) -> int:
    return get_lib().attn_bwd_workspace_bytes(B, H, N, d_qk, d_v, int(deterministic))


def attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d_qk, d_v, causal, scale, deterministic, workspace,
             workspace_bytes, stream=None, check=True) -> int:
    st = get_lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N,
                      d_qk, d_v, int(causal), float(scale), int(deterministic), _ptr(workspace), int(workspace_bytes),
                      _stream(stream))
    if check:
        _check(st)
    return st


def attn_fwd_splitkv(q, k, v, o, lse, B, H, N_q, N_k, d_qk, d_v, scale, n_splits, workspace, workspace_bytes,
                     stream=None, check=True) -> int:
    st = get_lib().attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N_q, N_k, d_qk, d_v,
                                    float(scale), int(n_splits), _ptr(workspace), int(workspace_bytes),
                                    _stream(stream))
    if check:
        _check(st)
    return st


def attn_fwd_splitkv_workspace_bytes(B, H, N_q, N_k, d_v, n_splits) -> int:
    return get_lib().attn_fwd_splitkv_workspace_bytes(B, H, N_q, N_k, d_v, int(n_splits))


def attn_splitkv_heuristic(B, H, N_q, N_k, d_qk, n_sms) -> int:
    return get_lib().attn_splitkv_heuristic(B, H, N_q, N_k, d_qk, int(n_sms))


def attn_merge(o_parts, lse_parts, n_parts, o, lse, BH, N, d_v, stream=None, check=True) -> int:
    st = get_lib().attn_merge(_ptr(o_parts), _ptr(lse_parts), int(n_parts), _ptr(o), _ptr(lse), BH, N, d_v,
                              _stream(stream))
    if check:
        _check(st)
    return st


def attn_fp8_quantize_workspace_bytes(B, H) -> int:
    return get_lib().attn_fp8_quantize_workspace_bytes(B, H)


def attn_fp8_quantize(q, k, v, signs, q8, k8, v8, sq, sk, sv, B, H, N, d, workspace, workspace_bytes, stream=None,
                      check=True) -> int:
    """``signs``: a host sequence of d values, each +1 or -1."""
    arr = (ctypes.c_byte * len(signs))(*[int(x) for x in signs])
    st = get_lib().attn_fp8_quantize(_ptr(q), _ptr(k), _ptr(v), ctypes.cast(arr, _P), _ptr(q8), _ptr(k8), _ptr(v8),
                                     _ptr(sq), _ptr(sk), _ptr(sv), B, H, N, d, _ptr(workspace), int(workspace_bytes),
                                     _stream(stream))
    if check:
        _check(st)
    return st


def attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, B, H, N, d, causal, scale, stream=None, check=True) -> int:
    st = get_lib().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(sq), _ptr(sk), _ptr(sv), _ptr(o), _ptr(lse), B, H,
                                N, d, int(causal), float(scale), _stream(stream))
    if check:
        _check(st)
    return st


def attn_fwd_masked(q, k, v, o, lse, B, H, N, d_qk, d_v, window_left, window_right, block_mask, scale, stream=None,
                    check=True) -> int:
    st = get_lib().attn_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d_qk, d_v, int(window_left),
                                   int(window_right), _ptr(block_mask), float(scale), _stream(stream))
    if check:
        _check(st)
    return st


def attn_bwd_masked(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d_qk, d_v, window_left, window_right, block_mask, scale,
                    deterministic, workspace, workspace_bytes, stream=None, check=True) -> int:
    st = get_lib().attn_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
                                   _ptr(dv), B, H, N, d_qk, d_v, int(window_left), int(window_right), _ptr(block_mask),
                                   float(scale), int(deterministic), _ptr(workspace), int(workspace_bytes),
                                   _stream(stream))
    if check:
        _check(st)
    return st


def attn_fwd_gqa(q, k, v, o, lse, B, H, H_kv, N, d_qk, d_v, causal, scale, stream=None, check=True) -> int:
    st = get_lib().attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, H_kv, N, d_qk, d_v, int(causal),
                                float(scale), _stream(stream))
    if check:
        _check(st)
    return st


def attn_fwd_splitkv_gqa(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d_qk, d_v, scale, n_splits, workspace,
                         workspace_bytes, stream=None, check=True) -> int:
    st = get_lib().attn_fwd_splitkv_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, H_kv, N_q, N_k, d_qk,
                                        d_v, float(scale), int(n_splits), _ptr(workspace), int(workspace_bytes),
                                        _stream(stream))
    if check:
        _check(st)
    return st


def attn_bwd_gqa(q, k, v, o, dO, lse, dq, dk, dv, B, H, H_kv, N, d_qk, d_v, causal, scale, deterministic, workspace,
                 workspace_bytes, stream=None, check=True) -> int:
    st = get_lib().attn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                                B, H, H_kv, N, d_qk, d_v, int(causal), float(scale), int(deterministic),
                                _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check:
        _check(st)
    return st


ATTN_NOALLOC_SCRATCH_BYTES = 32 << 20


def attn_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d_qk, d_v, causal, scale, deterministic, stream=None,
                     check=True) -> int:
    """attn_bwd with the library's built-in scratch array as workspace (no allocation)."""
    st = get_lib().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
                                    _ptr(dv), B, H, N, d_qk, d_v, int(causal), float(scale), int(deterministic),
                                    _stream(stream))
    if check:
        _check(st)
    return st


def attn_get_device_status(stream=None):
    """(status, where) after synchronising ``stream``; clears the device word."""
    where = ctypes.c_int(0)
    st = get_lib().attn_get_device_status(_stream(stream), ctypes.byref(where))
    return st, where.value


def attn_exp2_probe(x, out, n, method, stream=None):
    _check(get_lib().attn_exp2_probe(_ptr(x), _ptr(out), n, method, _stream(stream)))


def attn_exp2_throughput(sink, blocks, iters, method, stream=None):
    _check(get_lib().attn_exp2_throughput(_ptr(sink), blocks, iters, method, _stream(stream)))


def attn_set_rescale_counter(counter):
    _check(get_lib().attn_set_rescale_counter(_ptr(counter)))


def attn_set_rescale_threshold(tau: float):
    _check(get_lib().attn_set_rescale_threshold(float(tau)))


def attn_set_bwd_pair(enable: int):
    _check(get_lib().attn_set_bwd_pair(int(enable)))


def attn_set_fwd_persist(mode: int):
    _check(get_lib().attn_set_fwd_persist(int(mode)))


def attn_set_bwd_persist(mode: int):
    _check(get_lib().attn_set_bwd_persist(int(mode)))


def attn_set_exp_poly(enable: int):
    _check(get_lib().attn_set_exp_poly(int(enable)))


def attn_set_det_schedule(head_group: int, descending: int):
    _check(get_lib().attn_set_det_schedule(int(head_group), int(descending)))


def attn_bwd_det_plan(n_heads: int, n_tiles: int, n_ctas: int, head_group: int, descending: int = 0,
                      causal: int = 0, rotated: int = 0) -> dict:
    """The deterministic backward's plan as the kernels compute it (host only):
    per unit u its head, key tile and first query tile, and rank[u, i], the
    ticket value at which its dQ addition to query tile i goes ahead (-1: not
    visited).  Returns numpy int32 arrays."""
    import numpy as np
    n_units = int(n_heads) * int(n_tiles)
    head = np.zeros(n_units, np.int32)
    key = np.zeros(n_units, np.int32)
    first = np.zeros(n_units, np.int32)
    rank = np.zeros((n_units, int(n_tiles)), np.int32)
    _check(get_lib().attn_bwd_det_plan(int(n_heads), int(n_tiles), int(n_ctas), int(head_group), int(descending),
                                       int(causal), int(rotated), head.ctypes.data, key.ctypes.data,
                                       first.ctypes.data, rank.ctypes.data))
    return {"head": head, "key_tile": key, "first_tile": first, "rank": rank}


def attn_selftest_wait_timeout(timeout_us: int, stream=None):
    _check(get_lib().attn_selftest_wait_timeout(int(timeout_us), _stream(stream)))


def attn_profile_start():
    _check(get_lib().attn_profile_start())


def attn_profile_stop() -> dict:
    """Stop per-kernel timing; returns launch counts and summed milliseconds per kernel."""
    t = attn_kernel_times_t()
    _check(get_lib().attn_profile_stop(ctypes.byref(t)))
    return {name: getattr(t, name) for name, _ in attn_kernel_times_t._fields_}
