"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers of this library run where they may not allocate: inside a host
callback, or within a runtime that owns every device buffer and refuses
allocations while serving.  attn_bwd_noalloc gives them the backward pass with
the workspace taken from a fixed array inside the library.  This test calls it
through the C ABI twice in a row (the second call sees the first call's
leftovers in the shared array) and checks dq, dk, dv against attn_bwd with a
caller-provided workspace, within the backward tolerance of the other tests.
It is collected last so that a failure here cannot hide another test's result.
"""
import math

import pytest

from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_77_gb300 as A

    A.get_lib()
    return A


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("det", [0, 1])
def test_noalloc_matches_workspace_backward_twice(A, causal, det):
    torch = G.torch_mod()
    B, H, N, d = 2, 4, 1000, 128
    assert A.attn_bwd_workspace_bytes(B, H, N, d, d, det) <= A.ATTN_NOALLOC_SCRATCH_BYTES
    t = G.inputs(B, H, N, d, d, seed=17)
    o, lse = G.run_fwd(A, t, causal)
    ref = G.run_bwd(A, t, o, lse, causal, det)
    scale = 1.0 / math.sqrt(d)
    for _ in range(2):
        out = [torch.full_like(x, float("nan")) for x in ref]
        A.attn_bwd_noalloc(t["q"], t["k"], t["v"], o, t["do"], lse, out[0], out[1], out[2], B, H, N, d, d, causal,
                           scale, det)
        G.check_status(A)
        for name, got, want in zip(("dq", "dk", "dv"), out, ref):
            G.assert_grad_close(name, G.f64(got), G.f64(want))
            if det:
                assert torch.equal(got.view(torch.int16), want.view(torch.int16)), name


def test_noalloc_without_the_cut_unit_region(A):
    # 352 units: the persistent kernel would cut its last round, but only the
    # workspace without the region for the pieces fits the array
    B, H, N, d = 1, 11, 4096, 128
    base = 2 * B * H * N * 4 + B * H * N * d * 4
    assert base <= A.ATTN_NOALLOC_SCRATCH_BYTES < A.attn_bwd_workspace_bytes(B, H, N, d, d, 0)
    torch = G.torch_mod()
    t = G.inputs(B, H, N, d, d, seed=18)
    o, lse = G.run_fwd(A, t, 0)
    ref = G.run_bwd(A, t, o, lse, 0, 0)
    out = [torch.full_like(x, float("nan")) for x in ref]
    A.attn_bwd_noalloc(t["q"], t["k"], t["v"], o, t["do"], lse, out[0], out[1], out[2], B, H, N, d, d, 0,
                       1.0 / math.sqrt(d), 0)
    G.check_status(A)
    for name, got, want in zip(("dq", "dk", "dv"), out, ref):
        G.assert_grad_close(name, G.f64(got), G.f64(want))


def test_noalloc_rejects_sizes_beyond_its_array(A):
    # 16 heads x 16384 rows x 128 dims of FP32 accumulator alone is 128 MiB
    p = 0x1000
    st = A.get_lib().attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 16, 16384, 128, 128, 0, 0.1, 0, None)
    assert st == A.ATTN_ERR_WORKSPACE
    st = A.get_lib().attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 2, 256, 96, 96, 0, 0.1, 0, None)
    assert st == A.ATTN_ERR_UNSUPPORTED
