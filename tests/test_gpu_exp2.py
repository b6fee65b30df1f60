"""GPU tests of the exponential step of the forward (softmax numerator 2^x).

"FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
Hardware Scaling" (abstract, Table 2) and "FlashAttention 3 and 4: When the
Bottleneck Moves" (section 3.2) compute part of the exponentials as
2^floor(x) * p(x - floor(x)) with a low-degree polynomial on the FMA pipe.
Two things are checked here on the device:

* Table 2 itself: 4M seeded uniform FP32 inputs on [0, 1) through the
  library's probe (the hardware ex2 unit and the degree-3/4/5 emulations,
  the cubic being the one the forward kernel uses), relative errors against
  FP64 2^x, compared with the table's FP32 and BF16 columns.
* The forward kernels built with the polynomial share (attn_set_exp_poly(1)),
  for every head-dim pair, causal and not, against the FP64 oracle at the
  forward's tolerances, and proof that those instances ran: their output
  differs from the hardware-only instances' in the last bits of some P.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import attention as ora
from oracle import exp2_poly
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fa4_table2_exp2_accuracy.json")


@pytest.fixture(scope="module")
def A():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_77_gb300 as A

    A.get_lib()
    yield A
    A.attn_set_exp_poly(0)
    G.check_status(A)


@pytest.fixture
def poly(A):
    A.attn_set_exp_poly(1)
    yield
    A.attn_set_exp_poly(0)


def _probe(A, x_np, method):
    torch = G.torch_mod()
    x = torch.from_numpy(np.ascontiguousarray(x_np, dtype=np.float32)).cuda()
    out = torch.empty_like(x)
    A.attn_exp2_probe(x, out, x.numel(), method)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.fixture(scope="module")
def table2_inputs():
    # the experiment of Table 2: 4M uniform inputs on [0, 1) in FP32
    rng = np.random.Generator(np.random.PCG64(0))
    f = rng.random(4_000_000).astype(np.float32)
    return f[f < 1.0]


@pytest.mark.parametrize("method,row", [(0, "mufu"), (3, "degree3"), (4, "degree4"), (5, "degree5")])
def test_table2_on_the_device(A, table2_inputs, method, row):
    """FP32 max / mean relative error within 25 % of Table 2's row (the pages
    print no coefficients, so each fit is our own), BF16 columns within 2 %."""
    want = json.load(open(GOLDEN))["rows"][row]
    got = exp2_poly.accuracy_row(_probe(A, table2_inputs, method), table2_inputs)
    for key in ("fp32_max", "fp32_mean"):
        assert abs(got[key] / want[key] - 1.0) < 0.25, (row, key, got[key], want[key])
    for key in ("bf16_max", "bf16_mean"):
        assert abs(got[key] / want[key] - 1.0) < 0.02, (row, key, got[key], want[key])


def test_cubic_over_the_softmax_range(A):
    """The forward's arguments are x = s*scale*log2(e) - m <= tau (8) and
    reach far below 0: relative error of the cubic stays at its [0, 1) level
    over [-126, 8]; integers are exact; arguments below -127 give results
    below 2^-126 (they are only ever summed against terms >= 1)."""
    rng = np.random.Generator(np.random.PCG64(1))
    x = rng.uniform(-126.0, 8.0, 1_000_000).astype(np.float32)
    y = _probe(A, x, 3).astype(np.float64)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(y - exact) / exact
    want = json.load(open(GOLDEN))["rows"]["degree3"]["fp32_max"]
    assert rel.max() < 1.25 * want, rel.max()
    ints = np.arange(-126, 9, dtype=np.float32)
    assert np.array_equal(_probe(A, ints, 3).astype(np.float64), np.exp2(ints.astype(np.float64)))
    tiny = _probe(A, np.array([-127.0, -150.0, -1e4, -np.inf], dtype=np.float32), 3)
    assert np.all(tiny >= 0.0) and np.all(tiny < 2.0 ** -126)


def _fwd_check(A, B, H, N, dqk, dv, causal, seed=0):
    t = G.inputs(B, H, N, dqk, dv, seed=seed, with_do=False)
    o, lse = G.run_fwd(A, t, causal)
    G.check_status(A)
    q, k, v = (G.f64(t[n]) for n in ("q", "k", "v"))
    o_ref, lse_ref = ora.forward(q, k, v, 1.0 / math.sqrt(dqk), bool(causal))
    G.assert_fwd_close(G.f64(o), G.f64(lse), o_ref, lse_ref, f"poly N{N} d{dqk}/{dv} causal{causal}")
    return o


@pytest.mark.parametrize("dqk,dv", [(64, 64), (128, 128), (192, 128)])
@pytest.mark.parametrize("N", [17, 129, 300])
@pytest.mark.parametrize("causal", [0, 1])
def test_poly_forward_ragged(A, poly, dqk, dv, N, causal):
    _fwd_check(A, 1, 3, N, dqk, dv, causal, seed=21)


@pytest.mark.parametrize("causal", [0, 1])
def test_poly_forward_pr1(A, poly, causal):
    """B=1, H=2, N=256, d=64, seed 0, in full."""
    _fwd_check(A, 1, 2, 256, 64, 64, causal)


@pytest.mark.parametrize("dqk,dv", [(128, 128), (192, 128)])
@pytest.mark.parametrize("causal", [0, 1])
def test_poly_forward_16k_sampled_head(A, poly, dqk, dv, causal):
    """B=1, H=16, N=16384: one seeded head, 512 seeded rows against all keys."""
    B, H, N = 1, 16, 16384
    t = G.inputs(B, H, N, dqk, dv, with_do=False)
    o, lse = G.run_fwd(A, t, causal)
    G.check_status(A)
    h = int(np.random.Generator(np.random.PCG64(80 + dqk + causal)).integers(H))
    rows = G.seeded_rows(N, 512, 81 + causal)
    o_ref, l_ref = ora.forward_head(G.f64(t["q"][0, h][rows]), G.f64(t["k"][0, h]), G.f64(t["v"][0, h]),
                                    1.0 / math.sqrt(dqk), bool(causal), rows)
    G.assert_fwd_close(G.f64(o[0, h][rows]), G.f64(lse[0, h][rows]), o_ref, l_ref, f"poly 16K d{dqk} c{causal}")


@pytest.mark.parametrize("dqk,dv", [(64, 64), (128, 128), (192, 128)])
def test_poly_instances_are_the_ones_that_ran(A, dqk, dv):
    """The polynomial's error (~1e-4 relative) moves the bf16 rounding of some
    P values, so its output differs in places from the hardware-only run on
    the same inputs; both are within tolerance of the oracle."""
    torch = G.torch_mod()
    t = G.inputs(1, 4, 1024, dqk, dv, seed=22, with_do=False)
    A.attn_set_exp_poly(0)
    o_hw, l_hw = G.run_fwd(A, t, 0)
    A.attn_set_exp_poly(1)
    try:
        o_po, l_po = G.run_fwd(A, t, 0)
    finally:
        A.attn_set_exp_poly(0)
    G.check_status(A)
    assert not torch.equal(o_hw.view(torch.int16), o_po.view(torch.int16))
    q, k, v = (G.f64(t[n]) for n in ("q", "k", "v"))
    o_ref, l_ref = ora.forward(q, k, v, 1.0 / math.sqrt(dqk), False)
    G.assert_fwd_close(G.f64(o_hw), G.f64(l_hw), o_ref, l_ref, "hardware")
    G.assert_fwd_close(G.f64(o_po), G.f64(l_po), o_ref, l_ref, "polynomial")
