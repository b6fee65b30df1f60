"""CPU pins for the oracle's exp2 polynomial and roofline cycle model.

The expected numbers are the pages' printed tables (fixtures under
tests/golden/, each carrying its citation).
"""
import json
import os

import numpy as np
import pytest

from oracle import exp2_poly, roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def table():
    return exp2_poly.accuracy_table(degrees=(3, 4, 5), n=4_000_000, seed=0)


@pytest.mark.parametrize("deg", [3, 4, 5])
def test_fit_is_levelled_minimax_with_unit_constant(deg):
    c = exp2_poly.fit_exp2_poly(deg)
    assert c[0] == 1.0
    grid = np.linspace(0, 1, 200_001)
    err = exp2_poly.relative_error_f64(c, grid)
    # equioscillation: deg + 1 interior/extreme points of alternating sign and
    # equal magnitude (the constant term is pinned, so one point fewer).
    sgn = np.where(err >= 0, 1, -1)
    segs = np.split(np.arange(len(grid)), np.nonzero(np.diff(sgn))[0] + 1)
    peaks = np.array([np.abs(err[s]).max() for s in segs])
    assert len(segs) >= deg + 1
    big = np.sort(peaks)[-(deg + 1):]
    assert big.min() > 0.98 * big.max()


@pytest.mark.parametrize("deg", [3, 4, 5])
def test_fp32_error_matches_table2(table, deg):
    want = _load("fa4_table2_exp2_accuracy.json")["rows"][f"degree{deg}"]
    got = table[f"degree{deg}"]
    # coefficients are not printed; our own fit must land within 25 % of the
    # table (degree 5 is at the FP32 rounding floor, where the evaluation
    # order decides the last bits).
    for key in ("fp32_max", "fp32_mean"):
        assert abs(got[key] / want[key] - 1.0) < 0.25, (deg, key, got[key], want[key])
    for key in ("bf16_max", "bf16_mean"):
        assert abs(got[key] / want[key] - 1.0) < 0.02, (deg, key, got[key], want[key])


def test_mean_errors_reproduce_closely(table):
    """The p(0)=1 minimax reading reproduces the table's mean errors to 2 %."""
    rows = _load("fa4_table2_exp2_accuracy.json")["rows"]
    for deg in (3, 4):
        assert abs(table[f"degree{deg}"]["fp32_mean"] / rows[f"degree{deg}"]["fp32_mean"] - 1) < 0.02


def test_ideal_bf16_rounding_row(table):
    want = _load("fa4_table2_exp2_accuracy.json")["rows"]["ideal"]
    got = table["ideal"]
    assert abs(got["bf16_max"] / want["bf16_max"] - 1) < 0.01
    assert abs(got["bf16_mean"] / want["bf16_mean"] - 1) < 0.02
    # closed form: bfloat16 keeps 8 significant bits, so RNE's relative error
    # is below 2^-8 / (1 + 2^-8), plus the FP32 rounding of the input (2^-24).
    assert got["bf16_max"] <= 2.0 ** -8 / (1 + 2.0 ** -8) + 2.0 ** -24


def test_emulated_exp2_on_wide_range():
    c = exp2_poly.fit_exp2_poly(3)
    x = np.linspace(-120.0, 8.0, 100_001).astype(np.float32)
    got = exp2_poly.exp2_emulated(c, x).astype(np.float64)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(got - exact) / exact
    assert rel.max() < 1.0e-4
    # integer arguments are exact: p(0) = 1 and 2^floor(x) is an exponent add
    xi = np.arange(-100, 9, dtype=np.float32)
    np.testing.assert_array_equal(exp2_poly.exp2_emulated(c, xi), np.exp2(xi.astype(np.float64)))


def test_forward_roofline_table1():
    g = _load("fa4_roofline_cycles.json")
    assert roofline.MMA_FLOPS_PER_CLK == g["rates"]["mma_flops_per_clk_per_sm"]
    assert roofline.EXP_PER_CLK == g["rates"]["exp_per_clk_per_sm"]
    assert roofline.forward_tile(128, 128, 128) == g["forward"]["128x128x128"]
    assert roofline.forward_tile(256, 128, 128) == g["forward"]["256x128x128"]


def test_backward_roofline_table3():
    g = _load("fa4_roofline_cycles.json")["backward"]
    assert roofline.backward_tile_1cta() == g["1cta_M128"]
    two = roofline.backward_tile_2cta()
    for key in ("mma", "smem_operands", "smem_ds_write", "smem_dq"):
        assert two[key] == g["2cta_M256"][key], key
    one = roofline.backward_tile_1cta()
    smem_total = one["smem_operands"] + one["smem_ds_write"] + one["smem_dq"]
    # Table 3's caption puts the 1-CTA shared-memory cycles about 30 % above the MMA cycles
    assert abs(smem_total / one["mma"] - 1.30) < 0.01
