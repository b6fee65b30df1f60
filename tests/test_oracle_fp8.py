"""CPU pins of the FP8 oracle (oracle/fp8.py): the e4m3 format against its bit
definition and torch's float8_e4m3fn, the Hadamard rotation against
scipy.linalg.hadamard and the rotation identity of "FlashAttention 3 and 4:
When the Bottleneck Moves" section 2.2, the power-of-two block scales, and the
FP8 forward against the exact attention when its roundings are switched off."""
import math

import numpy as np
import pytest

from oracle import attention as ora
from oracle import fp8


def test_e4m3_table_from_the_bit_definition():
    vals = fp8.e4m3_positive_values()
    assert vals.size == 127 and vals[0] == 0.0
    assert np.all(np.diff(vals) > 0)
    assert vals[-1] == 448.0  # S.1111.110
    assert vals[1] == 2.0 ** -9  # smallest subnormal
    assert vals[8] == 2.0 ** -6  # smallest normal
    assert fp8.e4m3_decode(0x38) == 1.0 and fp8.e4m3_decode(0xB8) == -1.0
    assert math.isnan(fp8.e4m3_decode(0x7F)) and math.isnan(fp8.e4m3_decode(0xFF))


def test_e4m3_table_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = torch.arange(0x7F, dtype=torch.uint8)
    np.testing.assert_array_equal(codes.view(torch.float8_e4m3fn).double().numpy(), fp8.e4m3_positive_values())


def test_e4m3_round_ties_to_even_and_saturates():
    vals = fp8.e4m3_positive_values()
    np.testing.assert_array_equal(fp8.e4m3_round(vals), vals)
    np.testing.assert_array_equal(fp8.e4m3_round(-vals), -vals)
    mid = (vals[:-1] + vals[1:]) / 2
    got = fp8.e4m3_round(mid)
    # each midpoint goes to the neighbour whose code is even (mantissa LSB 0)
    lo_even = (np.arange(126) % 2) == 0
    np.testing.assert_array_equal(got, np.where(lo_even, vals[:-1], vals[1:]))
    np.testing.assert_array_equal(fp8.e4m3_round([449.0, 1e9, -500.0]), [448.0, 448.0, -448.0])
    assert fp8.e4m3_round(2.0 ** -10) == 0.0 and fp8.e4m3_round(2.0 ** -10 * 1.01) == 2.0 ** -9


def test_e4m3_round_matches_torch_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200_000) * np.exp2(rng.integers(-12, 8, 200_000))
    x = np.clip(x, -448, 448).astype(np.float32).astype(np.float64)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(fp8.e4m3_round(x), want)


def test_hadamard_and_rotation_identity():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    for d in (1, 2, 8, 64, 128):
        np.testing.assert_array_equal(fp8.hadamard(d), scipy_linalg.hadamard(d))
    rng = np.random.default_rng(1)
    d = 128
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    r = fp8.rotation(signs)
    np.testing.assert_allclose(r @ r.T, np.eye(d), atol=1e-13)
    q, k = rng.standard_normal((5, d)), rng.standard_normal((7, d))
    # (QR)(KR)^T = Q K^T, and the unnormalised form carries exactly a factor d
    np.testing.assert_allclose((q @ r) @ (k @ r).T, q @ k.T, atol=1e-12)
    qr, kr = fp8.rotate_unnormalised(q, signs), fp8.rotate_unnormalised(k, signs)
    np.testing.assert_allclose(qr @ kr.T / d, q @ k.T, atol=1e-11)
    # an outlying coordinate is spread evenly over all coordinates
    e = np.zeros(d)
    e[17] = 100.0
    np.testing.assert_allclose(np.abs(e @ r), np.full(d, 100.0 / math.sqrt(d)), rtol=1e-14)


def test_pow2_scale_rule():
    for amax in (448.0, 448.0 * 2 ** 5, 448.0 * 2 ** -7, 449.0, 224.0, 224.5, 1.0, 3.3e-3, 1e30):
        s = fp8.pow2_scale(amax)
        m, _ = math.frexp(s)
        assert m == 0.5  # a power of two
        assert amax <= 448.0 * s and amax > 224.0 * s, (amax, s)
    assert fp8.pow2_scale(448.0) == 1.0 and fp8.pow2_scale(449.0) == 2.0 and fp8.pow2_scale(0.0) == 1.0


def test_quantize_rows_blocks_and_bounds():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 3, 300, 16)) * np.exp2(rng.integers(-4, 4, (2, 3, 300, 1)))
    x[1, 2, 128:256] = 0.0  # an all-zero block
    codes, scales = fp8.quantize_rows(x, 128)
    assert scales.shape == (2, 3, 3)
    assert scales[1, 2, 1] == 1.0 and np.all(codes[1, 2, 128:256] == 0)
    grid = fp8.e4m3_positive_values()
    assert np.all(np.isin(np.abs(codes), grid))
    for b in range(3):
        blk = slice(b * 128, (b + 1) * 128)
        xs = x[..., blk, :] / scales[..., b, None, None]
        assert np.abs(xs).max() <= 448.0
        # rounding error at most half a grid step (relative 2^-4 above 2^-6, 2^-10 below)
        err = np.abs(codes[..., blk, :] - xs)
        assert np.all(err <= np.maximum(np.abs(xs) * 2.0 ** -4, 2.0 ** -10) + 1e-15)


def _inputs(B, H, N, d, seed, frac=0.0, mag=1.0):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(3):
        x = rng.standard_normal((B, H, N, d))
        out.append(np.where(rng.random(x.shape) < frac, x * mag, x))
    return out, np.where(rng.random(d) < 0.5, -1.0, 1.0)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tau", [0.0, 4.0, 8.0])
def test_forward_without_p_rounding_is_exact_attention_of_the_quantised_inputs(causal, tau):
    (q, k, v), signs = _inputs(1, 2, 300, 128, 3)
    # tiles of different magnitudes, so every tile gets its own scale
    q[..., 128:256, :] *= 8.0
    k[..., 0:128, :] *= 0.25
    k[..., 256:, :] *= 4.0
    qz = fp8.quantize_qkv(q, k, v, signs)
    assert len(set(qz["sq"][0, 0].tolist())) == 2 and len(set(qz["sk"][0, 0].tolist())) == 3
    o, lse = fp8.forward(qz, 0.09, causal, quantize_p=False, tau=tau)
    # dequantised, un-rotated: Q8 sq (sqrt(d) R)^T etc.; the scores equal those
    # of the dequantised rotated tensors divided by d
    tile_q = np.repeat(qz["sq"], 128, axis=-1)[..., :300, None]
    tile_k = np.repeat(qz["sk"], 128, axis=-1)[..., :300, None]
    qd, kd = qz["q8"] * tile_q, qz["k8"] * tile_k
    vd = qz["v8"] * qz["sv"][..., None, None]
    o_ref, lse_ref = ora.forward(qd, kd, vd, 0.09 / 128, causal)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)


def test_forward_with_exact_quantiser_is_the_attention_of_the_inputs():
    """Rotation alone changes nothing: with the e4m3 rounding replaced by the
    identity (scales kept), the FP8 forward returns the exact attention of the
    original Q, K, V."""
    (q, k, v), signs = _inputs(1, 2, 256, 128, 4)
    saved = fp8.e4m3_round
    try:
        fp8.e4m3_round = lambda x: np.asarray(x, dtype=np.float64)
        qz = fp8.quantize_qkv(q, k, v, signs)
        o, lse = fp8.forward(qz, 1 / math.sqrt(128), False)
    finally:
        fp8.e4m3_round = saved
    o_ref, lse_ref = ora.forward(q, k, v, 1 / math.sqrt(128), False)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)


def test_p_rounding_error_is_within_the_format_bound():
    (q, k, v), signs = _inputs(1, 1, 256, 128, 5)
    qz = fp8.quantize_qkv(q, k, v, signs)
    o1, l1 = fp8.forward(qz, 1 / math.sqrt(128), False)
    o0, l0 = fp8.forward(qz, 1 / math.sqrt(128), False, quantize_p=False)
    # each P' is off by at most 2^-4 relative (or 2^-10 absolute below 2^-6),
    # so O moves by at most that fraction of sum |P'| |v| / l
    vmax = np.abs(qz["v8"] * qz["sv"][..., None, None]).max()
    assert np.abs(o1 - o0).max() <= 2.0 ** -4 * vmax * 1.01
    np.testing.assert_array_equal(l1, l0)  # the row sums use P' before rounding


def test_rotation_reduces_the_error_on_outlier_inputs():
    """The direction of the section 2.2 claim: with outliers, rotating Q and K
    lowers the error against the exact attention; without outliers it changes
    nothing.  (The page's 2.6x depends on an input mix it does not state.)"""
    def rmse(frac, mag, seed):
        (q, k, v), signs = _inputs(1, 2, 512, 128, seed, frac, mag)
        o_ref, _ = ora.forward(q, k, v, 1 / math.sqrt(128), False)
        o_new, _ = fp8.forward(fp8.quantize_qkv(q, k, v, signs), 1 / math.sqrt(128), False)
        o_old, _ = fp8.forward_per_tensor_unrotated(q, k, v, 1 / math.sqrt(128), False)
        return math.sqrt(np.mean((o_old - o_ref) ** 2)) / math.sqrt(np.mean((o_new - o_ref) ** 2))

    assert 0.9 < rmse(0.0, 1.0, 6) < 1.1
    assert rmse(0.001, 10.0, 7) > 1.3
    assert rmse(0.01, 10.0, 8) > 1.8


def test_stale_max_keeps_p_within_the_format():
    """With threshold tau = 4 the stored P' = 2^(8 - tau) P never exceeds 2^8
    (no saturation), and on a rising-max input it does exceed 2^4, i.e. P is
    taken against a stale max."""
    (q, k, v), signs = _inputs(1, 1, 512, 128, 9)
    # a rising max: later keys score higher
    k *= np.linspace(0.2, 3.0, 512)[None, None, :, None]
    qz = fp8.quantize_qkv(q, k, v, signs)
    seen = []
    saved = fp8.e4m3_round

    def spy(x):
        seen.append(float(np.max(x)))
        return saved(x)

    try:
        fp8.e4m3_round = spy
        fp8.forward(qz, 1 / math.sqrt(128), False, tau=4.0)
    finally:
        fp8.e4m3_round = saved
    assert max(seen) <= 256.0 and max(seen) > 16.0
