"""CPU checks of the seeded input generator."""
import numpy as np

import synth


def test_splitmix64_published_outputs():
    # the first outputs of splitmix64 seeded with 0 (Steele, Lea & Flood's
    # generator as in the public reference implementation)
    got = synth.splitmix64(0, np.arange(3, dtype=np.uint64))
    assert [int(x) for x in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, -2.5, 0.0], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(bits)
    np.testing.assert_array_equal(back, np.array([1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -2.5, 0.0], np.float32))


def test_normal_stream_is_counter_based_and_standard():
    a = synth.normal_f64(0, 0, 200_000)
    b = synth.normal_f64(0, 1000, 500)
    np.testing.assert_array_equal(a[1000:1500], b)
    assert abs(a.mean()) < 0.01 and abs(a.var() - 1) < 0.01
    # chunk boundaries do not change values
    c = synth.normal_f64(0, 2 * (1 << 22) - 4, 10)
    d = synth.normal_f64(0, 0, 2 * (1 << 22) + 6)[-10:]
    np.testing.assert_array_equal(c, d)


def test_attention_inputs_order_and_shapes():
    s = synth.AttentionShape(1, 2, 8, 4, 6)
    t = synth.attention_inputs(s, seed=0)
    assert t["q"].shape == (1, 2, 8, 4) and t["v"].shape == (1, 2, 8, 6) and t["do"].shape == (1, 2, 8, 6)
    # K starts where Q ended in the one stream
    k_direct = synth.normal_bf16_bits(0, 64, (1, 2, 8, 4))
    np.testing.assert_array_equal(t["k"], k_direct)
    t2 = synth.attention_inputs(s, seed=0)
    for name in t:
        np.testing.assert_array_equal(t[name], t2[name])


def test_torch_generator_matches_numpy_on_cpu():
    torch = __import__("pytest").importorskip("torch")
    s = synth.AttentionShape(1, 2, 40, 8, 6)
    a = synth.attention_inputs(s, seed=0)
    b = synth.attention_inputs_torch(s, seed=0, device="cpu")
    for name in a:
        bits = b[name].view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(bits, a[name])


def test_decode_inputs_order_and_shapes():
    s = synth.DecodeShape(1, 2, 3, 10, 4, 6)
    t = synth.decode_inputs(s, seed=0)
    assert t["q"].shape == (1, 2, 3, 4) and t["k"].shape == (1, 2, 10, 4) and t["v"].shape == (1, 2, 10, 6)
    np.testing.assert_array_equal(t["k"], synth.normal_bf16_bits(0, 24, (1, 2, 10, 4)))
    np.testing.assert_array_equal(t["v"], synth.normal_bf16_bits(0, 104, (1, 2, 10, 6)))

    torch = __import__("pytest").importorskip("torch")
    b = synth.decode_inputs_torch(s, seed=0, device="cpu")
    for name in t:
        np.testing.assert_array_equal(b[name].view(torch.int16).numpy().view(np.uint16), t[name])
