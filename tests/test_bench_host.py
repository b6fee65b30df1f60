"""CPU checks of bench.py's host logic: FLOP counting, the multi-rank timing
reduction (two gloo ranks on CPU), and the oracle baseline sample."""
import math
import os
import socket

import numpy as np
import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    out[rank] = bench.max_over_ranks(10.0 + rank * 5.0, world)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_flop_convention():
    a = type("A", (), dict(B=1, H=16, N=16384, d=128, causal=0))()
    assert bench.flops_fwd(a) == 4 * 16 * 16384 ** 2 * 128
    a.causal = 1
    assert bench.flops_fwd(a) == 2 * 16 * 16384 ** 2 * 128
    # d_qk != d_v: the S product counts d_qk, the O product d_v
    b = type("A", (), dict(B=1, H=16, N=4096, d=192, dv=128, causal=0))()
    assert bench.flops_fwd(b) == 2 * 16 * 4096 ** 2 * (192 + 128)


def test_oracle_sample_runs_small():
    a = type("A", (), dict(B=1, H=1, N=256, d=64, causal=0))()
    dt, fl, desc = bench.oracle_sample(a, rows=64)
    assert dt > 0 and fl == 3.5 * 4 * 64 * 256 * 64 and "64 of 256" in desc
    b = type("A", (), dict(B=1, H=1, N=256, d=192, dv=128, causal=1))()
    dt, fl, desc = bench.oracle_sample(b, rows=64)
    assert dt > 0 and fl == 3.5 * 2 * 64 * 256 * (192 + 128) / 2


def test_source_hash_ignores_comments_only():
    src = 'const char* s = "a // b /* c */";  // note\nint x = 1; /* block\n comment */ int y = \'/\';\n'
    assert bench.strip_c_comments(src) == 'const char* s = "a // b /* c */";  \nint x = 1;  int y = \'/\';\n'
    assert bench.strip_c_comments("a = 1; // x") == bench.strip_c_comments("a = 1; // y")
    assert bench.strip_c_comments("a = 1;") != bench.strip_c_comments("a = 2;")


@pytest.mark.parametrize("d,dv", [(64, 64), (192, 128)])
def test_oracle_sample_draws_head_zero_of_the_workload(d, dv):
    """The CPU baseline's sample is head (0, 0) of the same seeded tensors the
    GPU step runs on."""
    import synth
    from oracle import attention as ora

    a = type("A", (), dict(B=2, H=3, N=130, d=d, dv=dv, causal=0))()
    q, k, v, do = bench.oracle_inputs(a, rows=17)
    full = synth.attention_inputs(synth.AttentionShape(2, 3, 130, d, dv), seed=0)
    f = {n: ora.bf16_to_f64(full[n])[0, 0] for n in ("q", "k", "v", "do")}
    assert np.array_equal(q, f["q"][:17]) and np.array_equal(k, f["k"])
    assert np.array_equal(v, f["v"]) and np.array_equal(do, f["do"][:17])


def test_roofline_peak_is_burst_unless_power_capped():
    peaks = {"bf16_tflops": 1943.4, "bf16_tflops_sustained": 1698.1}
    p, note = bench.roofline_peak(peaks, {"reasons": []})
    assert p == 1943.4 and "burst" in note
    p, note = bench.roofline_peak(peaks, {"reasons": ["sw_power_cap"]})
    assert p == 1698.1 and "power cap" in note
    p, _ = bench.roofline_peak({}, {"reasons": None})
    assert p == bench.FALLBACK_PEAKS["bf16_tflops"]


def test_e2e_groups_cover_every_head_once():
    for BH, chunks in ((16, 8), (16, 16), (16, 4), (12, 8), (1, 8), (7, 3)):
        for taper in (False, True):
            groups = bench.e2e_groups(BH, chunks, taper)
            heads = [h for g0, gn in groups for h in range(g0, g0 + gn)]
            assert heads == list(range(BH)), (BH, chunks, taper)
            assert all(gn >= 1 for _, gn in groups)


def test_e2e_groups_taper_halves_the_ends():
    assert [gn for _, gn in bench.e2e_groups(16, 8, False)] == [2] * 8
    assert [gn for _, gn in bench.e2e_groups(16, 8, True)] == [1, 1, 2, 2, 2, 2, 2, 2, 1, 1]
    assert [gn for _, gn in bench.e2e_groups(16, 4, True)] == [2, 2, 4, 4, 2, 2]
    # one-head groups cannot be halved; a single group is not tapered
    assert [gn for _, gn in bench.e2e_groups(16, 16, True)] == [1] * 16
    assert [gn for _, gn in bench.e2e_groups(16, 1, True)] == [16]
