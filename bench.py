#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300.

One step = the whole hot path over one batch: forward (O, LSE) then backward
(dQ, dK, dV) through the C ABI, on the workload B=1, H=16, N=16384,
d_qk=d_v=128, non-causal, atomic dQ mode (the d=128, 16K-token point of the
forward sweep and of the backward sweep).  Inputs are seeded synthetic BF16
N(0,1) tensors already resident in HBM.

Metric: BF16 attention TFLOPS (forward 4*B*H*N^2*d, halved for causal;
backward 2.5x the forward) over the timed steps, and the dominant kernel's
fraction of the measured dense BF16 peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the FP64 CPU oracle on the host cores (a bounded sample
of the same workload per step).

  python bench.py --case fp8|splitkv|masked|exp2|detsched|sweep [--B --H --N ...]

times one of the library's other paths instead (one GPU; a JSON line with its
own fields; no contract line): the FP8 quantiser + FP8 forward, the split-KV
decode forward (--Nq queries against --Nk keys, the heuristic's ranges), or
the masked forward + backward (--window-left / --window-right, --block-density
for a seeded random block map), or the exponential paths' accuracy (the
experiment of Table 2 of the FlashAttention-4 paper) and throughput per SM
per clock, the deterministic backward under each unit order (detsched), or
every configuration of the workload list, forward and backward (sweep).
Under torchrun every rank runs the same
workload on its own GPU (independent replicas: no data exchange), timing is
bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BF16 attention fwd+bwd TFLOPS on 1 GB300 (% of dense BF16 peak via roofline)"
UNIT = "TFLOPS"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def d_v(args) -> int:
    """Head dim of V, O and dO (--dv; 0: the same as --d)."""
    return getattr(args, "dv", 0) or args.d


def workload(args):
    dims = f"d={args.d}" if d_v(args) == args.d else f"d_qk={args.d} d_v={d_v(args)}"
    return {"workload": f"attention fwd+bwd B={args.B} H={args.H} N={args.N} {dims} "
                        f"{'causal' if args.causal else 'non-causal'} {'deterministic' if args.det else 'atomic'} dQ",
            "B": args.B, "H": args.H, "N": args.N, "d_qk": args.d, "d_v": d_v(args), "causal": bool(args.causal),
            "dq_mode": "deterministic" if args.det else "atomic", "scale": "1/sqrt(d_qk)", "seed": 0,
            "dtype_inputs": "bf16", "l2": "256 MiB write between timed steps (outside the timed events); "
                                         "inputs 320 MiB > 129 MB L2"}


def flops_fwd(a) -> float:
    # the two forward products: 2 N^2 d_qk for S plus 2 N^2 d_v for O per head
    f = 2.0 * a.B * a.H * a.N * a.N * (a.d + d_v(a))
    return f / 2 if a.causal else f


# ------------------------------------------------------------------ ranks
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of ``x`` across ranks (identity when world == 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.lines: list[str] = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if gpu_id:
            cmd.insert(1, f"--id={gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


def roofline_peak(peaks: dict, clk: dict):
    """Denominator of the roofline fractions: the burst bf16 peak (cuBLAS timed
    alone, at full clock), unless the clock record of the timed region shows
    the power cap acting, in which case the sustained (power-capped) peak."""
    if "sw_power_cap" in (clk.get("reasons") or []):
        return peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]), \
            "bf16_tflops_sustained (power cap active during the timed region)"
    return peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]), "bf16_tflops (burst; no power cap in the timed region)"


def gpu_uuid(torch, dev):
    """nvidia-smi id of the torch device (its UUID), or None."""
    try:
        g = str(torch.cuda.get_device_properties(dev).uuid)
        return g if g.startswith("GPU-") else "GPU-" + g
    except Exception:
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def strip_c_comments(text: str) -> str:
    """C/C++ source without its // and /* */ comments (string and character
    literals kept as they are), so an edit to comments alone leaves the
    source hash unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join(out)


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (comments excluded; the C-ABI host file
    left out): the committed DRAM counters stay valid while it is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_77_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        # the kernels and their headers (the C-ABI host code does not change a kernel's traffic)
        if name.endswith((".cu", ".cuh", ".h")) and name != "attn_api.cu":
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode() + strip_c_comments(f.read()).encode())
    return h.hexdigest()[:16]


def e2e_groups(BH: int, chunks: int, taper: bool) -> list:
    """(first head, heads) of each head group of the end-to-end leg: ``chunks``
    equal groups (fewer if they do not divide BH).  With ``taper`` the first
    and last groups are halved, so the pipeline fills (the first group's
    inputs going up before any kernel runs) and drains (the last group's
    results coming down after the last kernel) with half as many bytes."""
    n = max(1, min(chunks, BH))
    while BH % n:
        n -= 1
    hc = BH // n
    sizes = [hc] * n
    if taper and hc >= 2 and n >= 2:
        sizes = [hc // 2, hc - hc // 2] + [hc] * (n - 2) + [hc - hc // 2, hc // 2]
    groups, h0 = [], 0
    for sz in sizes:
        groups.append((h0, sz))
        h0 += sz
    return groups


def recorded_traffic(kernel: str, args):
    """DRAM bytes per launch from the committed ncu summary, if it still matches the sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    dims = f"d{args.d}" if d_v(args) == args.d else f"d{args.d}v{d_v(args)}"
    key = f"{kernel}:B{args.B}H{args.H}N{args.N}{dims}c{int(args.causal)}"
    return rec.get("per_launch_bytes", {}).get(key)


# ---------------------------------------------------------- CPU oracle
def oracle_inputs(args, rows: int):
    """FP64 values of head (0, 0) of the workload's seeded stream: the first
    ``rows`` query rows of Q and dO, every row of K and V.  Q, K, V, dO each
    start after the whole previous tensor (B*H*N*d draws)."""
    import synth
    from oracle import attention as ora

    dv = d_v(args)
    per_qk, per_v = args.B * args.H * args.N * args.d, args.B * args.H * args.N * dv
    draw = lambda start, n_rows, d: ora.bf16_to_f64(synth.normal_bf16_bits(0, start, (n_rows, d)))
    q, k = draw(0, rows, args.d), draw(per_qk, args.N, args.d)
    v, do = draw(2 * per_qk, args.N, dv), draw(2 * per_qk + per_v, rows, dv)
    return q, k, v, do


def oracle_sample(args, rows: int = 1024):
    """The oracle's forward and backward for ``rows`` query rows of head (0, 0)
    against all N keys (non-causal rows are independent, so this is exactly
    those rows' share of the workload).  Returns (seconds, flops, description)."""
    import numpy as np

    from oracle import attention as ora

    dv = d_v(args)
    q, k, v, do = oracle_inputs(args, rows)
    scale = 1.0 / math.sqrt(args.d)
    t0 = time.perf_counter()
    ora.forward_head(q, k, v, scale, bool(args.causal), np.arange(rows))
    ora.backward_head(q, k, v, do, scale, bool(args.causal))
    dt = time.perf_counter() - t0
    fl = 3.5 * 2.0 * rows * args.N * (args.d + dv) / (2 if args.causal else 1)
    return dt, fl, f"head (0,0): {rows} of {args.N} query rows x {args.N} keys, forward + backward, FP64"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(args, min_seconds: float = 10.0) -> dict:
    tot_t, tot_f, reps, desc = 0.0, 0.0, 0, ""
    while tot_t < min_seconds and reps < 50:
        dt, fl, desc = oracle_sample(args)
        tot_t += dt
        tot_f += fl
        reps += 1
    return {"value": tot_f / tot_t / 1e12, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
            "sample": f"{desc}; {reps} repetitions, {tot_t:.1f} s"}


# -------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import torch

    import exact_attention_77_gb300 as A
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    A.get_lib()
    B, H, N, d, dvh = args.B, args.H, args.N, args.d, d_v(args)
    scale = 1.0 / math.sqrt(d)
    t = synth.attention_inputs_torch(synth.AttentionShape(B, H, N, d, dvh), seed=0, device=dev)
    q, k, v, do = t["q"], t["k"], t["v"], t["do"]
    o = torch.empty_like(v)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nws = A.attn_bwd_workspace_bytes(B, H, N, d, dvh, args.det)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        A.attn_fwd(q, k, v, o, lse, B, H, N, d, dvh, args.causal, scale, stream)
        A.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, dvh, args.causal, scale, args.det, ws, nws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st, where = A.attn_get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {A.status_string(st)} at {where}")

    gpu_id = gpu_uuid(torch, dev)
    clocks = ClockSampler(gpu_id)
    time.sleep(0.5)
    barrier(world)
    torch.cuda.synchronize(dev)
    A.attn_profile_start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i & 0xFF)  # evict the previous step's data from L2 (not timed)
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    prof = A.attn_profile_stop()
    barrier(world)
    clk = clocks.stop()
    st, where = A.attn_get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {A.status_string(st)} at {where}")
    step_ms = sum(a.elapsed_time(b) for a, b in evs)
    total_ms = max_over_ranks(step_ms, world, dev)

    # sustained leg: the same step back to back for >= --sustain-seconds with
    # clocks sampled, to show whether the rates hold under the power limit
    # (inputs and outputs are 320 MiB > 129 MB of L2, so no flush between steps)
    sustained = None
    if args.sustain_seconds > 0:
        n_sus = max(args.steps, int(math.ceil(args.sustain_seconds / max(step_ms / args.steps / 1e3, 1e-6))))
        clocks_s = ClockSampler(gpu_id)
        time.sleep(0.5)
        barrier(world)
        torch.cuda.synchronize(dev)
        A.attn_profile_start()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(n_sus):
            step()
        s1.record(stream)
        torch.cuda.synchronize(dev)
        prof_s = A.attn_profile_stop()
        barrier(world)
        clk_s = clocks_s.stop()
        sus_ms = max_over_ranks(s0.elapsed_time(s1), world, dev)
        f1 = flops_fwd(args)
        sustained = {
            "steps": n_sus, "seconds": sus_ms / 1e3, "value": world * 3.5 * f1 * n_sus / (sus_ms / 1e3) / 1e12,
            "forward_tflops": f1 * prof_s["launches_fwd"] / (prof_s["ms_fwd"] / 1e3) / 1e12,
            "backward_main_tflops": 2.5 * f1 * prof_s["launches_bwd_main"] / (prof_s["ms_bwd_main"] / 1e3) / 1e12,
            "clocks": clk_s, "l2": "no flush: 320 MiB of inputs and outputs per step > 129 MB L2"}

    # end to end through the public API: pinned host buffers in, results out.
    # Every (b, h) is independent, so the step runs as n_chunks groups of
    # heads: inputs go up on one stream, results come down on another, and
    # the groups' kernels run on n_cs compute streams (round-robin, one
    # workspace each), so copies overlap kernels and neighbouring groups'
    # small grids share the GPU (every byte still crosses the link inside the
    # timed region, every step).
    hq, hk, hv, hdo = (x.cpu().pin_memory() for x in (q, k, v, do))
    ho, hlse, hdq, hdk, hdv = (torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (o, lse, dq, dk, dv))
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdo))
    d2h = sum(x.numel() * x.element_size() for x in (ho, hlse, hdq, hdk, hdv))
    BH = B * H
    groups = e2e_groups(BH, args.e2e_chunks, bool(args.e2e_taper))
    sizes = [gn for _, gn in groups]
    hc = max(sizes)
    n_chunks = len(groups)
    flat = lambda x: x.reshape(BH, *x.shape[2:])
    # the forward needs Q, K, V only, and O / LSE are final once it has run:
    # dO goes up after them and O / LSE come down before the gradients
    pairs_fwd_in = [(flat(dst), flat(src)) for dst, src in ((q, hq), (k, hk), (v, hv))]
    pairs_bwd_in = [(flat(do), flat(hdo))]
    pairs_fwd_out = [(flat(dst), flat(src)) for dst, src in ((ho, o), (hlse, lse))]
    pairs_bwd_out = [(flat(dst), flat(src)) for dst, src in ((hdq, dq), (hdk, dk), (hdv, dv))]
    dev_t = [flat(x) for x in (q, k, v, o, do, lse, dq, dk, dv)]
    cws = A.attn_bwd_workspace_bytes(1, hc, N, d, dvh, args.det)
    n_cs = max(1, min(args.e2e_streams, n_chunks))  # compute streams, groups dealt round-robin
    cwsb = [torch.empty(cws, dtype=torch.uint8, device=dev) for _ in range(n_cs)]
    s_comp = [stream] + [torch.cuda.Stream(dev) for _ in range(n_cs - 1)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    ev_in, ev_done, ev_out = [ev() for _ in range(n_chunks)], [ev() for _ in range(n_chunks)], [ev() for _ in range(n_chunks)]
    ev_fin, ev_fdone = [ev() for _ in range(n_chunks)], [ev() for _ in range(n_chunks)]
    ev_start = ev()
    first = [True]

    def e2e_step():
        ev_start.record(stream)
        s_in.wait_event(ev_start)
        s_out.wait_event(ev_start)
        for cs in s_comp[1:]:
            cs.wait_event(ev_start)
        for c, (g0, gn) in enumerate(groups):
            sl = slice(g0, g0 + gn)
            cs = s_comp[c % n_cs]
            if not first[0]:
                s_in.wait_event(ev_done[c])  # the previous step's group c no longer reads these inputs
            with torch.cuda.stream(s_in):
                for dst, src in pairs_fwd_in:
                    dst[sl].copy_(src[sl], non_blocking=True)
                ev_fin[c].record(s_in)
                for dst, src in pairs_bwd_in:
                    dst[sl].copy_(src[sl], non_blocking=True)
            ev_in[c].record(s_in)
            cs.wait_event(ev_fin[c])
            if not first[0]:
                cs.wait_event(ev_out[c])  # the previous step's results of group c are out
            cq, ck, cv, co, cdo, clse, cdq, cdk, cdv = (x[sl] for x in dev_t)
            A.attn_fwd(cq, ck, cv, co, clse, 1, gn, N, d, dvh, args.causal, scale, cs)
            ev_fdone[c].record(cs)
            cs.wait_event(ev_in[c])
            A.attn_bwd(cq, ck, cv, co, cdo, clse, cdq, cdk, cdv, 1, gn, N, d, dvh, args.causal, scale, args.det,
                       cwsb[c % n_cs], cws, cs)
            ev_done[c].record(cs)
            s_out.wait_event(ev_fdone[c])
            with torch.cuda.stream(s_out):
                for dst, src in pairs_fwd_out:
                    dst[sl].copy_(src[sl], non_blocking=True)
            s_out.wait_event(ev_done[c])
            with torch.cuda.stream(s_out):
                for dst, src in pairs_bwd_out:
                    dst[sl].copy_(src[sl], non_blocking=True)
            ev_out[c].record(s_out)
        first[0] = False
        for cs in s_comp[1:]:
            stream.wait_stream(cs)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)

    e2e_steps = max(2, args.steps // 2)
    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    # the pipelined results are the device-resident step's results
    if not (torch.equal(ho.view(torch.int16), o.cpu().view(torch.int16)) and
            torch.equal(hdq.view(torch.int16), dq.cpu().view(torch.int16))):
        raise RuntimeError("end-to-end results differ from the device-resident step")

    f_fwd = flops_fwd(args)
    f_step = 3.5 * f_fwd
    value = world * f_step * args.steps / (total_ms / 1e3) / 1e12
    peaks, peak_src = measured_peaks()
    kernels = {
        "attn_fwd_kernel": (prof["ms_fwd"], prof["launches_fwd"], f_fwd),
        "attn_bwd_main_kernel": (prof["ms_bwd_main"], prof["launches_bwd_main"], 2.5 * f_fwd),
    }
    per_kernel = {}
    for name, (ms, n, fl) in kernels.items():
        avg = ms / max(n, 1)
        ach = fl / (avg / 1e3) / 1e12 if avg > 0 else None
        per_kernel[name] = {"launches": n, "avg_ms": avg, "achieved_tflops": ach}
    dom = max(kernels, key=lambda n: kernels[n][0])
    peak, peak_note = roofline_peak(peaks, clk)

    def roof(name):
        a = per_kernel[name]["achieved_tflops"]
        return {"bound": "tensor", "kernel": name, "achieved": a, "peak": peak, "unit": "TFLOP/s",
                "frac": a / peak if a else None, "traffic": recorded_traffic(name, args),
                "peak_source": f"{peak_src} {peak_note}", "frac_of_nominal_2250": a / 2250.0 if a else None}

    roofline = roof(dom)
    roofline_fwd = roof("attn_fwd_kernel")
    launches = prof["launches_fwd"] + prof["launches_bwd_pre"] + prof["launches_bwd_main"] + prof["launches_bwd_convert"]
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16; splitmix64 + Box-Muller, seed 0)",
        "config": dict(workload(args), parallelism=f"replicas{world}" if world > 1 else "single"),
        "roofline": roofline, "roofline_fwd": roofline_fwd, "kernels": per_kernel,
        "breakdown_tflops": {"forward": per_kernel["attn_fwd_kernel"]["achieved_tflops"], "backward_main": per_kernel["attn_bwd_main_kernel"]["achieved_tflops"],
                             "backward_incl_pre_convert": 2.5 * f_fwd / ((prof["ms_bwd_pre"] + prof["ms_bwd_main"] + prof["ms_bwd_convert"]) / max(prof["launches_bwd_main"], 1) / 1e3) / 1e12 if prof["launches_bwd_main"] else None},
        "clocks": clk, "gpu_launches": launches, "sustained": sustained,
        "e2e": {"value": world * f_step / (e2e_ms / 1e3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "head_groups": n_chunks,
                "group_heads": sizes, "compute_streams": n_cs},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference(args, world, rank):
    """The oracle on the host cores: each step one bounded sample of the workload."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample(args)
    tot_t, tot_f, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        dt, fl, desc = oracle_sample(args)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1) bf16; splitmix64 + Box-Muller, seed 0)",
           "config": dict(workload(args), parallelism="host cores"),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle", "sample": desc},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(out), flush=True)


# ------------------------------------------------- other library paths
def run_exp2_case(args, A, torch, dev, out):
    """The exponential paths of the forward measured on the device: the
    relative error of 2^x on 4M uniform FP32 inputs on [0, 1) against FP64
    (the experiment of "FlashAttention-4 ...", Table 2; BF16 columns after
    rounding to bfloat16), and the throughput of each path in exponentials
    per SM per clock, from CUDA events and the SM clock sampled while the
    throughput kernel runs."""
    import numpy as np

    names = {0: "mufu", 3: "degree3", 4: "degree4", 5: "degree5"}
    rng = np.random.Generator(np.random.PCG64(0))
    f = rng.random(4_000_000).astype(np.float32)
    f = f[f < 1.0]
    x = torch.from_numpy(f).to(dev)
    y = torch.empty_like(x)
    exact = np.exp2(f.astype(np.float64))

    def bf16(v):
        b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
        r = ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)) << np.uint32(16)
        return r.view(np.float32).astype(np.float64)

    acc = {}
    for m, name in names.items():
        A.attn_exp2_probe(x, y, x.numel(), m)
        torch.cuda.synchronize(dev)
        v = y.cpu().numpy()
        r32 = np.abs(v.astype(np.float64) - exact) / exact
        rbf = np.abs(bf16(v) - exact) / exact
        acc[name] = {"fp32_max": float(r32.max()), "fp32_mean": float(r32.mean()),
                     "bf16_max": float(rbf.max()), "bf16_mean": float(rbf.mean())}
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = sms * 8, 20000
    sink = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    thr = {}
    for m, name in names.items():
        A.attn_exp2_throughput(sink, blocks, 100, m)  # warm-up
        torch.cuda.synchronize(dev)
        clocks = ClockSampler(gpu_uuid(torch, dev))
        time.sleep(0.3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        reps = 0
        t_end = time.perf_counter() + 1.5
        while time.perf_counter() < t_end:
            A.attn_exp2_throughput(sink, blocks, iters, m)
            reps += 1
            if reps % 4 == 0:
                torch.cuda.synchronize(dev)
        e1.record()
        torch.cuda.synchronize(dev)
        clk = clocks.stop()
        sec = e0.elapsed_time(e1) / 1e3
        n_exp = reps * blocks * 256 * iters * 8
        mhz = clk.get("sm_mhz") or 0.0
        thr[name] = {"exp_per_s": n_exp / sec, "sm_mhz_median": mhz, "reasons": clk.get("reasons"),
                     "exp_per_clk_per_sm": n_exp / sec / (mhz * 1e6) / sms if mhz else None}
    out.update({"config": {"inputs": "4M uniform FP32 on [0,1), PCG64 seed 0", "throughput_grid": f"{blocks}x256",
                           "chained_exponentials_per_thread": iters * 8}, "accuracy": acc, "throughput": thr})


def run_detsched_case(args, A, torch, dev, out):
    """The deterministic backward under each unit order of attn_set_det_schedule
    (head groups x ascending / descending key tiles), next to the atomic mode,
    on the --B --H --N --d --causal workload: main-kernel time from the
    library's per-kernel events, L2 flushed before each call, median of --steps."""
    import synth

    B, H, N, d = args.B, args.H, args.N, args.d
    t = synth.attention_inputs_torch(synth.AttentionShape(B, H, N, d, d), seed=0, device=dev)
    o = torch.empty_like(t["v"])
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    scale = 1.0 / math.sqrt(d)
    A.attn_fwd(t["q"], t["k"], t["v"], o, lse, B, H, N, d, d, args.causal, scale)
    nb = A.attn_bwd_workspace_bytes(B, H, N, d, d, 1)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    fl = 2.5 * flops_fwd(args)

    def main_ms(det):
        ts = []
        for i in range(args.warmup + args.steps):
            flush.fill_(i & 0xFF)
            A.attn_profile_start()
            A.attn_bwd(t["q"], t["k"], t["v"], o, t["do"], lse, dq, dk, dv, B, H, N, d, d, args.causal, scale, det,
                       ws, nb)
            prof = A.attn_profile_stop()
            if i >= args.warmup:
                ts.append(prof["ms_bwd_main"])
        return statistics.median(ts)

    rows = {"atomic": main_ms(0)}
    groups = [g for g in (1, 2, 4, 8) if g < B * H] + [B * H]  # the last: one group of all heads
    # both main kernels: one CTA per unit, and persistent CTAs (all resident;
    # without the causal mask they take the rotated walk)
    for persist in (0, 1):
        A.attn_set_bwd_persist(persist)
        kind = "persistent" if persist else "one-unit"
        rows[f"atomic {kind}"] = main_ms(0)
        for desc in (0, 1):
            for g in groups:
                A.attn_set_det_schedule(g, desc)
                rows[f"{kind} group={g if g < B * H else 'all'} {'desc' if desc else 'asc'}"] = main_ms(1)
    A.attn_set_det_schedule(0, 0)
    A.attn_set_bwd_persist(-1)
    out.update({"config": {"B": B, "H": H, "N": N, "d": d, "causal": bool(args.causal)},
                "backward_main_ms": rows,
                "backward_main_tflops": {k: fl / v / 1e9 for k, v in rows.items()},
                "note": ("deterministic backward main kernel per unit order and main kernel; group = heads per "
                         "key-tile-major group; 'atomic' = the library's default kernel choice")})


def run_sweep_case(args, A, torch, dev, out):
    """Every configuration of the workload list: forward TFLOP/s (configs 1-4)
    and backward TFLOP/s in both dQ modes (configs 1, 5 and the d_qk = 192
    backward), each the median of --steps calls after --warmup, the L2
    flushed before each call; kernel times from the library's per-kernel
    events (backward: the main kernel, and the whole call with its
    preprocess and dQ conversion)."""
    import synth

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def med(fn, key):
        ts = []
        for i in range(args.warmup + args.steps):
            flush.fill_(i & 0xFF)
            A.attn_profile_start()
            fn()
            pr = A.attn_profile_stop()
            if i >= args.warmup:
                ts.append(pr[key] if isinstance(key, str) else sum(pr[k] for k in key))
        return statistics.median(ts)

    rows = []

    def point(name, B, H, N, dqk, dvh, causal, bwd):
        t = synth.attention_inputs_torch(synth.AttentionShape(B, H, N, dqk, dvh), seed=0, with_do=bwd, device=dev)
        o = torch.empty((B, H, N, dvh), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        sc = 1.0 / math.sqrt(dqk)
        f = 2.0 * B * H * N * N * (dqk + dvh) / (2 if causal else 1)
        fwd = lambda: A.attn_fwd(t["q"], t["k"], t["v"], o, lse, B, H, N, dqk, dvh, causal, sc)
        row = {"config": name, "B": B, "H": H, "N": N, "d_qk": dqk, "d_v": dvh, "causal": bool(causal),
               "forward_tflops": f / med(fwd, "ms_fwd") / 1e9}
        if bwd:
            fwd()
            dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
            for det in (0, 1):
                nb = A.attn_bwd_workspace_bytes(B, H, N, dqk, dvh, det)
                ws = torch.empty(nb, dtype=torch.uint8, device=dev)
                bw = lambda: A.attn_bwd(t["q"], t["k"], t["v"], o, t["do"], lse, dq, dk, dv, B, H, N, dqk, dvh,
                                        causal, sc, det, ws, nb)
                tag = "deterministic" if det else "atomic"
                row[f"backward_main_tflops_{tag}"] = 2.5 * f / med(bw, "ms_bwd_main") / 1e9
                row[f"backward_call_tflops_{tag}"] = 2.5 * f / med(
                    bw, ("ms_bwd_pre", "ms_bwd_main", "ms_bwd_convert")) / 1e9
        rows.append(row)
        torch.cuda.synchronize(dev)

    point("1 (PR1)", 1, 2, 256, 64, 64, 0, True)
    point("2", 2, 16, 2048, 128, 128, 0, False)
    for N in (1024, 2048, 4096, 8192, 16384):
        for c in (0, 1):
            point("3/5", 16384 // N, 16, N, 128, 128, c, True)
    for N in (1024, 2048, 4096, 8192, 16384):
        point("4", 16384 // N, 16, N, 192, 128, 1, True)
        point("4 (non-causal backward)", 16384 // N, 16, N, 192, 128, 0, True)
    out.update({"config": {"sweep": "BASELINE configurations", "l2": "256 MiB flushed before each call"},
                "rows": rows})


def run_case(args):
    """Time the FP8, split-KV or masked path (CUDA events, L2 flushed before
    each timed call, median of --steps after --warmup)."""
    import numpy as np
    import torch

    import exact_attention_77_gb300 as A
    import synth

    A.get_lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    B, H, N, d = args.B, args.H, args.N, args.d
    scale = 1.0 / math.sqrt(d)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        ts = []
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    out = {"case": args.case, "steps": args.steps, "warmup": args.warmup, "data": "synthetic (seeded N(0,1) bf16)"}
    if args.case in ("exp2", "detsched", "sweep"):
        {"exp2": run_exp2_case, "detsched": run_detsched_case, "sweep": run_sweep_case}[args.case](args, A, torch, dev,
                                                                                              out)
        print(json.dumps(out), flush=True)
        return
    if args.case == "fp8":
        t = synth.attention_inputs_torch(synth.AttentionShape(B, H, N, d, d), seed=0, with_do=False, device=dev)
        nt = (N + 127) // 128
        q8, k8, v8 = (torch.empty((B, H, N, d), dtype=torch.uint8, device=dev) for _ in range(3))
        sq, sk = torch.empty((B, H, nt), device=dev), torch.empty((B, H, nt), device=dev)
        sv = torch.empty((B, H), device=dev)
        nb = A.attn_fp8_quantize_workspace_bytes(B, H)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        signs = [1 if (i * 2654435761) & 0x100 else -1 for i in range(d)]
        quant = lambda: A.attn_fp8_quantize(t["q"], t["k"], t["v"], signs, q8, k8, v8, sq, sk, sv, B, H, N, d, ws, nb)
        fwd = lambda: A.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, B, H, N, d, args.causal, scale)
        mq = timed(quant)
        mf = timed(fwd)
        fl = flops_fwd(args)
        out.update({"config": {"B": B, "H": H, "N": N, "d": d, "causal": bool(args.causal)}, "quantize_ms": mq,
                    "forward_ms": mf, "forward_tflops": fl / mf / 1e9, "end_to_end_tflops": fl / (mq + mf) / 1e9})
    elif args.case == "splitkv":
        Hkv = args.Hkv if args.Hkv > 0 else H
        tq = synth.decode_inputs_torch(synth.DecodeShape(B, H, args.Nq, 1, d, d), seed=0, device=dev)
        tk = synth.decode_inputs_torch(synth.DecodeShape(B, Hkv, 1, args.Nk, d, d), seed=1, device=dev)
        rows = (H // Hkv) * args.Nq  # query rows per K/V head (grouped-query heads packed)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        ns = A.attn_splitkv_heuristic(B, Hkv, rows, args.Nk, d, sms)
        nb = A.attn_fwd_splitkv_workspace_bytes(B, Hkv, rows, args.Nk, d, ns)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        o = torch.empty((B, H, args.Nq, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, args.Nq), dtype=torch.float32, device=dev)
        fn = lambda: A.attn_fwd_splitkv_gqa(tq["q"], tk["k"], tk["v"], o, lse, B, H, Hkv, args.Nq, args.Nk, d, d, scale,
                                            ns, ws, nb)
        ms = timed(fn)
        byts = B * (2 * Hkv * args.Nk + 2 * H * args.Nq) * d * 2
        out.update({"config": {"B": B, "H": H, "H_kv": Hkv, "N_q": args.Nq, "N_k": args.Nk, "d": d, "ranges": ns},
                    "ms": ms, "gbs": byts / ms / 1e6, "note": "one call (split forward + merge), bytes = K, V, Q, O"})
    else:
        t = synth.attention_inputs_torch(synth.AttentionShape(B, H, N, d, d), seed=0, device=dev)
        T = (N + 127) // 128
        block = None
        if args.block_density < 1.0:
            rng = np.random.Generator(np.random.PCG64(0))
            block = torch.from_numpy((rng.random((T, T)) < args.block_density).astype(np.uint8)).to(dev)
        o = torch.empty_like(t["v"])
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
        nb = A.attn_bwd_workspace_bytes(B, H, N, d, d, args.det)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        wl, wr = args.window_left, args.window_right
        fwd = lambda: A.attn_fwd_masked(t["q"], t["k"], t["v"], o, lse, B, H, N, d, d, wl, wr, block, scale)
        bwd = lambda: A.attn_bwd_masked(t["q"], t["k"], t["v"], o, t["do"], lse, dq, dk, dv, B, H, N, d, d, wl, wr,
                                        block, scale, args.det, ws, nb)
        mf = timed(fwd)
        fwd()
        mb = timed(bwd)
        # visible pairs from the window per row, times the kept share of tiles when a block map is used
        i = np.arange(N)
        lo = np.maximum(0, i - wl) if wl >= 0 else np.zeros(N, np.int64)
        hi = np.minimum(N - 1, i + wr) if wr >= 0 else np.full(N, N - 1)
        pairs = float((hi - lo + 1).clip(min=0).sum())
        if block is not None:
            pairs *= float(block.float().mean())
        fl = 4.0 * B * H * d * pairs
        out.update({"config": {"B": B, "H": H, "N": N, "d": d, "window": [wl, wr], "block_density": args.block_density,
                               "dq_mode": "deterministic" if args.det else "atomic"},
                    "forward_ms": mf, "backward_ms": mb, "forward_tflops": fl / mf / 1e9,
                    "backward_tflops": 2.5 * fl / mb / 1e9,
                    "note": "TFLOP/s over the visible pairs (with a block map: window pairs x kept share of tiles)"})
    st, where = A.attn_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status: {A.status_string(st)} at {where}")
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--N", type=int, default=16384)
    ap.add_argument("--d", type=int, default=128, help="head dim of Q and K (d_qk)")
    ap.add_argument("--dv", type=int, default=0, help="head dim of V, O and dO (0: the same as --d)")
    ap.add_argument("--causal", type=int, default=0)
    ap.add_argument("--det", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustain-seconds", type=float, default=2.0,
                    help="length of the back-to-back sustained leg (0: skip it)")
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="head groups pipelined through host copies and compute in the e2e leg")
    ap.add_argument("--e2e-streams", type=int, default=3, help="compute streams the e2e leg deals its groups to")
    ap.add_argument("--e2e-taper", type=int, default=1, choices=(0, 1),
                    help="1: halve the e2e leg's first and last head groups (shorter pipeline fill and drain)")
    ap.add_argument("--case", choices=("step", "fp8", "splitkv", "masked", "exp2", "detsched", "sweep"), default="step",
                    help="step: the benchmark contract; others time the library's other paths")
    ap.add_argument("--Nq", type=int, default=1)
    ap.add_argument("--Nk", type=int, default=16384)
    ap.add_argument("--Hkv", type=int, default=0, help="splitkv case: K/V heads (grouped-query; 0 = --H)")
    ap.add_argument("--window-left", type=int, default=-1)
    ap.add_argument("--window-right", type=int, default=0)
    ap.add_argument("--block-density", type=float, default=1.0)
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.case != "step":
        run_case(args)
        return
    world, rank, local = dist_env()
    if world != args.gpus and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
