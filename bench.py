#!/usr/bin/env python
"""Benchmark of the ring-attention fold hot path on GB300.

One step = one ra_forward over the N = 131072, d = 128, H = 8, P = 32 bf16
workload: every query block folds all 32 visiting K/V blocks in ring order
and writes out and lse.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W]      # this library
  python bench.py --impl reference [--steps K] [--warmup W] # the fp64 CPU oracle

Several GPUs (torchrun) run independent replicas of the same workload (the
virtual ring lives on one GPU; there is no exchange between ranks).

  python bench.py --ring R   # the compute of an R-rank ring, played on one GPU

--ring times what the ranks of a multi-device ring (long_context_ra_gb300.ring)
compute, without the exchange: every rank's state initialisation, its R
ra_fold steps over the blocks (i - t) mod R, and its final ra_merge, for all
R ranks one after another on this GPU.  Each of those launches is the one a
rank makes on its own device, so the figure is the per-device efficiency of
the ring's compute.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "attention TFLOP/s (4·B·H·N²·d) at 1 GB300 and % of dense bf16 tensor peak"
UNIT = "TFLOP/s"
KERNEL_SOURCES = ["long_context_ra_gb300/csrc/ra_fold_sm103.cu",
                  "long_context_ra_gb300/csrc/sm103_pipeline.cuh",
                  "long_context_ra_gb300/csrc/sm103_ptx.cuh",
                  "long_context_ra_gb300/csrc/ra_layout.cuh"]


def kernel_sha() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update((ROOT / f).read_bytes())
    return h.hexdigest()[:16]


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {"bf16": d["bf16_tflops"], "bf16_sustained": d.get("bf16_tflops_sustained"),
                "hbm": d["hbm_gbs"], "source": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel as it is now (same source hash) and the same workload."""
    for f in sorted((ROOT / "profiles").glob("*.md")):
        text = f.read_text()
        m_sha = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
        m_wl = re.search(r"bench_workload:\s*(\S+)", text)
        m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
        if m_sha and m_b and m_wl and m_sha.group(1) == kernel_sha() and m_wl.group(1) == workload:
            return float(m_b.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str | None):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if gpu_id:
            cmd.insert(1, f"--id={gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.4)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.tmp.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:]):
                if val.lower() == "active":
                    reasons.add(n)
        os.unlink(self.tmp.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def max_over_ranks(x: float, device, world: int) -> float:
    """Largest value of x over all ranks (the slowest replica sets the time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def causal_flops(w) -> float:
    """Work of causal attention: 4 d flops per visible (query, key) pair,
    N (N + 1) / 2 pairs per head."""
    return 4.0 * w.B * w.H * w.d * w.N * (w.N + 1) / 2.0


L2_BYTES = 129 * 2**20  # GB300 L2
FLUSH_BYTES = 512 * 2**20  # written between timed steps when the inputs fit in L2


def input_bytes(w) -> int:
    esize = 2 if "bf16" in w.name else 4
    return 3 * w.rows * w.d * esize


def flushes_l2(w) -> bool:
    """True when q, k and v together fit in twice the L2: the timed steps are
    then separated by an L2 flush instead of relying on the input size."""
    return input_bytes(w) < 2 * L2_BYTES


def l2_note(w) -> str:
    """How the timed steps avoid an L2-resident working set (both arms)."""
    mib = input_bytes(w) / 2**20
    if flushes_l2(w):
        return (f"L2 flushed before every timed step ({FLUSH_BYTES >> 20} MiB written, "
                f"outside the timed events; q+k+v = {mib:.0f} MiB)")
    return f"inputs larger than L2 (q+k+v = {mib:.0f} MiB)"


def host_pipeline_stages(host_in, host_out, dev_in, results, w, stream) -> dict:
    """The parts of ra_forward_host's pipeline that the compute cannot hide:
    the upload of its first chunk and the download of its last (each timed
    alone with CUDA events), next to the whole device-resident call."""
    import torch

    slices = w.B * w.H
    # ra_forward_host's chunk count: at most 8, at least 16 MiB of q, k, v each
    chunks = max(1, min(slices, 8, input_bytes(w) // (16 << 20)))
    first = slices // chunks  # slices in the first chunk
    last = slices - (chunks - 1) * slices // chunks
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def up():
        for dst, src in zip(dev_in, host_in):
            n = src.numel() // slices * first
            dst.view(-1)[:n].copy_(src.view(-1)[:n], non_blocking=True)

    def down():
        for dst, src in zip(host_out, results):
            n = src.numel() // slices * last
            dst.view(-1)[-n:].copy_(src.view(-1)[-n:], non_blocking=True)

    return {"first_chunk_upload": timed(up), "last_chunk_download": timed(down),
            "chunks": chunks}


def job_throughput(flops_per_replica: float, world: int, ms_max: float) -> float:
    """Whole-job TFLOP/s: every replica's work over the slowest replica's time."""
    return world * flops_per_replica / (ms_max * 1e-3) / 1e12


def oracle_view(t, w):
    """(array, dtype tag) of a [B, H, N, d] tensor for the oracle: bf16 as its
    bit patterns, fp32 as is (the oracle widens both exactly)."""
    import numpy as np
    import torch

    t = t.reshape(w.B * w.H, w.N, w.d).cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), "bf16"
    return t.float().numpy(), "f32"


def cpu_oracle_baseline(w, q, k, v, target_s: float):
    """Time the fp64 oracle (as it stands) on a bounded, seeded sample of the
    workload's query rows on all host cores; scale to TFLOP/s."""
    import numpy as np
    import torch

    from oracle import ra_oracle

    O = ra_oracle.get()
    (qa, tag), (ka, _), (va, _) = oracle_view(q, w), oracle_view(k, w), oracle_view(v, w)
    g = np.random.default_rng(99)
    pool = np.sort(g.choice(w.rows, size=min(w.rows, 65536), replace=False))
    per_row = 4.0 * w.N * w.d
    probe = pool[:: max(1, len(pool) // 16)][:16]
    t0 = time.perf_counter()
    O.ring(qa, ka, va, w.P, dtype=tag, rows=probe)
    t_probe = time.perf_counter() - t0
    n = int(min(len(pool), max(16, len(probe) * target_s / max(t_probe, 1e-6))))
    rows = pool[np.linspace(0, len(pool) - 1, n).astype(np.int64)]
    t0 = time.perf_counter()
    want = O.ring(qa, ka, va, w.P, dtype=tag, rows=rows)
    dt = time.perf_counter() - t0
    # the same oracle on one core, on a sample sized for about 3 s
    O1 = ra_oracle.Oracle(threads=1)
    n1 = int(min(n, max(4, 3.0 * n / (max(dt, 1e-6) * O.threads))))
    rows1 = rows[np.linspace(0, len(rows) - 1, n1).astype(np.int64)]
    t0 = time.perf_counter()
    O1.ring(qa, ka, va, w.P, dtype=tag, rows=rows1)
    dt1 = time.perf_counter() - t0
    return {"value": n * per_row / dt / 1e12, "unit": UNIT, "cores": O.threads, "kind": "oracle",
            "sample": f"{n} seeded query rows of {w.name} (ring recurrence, fp64), {dt:.1f} s; "
                      f"value = rows x 4*N*d flops / time",
            "value_1core": n1 * per_row / dt1 / 1e12,
            "sample_1core": f"{n1} of those rows on one core, {dt1:.1f} s",
            "projected_full_s": dt * w.rows / n}, rows, want


def sampled_parity(out, lse, rows, w_out, w_lse, w) -> dict:
    """The timed run's out and lse on the rows the CPU baseline computed,
    against those oracle values (the parity bars of the tests)."""
    import numpy as np
    import torch

    idx = torch.as_tensor(rows, device=out.device)
    got_out = out.reshape(-1, w.d).index_select(0, idx).double().cpu().numpy()
    got_lse = lse.reshape(-1).index_select(0, idx).double().cpu().numpy()
    e_out = float(np.abs(got_out - w_out).max())
    e_lse = float(np.abs(got_lse - w_lse).max())
    ref = float(np.abs(w_out).max())
    rms = float(np.sqrt(np.mean((got_out - w_out) ** 2)) / np.sqrt(np.mean(w_out ** 2)))
    if w.dtype == torch.float32:  # the FFMA path's bars
        bars = {"max_abs_out": 1e-5, "max_abs_lse": 1e-5, "rel_max_out": 2.0 ** -13,
                "rel_rms_out": 2.0 ** -14}
    else:
        bars = {"max_abs_out": 2e-2, "max_abs_lse": 1e-3, "rel_max_out": 2.0 ** -6,
                "rel_rms_out": 2.0 ** -7}
    got = {"max_abs_out": e_out, "max_abs_lse": e_lse, "rel_max_out": e_out / ref,
           "rel_rms_out": rms}
    return {"rows": int(len(rows)), "against": "the fp64 oracle on the rows of cpu_baseline",
            **got, "bars": bars, "pass": all(got[x] <= bars[x] for x in bars)}


def ring_parity(ra, q, k, v, r_out, r_lse, w, R: int) -> dict:
    """Every rank's out and lse of the played ring against the fused forward
    of the same inputs (two routes of the library to the same rows)."""
    import torch

    out, lse = ra.ra_forward(q, k, v, w.P)
    c, bh = w.N // R, w.B * w.H
    e_out = e_lse = ref = 0.0
    for i in range(R):
        want = out[:, :, i * c:(i + 1) * c].reshape(bh * c, w.d).float()
        e_out = max(e_out, (r_out[i].float() - want).abs().max().item())
        ref = max(ref, want.abs().max().item())
        wl = lse[:, :, i * c:(i + 1) * c].reshape(-1)
        e_lse = max(e_lse, (r_lse[i] - wl).abs().max().item())
    torch.cuda.synchronize()
    bars = {"max_abs_out": 2e-2, "max_abs_lse": 1e-3, "rel_max_out": 2.0 ** -6}
    got = {"max_abs_out": e_out, "max_abs_lse": e_lse, "rel_max_out": e_out / ref}
    return {"rows": bh * w.N, "against": "ra_forward on the same inputs (every row)", **got,
            "bars": bars, "pass": all(got[x] <= bars[x] for x in bars)}


def cpu_oracle_baseline_causal(w, q, k, v, layout: str, target_s: float):
    """The CPU baseline of a causal forward: the fp64 oracle's causal ring
    (same layout) timed on seeded query rows on all host cores, about
    `target_s` seconds; a row at position n costs 4 d (n + 1) flops.
    Returns (baseline, rows, the oracle's (out, lse) of those rows)."""
    import numpy as np
    import torch

    from long_context_ra_gb300 import synth
    from oracle import ra_oracle

    O = ra_oracle.get()
    (qa, tag), (ka, _), (va, _) = oracle_view(q, w), oracle_view(k, w), oracle_view(v, w)
    probe = synth.sample_rows(w, 16, seed=11).numpy()
    t0 = time.perf_counter()
    O.ring(qa, ka, va, w.P, dtype=tag, rows=probe, causal=True, layout=layout)
    t_probe = time.perf_counter() - t0
    n = int(min(4096, max(64, len(probe) * target_s / max(t_probe, 1e-6))))
    rows = synth.sample_rows(w, n, seed=11).numpy()
    t0 = time.perf_counter()
    want = O.ring(qa, ka, va, w.P, dtype=tag, rows=rows, causal=True, layout=layout)
    dt = time.perf_counter() - t0
    flops = float(np.sum(4.0 * w.d * (rows % w.N + 1)))
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": O.threads, "kind": "oracle",
            "sample": f"{len(rows)} seeded query rows of {w.name} under the causal mask "
                      f"({layout}; fp64 ring), {dt:.1f} s; value = the rows' visible "
                      f"4*d*(n+1) flops / time"}, rows, want


def cpu_oracle_baseline_backward(w, q, k, v, out, dout, lse, causal: bool):
    """The CPU baseline of a backward: the fp64 oracle's per-row backward
    timed on all host cores for dq of 64 seeded query rows and dk, dv of 64
    seeded key rows (a dq row costs 6 N d flops, a dk, dv row 8 N d).
    Returns (baseline, rows, the oracle's (dq, dk, dv) of those rows)."""
    import numpy as np
    import torch

    from long_context_ra_gb300 import synth
    from oracle import ra_oracle

    O = ra_oracle.get()
    rows = synth.sample_rows(w, 64, seed=5).numpy()
    views = [oracle_view(t, w) for t in (q, k, v, out, dout)]
    args = tuple(a for a, _ in views) + (lse.double().cpu().numpy(),)
    t0 = time.perf_counter()
    want = O.backward_rows(*args, rows, rows, dtype=views[0][1], causal=causal)
    dt = time.perf_counter() - t0
    pos = (rows % w.N).astype(np.float64)
    if causal:  # a query at position n meets n + 1 keys, a key N - n queries
        flops = float(np.sum(6.0 * w.d * (pos + 1) + 8.0 * w.d * (w.N - pos)))
    else:
        flops = len(rows) * 14.0 * w.N * w.d
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": O.threads, "kind": "oracle",
            "sample": f"dq of {len(rows)} seeded query rows and dk, dv of {len(rows)} seeded "
                      f"key rows of {w.name} (fp64 per-row backward"
                      f"{', causal' if causal else ''}), {dt:.2f} s; value = 6 d flops per "
                      f"visible key of a dq row + 8 d per visible query of a dk, dv row, "
                      f"/ time"}, rows, want


def backward_parity(grads, rows, want, w) -> dict:
    """dq, dk, dv of the timed backward on the rows of its CPU baseline,
    against those oracle values (the tests' bars)."""
    import numpy as np
    import torch

    idx = torch.as_tensor(rows, device=grads[0].device)
    res = {}
    ok = True
    for name, got, wt in zip(("dq", "dk", "dv"), grads, want):
        g = got.reshape(-1, w.d).index_select(0, idx).double().cpu().numpy()
        e = float(np.abs(g - wt).max())
        ref = float(np.abs(wt).max())
        rms = float(np.sqrt(np.mean((g - wt) ** 2)) / np.sqrt(np.mean(wt ** 2)))
        res[name] = {"max_abs": e, "rel_max": e / ref, "rel_rms": rms}
        ok = ok and e <= 2e-2 * max(1.0, ref) and e / ref <= 2.0 ** -6 and rms <= 2.0 ** -7
    return {"rows": int(len(rows)), "against": "the fp64 oracle's per-row backward (the rows "
            "of cpu_baseline)", **res,
            "bars": {"max_abs": "2e-2 max(1, max|ref|)", "rel_max": 2.0 ** -6,
                     "rel_rms": 2.0 ** -7}, "pass": ok}


def run_reference(args, w) -> None:
    """The CPU oracle as the reference arm, on this arm's workload and metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import torch

    from long_context_ra_gb300 import synth
    from oracle import ra_oracle

    O = ra_oracle.get()
    q, k, v = synth.make_inputs(w, "cpu")
    (qa, tag), (ka, _), (va, _) = oracle_view(q, w), oracle_view(k, w), oracle_view(v, w)
    per_row = 4.0 * w.N * w.d
    g = np.random.default_rng(7)
    probe = np.sort(g.choice(w.rows, size=8, replace=False))
    t0 = time.perf_counter()
    O.ring(qa, ka, va, w.P, dtype=tag, rows=probe)
    t_probe = (time.perf_counter() - t0) / len(probe)
    budget = args.ref_seconds / max(1, args.steps + args.warmup)  # whole run ~2 minutes
    n = int(min(w.rows, max(4, min(4096, budget / max(t_probe, 1e-6)))))
    times = []
    for s in range(args.warmup + args.steps):
        rows = np.sort(g.choice(w.rows, size=n, replace=False))
        t0 = time.perf_counter()
        O.ring(qa, ka, va, w.P, dtype=tag, rows=rows)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    t_step = sum(times) / len(times)
    value = n * per_row / t_step / 1e12
    sample = f"{n} seeded query rows of {w.name} per step (fp64 ring recurrence)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {**w.describe(), "parallelism": "replicas",
                                        "l2": l2_note(w)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": O.threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_ours(args, w) -> None:
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    if rank == 0:
        from long_context_ra_gb300.build import build
        build()
    barrier()
    import long_context_ra_gb300 as ra
    from long_context_ra_gb300 import synth

    q, k, v = synth.make_inputs(w, dev)
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream()

    if args.backward:
        if args.causal:
            out0, lse0 = ra.ra_forward_causal(q, k, v, w.P, layout=args.causal)
        else:
            out0, lse0 = ra.ra_forward(q, k, v, w.P)
        g = torch.Generator(device=dev).manual_seed(4242)
        dout = torch.randn(q.shape, device=dev, generator=g).to(q.dtype)
        ws = torch.empty(2 * w.rows, device=dev, dtype=torch.float32)

        def step():
            return ra.ra_backward(q, k, v, out0, dout, lse0, w.P, workspace=ws,
                                  causal=args.causal)
    elif args.ring is not None:
        R = args.ring
        c, bh = w.N // R, w.B * w.H
        if R < 1 or w.N % R or c % 128:
            raise SystemExit(f"--ring {R}: the block N / R must be a multiple of 128")

        def blocks(t):
            return [t[:, :, i * c:(i + 1) * c].reshape(bh, c, w.d).contiguous() for i in range(R)]

        qs, ks, vs = blocks(q), blocks(k), blocks(v)  # what each rank holds
        states = [ra.new_state(bh * c, w.d, dev) for _ in range(R)]
        r_out = [torch.empty(bh * c, w.d, device=dev, dtype=q.dtype) for _ in range(R)]
        r_lse = [torch.empty(bh * c, device=dev, dtype=torch.float32) for _ in range(R)]

        def step():
            for st in states:
                ra.ra_state_init(st)
            for t in range(R):
                for i in range(R):
                    j = (i - t) % R
                    ra.ra_fold(states[i], qs[i], ks[j], vs[j], batch=bh)
            for i in range(R):
                ra.ra_merge([states[i]], out=r_out[i], lse=r_lse[i])
            return r_out + r_lse
    elif args.split is not None:
        G = args.split or ra.ra_forward_split_segments(w.B, w.H, w.N, w.d, w.P, w.dtype)
        ws = torch.empty(ra.ra_forward_split_workspace_bytes(w.B, w.H, w.N, w.d, G), device=dev,
                         dtype=torch.uint8)

        def step():
            return ra.ra_forward_split(q, k, v, w.P, G=G, workspace=ws, out=out, lse=lse)
    elif args.causal:
        def step():
            return ra.ra_forward_causal(q, k, v, w.P, layout=args.causal, out=out, lse=lse)
    else:
        def step():
            return ra.ra_forward(q, k, v, w.P, out=out, lse=lse)
    flops = causal_flops(w) if args.causal else w.flops
    if args.backward:
        # five products of 2 N^2 d per head (S, dP, dV, dQ, dK)
        flops = 2.5 * (causal_flops(w) if args.causal else w.flops)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ra.ra_last_device_status() != 0:
        raise RuntimeError("kernel watchdog fired during warm-up")

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    if flushes_l2(w):
        # small inputs: each step timed alone, after a write larger than L2
        flush = torch.empty(FLUSH_BYTES, device=dev, dtype=torch.uint8)
        marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
        for a, b in marks:
            flush.fill_(1)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in marks) / args.steps
    else:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
    barrier()
    clocks = sampler.stop()
    if ra.ra_last_device_status() != 0:
        raise RuntimeError("kernel watchdog fired in the timed region")
    ms_max = max_over_ranks(ms, dev, world)
    value = job_throughput(flops, world, ms_max)

    # end to end through the C ABI: the step's inputs from pinned host memory
    # to the device, the call, its results back to pinned host memory, every
    # step
    dev_in = [q, k, v] + ([out0, dout, lse0] if args.backward else [])
    if args.ring is not None:
        dev_in = qs + ks + vs  # each rank's blocks
    host_in = [x.cpu().pin_memory() for x in dev_in]
    results = step()
    host_out = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in results]
    if not args.backward and args.split is None and args.ring is None:
        # the host-buffer entry point: chunked upload / compute / download
        e2e_path = "ra_forward_host"
        ws_host = torch.empty(ra.ra_forward_host_workspace_bytes(w.B, w.H, w.N, w.d, q.dtype),
                              device=dev, dtype=torch.uint8)

        def e2e_step():
            ra.ra_forward_host(*host_in, w.P, out=host_out[0], lse=host_out[1],
                               workspace=ws_host, causal=args.causal)
    else:
        e2e_path = "copies + device call"

        def e2e_step():
            for dst, src in zip(dev_in, host_in):
                dst.copy_(src, non_blocking=True)
            for dst, src in zip(host_out, step()):
                dst.copy_(src, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    n_e2e = args.steps  # the same step count as the device leg
    barrier()
    w0 = time.perf_counter()
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - w0) / n_e2e
    ms_e2e = max(e0.elapsed_time(e1) / n_e2e, wall * 1e3)
    ms_e2e_max = max_over_ranks(ms_e2e, dev, world)
    e2e_value = job_throughput(flops, world, ms_e2e_max)
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    stages = None
    if e2e_path == "ra_forward_host":
        stages = host_pipeline_stages(host_in, host_out, dev_in, results, w, stream)

    peaks = load_peaks()
    achieved = flops / (ms * 1e-3) / 1e12  # one fold launch per step
    traffic = None if (args.causal or args.backward or args.ring is not None) \
        else profiled_traffic(w.name)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"], "unit": UNIT,
                "frac": achieved / peaks["bf16"], "traffic": traffic,
                "kernel": (f"dkv_kernel<{w.d}> + dq_kernel<{w.d}> (the whole backward step)"
                           if args.backward else
                           f"fold_sm103_kernel<{w.d}> partials + merge (the whole step)"
                           if args.split is not None else
                           f"fold_sm103_kernel<{w.d}> in fold mode + merge (all ranks' steps)"
                           if args.ring is not None else
                           f"fold_sm103_kernel<{w.d}, causal>" if args.causal else
                           f"fold_sm103_kernel<{w.d}>"),
                "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)"
                if peaks["source"] == "measured" else "fallback 1.9 PFLOP/s bf16 burst"}
    if w.dtype == torch.float32:
        # the FFMA path: bound by fp32 FMA issue, not the tensor cores.  Peak =
        # SMs x 128 FP32 lanes x 2 flops x the maximum SM clock seen.
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = clocks.get("sm_max_mhz") or 2070.0
        alu_peak = sms * 128 * 2 * mhz * 1e6 / 1e12
        roofline.update({"bound": "alu", "peak": alu_peak, "frac": achieved / alu_peak,
                         "traffic": None,
                         "kernel": "fold_f32 (tiled, split over clusters on small grids, or rows split over warps on the smallest)",
                         "peak_source": f"derived: {sms} SMs x 128 FP32 lanes x 2 flops x "
                                        f"{mhz:.0f} MHz"})
        if ms < 0.1:
            roofline["note"] = (f"a {flops / 1e6:.1f} MFLOP problem in {ms * 1e3:.1f} us a "
                                "call: launch- and latency-bound, not ALU-bound")

    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.causal \
            and not args.backward and args.ring is None:
        cpu, rows, (w_out, w_lse) = cpu_oracle_baseline(w, q, k, v, args.cpu_seconds)
        parity = sampled_parity(out, lse, rows, w_out, w_lse, w)
    elif rank == 0 and world == 1 and args.ring is not None:
        parity = ring_parity(ra, q, k, v, r_out, r_lse, w, args.ring)
    elif rank == 0 and world == 1 and not args.no_cpu_baseline and args.causal \
            and not args.backward:
        cpu, rows, (w_out, w_lse) = cpu_oracle_baseline_causal(w, q, k, v, args.causal,
                                                                args.cpu_seconds)
        parity = sampled_parity(out, lse, rows, w_out, w_lse, w)
        parity["against"] = f"the fp64 oracle's causal ring ({args.causal}) on the rows of " \
                            "cpu_baseline"
    elif rank == 0 and world == 1 and not args.no_cpu_baseline and args.backward \
            and args.causal in (None, "contiguous"):
        cpu, rows, want = cpu_oracle_baseline_backward(w, q, k, v, out0, dout, lse0,
                                                       args.causal is not None)
        parity = backward_parity(results, rows, want, w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if w.dtype == torch.float32 else "bf16", "data": "synthetic",
            "config": {**w.describe(), "parallelism": "replicas",
                       **({"causal": args.causal} if args.causal else {}),
                       **({"split_segments": G} if args.split is not None else {}),
                       **({"pass": "backward"} if args.backward else {}),
                       **({"ring_ranks": args.ring, "block": w.N // args.ring,
                           "pass": "ring compute: every rank's state init, R ra_fold steps "
                                   "and ra_merge, played on one GPU, no exchange"}
                          if args.ring is not None else {}),
                       "l2": l2_note(w)},
            "roofline": roofline, "cpu_baseline": cpu,
            **({"parity": parity} if parity else {}),
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e_max, "path": e2e_path,
                    "steps": n_e2e, "of_device_value": e2e_value / value,
                    **({"stages_ms": stages} if stages else {})},
            "gpu_launches": args.steps * (3 if args.backward else 2 if args.split is not None
                                          else args.ring * (args.ring + 2)
                                          if args.ring is not None else 1),
            "clocks": clocks,
            "pct_of_peak": 100.0 * achieved / peaks["bf16"],
            "exps_per_s": (flops / (4.0 * w.d)) / (ms * 1e-3),
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4, help="workload key (default 4)")
    ap.add_argument("--heads", type=int, default=None, help="override the head count")
    ap.add_argument("--tokens", type=int, default=None, help="override N")
    ap.add_argument("--head-dim", type=int, default=None, help="override d")
    ap.add_argument("--blocks", type=int, default=None, help="override P")
    ap.add_argument("--causal", choices=["contiguous", "zigzag", "striped"], default=None,
                    help="time ra_forward_causal with this layout instead of ra_forward")
    ap.add_argument("--split", type=int, default=None,
                    help="time ra_forward_split with G segments (0 = recommended)")
    ap.add_argument("--backward", action="store_true",
                    help="time ra_backward (5 products per head counted: 10 B H N^2 d)")
    ap.add_argument("--ring", type=int, default=None,
                    help="time the compute of an R-rank multi-device ring on this GPU")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="CPU time of the whole --impl reference run (default 120 s)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # timing rule: at least 3 warm-up steps
    from long_context_ra_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    if args.heads is not None and args.heads != w.H:
        # a smaller case of the same workload (for profiler captures)
        w = dataclasses.replace(w, H=args.heads, name=f"{w.name.replace(f'_H{w.H}_', f'_H{args.heads}_')}")
    # other shapes with the same recipe and dtype (profiler captures, sweeps):
    # the name states every size
    shape = {"N": args.tokens, "d": args.head_dim, "P": args.blocks}
    if any(x is not None for x in shape.values()):
        kw = {k: x for k, x in shape.items() if x is not None}
        w = dataclasses.replace(w, **kw)
        w = dataclasses.replace(w, name=f"{str(w.dtype).replace('torch.', '').replace('bfloat16', 'bf16').replace('float32', 'fp32')}"
                                        f"_B{w.B}_H{w.H}_N{w.N}_d{w.d}_P{w.P}_{w.recipe}")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
