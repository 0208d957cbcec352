"""The benchmark's JSON line (no GPU): the reference arm, which times the CPU
oracle, prints one line with every key of the contract."""
import json
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parent.parent


def test_reference_arm_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "2",
                        "--steps", "1", "--warmup", "3", "--ref-seconds", "4"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 1 and line["warmup"] == 3
    assert line["config"]["workload"].startswith("bf16_B1_H8_N4096_d64_P8")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_warmup_floor():
    # fewer than three warm-up steps are raised to three
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "2",
                        "--steps", "1", "--warmup", "1", "--ref-seconds", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert json.loads(r.stdout.strip().splitlines()[-1])["warmup"] == 3


def _bench():
    sys.path.insert(0, str(ROOT))
    import bench
    return bench


def test_line_parity_can_fail():
    """The bench line's parity record (its own results on the CPU baseline's
    oracle rows) passes for results within rounding and fails for a planted
    mistake: a 0.9 x scaled out, a sign flip, one wrong row, a shifted lse."""
    import numpy as np
    import torch

    bench = _bench()
    from long_context_ra_gb300 import synth

    w = synth.WORKLOADS[2]
    rows = np.arange(0, w.rows, 97)
    g = np.random.default_rng(3)
    w_out = g.standard_normal((len(rows), w.d)) * 0.2
    w_lse = g.standard_normal(len(rows)) + 8.0

    def line(out_rows, lse_rows):
        out = torch.zeros(w.rows, w.d, dtype=torch.bfloat16)
        lse = torch.zeros(w.rows)
        out[torch.as_tensor(rows)] = torch.as_tensor(out_rows, dtype=torch.float64).to(torch.bfloat16)
        lse[torch.as_tensor(rows)] = torch.as_tensor(lse_rows, dtype=torch.float32)
        return bench.sampled_parity(out, lse, rows, w_out, w_lse, w)

    assert line(w_out, w_lse)["pass"]  # bf16 rounding of the right answer
    assert not line(0.9 * w_out, w_lse)["pass"]
    assert not line(-w_out, w_lse)["pass"]
    bad = w_out.copy()
    bad[5] += 0.05
    assert not line(bad, w_lse)["pass"]
    assert not line(w_out, w_lse + 2e-3)["pass"]


def test_backward_line_parity_can_fail():
    import numpy as np
    import torch

    bench = _bench()
    from long_context_ra_gb300 import synth

    w = synth.WORKLOADS[2]
    rows = np.arange(0, w.rows, 511)
    g = np.random.default_rng(4)
    want = [g.standard_normal((len(rows), w.d)) * s for s in (0.05, 0.03, 0.2)]

    def grads(scale=(1.0, 1.0, 1.0)):
        out = []
        for wt, s in zip(want, scale):
            t = torch.zeros(w.rows, w.d, dtype=torch.bfloat16)
            t[torch.as_tensor(rows)] = torch.as_tensor(wt * s).to(torch.bfloat16)
            out.append(t)
        return out

    assert bench.backward_parity(grads(), rows, want, w)["pass"]
    assert not bench.backward_parity(grads((1.0, 0.9, 1.0)), rows, want, w)["pass"]
    assert not bench.backward_parity(grads((1.0, 1.0, -1.0)), rows, want, w)["pass"]
