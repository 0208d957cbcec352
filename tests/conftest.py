import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parent.parent
for p in (str(ROOT), str(ROOT / "tests")):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Achieved parity errors of the GPU tests: per checked tensor, the
    worst max-abs error and the worst errors relative to the signal."""
    mod = sys.modules.get("gpu_util")
    recs = getattr(mod, "RECORDS", None)
    if not recs:
        return
    worst = {}
    for r in recs:
        key = (r["test"].split("::")[0].split("/")[-1], r["test"].split("::")[-1].split("[")[0],
               r["what"], r["dtype"])
        w = worst.setdefault(key, {"abs": 0.0, "rel_max": 0.0, "rel_rms": 0.0, "ref_max": 0.0,
                                   "checks": 0})
        for f in ("abs", "rel_max", "rel_rms", "ref_max"):
            w[f] = max(w[f], r[f])
        w["checks"] += 1
    tr = terminalreporter
    tr.write_sep("-", "achieved parity errors (worst per test and tensor)")
    tr.write_line(f"{'test':58s} {'tensor':22s} {'dtype':8s} {'max-abs':>9s} {'max|ref|':>9s} "
                  f"{'rel-max':>9s} {'rel-rms':>9s} {'n':>4s}")
    for (f, t, what, dt), w in sorted(worst.items()):
        tr.write_line(f"{(f + '::' + t)[-58:]:58s} {what[:22]:22s} {dt:8s} {w['abs']:9.2e} "
                      f"{w['ref_max']:9.2e} {w['rel_max']:9.2e} {w['rel_rms']:9.2e} "
                      f"{w['checks']:4d}")
