"""Helpers shared by the GPU parity tests: tensor conversion for the oracle,
error measurement and the tolerances.

Every floating-point comparison applies two kinds of bars.

Absolute bars (the stated parity target): max-abs(out) <= 2e-2 on the bf16
path and <= 1e-5 on the fp32 path, max-abs(lse) <= 1e-3.

Signal-relative bars, so that a check can still fail where the outputs are
small.  For i.i.d. inputs the attention output has rms about sqrt(e / N)
(0.0045 at N = 131072, 0.0017 at N = 1048576), far below 2e-2, so the
absolute bar alone would pass an all-zero output there.  For a tensor x with
reference r:

    max|x - r|  <= REL_MAX * max|r|
    rms(x - r)  <= REL_RMS * rms(r)

Where the bf16 numbers come from: the tensor path rounds every p to bf16
before the P.V product (relative error <= 2^-9 per term, with independent
signs) and rounds out to bf16 (relative error <= 2^-9 per element).  The
expected error is therefore about 2^-9 |out| per element plus a noise of
rms about 2^-9 / sqrt(3) * rms(out): max-abs about 2^-8 max|r| and rms about
2^-9 rms(r).  The backward's dS = p (dP - D) is rounded to bf16 once more,
which adds a term of the same size.  The bars keep a margin of 4 or more
above those estimates: REL_MAX = 2^-6, REL_RMS = 2^-7.  A uniformly 10 %
small output misses REL_MAX six times over, and a zero or sign-flipped one
misses both bars.  The fp32 path (FFMA, expf, fp32 sums) is expected near
1e-6 relative; its bars are 2^-13 and 2^-14.

The achieved errors of every check are recorded (RECORDS) and printed in the
test summary; with RA_PARITY_LOG=<path> they are also written there as JSON
lines.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

# Absolute tolerances: max-abs error of out and lse against the fp64 oracle.
TOL_OUT = {torch.bfloat16: 2e-2, torch.float32: 1e-5}
TOL_LSE = 1e-3
# Signal-relative tolerances (see the module docstring).
REL_MAX = {torch.bfloat16: 2.0 ** -6, torch.float32: 2.0 ** -13}
REL_RMS = {torch.bfloat16: 2.0 ** -7, torch.float32: 2.0 ** -14}

RECORDS: list[dict] = []


def to_oracle(t: torch.Tensor):
    """(numpy array, dtype tag) of a [B, H, N, d] tensor as [B*H, N, d]."""
    B, H, N, d = t.shape
    t = t.reshape(B * H, N, d).cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), "bf16"
    if t.dtype == torch.float32:
        return t.numpy(), "f32"
    raise TypeError(t.dtype)


def oracle_ring(O, q, k, v, P, rows=None, **kw):
    qa, tag = to_oracle(q)
    ka, _ = to_oracle(k)
    va, _ = to_oracle(v)
    r = None if rows is None else np.asarray(rows, dtype=np.int64)
    return O.ring(qa, ka, va, P, dtype=tag, rows=r, **kw)


def _as_f64(x, shape) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().double().cpu().numpy()
    return np.asarray(x, dtype=np.float64).reshape(shape)


def max_err(got, want: np.ndarray) -> float:
    g = _as_f64(got, np.shape(want))
    return float(np.max(np.abs(g - want))) if np.size(want) else 0.0


def error_stats(got, want) -> dict:
    """Absolute and signal-relative errors of `got` against `want`."""
    w = np.asarray(want, dtype=np.float64)
    g = _as_f64(got, w.shape)
    if w.size == 0:
        return {"abs": 0.0, "ref_max": 0.0, "rel_max": 0.0, "rel_rms": 0.0, "n": 0}
    e = np.abs(g - w)
    ref_max = float(np.max(np.abs(w)))
    ref_rms = float(np.sqrt(np.mean(w * w)))
    err_rms = float(np.sqrt(np.mean(e * e)))
    return {"abs": float(np.max(e)), "ref_max": ref_max,
            "rel_max": float(np.max(e)) / ref_max if ref_max > 0 else float(np.max(e)),
            "rel_rms": err_rms / ref_rms if ref_rms > 0 else err_rms, "n": int(w.size)}


def _record(what: str, dtype, st: dict) -> None:
    rec = {"test": os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], "what": what,
           "dtype": str(dtype).replace("torch.", ""), **st}
    RECORDS.append(rec)
    path = os.environ.get("RA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def _assert_bars(st: dict, dtype, what: str, tol_abs: float | None, relative: bool) -> dict:
    _record(what, dtype, st)
    if tol_abs is not None:
        assert st["abs"] <= tol_abs, f"{what}: max-abs error {st['abs']:.3e} > {tol_abs:.1e}"
    if relative and st["n"] and st["ref_max"] > 0:
        assert st["rel_max"] <= REL_MAX[dtype], (
            f"{what}: max-abs error {st['abs']:.3e} is {st['rel_max']:.2e} of max|ref| "
            f"{st['ref_max']:.3e} (bar {REL_MAX[dtype]:.2e})")
        assert st["rel_rms"] <= REL_RMS[dtype], (
            f"{what}: rms error is {st['rel_rms']:.2e} of rms(ref) (bar {REL_RMS[dtype]:.2e})")
    return st


def check_close(got, want, dtype, what: str, tol_abs: float | None = None,
                relative: bool = True) -> dict:
    """Assert the absolute bar `tol_abs` (None: none) and, if `relative`, the
    signal-relative bars of `dtype` on `got` (tensor or array) against the
    oracle's `want`; record the achieved errors."""
    return _assert_bars(error_stats(got, want), dtype, what, tol_abs, relative)


def assert_finite(*ts):
    for t in ts:
        assert torch.isfinite(t).all(), "NaN or Inf in output"


def check_out_lse(out, lse, want_out, want_lse, dtype, what: str = "forward",
                  rows=None):
    """out/lse of a forward (all rows, or the listed flat rows) against the
    oracle's: the absolute bars on both, the relative bars on out."""
    d = want_out.shape[-1]
    o2 = out.reshape(-1, d)
    l2 = lse.reshape(-1)
    if rows is not None:
        idx = torch.as_tensor(np.asarray(rows), device=out.device)
        o2 = o2.index_select(0, idx)
        l2 = l2.index_select(0, idx)
    so = check_close(o2, want_out, dtype, f"{what} out", TOL_OUT[dtype])
    sl = check_close(l2, want_lse, dtype, f"{what} lse", TOL_LSE, relative=False)
    return so["abs"], sl["abs"]


def check_forward(O, q, k, v, P, out, lse, rows=None, **kw):
    """Compare out/lse of a forward call (all rows or the listed flat rows)
    with the oracle's ring; keyword arguments go to the oracle (causal, layout)."""
    want_out, want_lse = oracle_ring(O, q, k, v, P, rows=rows, **kw)
    return check_out_lse(out, lse, want_out, want_lse, q.dtype, rows=rows)


def check_same(got: torch.Tensor, ref: torch.Tensor, dtype, what: str,
               tol_abs: float | None = None, relative: bool = True) -> dict:
    """Two results of this library that compute the same thing by different
    routes (tensors on the device), under the same bars; the statistics are
    taken on the device."""
    g = got.detach().reshape(-1).double()
    r = ref.detach().reshape(-1).double()
    if r.numel() == 0:
        st = {"abs": 0.0, "ref_max": 0.0, "rel_max": 0.0, "rel_rms": 0.0, "n": 0}
    else:
        e = (g - r).abs()
        ref_max = r.abs().max().item()
        ref_rms = r.square().mean().sqrt().item()
        err_max = e.max().item()
        err_rms = e.square().mean().sqrt().item()
        st = {"abs": err_max, "ref_max": ref_max,
              "rel_max": err_max / ref_max if ref_max > 0 else err_max,
              "rel_rms": err_rms / ref_rms if ref_rms > 0 else err_rms, "n": int(r.numel())}
    return _assert_bars(st, dtype, what, tol_abs, relative)
