"""Helpers shared by the GPU parity tests: tensor conversion for the oracle,
error measurement and the tolerances."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances: max-abs error of out and lse against the fp64 oracle.
TOL_OUT = {torch.bfloat16: 2e-2, torch.float32: 1e-5}
TOL_LSE = 1e-3


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


def max_err(got: torch.Tensor, want: np.ndarray) -> float:
    g = got.detach().float().cpu().numpy().astype(np.float64).reshape(want.shape)
    return float(np.max(np.abs(g - want))) if want.size else 0.0


def assert_finite(*ts):
    for t in ts:
        assert torch.isfinite(t).all(), "NaN or Inf in output"


def check_forward(O, q, k, v, P, out, lse, rows=None):
    """Compare out/lse of a forward call (all rows or the listed flat rows)."""
    want_out, want_lse = oracle_ring(O, q, k, v, P, rows=rows)
    d = q.shape[-1]
    o2 = out.reshape(-1, d)
    l2 = lse.reshape(-1)
    if rows is not None:
        idx = torch.as_tensor(rows, device=out.device)
        o2 = o2.index_select(0, idx)
        l2 = l2.index_select(0, idx)
    eo = max_err(o2, want_out)
    el = max_err(l2, want_lse)
    assert eo <= TOL_OUT[q.dtype], f"out max-abs error {eo:.3e}"
    assert el <= TOL_LSE, f"lse max-abs error {el:.3e}"
    return eo, el
