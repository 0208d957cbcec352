"""ctypes front end of the fp64 Ring Attention oracle (``ra_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``.  The product library never loads
it and it loads nothing from the product library.

Arrays are numpy; bf16 inputs are passed as their raw ``uint16`` bit patterns
(``dtype="bf16"``) and widened exactly inside the oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "ra_oracle.cpp"

_DTYPES = {"f64": 0, "f32": 1, "bf16": 2}
LAYOUTS = {"contiguous": 0, "zigzag": 1, "striped": 2}
_NP = {"f64": np.float64, "f32": np.float32, "bf16": np.uint16}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int


def lib_path(mutant: int = 0, outdir: Path | None = None) -> Path:
    name = "libra_oracle.so" if mutant == 0 else f"libra_oracle_m{mutant}.so"
    return (outdir or HERE) / name


def compile_oracle(mutant: int = 0, outdir: Path | None = None) -> Path:
    """Compile the oracle with g++ (optionally with a planted mistake)."""
    out = lib_path(mutant, outdir)
    if out.exists() and out.stat().st_mtime >= SRC.stat().st_mtime:
        return out
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", f"-DORA_MUTANT={mutant}", str(SRC), "-o", str(out) + ".tmp"]
    subprocess.run(cmd, check=True)
    os.replace(str(out) + ".tmp", out)
    return out


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


class Oracle:
    """Thin typed wrapper over the oracle's C entry points."""

    def __init__(self, mutant: int = 0, outdir: Path | None = None, threads: int | None = None):
        self.path = compile_oracle(mutant, outdir)
        self.lib = ctypes.CDLL(str(self.path))
        self.threads = threads or default_threads()
        L = self.lib
        L.ora_ring_order.argtypes = [_I64, _P]
        L.ora_dense.argtypes = [_P, _P, _P, _I32, _I64, _I64, _I32, _I32, _P, _I64, _P, _P, _I32]
        L.ora_ring.argtypes = [_P, _P, _P, _I32, _I64, _I64, _I32, _I64, _P, _I64, _I64,
                               _I64, _I32, _I32, _P, _I64, _P, _P, _P, _P, _P, _I32]
        L.ora_layout_positions.argtypes = [_I32, _I64, _I64, _P]
        L.ora_backward_rows.argtypes = [_P, _P, _P, _I32, _P, _P, _P, _I64, _I64, _I32, _I32,
                                        _P, _I64, _P, _P, _I64, _P, _P, _I32]
        L.ora_backward.argtypes = [_P, _P, _P, _I32, _P, _P, _P, _I64, _I64, _I32, _I64, _I32,
                                   _I32, _P, _P, _P, _I32]
        L.ora_fold.argtypes = [_P, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _I32, _I32]
        L.ora_merge.argtypes = [_P, _P, _P, _I64, _I64, _I32, _P, _P, _P, _P, _P]
        for f in (L.ora_ring_order, L.ora_dense, L.ora_ring, L.ora_fold, L.ora_merge,
                  L.ora_layout_positions, L.ora_backward, L.ora_backward_rows):
            f.restype = _I32
        L.ora_mutant.restype = _I32
        self.mutant = L.ora_mutant()

    # -- helpers -----------------------------------------------------------
    @staticmethod
    def _arr(x, dtype: str):
        a = np.ascontiguousarray(x, dtype=_NP[dtype])
        return a, a.ctypes.data

    @staticmethod
    def _rows(rows):
        if rows is None:
            return None, None, 0
        r = np.ascontiguousarray(rows, dtype=np.int64)
        return r, r.ctypes.data, r.size

    @staticmethod
    def _check(rc: int, what: str):
        if rc != 0:
            raise ValueError(f"oracle {what} rejected its arguments (code {rc})")

    # -- entry points --------------------------------------------------------
    def ring_order(self, P: int) -> np.ndarray:
        out = np.zeros((P, P), dtype=np.int64)
        self._check(self.lib.ora_ring_order(P, out.ctypes.data), "ring_order")
        return out

    def layout_positions(self, layout: str, P: int, c: int) -> np.ndarray:
        """[P, c]: position of local row r of block j under `layout`."""
        out = np.zeros((P, c), dtype=np.int64)
        self._check(self.lib.ora_layout_positions(LAYOUTS[layout], P, c, out.ctypes.data),
                    "layout_positions")
        return out

    def dense(self, q, k, v, dtype="f64", rows=None, causal=False):
        """q, k, v: [BH, N, d].  Returns out [R, d], lse [R] (float64)."""
        BH, N, d = q.shape
        qa, qp = self._arr(q, dtype)
        ka, kp = self._arr(k, dtype)
        va, vp = self._arr(v, dtype)
        ra, rp, R = self._rows(rows)
        if ra is None:
            R = BH * N
        out = np.empty((R, d), np.float64)
        lse = np.empty((R,), np.float64)
        self._check(self.lib.ora_dense(qp, kp, vp, _DTYPES[dtype], BH, N, d, int(causal), rp, R,
                                       out.ctypes.data, lse.ctypes.data, self.threads), "dense")
        return out, lse

    def ring(self, q, k, v, P, dtype="f64", order=None, t0=0, t1=None, tile=0, rows=None,
             state=False, causal=False, layout="contiguous"):
        """Ring recurrence over steps [t0, t1) of the visiting order.

        Returns (out, lse) or, with ``state=True``, (out, lse, m, l, o)."""
        BH, N, d = q.shape
        t1 = P if t1 is None else t1
        qa, qp = self._arr(q, dtype)
        ka, kp = self._arr(k, dtype)
        va, vp = self._arr(v, dtype)
        ra, rp, R = self._rows(rows)
        if ra is None:
            R = BH * N
        oa = None
        op = None
        if order is not None:
            oa = np.ascontiguousarray(order, dtype=np.int64)
            op = oa.ctypes.data
        out = np.empty((R, d), np.float64)
        lse = np.empty((R,), np.float64)
        m = np.empty((R,), np.float64)
        l = np.empty((R,), np.float64)
        o = np.empty((R, d), np.float64)
        rc = self.lib.ora_ring(qp, kp, vp, _DTYPES[dtype], BH, N, d, P, op, t0, t1, tile,
                               int(causal), LAYOUTS[layout], rp, R,
                               out.ctypes.data, lse.ctypes.data, m.ctypes.data, l.ctypes.data,
                               o.ctypes.data, self.threads)
        self._check(rc, "ring")
        return (out, lse, m, l, o) if state else (out, lse)

    def fold(self, m, l, o, q, kb, vb, dtype="f64", batch=1):
        """One fold of a visiting block into state (m, l, o); returns the new state."""
        m = np.array(m, dtype=np.float64, copy=True)
        l = np.array(l, dtype=np.float64, copy=True)
        o = np.array(o, dtype=np.float64, copy=True)
        R, d = o.shape
        Nk = kb.shape[-2] if kb.ndim >= 2 else 0
        qa, qp = self._arr(q, dtype)
        ka, kp = self._arr(kb, dtype)
        va, vp = self._arr(vb, dtype)
        rc = self.lib.ora_fold(m.ctypes.data, l.ctypes.data, o.ctypes.data, qp, kp, vp,
                               _DTYPES[dtype], batch, R, Nk, d, self.threads)
        self._check(rc, "fold")
        return m, l, o

    def backward(self, q, k, v, out, dout, lse, P, dtype="f64", causal=False,
                 layout="contiguous"):
        """Gradients (dq, dk, dv) of L = sum(dout * out); q, k, v, out, dout:
        [BH, N, d]; lse: [BH, N] (the forward's)."""
        BH, N, d = q.shape
        qa, qp = self._arr(q, dtype)
        ka, kp = self._arr(k, dtype)
        va, vp = self._arr(v, dtype)
        oa = np.ascontiguousarray(out, dtype=np.float64)
        da = np.ascontiguousarray(dout, dtype=np.float64)
        la = np.ascontiguousarray(lse, dtype=np.float64)
        dq = np.empty((BH, N, d), np.float64)
        dk = np.empty((BH, N, d), np.float64)
        dv = np.empty((BH, N, d), np.float64)
        rc = self.lib.ora_backward(qp, kp, vp, _DTYPES[dtype], oa.ctypes.data, da.ctypes.data,
                                   la.ctypes.data, BH, N, d, P, int(causal), LAYOUTS[layout],
                                   dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, self.threads)
        self._check(rc, "backward")
        return dq, dk, dv

    def backward_rows(self, q, k, v, out, dout, lse, qrows, krows, dtype="f64", causal=False):
        """dq for flat rows `qrows`, (dk, dv) for flat rows `krows`.
        out and dout have q's dtype; lse is [BH*N]."""
        BH, N, d = q.shape
        qa, qp = self._arr(q, dtype)
        ka, kp = self._arr(k, dtype)
        va, vp = self._arr(v, dtype)
        oa, op = self._arr(out, dtype)
        ga, gp = self._arr(dout, dtype)
        la = np.ascontiguousarray(lse, dtype=np.float64).reshape(-1)
        qr = np.ascontiguousarray(qrows, dtype=np.int64)
        kr = np.ascontiguousarray(krows, dtype=np.int64)
        dq = np.empty((qr.size, d), np.float64)
        dk = np.empty((kr.size, d), np.float64)
        dv = np.empty((kr.size, d), np.float64)
        rc = self.lib.ora_backward_rows(qp, kp, vp, _DTYPES[dtype], op, gp, la.ctypes.data, BH,
                                        N, d, int(causal), qr.ctypes.data, qr.size, dq.ctypes.data,
                                        kr.ctypes.data, kr.size, dk.ctypes.data, dv.ctypes.data,
                                        self.threads)
        self._check(rc, "backward_rows")
        return dq, dk, dv

    def merge(self, m, l, o, state=False):
        """m, l: [G, R]; o: [G, R, d].  Returns out, lse (and the merged state)."""
        m = np.ascontiguousarray(m, dtype=np.float64)
        l = np.ascontiguousarray(l, dtype=np.float64)
        o = np.ascontiguousarray(o, dtype=np.float64)
        G, R, d = o.shape
        out = np.empty((R, d), np.float64)
        lse = np.empty((R,), np.float64)
        mo = np.empty((R,), np.float64)
        lo = np.empty((R,), np.float64)
        oo = np.empty((R, d), np.float64)
        rc = self.lib.ora_merge(m.ctypes.data, l.ctypes.data, o.ctypes.data, G, R, d,
                                out.ctypes.data, lse.ctypes.data, mo.ctypes.data,
                                lo.ctypes.data, oo.ctypes.data)
        self._check(rc, "merge")
        return (out, lse, mo, lo, oo) if state else (out, lse)


_DEFAULT: Oracle | None = None


def get() -> Oracle:
    """The correct (non-mutant) oracle, compiled on first use."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
