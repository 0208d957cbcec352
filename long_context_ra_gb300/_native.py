"""ctypes loader of the CUDA library ``_lib/libra_gb300.so``.

There is no fallback: if the library has not been built (see ``build.py``)
or cannot be loaded, every entry point raises.  The prototypes below mirror
``include/ra.h`` one for one.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "_lib" / "libra_gb300.so"

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_MISALIGNED, RA_ERR_ARCH, RA_ERR_CUDA, \
    RA_ERR_TIMEOUT = range(7)
RA_F32, RA_BF16 = 0, 1
RA_LAYOUTS = {"contiguous": 0, "zigzag": 1, "striped": 2}
RA_MAX_PARTIALS = 64
RA_SPLIT_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


class RaStateC(ctypes.Structure):
    """``ra_state``: device pointers m [rows], l [rows], o [rows, d] (fp32)."""

    _fields_ = [("m", ctypes.c_void_p), ("l", ctypes.c_void_p), ("o", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("d", ctypes.c_int32)]


# Exported symbol -> (restype, argtypes).
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SP = ctypes.POINTER(RaStateC)
PROTOTYPES = {
    "ra_forward": (_I32, [_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _P]),
    "ra_forward_causal": (_I32, [_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _I32,
                                 _P]),
    "ra_forward_partial": (_I32, [_P, _P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _SP, _I32, _P]),
    "ra_forward_partial_causal": (_I32, [_P, _P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _SP,
                                         _I32, _I32, _P]),
    "ra_forward_split": (_I32, [_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _P, _I64,
                                _I32, _P]),
    "ra_forward_split_workspace_bytes": (_I64, [_I32, _I32, _I64, _I32, _I32]),
    "ra_forward_split_noalloc": (_I32, [_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _I32, _I32,
                                        _I32, _P]),
    "ra_forward_split_segments": (_I32, [_I32, _I32, _I64, _I32, _I32, _I32]),
    "ra_forward_host": (_I32, [_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _I32, _I32, _I32, _I32,
                               _P, _I64, _P]),
    "ra_forward_host_workspace_bytes": (_I64, [_I32, _I32, _I64, _I32, _I32]),
    "ra_backward": (_I32, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _I32,
                           _I32, _P]),
    "ra_backward_causal": (_I32, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I64, _I32,
                                  _I32, _I32, _I32, _P]),
    "ra_backward_rowterms": (_I32, [_P, _P, _P, _I64, _I32, _I32, _P, _P]),
    "ra_backward_block": (_I32, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32,
                                 _P]),
    "ra_state_init": (_I32, [_SP, _P]),
    "ra_fold": (_I32, [_SP, _P, _P, _P, _I64, _I64, _I32, _P]),
    "ra_merge": (_I32, [_SP, _I32, _P, _P, _I32, _P]),
    "ra_last_device_status": (_I32, [_P]),
    "ra_watchdog_config": (None, [_I64, _I64]),
    "ra_status_string": (ctypes.c_char_p, [_I32]),
    "ra_version": (_I32, []),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (loaded on first use; raises if it is missing)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m long_context_ra_gb300.build` "
                "(there is no CPU fallback)")
        L = ctypes.CDLL(str(LIB_PATH))
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib
