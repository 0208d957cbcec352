"""GB300-native Ring Attention fold: Python binding of ``include/ra.h``.

The functions below have the names of the C entry points and only marshal
arguments (tensor pointers, sizes, the current CUDA stream); every step of
the computation runs in the library's kernels.  PyTorch provides device
memory and streams.

Layout: attention tensors are [B, H, N, d], contiguous, on one CUDA device;
bf16 (tensor cores) or float32 (FFMA path).  States are fp32 (m, l, o).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _native
from ._native import RA_BF16, RA_F32, RA_MAX_PARTIALS, RaStateC

__all__ = ["RaError", "RaState", "ra_forward", "ra_forward_causal", "ra_forward_partial",
           "ra_forward_partial_causal", "ra_forward_split", "ra_forward_split_workspace_bytes",
           "ra_forward_split_segments", "ra_forward_host", "ra_forward_host_workspace_bytes",
           "ra_backward", "ra_backward_causal", "ra_backward_rowterms", "ra_backward_block",
           "ra_state_init",
           "ra_fold", "ra_merge",
           "ra_last_device_status", "ra_watchdog_config", "new_state", "library_path"]


class RaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _native.lib().ra_status_string(code).decode()
        super().__init__(f"{where}: {msg}")


def library_path() -> str:
    return str(_native.LIB_PATH)


def _check(code: int, where: str) -> None:
    if code != 0:
        raise RaError(code, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return RA_BF16
    if t.dtype == torch.float32:
        return RA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use bfloat16 or float32")


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    """The CUDA stream handle (an int, which ctypes passes as a pointer): the
    given stream, or the current one of the current device."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: torch.Tensor) -> int:
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


@dataclass
class RaState:
    """Running online-softmax state of `rows` query rows (fp32 device tensors)."""

    m: torch.Tensor  # [rows]
    l: torch.Tensor  # [rows]
    o: torch.Tensor  # [rows, d]

    @property
    def rows(self) -> int:
        return self.o.shape[0]

    @property
    def d(self) -> int:
        return self.o.shape[1]

    def c(self) -> RaStateC:
        for t in (self.m, self.l, self.o):
            if t.dtype != torch.float32:
                raise TypeError("state tensors must be float32")
        return RaStateC(_ptr(self.m), _ptr(self.l), _ptr(self.o), self.rows,
                        self.d)


def new_state(rows: int, d: int, device=None) -> RaState:
    """Allocate (uninitialised) state storage; see ra_state_init."""
    dev = device if device is not None else torch.device("cuda")
    return RaState(torch.empty(rows, device=dev, dtype=torch.float32),
                   torch.empty(rows, device=dev, dtype=torch.float32),
                   torch.empty(rows, d, device=dev, dtype=torch.float32))


def ra_forward(q, k, v, P: int, out=None, lse=None, stream=None):
    """Ring attention forward; returns (out [B,H,N,d], lse [B,H,N] fp32)."""
    B, H, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share shape and dtype")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, N, device=q.device, dtype=torch.float32)
    code = _native.lib().ra_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                                    P, _dtype_code(q), _stream(stream))
    _check(code, "ra_forward")
    return out, lse


def ra_forward_causal(q, k, v, P: int, layout: str = "contiguous", out=None, lse=None,
                      stream=None):
    """Causal ring attention forward (query n sees keys 0..n); `layout` is
    "contiguous", "zigzag" or "striped".  Returns (out, lse)."""
    B, H, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share shape and dtype")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, N, device=q.device, dtype=torch.float32)
    code = _native.lib().ra_forward_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H,
                                           N, d, P, _native.RA_LAYOUTS[layout], _dtype_code(q),
                                           _stream(stream))
    _check(code, "ra_forward_causal")
    return out, lse


def _state_array(states):
    arr = (RaStateC * len(states))()
    for i, s in enumerate(states):
        arr[i] = s.c()
    return arr


def ra_forward_partial(q, k, v, P: int, G: int, partials=None, stream=None):
    """Ring split into G segments; returns G partial RaStates (rows = B*H*N)."""
    B, H, N, d = q.shape
    if partials is None:
        partials = [new_state(B * H * N, d, q.device) for _ in range(G)]
    arr = _state_array(partials)
    code = _native.lib().ra_forward_partial(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, P, G, arr,
                                            _dtype_code(q), _stream(stream))
    _check(code, "ra_forward_partial")
    return partials


def ra_forward_partial_causal(q, k, v, P: int, G: int, layout: str = "contiguous",
                              partials=None, stream=None):
    """Causal ring split into G segments; returns G partial RaStates."""
    B, H, N, d = q.shape
    if partials is None:
        partials = [new_state(B * H * N, d, q.device) for _ in range(G)]
    arr = _state_array(partials)
    code = _native.lib().ra_forward_partial_causal(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, P, G,
                                                   arr, _native.RA_LAYOUTS[layout],
                                                   _dtype_code(q), _stream(stream))
    _check(code, "ra_forward_partial_causal")
    return partials


def ra_forward_split_workspace_bytes(B: int, H: int, N: int, d: int, G: int) -> int:
    return int(_native.lib().ra_forward_split_workspace_bytes(B, H, N, d, G))


def ra_forward_split_segments(B: int, H: int, N: int, d: int, P: int, dtype) -> int:
    code = RA_BF16 if dtype == torch.bfloat16 else RA_F32
    return int(_native.lib().ra_forward_split_segments(B, H, N, d, P, code))


def ra_forward_split(q, k, v, P: int, G: int | None = None, workspace=None, out=None, lse=None,
                     stream=None):
    """Ring split into G segments folded in parallel, then merged.

    G=None takes ra_forward_split_segments' choice; `workspace` (a CUDA
    uint8 tensor of ra_forward_split_workspace_bytes bytes) is allocated
    when not given.  Returns (out, lse)."""
    B, H, N, d = q.shape
    if G is None:
        G = ra_forward_split_segments(B, H, N, d, P, q.dtype)
    nbytes = ra_forward_split_workspace_bytes(B, H, N, d, G)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), device=q.device, dtype=torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, N, device=q.device, dtype=torch.float32)
    code = _native.lib().ra_forward_split(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H,
                                          N, d, P, G, _ptr(workspace), workspace.numel(),
                                          _dtype_code(q), _stream(stream))
    _check(code, "ra_forward_split")
    return out, lse


def _host_ptr(t: torch.Tensor) -> ctypes.c_void_p:
    if t.is_cuda:
        raise ValueError("ra_forward_host takes host (CPU) tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def ra_forward_host_workspace_bytes(B: int, H: int, N: int, d: int, dtype) -> int:
    code = RA_BF16 if dtype == torch.bfloat16 else RA_F32
    return int(_native.lib().ra_forward_host_workspace_bytes(B, H, N, d, code))


def ra_forward_host(q, k, v, P: int, out=None, lse=None, workspace=None, causal=None,
                    stream=None):
    """Forward for HOST tensors q, k, v ([B,H,N,d], pinned for overlap): the
    library uploads, computes and downloads in overlapped chunks of (batch,
    head) slices.  causal=<layout> for the causal forward.  `workspace` is a
    CUDA uint8 tensor of ra_forward_host_workspace_bytes bytes (allocated on
    the current device when not given).  Returns host (out, lse); the call
    is asynchronous on `stream`, so synchronize before reading them."""
    B, H, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share shape and dtype")
    pinned = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=pinned)
    if lse is None:
        lse = torch.empty(B, H, N, dtype=torch.float32, pin_memory=pinned)
    nbytes = ra_forward_host_workspace_bytes(B, H, N, d, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), device=torch.cuda.current_device(),
                                dtype=torch.uint8)
    layout = _native.RA_LAYOUTS[causal] if causal is not None else 0
    code = _native.lib().ra_forward_host(_host_ptr(q), _host_ptr(k), _host_ptr(v), _host_ptr(out),
                                         _host_ptr(lse), B, H, N, d, P,
                                         0 if causal is None else 1, layout, _dtype_code(q),
                                         _ptr(workspace), workspace.numel(), _stream(stream))
    _check(code, "ra_forward_host")
    return out, lse


def ra_backward(q, k, v, out, dout, lse, P: int, workspace=None, stream=None, causal=None):
    """Gradients (dq, dk, dv) of L = sum(dout * out) for ra_forward's out/lse;
    causal=<layout> for ra_forward_causal's."""
    B, H, N, d = q.shape
    for t in (k, v, out, dout):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("q, k, v, out, dout must share shape and dtype")
    if workspace is None:
        workspace = torch.empty(2 * B * H * N, device=q.device, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ptrs = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
            _ptr(dv), _ptr(workspace))
    if causal is None:
        code = _native.lib().ra_backward(*ptrs, B, H, N, d, P, _dtype_code(q), _stream(stream))
    else:
        code = _native.lib().ra_backward_causal(*ptrs, B, H, N, d, P, _native.RA_LAYOUTS[causal],
                                                _dtype_code(q), _stream(stream))
    _check(code, "ra_backward")
    return dq, dk, dv


def ra_backward_causal(q, k, v, out, dout, lse, P: int, layout: str = "contiguous",
                       workspace=None, stream=None):
    """Gradients for ra_forward_causal (same mask and layout)."""
    return ra_backward(q, k, v, out, dout, lse, P, workspace=workspace, stream=stream,
                       causal=layout)


def ra_backward_rowterms(out, dout, lse, workspace=None, stream=None):
    """Row terms (D, -lse log2 e) of a query block: out, dout [..., d] of one
    dtype, lse of their rows; returns the fp32 workspace [2 * rows]."""
    d = out.shape[-1]
    rows = out.numel() // d
    if dout.shape != out.shape or dout.dtype != out.dtype or lse.numel() != rows:
        raise ValueError("out, dout must match and lse must have one value per row")
    if workspace is None:
        workspace = torch.empty(2 * rows, device=out.device, dtype=torch.float32)
    code = _native.lib().ra_backward_rowterms(_ptr(out), _ptr(dout), _ptr(lse), rows, d,
                                              _dtype_code(out), _ptr(workspace), _stream(stream))
    _check(code, "ra_backward_rowterms")
    return workspace


def ra_backward_block(q, k, v, dout, lse, rowterms, dq_acc, dk_acc, dv_acc, causal=False,
                      stream=None):
    """One ring-backward step: the query block (q, dout [batch, c, d], lse
    [batch, c], rowterms) against the visiting block (k, v), added into the
    fp32 accumulators dq_acc (query block) and dk_acc, dv_acc (visiting
    block).  causal=True for the query block's own block (diagonal mask)."""
    batch, c, d = q.shape
    for t in (k, v, dout):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("q, k, v, dout must share shape and dtype")
    for t in (dq_acc, dk_acc, dv_acc):
        if t.shape != q.shape or t.dtype != torch.float32:
            raise ValueError("accumulators are fp32 tensors of q's shape")
    code = _native.lib().ra_backward_block(
        _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse), _ptr(rowterms), _ptr(dq_acc),
        _ptr(dk_acc), _ptr(dv_acc), batch, c, d, 1 if causal else 0, _dtype_code(q),
        _stream(stream))
    _check(code, "ra_backward_block")


def ra_state_init(state: RaState, stream=None) -> RaState:
    sc = state.c()
    _check(_native.lib().ra_state_init(ctypes.byref(sc), _stream(stream)), "ra_state_init")
    return state


def ra_fold(state: RaState, q, kblk, vblk, batch: int = 1, stream=None) -> RaState:
    """Fold one visiting block: q [batch, rq, d], kblk/vblk [batch, kv_rows, d]."""
    if kblk.shape != vblk.shape or kblk.dtype != q.dtype or vblk.dtype != q.dtype:
        raise ValueError("kblk and vblk must match each other and q's dtype")
    kv_rows = kblk.numel() // (batch * state.d) if kblk.numel() else 0
    sc = state.c()
    code = _native.lib().ra_fold(ctypes.byref(sc), _ptr(q), _ptr(kblk), _ptr(vblk), batch,
                                 kv_rows, _dtype_code(q), _stream(stream))
    _check(code, "ra_fold")
    return state


def ra_merge(partials, out_dtype=torch.bfloat16, out=None, lse=None, stream=None):
    """Merge partial states; returns (out [rows, d], lse [rows])."""
    rows, d = partials[0].rows, partials[0].d
    dev = partials[0].o.device
    if out is None:
        out = torch.empty(rows, d, device=dev, dtype=out_dtype)
    if lse is None:
        lse = torch.empty(rows, device=dev, dtype=torch.float32)
    arr = _state_array(partials)
    code = _native.lib().ra_merge(arr, len(partials), _ptr(out), _ptr(lse), _dtype_code(out),
                                  _stream(stream))
    _check(code, "ra_merge")
    return out, lse


def ra_last_device_status(stream=None) -> int:
    """Synchronise and return (and clear) the device watchdog status code."""
    return _native.lib().ra_last_device_status(_stream(stream))


def ra_watchdog_config(wait_cycles: int = 0, stall_cta: int = -1) -> None:
    """Bounded-wait limit of the tensor-core kernels in SM cycles (<= 0: the
    default of 2^31) and the test aid `stall_cta` (>= 0: that CTA of later
    fold, dK/dV and dQ launches loads nothing, so its waits run out; -1:
    off)."""
    _native.lib().ra_watchdog_config(int(wait_cycles), int(stall_cta))
