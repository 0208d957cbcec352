"""The C ABI on the host: the library loads, exports every declared entry
point, and validates arguments before touching the GPU (no GPU needed)."""
import ctypes
import re
from pathlib import Path

import pytest

from long_context_ra_gb300 import _native
from long_context_ra_gb300.build import build

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def L():
    build()
    return _native.lib()


def declared_symbols():
    text = (ROOT / "include" / "ra.h").read_text()
    return sorted(set(re.findall(r"RA_API\s+[\w\s\*]+?\b(ra_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 8, names
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_native.PROTOTYPES), "binding prototypes drift from the header"


def test_status_strings(L):
    for code in range(7):
        s = L.ra_status_string(code).decode()
        assert s.startswith("RA_"), s
    assert b"unknown" in L.ra_status_string(99)
    assert L.ra_version() >= 100


BF16, F32 = _native.RA_BF16, _native.RA_F32
A = 1 << 20  # a fake, 16-byte-aligned "device" address: never dereferenced


def fwd(L, q=A, k=A, v=A, out=A, lse=A, B=1, H=1, N=256, d=64, P=2, dt=BF16):
    return L.ra_forward(q, k, v, out, lse, B, H, N, d, P, dt, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), _native.RA_ERR_INVALID_ARG),
    (dict(lse=None), _native.RA_ERR_INVALID_ARG),
    (dict(B=-1), _native.RA_ERR_INVALID_ARG),
    (dict(N=-4), _native.RA_ERR_INVALID_ARG),
    (dict(d=0), _native.RA_ERR_INVALID_ARG),
    (dict(P=0), _native.RA_ERR_INVALID_ARG),
    (dict(dt=7), _native.RA_ERR_INVALID_ARG),
    (dict(N=250, P=4), _native.RA_ERR_UNSUPPORTED),            # P does not divide N
    (dict(d=96), _native.RA_ERR_UNSUPPORTED),                  # bf16 head dim
    (dict(N=256, P=4), _native.RA_ERR_UNSUPPORTED),            # bf16 c = 64 not a multiple of 128
    (dict(d=300, dt=F32), _native.RA_ERR_UNSUPPORTED),         # f32 head dim
    (dict(q=A + 8), _native.RA_ERR_MISALIGNED),                # TMA needs 16 bytes
    (dict(out=A + 8), _native.RA_ERR_MISALIGNED),
    (dict(q=A + 2, dt=F32), _native.RA_ERR_MISALIGNED),
])
def test_forward_validation(L, kw, code):
    assert fwd(L, **kw) == code


def test_empty_problem_launches_nothing(L):
    # zero rows: RA_OK without any CUDA call (no device here)
    assert fwd(L, B=0) == _native.RA_OK
    assert fwd(L, N=0, P=1) == _native.RA_OK
    # an empty tensor's data pointer is NULL: still fine when there is no row
    assert fwd(L, q=None, k=None, v=None, out=None, lse=None, H=0) == _native.RA_OK


def test_valid_call_without_device_reports_arch(L):
    # arguments are fine; with no CUDA device the call stops at the device check
    assert fwd(L) == _native.RA_ERR_ARCH


def test_fold_and_merge_validation(L):
    st = _native.RaStateC(A, A, A, 256, 64)
    ref = ctypes.byref(st)
    assert L.ra_fold(None, A, A, A, 1, 128, BF16, None) == _native.RA_ERR_INVALID_ARG
    assert L.ra_fold(ref, A, A, A, 0, 128, BF16, None) == _native.RA_ERR_INVALID_ARG
    assert L.ra_fold(ref, A, A, A, 3, 128, BF16, None) == _native.RA_ERR_UNSUPPORTED  # 256 % 3
    assert L.ra_fold(ref, A, A, A, 1, 100, BF16, None) == _native.RA_ERR_UNSUPPORTED  # kv % 128
    assert L.ra_fold(ref, A, A, A, 1, 0, BF16, None) == _native.RA_OK  # nothing to fold
    arr = (_native.RaStateC * 2)(st, _native.RaStateC(A, A, A, 128, 64))
    assert L.ra_merge(arr, 2, A, A, BF16, None) == _native.RA_ERR_INVALID_ARG  # rows differ
    assert L.ra_merge(arr, 0, A, A, BF16, None) == _native.RA_ERR_INVALID_ARG
    assert L.ra_merge(arr, 65, A, A, BF16, None) == _native.RA_ERR_INVALID_ARG
    assert L.ra_forward_partial(A, A, A, 1, 1, 256, 64, 2, 3, arr, BF16, None) == \
        _native.RA_ERR_INVALID_ARG  # G > P
    empty = _native.RaStateC(A, A, A, 0, 64)
    assert L.ra_state_init(ctypes.byref(empty), None) == _native.RA_OK
    assert L.ra_state_init(None, None) == _native.RA_ERR_INVALID_ARG


def test_causal_validation(L):
    def fc(layout=0, N=1024, P=4, d=64, dt=BF16):
        return L.ra_forward_causal(A, A, A, A, A, 1, 1, N, d, P, layout, dt, None)
    assert fc(layout=3) == _native.RA_ERR_INVALID_ARG
    assert fc(layout=-1) == _native.RA_ERR_INVALID_ARG
    assert fc(layout=1, N=1536, P=4) == _native.RA_ERR_UNSUPPORTED   # zigzag bf16: c % 256
    assert fc(layout=1, N=12, P=4, dt=F32) == _native.RA_ERR_UNSUPPORTED  # zigzag: c odd
    assert fc(layout=0, N=2048 * 128, P=2048) == _native.RA_ERR_UNSUPPORTED  # bf16 P > 1024
    assert fc(layout=2, N=1024, P=8) == _native.RA_ERR_ARCH  # valid: stops at the device check
    assert fc(layout=1, N=16, P=4, dt=F32) == _native.RA_ERR_ARCH


def test_split_validation(L):
    need = L.ra_forward_split_workspace_bytes(1, 2, 1024, 64, 4)
    rows = 2 * 1024
    up = lambda x: (x + 255) // 256 * 256
    assert need == 4 * (2 * up(rows * 4) + up(rows * 64 * 4))
    assert L.ra_forward_split_workspace_bytes(1, 2, 1024, 64, 0) == -1
    assert L.ra_forward_split_workspace_bytes(1, 2, 1024, 64, 65) == -1

    def fs(ws=A, nbytes=need, G=4, P=4):
        return L.ra_forward_split(A, A, A, A, A, 1, 2, 1024, 64, P, G, ws, nbytes, BF16, None)
    assert fs(ws=None) == _native.RA_ERR_INVALID_ARG
    assert fs(nbytes=need - 1) == _native.RA_ERR_INVALID_ARG
    assert fs(ws=A + 16) == _native.RA_ERR_MISALIGNED   # needs 256-byte alignment
    assert fs(G=0) == _native.RA_ERR_INVALID_ARG
    assert fs(G=8, P=4) == _native.RA_ERR_INVALID_ARG   # G > P
    assert fs() == _native.RA_ERR_ARCH                  # valid; no device here


def test_noalloc_split_rejects_oversize_without_device(L):
    # the size check comes before any device work
    assert L.ra_forward_split_noalloc(A, A, A, A, A, 1, 1, 65536, 128, 8, 8, BF16, None) == \
        _native.RA_ERR_UNSUPPORTED
    assert L.ra_forward_split_noalloc(A, A, A, A, A, 1, 1, 65536, 128, 8, 0, BF16, None) == \
        _native.RA_ERR_INVALID_ARG
    assert L.ra_forward_split_noalloc(A, A, A, A, A, 1, 2, 4096, 128, 8, 2, BF16, None) == \
        _native.RA_ERR_ARCH


def test_noalloc_split_checks_arguments_before_the_scratch_size(L):
    # oversize for the scratch AND wrong otherwise: the argument error wins
    big = dict(B=1, H=1, N=65536, d=128, P=8)

    def fn(q=A, out=A, lse=A, G=8, dt=BF16, **kw):
        a = {**big, **kw}
        return L.ra_forward_split_noalloc(q, A, A, out, lse, a["B"], a["H"], a["N"], a["d"],
                                          a["P"], G, dt, None)
    assert fn() == _native.RA_ERR_UNSUPPORTED                    # valid, too large
    assert fn(G=16) == _native.RA_ERR_INVALID_ARG                 # G > P
    assert fn(q=None) == _native.RA_ERR_INVALID_ARG
    assert fn(lse=None) == _native.RA_ERR_INVALID_ARG
    assert fn(dt=9) == _native.RA_ERR_INVALID_ARG
    assert fn(q=A + 8) == _native.RA_ERR_MISALIGNED
    assert fn(out=A + 8) == _native.RA_ERR_MISALIGNED
    assert fn(N=65536 - 8) == _native.RA_ERR_UNSUPPORTED         # P does not divide N
    assert fn(N=1 << 31, P=1 << 14) == _native.RA_ERR_UNSUPPORTED  # too many rows, no overflow


def test_watchdog_config_is_host_only(L):
    # settings only; no device needed, nothing returned
    L.ra_watchdog_config(1 << 20, 3)
    L.ra_watchdog_config(0, -1)


def test_backward_validation(L):
    def fb(ws=A, N=1024, P=4, d=64, dt=BF16):
        return L.ra_backward(A, A, A, A, A, A, A, A, A, ws, 1, 1, N, d, P, dt, None)
    assert fb(ws=None) == _native.RA_ERR_INVALID_ARG
    assert fb(ws=A + 4) == _native.RA_ERR_MISALIGNED
    assert fb(N=1000) == _native.RA_ERR_UNSUPPORTED
    assert fb() == _native.RA_ERR_ARCH
    assert L.ra_backward_causal(A, A, A, A, A, A, A, A, A, A, 1, 1, 1024, 64, 4, 7, BF16,
                                None) == _native.RA_ERR_INVALID_ARG


def test_host_forward_validation(L):
    rows, d = 2 * 1024, 64
    up = lambda x: (x + 255) // 256 * 256
    need = L.ra_forward_host_workspace_bytes(1, 2, 1024, d, BF16)
    assert need == 4 * up(rows * d * 2) + up(rows * 4)
    assert L.ra_forward_host_workspace_bytes(1, 2, 1024, d, F32) == 4 * up(rows * d * 4) + up(rows * 4)
    assert L.ra_forward_host_workspace_bytes(-1, 2, 1024, d, BF16) == -1
    assert L.ra_forward_host_workspace_bytes(1, 2, 1024, d, 9) == -1

    def fh(q=A, out=A, ws=A, nbytes=need, N=1024, P=4, dd=d, causal=0, layout=0, dt=BF16, H=2):
        return L.ra_forward_host(q, A, A, out, A, 1, H, N, dd, P, causal, layout, dt, ws, nbytes,
                                 None)
    assert fh(q=None) == _native.RA_ERR_INVALID_ARG
    assert fh(out=None) == _native.RA_ERR_INVALID_ARG
    assert fh(ws=None) == _native.RA_ERR_INVALID_ARG
    assert fh(nbytes=need - 1) == _native.RA_ERR_INVALID_ARG
    assert fh(ws=A + 16) == _native.RA_ERR_MISALIGNED       # workspace: 256-byte alignment
    assert fh(causal=2) == _native.RA_ERR_INVALID_ARG
    assert fh(causal=1, layout=5) == _native.RA_ERR_INVALID_ARG
    assert fh(N=1000) == _native.RA_ERR_UNSUPPORTED          # P does not divide N
    assert fh(dd=96) == _native.RA_ERR_UNSUPPORTED           # bf16 head dim
    assert fh(causal=1, layout=1, N=1536, P=4) == _native.RA_ERR_UNSUPPORTED  # zigzag c % 256
    assert fh(H=0, q=None, ws=None) == _native.RA_OK        # nothing to do
    assert fh() == _native.RA_ERR_ARCH                      # valid; no device here


def test_largest_sizes(L):
    # TMA coordinates are int32: B*H*N rows must stay below 2^31
    big = 1 << 31
    assert fwd(L, N=big, P=1 << 14, d=128) == _native.RA_ERR_UNSUPPORTED
    assert fwd(L, B=2, H=1 << 14, N=1 << 16, P=1 << 9, d=128) == _native.RA_ERR_UNSUPPORTED
    # one row less than the limit passes the size rules (then stops at the device check)
    assert fwd(L, B=1, H=(1 << 14) - 1, N=1 << 17, P=1 << 10, d=128) == _native.RA_ERR_ARCH
    # the causal bf16 path keeps one step-table entry per ring step: P <= 1024
    assert L.ra_forward_causal(A, A, A, A, A, 1, 1, 1024 * 128, 128, 1024, 0, BF16, None) == \
        _native.RA_ERR_ARCH
    assert L.ra_forward_causal(A, A, A, A, A, 1, 1, 1025 * 128, 128, 1025, 0, BF16, None) == \
        _native.RA_ERR_UNSUPPORTED


def test_backward_block_validation(L):
    def fb(q=A, dq=A, rt=A, batch=2, c=256, d=64, causal=0, dt=BF16):
        return L.ra_backward_block(q, A, A, A, A, rt, dq, A, A, batch, c, d, causal, dt, None)
    assert fb(q=None) == _native.RA_ERR_INVALID_ARG
    assert fb(rt=None) == _native.RA_ERR_INVALID_ARG
    assert fb(causal=2) == _native.RA_ERR_INVALID_ARG
    assert fb(batch=-1) == _native.RA_ERR_INVALID_ARG
    assert fb(c=200) == _native.RA_ERR_UNSUPPORTED          # bf16 block of 200 rows
    assert fb(d=96) == _native.RA_ERR_UNSUPPORTED           # bf16 head dim
    assert fb(dq=A + 4) == _native.RA_ERR_MISALIGNED        # fp32 accumulator, 16 bytes on bf16
    assert fb(batch=0, q=None, dq=None, rt=None) == _native.RA_OK
    assert fb() == _native.RA_ERR_ARCH                      # valid; no device here
    assert fb(c=24, d=40, dt=F32) == _native.RA_ERR_ARCH    # fp32: any block length
    rt = L.ra_backward_rowterms
    assert rt(A, A, A, 128, 64, BF16, None, None) == _native.RA_ERR_INVALID_ARG
    assert rt(A, A, A, -1, 64, BF16, A, None) == _native.RA_ERR_INVALID_ARG
    assert rt(A, A, A, 0, 64, BF16, None, None) == _native.RA_OK
    assert rt(A, A, A, 128, 64, BF16, A + 4, None) == _native.RA_ERR_MISALIGNED
    assert rt(A, A, A, 128, 64, BF16, A, None) == _native.RA_ERR_ARCH
