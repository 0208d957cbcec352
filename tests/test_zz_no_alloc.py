"""The allocation-free split forward, called through the C ABI.

Some callers of this library may not allocate device memory while they run:
a plug-in whose host process already owns the device's memory pool, or a
latency-bound loop that cannot take the implicit synchronisation of
cudaMalloc.  ra_forward_split_noalloc serves them by keeping its scratch (the
partial states of the split) in a device array owned by the library.

The test makes two calls in a row, on different inputs, and checks each
against ra_forward_split, which takes its scratch from the caller, within
the tolerances the other tests use.  This file is collected last so that a
run stopping at the first failure has run every other test first.
"""
import ctypes

import pytest
import torch

from gpu_util import TOL_LSE, TOL_OUT, check_same
import long_context_ra_gb300 as ra
from long_context_ra_gb300 import _native
from long_context_ra_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def L():
    build()
    return _native.lib()


def _inputs(shape, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return [torch.randn(shape, device=DEV, generator=g).to(torch.bfloat16) for _ in range(3)]


def _noalloc(L, q, k, v, P, G, out=None, lse=None):
    B, H, N, d = q.shape
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(B, H, N, device=DEV, dtype=torch.float32) if lse is None else lse
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = L.ra_forward_split_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                      lse.data_ptr(), B, H, N, d, P, G, _native.RA_BF16, stream)
    assert code == _native.RA_OK, L.ra_status_string(code)
    return out, lse


def test_noalloc_matches_caller_scratch_twice(L):
    B, H, N, d, P, G = 1, 2, 4096, 128, 8, 2
    assert ra.ra_forward_split_workspace_bytes(B, H, N, d, G) <= \
        _native.RA_SPLIT_NOALLOC_SCRATCH_BYTES
    for call in range(2):  # the second call runs over the first call's scratch
        q, k, v = _inputs((B, H, N, d), 500 + call)
        out, lse = _noalloc(L, q, k, v, P, G)
        ref_out, ref_lse = ra.ra_forward_split(q, k, v, P, G=G)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        check_same(out, ref_out, torch.bfloat16, "noalloc vs split out", TOL_OUT[torch.bfloat16])
        check_same(lse, ref_lse, torch.bfloat16, "noalloc vs split lse", TOL_LSE, relative=False)
    assert ra.ra_last_device_status() == 0


def test_noalloc_call_takes_no_device_memory(L):
    """After a first call (which looks up the scratch address), a call leaves
    the device's free memory exactly as it was: it allocated nothing."""
    B, H, N, d, P, G = 1, 2, 4096, 128, 8, 2
    q, k, v = _inputs((B, H, N, d), 600)
    out = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=DEV, dtype=torch.float32)
    _noalloc(L, q, k, v, P, G, out, lse)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    _noalloc(L, q, k, v, P, G, out, lse)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert ra.ra_last_device_status() == 0


def test_noalloc_rejects_partials_beyond_the_scratch(L):
    # 8 partial states of 65536 rows x 130 floats do not fit 32 MiB
    B, H, N, d, P, G = 1, 1, 65536, 128, 8, 8
    assert ra.ra_forward_split_workspace_bytes(B, H, N, d, G) > \
        _native.RA_SPLIT_NOALLOC_SCRATCH_BYTES
    q = torch.empty(B, H, N, d, device=DEV, dtype=torch.bfloat16)
    lse = torch.empty(B, H, N, device=DEV)
    code = L.ra_forward_split_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(),
                                      lse.data_ptr(), B, H, N, d, P, G, _native.RA_BF16, None)
    assert code == _native.RA_ERR_UNSUPPORTED
