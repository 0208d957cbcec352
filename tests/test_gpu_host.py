"""Host-buffer forward (ra_forward_host: chunked upload / compute / download)
against the device entry points and the fp64 oracle, through the C ABI."""
import pytest
import torch

import long_context_ra_gb300 as ra
from gpu_util import assert_finite, check_forward

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def O():
    from oracle import ra_oracle
    return ra_oracle.get()


def host_rnd(shape, seed, dtype=torch.bfloat16, pinned=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g).to(dtype)
    return x.pin_memory() if pinned else x


def device_reference(q, k, v, P, causal):
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    if causal is None:
        return ra.ra_forward(qd, kd, vd, P)
    return ra.ra_forward_causal(qd, kd, vd, P, layout=causal)


# slices = B*H: one chunk, an odd count, and more slices than chunks (uneven
# chunks of 1 and 2 slices)
@pytest.mark.parametrize("B,H", [(1, 1), (1, 3), (2, 5)])
@pytest.mark.parametrize("causal", [None, "zigzag"])
def test_host_equals_device_call(B, H, causal):
    N, d, P = 1024, 64, 4
    q, k, v = (host_rnd((B, H, N, d), 10 + s) for s in range(3))
    out, lse = ra.ra_forward_host(q, k, v, P, causal=causal)
    torch.cuda.synchronize()
    assert not out.is_cuda and not lse.is_cuda
    ref_out, ref_lse = device_reference(q, k, v, P, causal)
    # the same kernels on the same data: identical bits
    assert torch.equal(out, ref_out.cpu())
    assert torch.equal(lse, ref_lse.cpu())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_host_matches_oracle(O, dtype):
    B, H, N, d, P = 1, 2, 512, 128, 4
    q, k, v = (host_rnd((B, H, N, d), 20 + s, dtype) for s in range(3))
    out, lse = ra.ra_forward_host(q, k, v, P)
    torch.cuda.synchronize()
    assert_finite(out, lse)
    check_forward(O, q.to(DEV), k.to(DEV), v.to(DEV), P, out.to(DEV), lse.to(DEV))


def test_host_pageable_memory():
    # pageable host memory: same results, the copies just do not overlap
    B, H, N, d, P = 1, 2, 1024, 128, 8
    q, k, v = (host_rnd((B, H, N, d), 30 + s, pinned=False) for s in range(3))
    out, lse = ra.ra_forward_host(q, k, v, P)
    torch.cuda.synchronize()
    ref_out, ref_lse = device_reference(q, k, v, P, None)
    assert torch.equal(out, ref_out.cpu()) and torch.equal(lse, ref_lse.cpu())


def test_host_two_calls_reuse_workspace():
    B, H, N, d, P = 1, 4, 1024, 64, 4
    ws = torch.empty(ra.ra_forward_host_workspace_bytes(B, H, N, d, torch.bfloat16), device=DEV,
                     dtype=torch.uint8)
    res = []
    for seed in (40, 50):
        q, k, v = (host_rnd((B, H, N, d), seed + s) for s in range(3))
        out, lse = ra.ra_forward_host(q, k, v, P, workspace=ws)
        res.append((q, k, v, out, lse))
    torch.cuda.synchronize()
    for q, k, v, out, lse in res:
        ref_out, ref_lse = device_reference(q, k, v, P, None)
        assert torch.equal(out, ref_out.cpu()) and torch.equal(lse, ref_lse.cpu())


def test_host_empty_problem():
    q = torch.empty(1, 0, 1024, 64, dtype=torch.bfloat16)
    out, lse = ra.ra_forward_host(q, q, q, 4)
    torch.cuda.synchronize()
    assert out.numel() == 0 and lse.numel() == 0
