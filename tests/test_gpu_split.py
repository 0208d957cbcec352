"""Split forward (ring segments folded in parallel into caller scratch, then
merged) against the fp64 oracle and the plain forward, through the C ABI."""
import pytest
import torch

import long_context_ra_gb300 as ra
from gpu_util import TOL_LSE, TOL_OUT, assert_finite, check_forward, check_same
from long_context_ra_gb300 import synth
from oracle import ra_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def O():
    return ra_oracle.get()


def rnd(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(shape, device=DEV, generator=g).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("G", [1, 2, 3, 8])
def test_split_matches_oracle(O, dtype, G):
    B, H, N, d, P = 1, 2, 1024, 64, 8
    q, k, v = (rnd((B, H, N, d), 60 + s, dtype) for s in range(3))
    out, lse = ra.ra_forward_split(q, k, v, P, G=G)
    assert_finite(out, lse)
    check_forward(O, q, k, v, P, out, lse)
    ref_out, ref_lse = ra.ra_forward(q, k, v, P)
    check_same(out, ref_out, dtype, "split vs forward out", TOL_OUT[dtype])
    check_same(lse, ref_lse, dtype, "split vs forward lse", TOL_LSE, relative=False)


def test_split_recommendation():
    # workload 2: 32 K/V tiles per query block, too few to split
    w = synth.WORKLOADS[2]
    assert ra.ra_forward_split_segments(w.B, w.H, w.N, w.d, w.P, w.dtype) == 1
    # one head of 16384 tokens, P = 1: 64 CTAs of 128 tiles each
    G = ra.ra_forward_split_segments(1, 1, 16384, 128, 1, torch.bfloat16)
    assert G == 1  # G <= P = 1
    G = ra.ra_forward_split_segments(1, 1, 16384, 128, 8, torch.bfloat16)
    assert G == 2  # 64 CTAs unsplit; 2 x 64 still fit in one wave of 152 SMs


def test_split_long_single_head(O):
    """One head, 16384 tokens, P = 8: the recommended split over sampled rows."""
    B, H, N, d, P = 1, 1, 16384, 128, 8
    q, k, v = (rnd((B, H, N, d), 80 + s) for s in range(3))
    G = ra.ra_forward_split_segments(B, H, N, d, P, q.dtype)
    out, lse = ra.ra_forward_split(q, k, v, P, G=G)
    rows = torch.randperm(N, generator=torch.Generator().manual_seed(3))[:512].sort().values
    check_forward(O, q, k, v, P, out, lse, rows=rows.numpy())


def test_split_workload2(O):
    """Workload 2 through the split path with G = 2."""
    w = synth.WORKLOADS[2]
    q, k, v = synth.make_inputs(w, DEV)
    out, lse = ra.ra_forward_split(q, k, v, w.P, G=2)
    check_forward(O, q, k, v, w.P, out, lse)
    assert ra.ra_last_device_status() == 0


def test_split_workspace_reuse_and_errors():
    B, H, N, d, P = 1, 1, 512, 128, 4
    q, k, v = (rnd((B, H, N, d), 70 + s) for s in range(3))
    nbytes = ra.ra_forward_split_workspace_bytes(B, H, N, d, 4)
    ws = torch.full((nbytes,), 0xFF, device=DEV, dtype=torch.uint8)  # stale contents
    a, la = ra.ra_forward_split(q, k, v, P, G=4, workspace=ws)
    b, lb = ra.ra_forward_split(q, k, v, P, G=4, workspace=ws)
    assert torch.equal(a, b) and torch.equal(la, lb)
    with pytest.raises(ra.RaError):
        ra.ra_forward_split(q, k, v, P, G=4, workspace=ws[: nbytes - 256])
