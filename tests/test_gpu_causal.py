"""Causal mask with contiguous, zigzag and striped layouts, through the C ABI,
against the fp64 oracle (query at position n sees keys 0..n; "Ring attention,
explained", section "The causal-mask catch")."""
import numpy as np
import pytest
import torch

import long_context_ra_gb300 as ra
from gpu_util import TOL_OUT, assert_finite, check_out_lse, check_same, oracle_ring
from long_context_ra_gb300 import synth
from oracle import ra_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
LAYOUTS = ["contiguous", "zigzag", "striped"]


@pytest.fixture(scope="module")
def O():
    return ra_oracle.get()


def rnd(shape, seed, dtype, scale=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(shape, device=DEV, generator=g) * scale).to(dtype)


def check(O, q, k, v, P, layout, out, lse, rows=None):
    want_out, want_lse = oracle_ring(O, q, k, v, P, rows=rows, causal=True, layout=layout)
    check_out_lse(out, lse, want_out, want_lse, q.dtype, f"causal {layout}", rows=rows)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape,P", [((1, 2, 48, 8), 4), ((2, 1, 36, 33), 6), ((1, 1, 64, 128), 1),
                                     ((1, 3, 40, 5), 2)])
def test_f32_causal(O, layout, shape, P):
    q, k, v = (rnd(shape, 7 + s, torch.float32, 1.5) for s in range(3))
    out, lse = ra.ra_forward_causal(q, k, v, P, layout=layout)
    check(O, q, k, v, P, layout, out, lse)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,H,N,P", [(1, 2, 1024, 4), (2, 1, 512, 2), (1, 1, 1536, 3),
                                     (1, 2, 512, 1), (1, 1, 2048, 8)])
def test_bf16_causal(O, layout, d, B, H, N, P):
    c = N // P
    if layout == "zigzag" and c % 256:
        pytest.skip("zigzag on the tensor path needs c % 256 == 0")
    shape = (B, H, N, d)
    q, k, v = (rnd(shape, 100 + N + d + s, torch.bfloat16) for s in range(3))
    out, lse = ra.ra_forward_causal(q, k, v, P, layout=layout)
    torch.cuda.synchronize()
    assert_finite(out, lse)
    check(O, q, k, v, P, layout, out, lse)
    assert ra.ra_last_device_status() == 0


@pytest.mark.parametrize("layout", LAYOUTS)
def test_bf16_first_token_is_v0(layout):
    """Position 0 sees only itself: out = v_0 exactly, lse = tau q_0 . k_0."""
    shape = (1, 2, 1024, 128)
    q, k, v = (rnd(shape, 300 + s, torch.bfloat16) for s in range(3))
    out, lse = ra.ra_forward_causal(q, k, v, 4, layout=layout)
    assert torch.equal(out[:, :, 0], v[:, :, 0])
    want = (q[:, :, 0].float() * k[:, :, 0].float()).sum(-1) / 128 ** 0.5
    assert (lse[:, :, 0] - want).abs().max().item() <= 1e-3


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_causal_partials_merge(O, layout, dtype):
    """One partial per ring step (G = P): many are empty for early rows."""
    B, H, N, d, P = 1, 2, 1024, 64, 4
    q, k, v = (rnd((B, H, N, d), 400 + s, dtype) for s in range(3))
    out_f, lse_f = ra.ra_forward_causal(q, k, v, P, layout=layout)
    parts = ra.ra_forward_partial_causal(q, k, v, P, G=P, layout=layout)
    assert any(torch.isneginf(p.m).any().item() for p in parts)  # empty partials exist
    out, lse = ra.ra_merge(parts, out_dtype=dtype)
    check(O, q, k, v, P, layout, out.reshape(B, H, N, d), lse.reshape(B, H, N))
    check_same(out, out_f.reshape(-1, d), dtype, f"causal {layout} merge vs forward",
               TOL_OUT[dtype])


@pytest.mark.parametrize("layout", LAYOUTS)
def test_causal_workload4_sampled(O, layout):
    """The N = 131072, d = 128, P = 32 workload under the mask, sampled rows."""
    w = synth.WORKLOADS[4]
    q, k, v = synth.make_inputs(w, DEV)
    out, lse = ra.ra_forward_causal(q, k, v, w.P, layout=layout)
    assert_finite(out, lse)
    rows = synth.sample_rows(w, 512, seed=11)
    check(O, q, k, v, w.P, layout, out, lse, rows=rows.numpy())
    assert ra.ra_last_device_status() == 0


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_causal_at_the_largest_step_count(O, layout):
    """P = 1024 ring blocks of one tile each: the largest step count of the
    causal tensor path (its per-unit step table holds 1024 entries)."""
    B, H, N, d, P = 1, 1, 1024 * 128, 128, 1024
    q, k, v = (rnd((B, H, N, d), 500 + s, torch.bfloat16) for s in range(3))
    out, lse = ra.ra_forward_causal(q, k, v, P, layout=layout)
    assert_finite(out, lse)
    g = torch.Generator().manual_seed(12)
    rows = torch.cat([torch.tensor([0, 127, 128, N - 129, N - 128, N - 1]),
                      torch.randint(0, N, (250,), generator=g)]).unique().numpy()
    check(O, q, k, v, P, layout, out, lse, rows=rows)
    assert ra.ra_last_device_status() == 0
