"""Backward pass (dQ, dK, dV) through the C ABI against the fp64 oracle.

Bars per gradient: the bf16 path must meet max-abs <= 2e-2 max(1, max|ref|)
(the forward's bf16 bar, for values of unit size; above that bf16's own
resolution, 2^-9 |x|, would exceed a flat 2e-2 once |x| > 10) and the
signal-relative bars of gpu_util (max-abs <= 2^-6 max|ref|, rms <= 2^-7
rms(ref)), which are what constrain small gradients; the bf16 path rounds P
and dS to bf16 before the tensor-core products and the gradients to bf16 at
the end, each a relative error of at most 2^-9.  The fp32 path must meet
max-abs <= 1e-5 max(1, max|ref|) and the fp32 relative bars."""
import numpy as np
import pytest
import torch

import long_context_ra_gb300 as ra
from gpu_util import check_close, to_oracle
from long_context_ra_gb300 import synth
from oracle import ra_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module")
def O():
    return ra_oracle.get()


def rnd(shape, seed, dtype, scale=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(shape, device=DEV, generator=g) * scale).to(dtype)


def close(got, want, dtype, what):
    tol = TOL[dtype] * max(1.0, float(np.abs(want).max()) if np.size(want) else 1.0)
    return check_close(got, want, dtype, what, tol)


def full_check(O, q, k, v, P, dtype, causal=None):
    B, H, N, d = q.shape
    if causal is None:
        out, lse = ra.ra_forward(q, k, v, P)
    else:
        out, lse = ra.ra_forward_causal(q, k, v, P, layout=causal)
    dout = rnd(q.shape, 999, dtype)
    dq, dk, dv = ra.ra_backward(q, k, v, out, dout, lse, P, causal=causal)
    torch.cuda.synchronize()
    qa, tag = to_oracle(q)
    ka, _ = to_oracle(k)
    va, _ = to_oracle(v)
    oa = out.double().reshape(B * H, N, d).cpu().numpy()
    ga = dout.double().reshape(B * H, N, d).cpu().numpy()
    la = lse.double().reshape(B * H, N).cpu().numpy()
    wq, wk, wv = O.backward(qa, ka, va, oa, ga, la, P, dtype=tag, causal=causal is not None,
                            layout=causal or "contiguous")
    for name, got, want in (("dq", dq, wq), ("dk", dk, wk), ("dv", dv, wv)):
        close(got, want, dtype, name)
    assert ra.ra_last_device_status() == 0


# Small fp32 problems run on the row kernels, each row split over up to 8
# warps: 256-row cases with 8 chunks a row take the 8-way split.
@pytest.mark.parametrize("shape,P", [((1, 2, 40, 8), 4), ((2, 1, 33, 5), 3), ((1, 1, 64, 128), 1),
                                     ((1, 2, 96, 64), 6), ((1, 1, 256, 64), 4)])
def test_f32_backward(O, shape, P):
    q, k, v = (rnd(shape, 10 + s, torch.float32, 1.3) for s in range(3))
    full_check(O, q, k, v, P, torch.float32)


# fp32 shapes large enough for the tiled kernels (d <= 128, 128 CTAs or more
# of 64 rows): ragged 64-row and 32-row tiles, d in both width classes
F32_TILED = [((1, 8, 1000, 100), 4), ((4, 8, 384, 40), 3), ((1, 32, 256, 128), 2),
             ((1, 16, 1024, 64), 1)]


@pytest.mark.parametrize("shape,P", F32_TILED)
def test_f32_backward_tiled(O, shape, P):
    q, k, v = (rnd(shape, 60 + s, torch.float32, 1.3) for s in range(3))
    full_check(O, q, k, v, P, torch.float32)


# fp32 shapes with too few 64-row tiles for the SMs: each tile's walk is
# split over a cluster of 2 or 4 CTAs, summed in distributed shared memory
F32_SPLIT = [((1, 4, 1024, 64), 4), ((1, 1, 2048, 128), 8), ((1, 2, 1024, 40), 2)]


@pytest.mark.parametrize("shape,P", F32_SPLIT)
def test_f32_backward_tiled_cluster_split(O, shape, P):
    q, k, v = (rnd(shape, 70 + s, torch.float32, 1.3) for s in range(3))
    full_check(O, q, k, v, P, torch.float32)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_f32_backward_tiled_cluster_split_causal(O, layout):
    q, k, v = (rnd((1, 2, 2048, 64), 74 + s, torch.float32, 1.3) for s in range(3))
    full_check(O, q, k, v, 4, torch.float32, causal=layout)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_f32_backward_tiled_causal(O, layout):
    q, k, v = (rnd((1, 8, 1024, 72), 64 + s, torch.float32, 1.3) for s in range(3))
    full_check(O, q, k, v, 4, torch.float32, causal=layout)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,H,N,P", [(1, 1, 256, 1), (1, 2, 512, 2), (2, 1, 768, 3),
                                     (1, 2, 1024, 8)])
def test_bf16_backward(O, d, B, H, N, P):
    q, k, v = (rnd((B, H, N, d), 20 + N + d + s, torch.bfloat16) for s in range(3))
    full_check(O, q, k, v, P, torch.bfloat16)


def test_bf16_backward_workload2(O):
    w = synth.WORKLOADS[2]
    q, k, v = synth.make_inputs(w, DEV)
    full_check(O, q, k, v, w.P, torch.bfloat16)


def test_bf16_backward_workload4_sampled(O):
    """The N = 131072, d = 128, P = 32 workload: gradients of sampled rows."""
    w = synth.WORKLOADS[4]
    q, k, v = synth.make_inputs(w, DEV)
    out, lse = ra.ra_forward(q, k, v, w.P)
    dout = rnd(q.shape, 4242, torch.bfloat16)
    dq, dk, dv = ra.ra_backward(q, k, v, out, dout, lse, w.P)
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    rows = synth.sample_rows(w, 256, seed=5).numpy()
    bits = lambda t: t.reshape(w.B * w.H, w.N, w.d).cpu().view(torch.int16).numpy().view(np.uint16)
    wq, wk, wv = O.backward_rows(bits(q), bits(k), bits(v), bits(out), bits(dout),
                                 lse.double().cpu().numpy(), rows, rows, dtype="bf16")
    idx = torch.as_tensor(rows, device=DEV)
    for name, got, want in (("dq", dq, wq), ("dk", dk, wk), ("dv", dv, wv)):
        close(got.reshape(-1, w.d).index_select(0, idx), want, torch.bfloat16, name)
    assert ra.ra_last_device_status() == 0


def test_bf16_backward_workload5_sampled(O):
    """The largest workload (N = 1048576, P = 64): gradients of sampled rows."""
    w = synth.WORKLOADS[5]
    q, k, v = synth.make_inputs(w, DEV)
    out, lse = ra.ra_forward(q, k, v, w.P)
    dout = rnd(q.shape, 4545, torch.bfloat16)
    dq, dk, dv = ra.ra_backward(q, k, v, out, dout, lse, w.P)
    torch.cuda.synchronize()
    assert ra.ra_last_device_status() == 0
    rows = synth.sample_rows(w, 64, seed=8).numpy()
    idx = torch.as_tensor(rows, device=DEV)
    got = [t.reshape(-1, w.d).index_select(0, idx) for t in (dq, dk, dv)]
    del dq, dk, dv
    bits = lambda t: t.reshape(w.B * w.H, w.N, w.d).cpu().view(torch.int16).numpy().view(np.uint16)
    wq, wk, wv = O.backward_rows(bits(q), bits(k), bits(v), bits(out), bits(dout),
                                 lse.double().cpu().numpy(), rows, rows, dtype="bf16")
    for name, g, want in zip(("dq", "dk", "dv"), got, (wq, wk, wv)):
        assert torch.isfinite(g.float()).all()
        close(g, want, torch.bfloat16, name)


LAYOUTS = ["contiguous", "zigzag", "striped"]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape,P", [((1, 2, 48, 8), 4), ((2, 1, 36, 33), 6), ((1, 1, 64, 64), 2),
                                     ((1, 1, 256, 40), 4)])
def test_f32_backward_causal(O, layout, shape, P):
    q, k, v = (rnd(shape, 40 + s, torch.float32, 1.3) for s in range(3))
    full_check(O, q, k, v, P, torch.float32, causal=layout)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,H,N,P", [(1, 2, 1024, 4), (2, 1, 512, 2), (1, 1, 1536, 3),
                                     (1, 1, 2048, 8)])
def test_bf16_backward_causal(O, layout, d, B, H, N, P):
    if layout == "zigzag" and (N // P) % 256:
        pytest.skip("zigzag on the tensor path needs c % 256 == 0")
    q, k, v = (rnd((B, H, N, d), 50 + N + d + s, torch.bfloat16) for s in range(3))
    full_check(O, q, k, v, P, torch.bfloat16, causal=layout)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_bf16_backward_causal_workload4_sampled(O, layout):
    w = synth.WORKLOADS[4]
    q, k, v = synth.make_inputs(w, DEV)
    out, lse = ra.ra_forward_causal(q, k, v, w.P, layout=layout)
    dout = rnd(q.shape, 4343, torch.bfloat16)
    dq, dk, dv = ra.ra_backward_causal(q, k, v, out, dout, lse, w.P, layout=layout)
    torch.cuda.synchronize()
    rows = synth.sample_rows(w, 128, seed=6).numpy()
    bits = lambda t: t.reshape(w.B * w.H, w.N, w.d).cpu().view(torch.int16).numpy().view(np.uint16)
    wq, wk, wv = O.backward_rows(bits(q), bits(k), bits(v), bits(out), bits(dout),
                                 lse.double().cpu().numpy(), rows, rows, dtype="bf16", causal=True)
    idx = torch.as_tensor(rows, device=DEV)
    for name, got, want in (("dq", dq, wq), ("dk", dk, wk), ("dv", dv, wv)):
        close(got.reshape(-1, w.d).index_select(0, idx), want, torch.bfloat16, name)
    assert ra.ra_last_device_status() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_backward_large_scores(O, d):
    """Scores of magnitude ~100: the probabilities the backward recomputes
    from lse stay finite and match."""
    shape = (1, 1, 512, d)
    q, k, v = (rnd(shape, 80 + s, torch.bfloat16, 4.0 if s < 2 else 1.0) for s in range(3))
    full_check(O, q, k, v, 2, torch.bfloat16)


@pytest.mark.parametrize("jump", [200.0, -200.0])
def test_bf16_backward_score_jump_closed_form(O, jump):
    """All queries equal and two key tiles whose scores differ by 200: every
    row's attention is uniform (p = 1/128, exact in bf16) over the dominant
    tile and zero elsewhere.  Then, with dO the upstream gradient, dV of a
    dominant key is the mean of dO over the queries, the other keys get
    dV = 0, and dQ = 0 (the dominant keys are all alike, and dS sums to zero
    over them; the bf16 path rounds each dS, and out inside D = dO.out, to
    bf16, so there dQ is zero up to tau |k| sum_k |dS| 2^-8, about six times
    what an emulation of that rounding gives).  dK of a dominant key is tau q sum_q dS, with
    dS = p (dO.v_k - dO.out).  Checked against those forms and against the
    oracle."""
    B, H, N, d, P = 1, 1, 256, 64, 1
    q = torch.zeros(B, H, N, d)
    q[..., 0] = 8.0
    k = torch.zeros(B, H, N, d)
    k[..., 128:, 0] = jump
    g = torch.Generator().manual_seed(62)
    v = torch.randn(B, H, N, d, generator=g)
    dout = torch.randn(B, H, N, d, generator=g)
    q, k, v, dout = (x.to(DEV, torch.bfloat16) for x in (q, k, v, dout))
    out, lse = ra.ra_forward(q, k, v, P)
    dq, dk, dv = ra.ra_backward(q, k, v, out, dout, lse, P)
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    dom = slice(128, 256) if jump > 0 else slice(0, 128)
    other = slice(0, 128) if jump > 0 else slice(128, 256)
    G = dout[0, 0].double().cpu().numpy()
    V = v[0, 0].double().cpu().numpy()
    p = 1.0 / 128
    o = V[dom].mean(0)
    want_dv = np.zeros((N, d))
    want_dv[dom] = G.sum(0) * p
    ds = p * (G @ V[dom].T - (G @ o)[:, None])  # [queries, dominant keys]
    want_dk = np.zeros((N, d))
    want_dk[dom] = (1 / np.sqrt(d)) * ds.sum(0)[:, None] * q[0, 0, 0].double().cpu().numpy()
    check_close(dv[0, 0], want_dv, torch.bfloat16, "dV closed form", 2e-2)
    check_close(dk[0, 0], want_dk, torch.bfloat16, "dK closed form", 2e-2)
    kmax = abs(jump) if jump > 0 else 0.0  # |k| of the dominant keys
    bound_q = (1 / np.sqrt(d)) * kmax * np.abs(ds).sum(1) * 2.0 ** -8 + 1e-6
    assert (dq[0, 0].double().abs().max(1).values.cpu().numpy() <= bound_q).all()
    assert dv[0, 0, other].abs().max().item() == 0.0 and dk[0, 0, other].abs().max().item() == 0.0
    full_check_grads = O.backward(*[to_oracle(x)[0] for x in (q, k, v)],
                                  out.double().reshape(1, N, d).cpu().numpy(),
                                  dout.double().reshape(1, N, d).cpu().numpy(),
                                  lse.double().reshape(1, N).cpu().numpy(), P, dtype="bf16")
    for name, got, want in zip(("dk", "dv"), (dk, dv), full_check_grads[1:]):
        close(got, want, torch.bfloat16, f"{name} vs oracle")
    assert ra.ra_last_device_status() == 0
