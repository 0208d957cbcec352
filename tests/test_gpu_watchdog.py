"""Failure detection on the GPU without a fault: every wait of the
tensor-core kernels is bounded, and a wait that runs out makes the kernel
record RA_ERR_TIMEOUT, let what it has in flight finish, free its tensor
memory and return, leaving the context usable.

The test makes such a wait run out on purpose through the library's test
aid: with ra_watchdog_config(wait_cycles, stall_cta) one CTA of the next
fold launches loads no input, so the barriers its MMA and softmax warps wait
on are never signalled.  Nothing faults, traps or hangs: the waits give up
after `wait_cycles` SM cycles."""
import time

import numpy as np
import pytest
import torch

import long_context_ra_gb300 as ra
from gpu_util import check_close, check_forward, oracle_ring
from long_context_ra_gb300 import _native

pytestmark = pytest.mark.gpu
DEV = "cuda"
SHORT = 1 << 20  # SM cycles: about half a millisecond


@pytest.fixture(scope="module")
def O():
    from oracle import ra_oracle
    return ra_oracle.get()


@pytest.fixture(autouse=True)
def restore_watchdog():
    ra.ra_last_device_status()  # start from a clear status word
    yield
    ra.ra_watchdog_config(0, -1)


def rnd(shape, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(shape, device=DEV, generator=g).to(torch.bfloat16)


def test_short_limit_alone_raises_nothing(O):
    """A short limit is long enough for every wait of a healthy launch."""
    B, H, N, d, P = 1, 2, 2048, 128, 4
    q, k, v = (rnd((B, H, N, d), 700 + s) for s in range(3))
    ra.ra_watchdog_config(SHORT, -1)
    out, lse = ra.ra_forward(q, k, v, P)
    assert ra.ra_last_device_status() == _native.RA_OK
    check_forward(O, q, k, v, P, out, lse)


@pytest.mark.parametrize("d", [64, 128])
def test_stalled_cta_times_out_and_the_context_recovers(O, d):
    # 2 heads x 4 query blocks of 256 rows = 8 CTAs of one 128-row tile pair;
    # CTA 3 is (head 0, query block 3): rows 768 .. 1023 of head 0
    B, H, N, P = 1, 2, 1024, 4
    q, k, v = (rnd((B, H, N, d), 710 + d + s) for s in range(3))
    out = torch.full((B, H, N, d), float("nan"), device=DEV, dtype=torch.bfloat16)
    lse = torch.full((B, H, N), float("nan"), device=DEV)
    ra.ra_watchdog_config(SHORT, 3)
    t0 = time.perf_counter()
    ra.ra_forward(q, k, v, P, out=out, lse=lse)
    status = ra.ra_last_device_status()
    elapsed = time.perf_counter() - t0
    ra.ra_watchdog_config(0, -1)
    assert status == _native.RA_ERR_TIMEOUT
    assert ra.ra_last_device_status() == _native.RA_OK  # read and cleared
    assert elapsed < 5.0
    # the stalled CTA wrote nothing; every other CTA finished its rows
    assert torch.isnan(out[0, 0, 768:].float()).all() and torch.isnan(lse[0, 0, 768:]).all()
    rows = [r for r in range(B * H * N) if not 768 <= r < 1024]
    want_out, want_lse = oracle_ring(O, q, k, v, P, rows=rows)
    idx = torch.tensor(rows, device=DEV)
    check_close(out.reshape(-1, d).index_select(0, idx), want_out, torch.bfloat16,
                "rows of the other CTAs", 2e-2)
    check_close(lse.reshape(-1).index_select(0, idx), want_lse, torch.bfloat16,
                "lse of the other CTAs", 1e-3, relative=False)
    # the context is intact: the same call with the default settings is right
    out2, lse2 = ra.ra_forward(q, k, v, P)
    assert ra.ra_last_device_status() == _native.RA_OK
    check_forward(O, q, k, v, P, out2, lse2)


def test_stalled_fold_call_times_out(O):
    """ra_fold (state in, state out) with its only CTA stalled: timeout
    reported, then the same fold from a fresh state is right."""
    rq, kv, d = 128, 256, 128
    q, kb, vb = rnd((1, rq, d), 720), rnd((1, kv, d), 721), rnd((1, kv, d), 722)
    st = ra.ra_state_init(ra.new_state(rq, d))
    ra.ra_watchdog_config(SHORT, 0)
    ra.ra_fold(st, q, kb, vb)
    assert ra.ra_last_device_status() == _native.RA_ERR_TIMEOUT
    ra.ra_watchdog_config(0, -1)
    st = ra.ra_state_init(ra.new_state(rq, d))
    ra.ra_fold(st, q, kb, vb)
    torch.cuda.synchronize()
    assert ra.ra_last_device_status() == _native.RA_OK
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    m0 = np.full(rq, -np.inf)
    l0 = np.zeros(rq)
    o0 = np.zeros((rq, d))
    m, l, o = O.fold(m0, l0, o0, bits(q), bits(kb), bits(vb), dtype="bf16")
    assert np.max(np.abs(st.m.double().cpu().numpy() - m)) <= 1e-4
    check_close(st.o / st.l[:, None], o / l[:, None], torch.bfloat16, "fold after timeout",
                2e-2)


def _backward_want(O, q, k, v, out, dout, lse, P):
    from gpu_util import to_oracle
    B, H, N, d = q.shape
    qa, tag = to_oracle(q)
    ka, _ = to_oracle(k)
    va, _ = to_oracle(v)
    oa = out.double().reshape(B * H, N, d).cpu().numpy()
    ga = dout.double().reshape(B * H, N, d).cpu().numpy()
    la = lse.double().reshape(B * H, N).cpu().numpy()
    return O.backward(qa, ka, va, oa, ga, la, P, dtype=tag)


def test_short_limit_alone_raises_nothing_in_the_backward(O):
    B, H, N, d, P = 1, 2, 1024, 128, 4
    q, k, v, dout = (rnd((B, H, N, d), 730 + s) for s in range(4))
    out, lse = ra.ra_forward(q, k, v, P)
    ra.ra_watchdog_config(SHORT, -1)
    grads = ra.ra_backward(q, k, v, out, dout, lse, P)
    assert ra.ra_last_device_status() == _native.RA_OK
    for name, got, want in zip(("dq", "dk", "dv"), grads,
                               _backward_want(O, q, k, v, out, dout, lse, P)):
        check_close(got.reshape(-1, d), want.reshape(-1, d), torch.bfloat16,
                    f"backward {name} under a short limit", 2e-2)


def test_stalled_backward_cta_times_out_and_the_context_recovers(O):
    """CTA 3 of the dK/dV kernel and of the dQ kernel loads nothing.  With
    2 heads, P = 4 and c = 256 both kernels have 16 CTAs of one 128-row tile;
    CTA 3 is head 0, block 1, tile 1 (rows 384 .. 511 of head 0) in both, so
    every other row of dq, dk and dv is still right."""
    B, H, N, d, P = 1, 2, 1024, 128, 4
    q, k, v, dout = (rnd((B, H, N, d), 740 + s) for s in range(4))
    out, lse = ra.ra_forward(q, k, v, P)
    assert ra.ra_last_device_status() == _native.RA_OK
    ra.ra_watchdog_config(SHORT, 3)
    t0 = time.perf_counter()
    grads = ra.ra_backward(q, k, v, out, dout, lse, P)
    status = ra.ra_last_device_status()
    elapsed = time.perf_counter() - t0
    ra.ra_watchdog_config(0, -1)
    assert status == _native.RA_ERR_TIMEOUT
    assert ra.ra_last_device_status() == _native.RA_OK
    assert elapsed < 5.0
    want = _backward_want(O, q, k, v, out, dout, lse, P)
    rows = [r for r in range(B * H * N) if not 384 <= r < 512]
    idx = torch.tensor(rows, device=DEV)
    for name, got, w in zip(("dq", "dk", "dv"), grads, want):
        check_close(got.reshape(-1, d).index_select(0, idx), w.reshape(-1, d)[rows],
                    torch.bfloat16, f"backward {name}, rows of the other CTAs", 2e-2)
    # the context is intact: the same call with the default settings is right
    grads = ra.ra_backward(q, k, v, out, dout, lse, P)
    assert ra.ra_last_device_status() == _native.RA_OK
    for name, got, w in zip(("dq", "dk", "dv"), grads, want):
        check_close(got.reshape(-1, d), w.reshape(-1, d), torch.bfloat16,
                    f"backward {name} after a timeout", 2e-2)
