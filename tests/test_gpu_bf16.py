"""Tensor-core (tcgen05) bf16 path against the fp64 oracle, through the C ABI.

Sizes are small enough for the oracle to check every row, yet span several
128-row query tiles, several 128-key tiles per block, a query block with an
odd number of tiles (a CTA with a single tile), P = 1 (plain attention) and
c = 128 (one tile per block)."""
import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch

import long_context_ra_gb300 as ra
from gpu_util import (TOL_LSE, TOL_OUT, assert_finite, check_close, check_forward,
                      check_out_lse, check_same, max_err, oracle_ring)
from oracle import ra_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = Path(__file__).resolve().parent / "golden"


@pytest.fixture(scope="module")
def O():
    return ra_oracle.get()


def rnd(shape, seed, scale=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(shape, device=DEV, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,H,N,P", [(1, 1, 256, 1), (1, 2, 512, 2), (2, 3, 768, 2),
                                     (1, 2, 1024, 8), (1, 1, 1536, 4)])
def test_forward_small(O, B, H, N, P, d):
    shape = (B, H, N, d)
    q, k, v = rnd(shape, 1 + N + d), rnd(shape, 2 + N + d), rnd(shape, 3 + N + d)
    out, lse = ra.ra_forward(q, k, v, P=P)
    torch.cuda.synchronize()
    assert_finite(out, lse)
    check_forward(O, q, k, v, P, out, lse)
    assert ra.ra_last_device_status() == 0


def test_growing_and_shrinking_max(O):
    """Key blocks with offsets that make the running max rise at every step for
    some query blocks and fall for others: the reference-max update and the O
    rescale in TMEM both fire."""
    B, H, N, d, P = 1, 2, 1024, 128, 8
    c = N // P
    q = rnd((B, H, N, d), 11).float()
    k = rnd((B, H, N, d), 12).float()
    v = rnd((B, H, N, d), 13)
    u = q.mean(dim=2, keepdim=True)
    u = u / u.norm(dim=-1, keepdim=True)
    for j in range(P):
        k[:, :, j * c:(j + 1) * c] += (6.0 * j - 20.0) * u
    q = (q * 3).to(torch.bfloat16)
    k = k.to(torch.bfloat16)
    out, lse = ra.ra_forward(q, k, v, P=P)
    check_forward(O, q, k, v, P, out, lse)


@pytest.mark.parametrize("d", [64, 128])
def test_max_rises_in_the_second_half_of_tiles(O, d):
    """Keys 64-127 of every 128-key tile lifted along the mean query, more
    for every later tile: in the forward's fast path the first half of each
    tile passes its check and goes to the tensor cores, and the second half
    then moves the reference max, so O and l are rescaled after that first
    half's product (and the second half redone).  Also the causal kernel."""
    B, H, N, P = 1, 2, 1024, 4
    q = rnd((B, H, N, d), 71).float()
    k = rnd((B, H, N, d), 72).float()
    v = rnd((B, H, N, d), 73)
    u = q.mean(dim=2, keepdim=True)
    u = u / u.norm(dim=-1, keepdim=True)
    for j in range(N // 128):
        k[:, :, j * 128 + 64:(j + 1) * 128] += (3.0 * j) * u
    q = (q * 3).to(torch.bfloat16)
    k = k.to(torch.bfloat16)
    out, lse = ra.ra_forward(q, k, v, P=P)
    check_forward(O, q, k, v, P, out, lse)
    out, lse = ra.ra_forward_causal(q, k, v, P, layout="contiguous")
    check_forward(O, q, k, v, P, out, lse, causal=True, layout="contiguous")
    assert ra.ra_last_device_status() == 0


def test_large_scores(O):
    """Scores of magnitude ~100: no overflow in exp or in l."""
    B, H, N, d, P = 1, 1, 512, 64, 2
    q, k, v = rnd((B, H, N, d), 21, 4.0), rnd((B, H, N, d), 22, 4.0), rnd((B, H, N, d), 23)
    out, lse = ra.ra_forward(q, k, v, P=P)
    assert_finite(out, lse)
    check_forward(O, q, k, v, P, out, lse)


@pytest.mark.parametrize("jump", [200.0, -200.0])
def test_score_jump_beyond_the_exponent_range(O, jump):
    """A later key tile whose scores differ from the first tile's by 200
    (about 289 in log2 units): far outside the range of a float exponent.
    Rising, the exponentials against the old reference overflow (the
    kernel must redo the tile with the new max); falling, they underflow to
    nothing.  out is the mean of V over the dominant tile."""
    B, H, N, d, P = 1, 1, 256, 64, 1
    q = torch.zeros(B, H, N, d)
    q[..., 0] = 8.0
    k = torch.zeros(B, H, N, d)
    k[..., 128:, 0] = jump  # tau q.k = 8 * jump / 8 on the second tile
    g = torch.Generator().manual_seed(61)
    v = torch.randn(B, H, N, d, generator=g)
    q, k, v = (x.to(DEV, torch.bfloat16) for x in (q, k, v))
    out, lse = ra.ra_forward(q, k, v, P=P)
    assert_finite(out, lse)
    check_forward(O, q, k, v, P, out, lse)
    dom = slice(128, 256) if jump > 0 else slice(0, 128)
    want = v[0, 0, dom].float().mean(0)
    assert (out[0, 0].float() - want).abs().max().item() <= 2e-2
    assert (lse[0, 0] - (max(jump, 0.0) + math.log(128))).abs().max().item() <= 1e-3


def test_deterministic():
    shape = (1, 2, 512, 128)
    q, k, v = rnd(shape, 31), rnd(shape, 32), rnd(shape, 33)
    a, la = ra.ra_forward(q, k, v, P=2)
    b, lb = ra.ra_forward(q, k, v, P=2)
    assert torch.equal(a, b) and torch.equal(la, lb)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_partial_merge(O, G):
    B, H, N, d, P = 1, 2, 1024, 128, 4
    q, k, v = rnd((B, H, N, d), 41), rnd((B, H, N, d), 42), rnd((B, H, N, d), 43)
    parts = ra.ra_forward_partial(q, k, v, P=P, G=G)
    out, lse = ra.ra_merge(parts, out_dtype=torch.bfloat16)
    check_forward(O, q, k, v, P, out.reshape(B, H, N, d), lse.reshape(B, H, N))
    # the partial states against the oracle's segment states
    seg = P // G
    for gi in range(G):
        _, _, m, l, o = oracle_ring(O, q, k, v, P, t0=gi * seg, t1=(gi + 1) * seg, state=True)
        assert max_err(parts[gi].m, m) <= 1e-4
        norm = parts[gi].o / parts[gi].l[:, None]
        check_close(norm, o / l[:, None], torch.bfloat16, f"partial {gi} o/l",
                    TOL_OUT[torch.bfloat16])
        # l relative to the true max: sum of p <= number of keys, >= 1
        lg = parts[gi].l.double().cpu().numpy()
        assert np.max(np.abs(lg / l - 1)) <= 2e-2


def test_fold_chain_in_ring_order(O):
    B, H, N, d, P = 1, 2, 768, 64, 3
    c = N // P
    q, k, v = rnd((B, H, N, d), 51, 1.5), rnd((B, H, N, d), 52, 1.5), rnd((B, H, N, d), 53)
    out_f, lse_f = ra.ra_forward(q, k, v, P=P)
    order = O.ring_order(P)
    for i in range(P):
        st = ra.ra_state_init(ra.new_state(B * H * c, d))
        qi = q[:, :, i * c:(i + 1) * c].reshape(B * H, c, d).contiguous()
        for t in range(P):
            j = int(order[i, t])
            kj = k[:, :, j * c:(j + 1) * c].reshape(B * H, c, d).contiguous()
            vj = v[:, :, j * c:(j + 1) * c].reshape(B * H, c, d).contiguous()
            ra.ra_fold(st, qi, kj, vj, batch=B * H)
        out, lse = ra.ra_merge([st], out_dtype=torch.bfloat16)
        want_out, want_lse = oracle_ring(
            O, q, k, v, P, rows=[b * N + i * c + r for b in range(B * H) for r in range(c)])
        check_out_lse(out, lse, want_out, want_lse, torch.bfloat16, "fold chain")
        # and against the fused forward of the same rows
        f = out_f[:, :, i * c:(i + 1) * c].reshape(-1, d)
        check_same(out, f, torch.bfloat16, "fold chain vs forward", TOL_OUT[torch.bfloat16])


def test_worked_example_embedded(O):
    """The worked example of 'Ring Attention: the math', embedded in d = 64.

    q = e1, k_j = 8 s_j e1 so that tau q.k_j = s_j exactly (tau = 1/8), v_j =
    v_j e1.  Each block is padded to 128 keys with scores of -100 (their
    weight e^-103 vanishes in fp32) and the query tile to 128 rows."""
    g = json.loads((GOLDEN / "worked_example.json").read_text())
    d = 64
    st = ra.ra_state_init(ra.new_state(128, d))
    q = torch.zeros(1, 128, d)
    q[0, :, 0] = 1.0
    q = q.to(DEV, torch.bfloat16)
    for name, step in (("A", "step_A"), ("B", "step_B")):
        blk = g["blocks"][name]
        kb = torch.zeros(1, 128, d)
        vb = torch.zeros(1, 128, d)
        kb[0, :, 0] = -100.0 * 8
        kb[0, :2, 0] = torch.tensor(blk["s"]) * 8
        vb[0, :2, 0] = torch.tensor(blk["v"])
        ra.ra_fold(st, q, kb.to(DEV, torch.bfloat16), vb.to(DEV, torch.bfloat16))
        pr = g["printed"][step]
        assert abs(st.m[0].item() - pr["m"]) <= 1e-5
        assert abs(st.l[0].item() - pr["l"]) <= g["printed_tolerance"]
        assert abs(st.o[0, 0].item() - pr["o"]) <= TOL_OUT[torch.bfloat16]
    out, lse = ra.ra_merge([st], out_dtype=torch.float32)
    assert abs(out[0, 0].item() - g["printed"]["out"]) <= TOL_OUT[torch.bfloat16]
    e1, e3 = math.exp(-1), math.exp(-3)
    lB = e1 * (1 + e1) + 1 + e3
    assert abs(lse[0].item() - (3 + math.log(lB))) <= 1e-3
    assert torch.all(out[:, 1:] == 0)


def test_misaligned_pointer_rejected():
    x = torch.zeros(1 * 1 * 256 * 64 + 8, device=DEV, dtype=torch.bfloat16)
    q = x[4:4 + 256 * 64].view(1, 1, 256, 64)  # 8-byte offset
    with pytest.raises(ra.RaError) as e:
        ra.ra_forward(q, q, q, P=1)
    assert e.value.code == 3


def test_state_checkpoint_and_resume(O):
    """The (m, l, o) state is the whole of a half-done ring: fold the first
    half of every query block's ring, copy the state to the host, restore it
    into fresh device buffers, fold the rest, and the result equals the
    one-call forward (and the oracle)."""
    B, H, N, d, P = 1, 2, 1024, 128, 4
    c = N // P
    q, k, v = rnd((B, H, N, d), 61), rnd((B, H, N, d), 62), rnd((B, H, N, d), 63)
    out_f, lse_f = ra.ra_forward(q, k, v, P=P)
    order = O.ring_order(P)
    blk = lambda t, j: t[:, :, j * c:(j + 1) * c].reshape(B * H, c, d).contiguous()
    outs, lses = [], []
    for i in range(P):
        st = ra.ra_state_init(ra.new_state(B * H * c, d))
        for t in range(P // 2):
            ra.ra_fold(st, blk(q, i), blk(k, int(order[i, t])), blk(v, int(order[i, t])),
                       batch=B * H)
        saved = [x.cpu() for x in (st.m, st.l, st.o)]  # the checkpoint
        del st
        st = ra.RaState(*(x.to(DEV) for x in saved))   # resumed elsewhere
        for t in range(P // 2, P):
            ra.ra_fold(st, blk(q, i), blk(k, int(order[i, t])), blk(v, int(order[i, t])),
                       batch=B * H)
        o, l = ra.ra_merge([st], out_dtype=torch.bfloat16)
        outs.append(o.reshape(B * H, c, d))
        lses.append(l.reshape(B * H, c))
    out = torch.cat(outs, dim=1).reshape(B, H, N, d)
    lse = torch.cat(lses, dim=1).reshape(B, H, N)
    check_forward(O, q, k, v, P, out, lse)
    check_same(out, out_f, torch.bfloat16, "resumed vs one call", TOL_OUT[torch.bfloat16])


def test_streams_and_concurrent_calls():
    """Calls are asynchronous on the caller's stream and share no state:
    the same call on a side stream gives the same bits, and two calls
    running at once on two streams each give their own result."""
    shape = (1, 4, 2048, 128)
    q, k, v = rnd(shape, 71), rnd(shape, 72), rnd(shape, 73)
    q2, k2, v2 = rnd(shape, 74), rnd(shape, 75), rnd(shape, 76)
    ref1 = ra.ra_forward(q, k, v, P=4)
    ref2 = ra.ra_forward(q2, k2, v2, P=4)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        got1 = ra.ra_forward(q, k, v, P=4)
    with torch.cuda.stream(s2):
        got2 = ra.ra_forward(q2, k2, v2, P=4)
    s1.synchronize()
    s2.synchronize()
    for got, ref in ((got1, ref1), (got2, ref2)):
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    assert ra.ra_last_device_status() == 0
