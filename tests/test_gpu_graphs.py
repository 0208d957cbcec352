"""The library's device calls inside CUDA graphs.

A step of the path (the fused forward, the causal and split forwards, the
backward, a query block's fold chain in ring order, "Ring Attention: the
math", section "The ring schedule: passing K/V around") is captured once on
static buffers and replayed with new inputs copied into them.  The calls
make no host synchronisation and no allocation of their own when given
their outputs and workspaces, so they capture as they are.  Every kernel
of the path is deterministic (no atomics, fixed reduction orders), so each
replay must equal the same calls made eagerly on the same inputs bit for
bit, and the last replay is also checked against the oracle."""
import pytest
import torch

import long_context_ra_gb300 as ra
from gpu_util import check_forward, check_same
from long_context_ra_gb300.ring import ring_block
from oracle import ra_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def O():
    return ra_oracle.get()


def rnd(shape, seed, scale=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(shape, device=DEV, generator=g) * scale).to(torch.bfloat16)


def capture(fn):
    """Warm `fn` up on a side stream, then capture it into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        res = fn()
    return g, res


def refill(tensors, seed):
    for x, t in enumerate(tensors):
        t.copy_(rnd(t.shape, seed + x))


def test_forward_backward_step_replays(O):
    """Forward then backward of one head group, captured as one graph."""
    B, H, N, d, P = 1, 2, 1024, 128, 4
    shape = (B, H, N, d)
    q, k, v, dout = (rnd(shape, 10 + x) for x in range(4))
    out = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=DEV, dtype=torch.float32)
    ws = torch.empty(2 * B * H * N, device=DEV, dtype=torch.float32)

    def step():
        ra.ra_forward(q, k, v, P, out=out, lse=lse)
        return ra.ra_backward(q, k, v, out, dout, lse, P, workspace=ws)

    g, (dq, dk, dv) = capture(step)
    for seed in (100, 200):
        refill((q, k, v, dout), seed)
        g.replay()
        e_out, e_lse = ra.ra_forward(q, k, v, P)
        e_dq, e_dk, e_dv = ra.ra_backward(q, k, v, e_out, dout, e_lse, P)
        torch.cuda.synchronize()
        assert torch.equal(out, e_out) and torch.equal(lse, e_lse)
        assert torch.equal(dq, e_dq) and torch.equal(dk, e_dk) and torch.equal(dv, e_dv)
    check_forward(O, q, k, v, P, out, lse)
    assert ra.ra_last_device_status() == 0


def test_causal_and_split_forwards_replay(O):
    B, H, N, d, P = 1, 2, 2048, 64, 4
    shape = (B, H, N, d)
    q, k, v = (rnd(shape, 30 + x) for x in range(3))
    out_c = torch.empty_like(q)
    lse_c = torch.empty(B, H, N, device=DEV, dtype=torch.float32)
    out_s = torch.empty_like(q)
    lse_s = torch.empty(B, H, N, device=DEV, dtype=torch.float32)
    G = 2
    ws = torch.empty(ra.ra_forward_split_workspace_bytes(B, H, N, d, G), device=DEV,
                     dtype=torch.uint8)

    def step():
        ra.ra_forward_causal(q, k, v, P, layout="zigzag", out=out_c, lse=lse_c)
        ra.ra_forward_split(q, k, v, P, G=G, workspace=ws, out=out_s, lse=lse_s)

    g, _ = capture(step)
    for seed in (300, 400):
        refill((q, k, v), seed)
        g.replay()
        e_out_c, e_lse_c = ra.ra_forward_causal(q, k, v, P, layout="zigzag")
        e_out_s, e_lse_s = ra.ra_forward_split(q, k, v, P, G=G)
        torch.cuda.synchronize()
        assert torch.equal(out_c, e_out_c) and torch.equal(lse_c, e_lse_c)
        assert torch.equal(out_s, e_out_s) and torch.equal(lse_s, e_lse_s)
    check_forward(O, q, k, v, P, out_s, lse_s)
    assert ra.ra_last_device_status() == 0


def test_fold_chain_replays(O):
    """Query block i's state folded over the blocks (i - t) mod P, then
    normalised: the per-step calls a multi-device ring makes, as one graph."""
    B, H, N, d, P = 1, 2, 1024, 128, 4
    c = N // P
    i = 1
    shape = (B, H, N, d)
    q, k, v = (rnd(shape, 50 + x) for x in range(3))
    st = ra.new_state(B * H * c, d)
    out = torch.empty(B * H * c, d, device=DEV, dtype=torch.bfloat16)
    lse = torch.empty(B * H * c, device=DEV, dtype=torch.float32)

    def blk(t, j):
        return t[:, :, j * c:(j + 1) * c].reshape(B * H, c, d).contiguous()

    def chain():
        ra.ra_state_init(st)
        qi = blk(q, i)
        for t in range(P):
            j = ring_block(i, t, P)
            ra.ra_fold(st, qi, blk(k, j), blk(v, j), batch=B * H)
        ra.ra_merge([st], out=out, lse=lse)

    g, _ = capture(chain)
    for seed in (500, 600):
        refill((q, k, v), seed)
        g.replay()
        e_out, e_lse = ra.ra_forward(q, k, v, P)
        torch.cuda.synchronize()
        want_out = e_out[:, :, i * c:(i + 1) * c].reshape(-1, d)
        want_lse = e_lse[:, :, i * c:(i + 1) * c].reshape(-1)
        # the fold chain and the fused forward round differently (the chain
        # keeps fp32 states between blocks): same bars as against the oracle
        check_same(out, want_out, torch.bfloat16, "graph fold chain vs forward", 2e-2)
        check_same(lse, want_lse, torch.float32, "graph fold chain lse vs forward", 1e-3,
                   relative=False)
    # the eager chain on the last inputs gives the replay's result bit for bit
    st2 = ra.new_state(B * H * c, d)
    ra.ra_state_init(st2)
    for t in range(P):
        j = ring_block(i, t, P)
        ra.ra_fold(st2, blk(q, i), blk(k, j), blk(v, j), batch=B * H)
    out2, lse2 = ra.ra_merge([st2])
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    assert ra.ra_last_device_status() == 0
