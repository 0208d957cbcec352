"""One step of the ring backward across devices (ra_backward_rowterms,
ra_backward_block) through the C ABI.  The ring of P devices is played out
on one GPU: every query block meets the blocks (i - t) mod P, adding its dQ
into its own fp32 accumulator and the visiting block's dK, dV into that
block's accumulators; the accumulated gradients must equal the oracle's
ring backward over the whole sequence (bars of gpu_util: bf16 and fp32
paths)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import long_context_ra_gb300 as ra
from gpu_util import check_close, to_oracle
from long_context_ra_gb300.ring import ring_backward, ring_forward

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def O():
    from oracle import ra_oracle
    return ra_oracle.get()


def rnd(shape, seed, dtype):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(shape, device=DEV, generator=g).to(dtype)


def oracle_grads(O, q, k, v, out, dout, lse, P, causal):
    B, H, N, d = q.shape
    qa, tag = to_oracle(q)
    ka, _ = to_oracle(k)
    va, _ = to_oracle(v)
    oa = out.double().reshape(B * H, N, d).cpu().numpy()
    ga = dout.double().reshape(B * H, N, d).cpu().numpy()
    la = lse.double().reshape(B * H, N).cpu().numpy()
    return O.backward(qa, ka, va, oa, ga, la, P, dtype=tag, causal=causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,d,c", [(torch.bfloat16, 128, 256), (torch.bfloat16, 64, 128),
                                       (torch.float32, 40, 24)])
def test_ring_of_blocks_on_one_gpu(O, dtype, d, c, causal):
    B, H, P = 1, 2, 4
    N, bh = P * c, B * H
    q, k, v, dout = (rnd((B, H, N, d), 800 + s, dtype) for s in range(4))
    out, lse = (ra.ra_forward_causal(q, k, v, P) if causal else ra.ra_forward(q, k, v, P))
    blk = lambda t, j: t.reshape(bh, N, -1)[:, j * c:(j + 1) * c].contiguous()
    lse3 = lse.reshape(bh, N, 1)
    rts = [ra.ra_backward_rowterms(blk(out, i), blk(dout, i), blk(lse3, i).reshape(bh, c))
           for i in range(P)]
    acc = lambda: torch.zeros(bh, c, d, device=DEV)
    dq = [acc() for _ in range(P)]
    dk = [acc() for _ in range(P)]
    dv = [acc() for _ in range(P)]
    for i in range(P):
        for t in range(P):
            j = (i - t) % P
            if causal and j > i:
                continue
            ra.ra_backward_block(blk(q, i), blk(k, j), blk(v, j), blk(dout, i),
                                 blk(lse3, i).reshape(bh, c), rts[i], dq[i], dk[j], dv[j],
                                 causal=causal and j == i)
    torch.cuda.synchronize()
    assert ra.ra_last_device_status() == 0
    wq, wk, wv = oracle_grads(O, q, k, v, out, dout, lse, P, causal)
    cat = lambda xs: torch.cat(xs, dim=1)  # [bh, N, d]
    for name, got, want in (("dq", cat(dq), wq), ("dk", cat(dk), wk), ("dv", cat(dv), wv)):
        tol = 2e-2 if dtype == torch.bfloat16 else 1e-5 * max(1.0, float(np.abs(want).max()))
        check_close(got, want, dtype, f"ring of blocks {name}", tol)


@pytest.mark.parametrize("causal", [False, True])
def test_ring_of_fp32_blocks_tiled(O, causal):
    """The fp32 block steps with enough rows for the tiled kernels (64 heads
    of 128-row blocks: 128 CTAs a step), accumulating across the ring."""
    B, H, P, c, d = 1, 64, 4, 128, 72
    N, bh = P * c, B * H
    q, k, v, dout = (rnd((B, H, N, d), 840 + s, torch.float32) for s in range(4))
    out, lse = (ra.ra_forward_causal(q, k, v, P) if causal else ra.ra_forward(q, k, v, P))
    blk = lambda t, j: t.reshape(bh, N, -1)[:, j * c:(j + 1) * c].contiguous()
    lse3 = lse.reshape(bh, N, 1)
    rts = [ra.ra_backward_rowterms(blk(out, i), blk(dout, i), blk(lse3, i).reshape(bh, c))
           for i in range(P)]
    dq = [torch.zeros(bh, c, d, device=DEV) for _ in range(P)]
    dk = [torch.zeros(bh, c, d, device=DEV) for _ in range(P)]
    dv = [torch.zeros(bh, c, d, device=DEV) for _ in range(P)]
    for i in range(P):
        for t in range(P):
            j = (i - t) % P
            if causal and j > i:
                continue
            ra.ra_backward_block(blk(q, i), blk(k, j), blk(v, j), blk(dout, i),
                                 blk(lse3, i).reshape(bh, c), rts[i], dq[i], dk[j], dv[j],
                                 causal=causal and j == i)
    torch.cuda.synchronize()
    assert ra.ra_last_device_status() == 0
    wq, wk, wv = oracle_grads(O, q, k, v, out, dout, lse, P, causal)
    cat = lambda xs: torch.cat(xs, dim=1)
    for name, got, want in (("dq", cat(dq), wq), ("dk", cat(dk), wk), ("dv", cat(dv), wv)):
        check_close(got, want, torch.float32, f"tiled fp32 ring of blocks {name}",
                    1e-5 * max(1.0, float(np.abs(want).max())))


def test_block_accumulates_into_existing_values():
    """Accumulators are added to, not overwritten."""
    bh, c, d = 2, 128, 64
    q, k, v, dout = (rnd((bh, c, d), 830 + s, torch.bfloat16) for s in range(4))
    out, lse = ra.ra_forward(q.reshape(1, bh, c, d), k.reshape(1, bh, c, d),
                             v.reshape(1, bh, c, d), 1)
    rt = ra.ra_backward_rowterms(out.reshape(bh, c, d), dout, lse.reshape(bh, c))
    zeros = [torch.zeros(bh, c, d, device=DEV) for _ in range(3)]
    ones = [torch.full((bh, c, d), 1.5, device=DEV) for _ in range(3)]
    for accs in (zeros, ones):
        ra.ra_backward_block(q, k, v, dout, lse.reshape(bh, c), rt, *accs)
    torch.cuda.synchronize()
    for z, o in zip(zeros, ones):
        assert torch.equal(o - 1.5, z) or (o - 1.5 - z).abs().max().item() <= 1e-6


@pytest.fixture(scope="module")
def group():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ["MASTER_PORT"] = str(port)
    mine = not dist.is_initialized()
    if mine:
        dist.init_process_group("gloo", rank=0, world_size=1)
    yield None
    if mine:
        dist.destroy_process_group()


@pytest.mark.parametrize("causal,layout", [(False, "contiguous"), (True, "contiguous"),
                                           (True, "zigzag")])
def test_one_rank_ring_backward_on_the_gpu(O, group, causal, layout):
    B, H, N, d = 1, 2, 1024, 128
    q, k, v, dout = (rnd((B, H, N, d), 850 + s, torch.bfloat16) for s in range(4))
    out, lse = ring_forward(q, k, v, causal=causal, layout=layout)
    dq, dk, dv = ring_backward(q, k, v, out, dout, lse, causal=causal, layout=layout)
    torch.cuda.synchronize()
    wq, wk, wv = oracle_grads(O, q, k, v, out, dout, lse, 1, causal)
    for name, got, want in (("dq", dq, wq), ("dk", dk, wk), ("dv", dv, wv)):
        check_close(got.reshape(want.shape), want, torch.bfloat16, f"one-rank ring {name}", 2e-2)
