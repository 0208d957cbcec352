"""The multi-device ring backward (ring.ring_backward) on CPU ranks over
gloo.  The K/V blocks move to the next rank with their dK, dV accumulators
("Ring attention, explained", step 6); each rank adds the gradients of its
queries against the block it holds.  The per-block gradient here is the
plain formula in fp64 numpy (on GPUs it is the library's kernel), so the
test checks the orchestration: each block meets every query block once,
its accumulators come home complete, the causal variant skips and masks
the right blocks (contiguous and zigzag splits), and dq, dk, dv equal the
oracle's ring backward over the whole sequence."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

B, H, C, D = 1, 2, 16, 8


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _numpy_ops(calls):
    from long_context_ra_gb300.ring import RingBackwardOps

    tau = 1.0 / np.sqrt(D)

    def rowterms(out, dout, lse):
        return (out.numpy() * dout.numpy()).sum(-1)  # D per row

    def block(q, k, v, dout, lse, rt, dq, dk, dv, causal):
        calls.append((k.clone(), causal))
        qn, kn, vn, gn = (x.numpy() for x in (q, k, v, dout))
        s = np.einsum("bqe,bke->bqk", qn, kn) * tau
        if causal:
            n = qn.shape[1]
            s = np.where(np.tril(np.ones((n, n), bool)), s, -np.inf)
        p = np.exp(s - lse.numpy()[:, :, None])
        dp = np.einsum("bqe,bke->bqk", gn, vn)
        ds = p * (dp - rt[:, :, None])
        dq += torch.from_numpy(tau * np.einsum("bqk,bke->bqe", ds, kn))
        dk += torch.from_numpy(tau * np.einsum("bqk,bqe->bke", ds, qn))
        dv += torch.from_numpy(np.einsum("bqk,bqe->bke", p, gn))

    def finish(acc, dtype):
        return acc.to(dtype)

    return RingBackwardOps(rowterms, block, finish)


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    from long_context_ra_gb300.ring import ring_backward
    from oracle import ra_oracle

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        O = ra_oracle.Oracle(threads=1)
        g = torch.Generator().manual_seed(91 + world)
        N = world * C
        q, k, v, dout = (torch.randn(B, H, N, D, generator=g, dtype=torch.float64)
                         for _ in range(4))
        bh = B * H
        arr = lambda t: t.reshape(bh, N, D).numpy()
        blk = lambda t: t[:, :, rank * C:(rank + 1) * C].contiguous()
        res = {}
        for causal in (False, True):
            out, lse = O.dense(arr(q), arr(k), arr(v), causal=causal)
            out = torch.from_numpy(out).reshape(B, H, N, D)
            lse = torch.from_numpy(lse).reshape(B, H, N)
            calls = []
            dq, dk, dv = ring_backward(blk(q), blk(k), blk(v), blk(out), blk(dout),
                                       lse[:, :, rank * C:(rank + 1) * C].contiguous(),
                                       ops=_numpy_ops(calls), causal=causal)
            wq, wk, wv = O.backward(arr(q), arr(k), arr(v), out.reshape(bh, N, D).numpy(),
                                    arr(dout), lse.reshape(bh, N).numpy(), world, causal=causal)
            sl = slice(rank * C, (rank + 1) * C)
            errs = [float(np.abs(got.reshape(bh, C, D).numpy() - want[:, sl]).max())
                    for got, want in ((dq, wq), (dk, wk), (dv, wv))]
            seen = [next(j for j in range(world)
                         if torch.equal(kk.reshape(B, H, C, D), k[:, :, j * C:(j + 1) * C]))
                    for kk, _ in calls]
            res[causal] = (errs, seen, [c for _, c in calls])
        # zigzag: rank i holds chunks i and 2P-1-i of 2P chunks of C/2 tokens
        h = C // 2
        pos = list(range(rank * h, rank * h + h)) + \
            list(range((2 * world - 1 - rank) * h, (2 * world - 1 - rank) * h + h))
        out, lse = O.dense(arr(q), arr(k), arr(v), causal=True)
        out = torch.from_numpy(out).reshape(B, H, N, D)
        lse = torch.from_numpy(lse).reshape(B, H, N)
        zz = lambda t: t[:, :, pos].contiguous()
        calls = []
        dq, dk, dv = ring_backward(zz(q), zz(k), zz(v), zz(out), zz(dout), zz(lse),
                                   ops=_numpy_ops(calls), causal=True, layout="zigzag")
        wq, wk, wv = O.backward(arr(q), arr(k), arr(v), out.reshape(bh, N, D).numpy(),
                                arr(dout), lse.reshape(bh, N).numpy(), world, causal=True)
        res["zigzag"] = [float(np.abs(got.reshape(bh, C, D).numpy() - want[:, pos]).max())
                         for got, want in ((dq, wq), (dk, wk), (dv, wv))]
        results[rank] = res
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ring_backward_over_gloo_equals_the_oracle(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world,
                           join=True, start_method="spawn")
        results = dict(results)
    assert sorted(results) == list(range(world))
    for rank, res in results.items():
        zz = res.pop("zigzag")
        assert max(zz) <= 1e-12, (rank, "zigzag", zz)
        for causal, (errs, seen, masked) in res.items():
            assert max(errs) <= 1e-12, (rank, causal, errs)
            want = [(rank - t) % world for t in range(world)]
            if causal:
                want = [j for j in want if j <= rank]
            assert seen == want, (rank, causal, seen, want)
            assert masked == [causal and j == rank for j in want], (rank, causal, masked)
