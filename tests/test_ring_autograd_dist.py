"""`ring_attention` (long_context_ra_gb300.autograd) on 2 CPU ranks over
gloo: loss.backward() through the autograd Function runs the forward ring
and then the backward ring, and the gradients each rank gets for its block
equal the oracle's backward over the whole sequence.  The per-block
arithmetic is the oracle's fold (forward) and the plain fp64 formula
(backward), as in the ring tests; on GPUs both are the library's kernels."""
import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp

B, H, C, D = 1, 2, 16, 8


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    from long_context_ra_gb300.autograd import ring_attention
    from oracle import ra_oracle
    from test_ring_backward_dist import _numpy_ops
    from test_ring_dist import _oracle_ops

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        O = ra_oracle.Oracle(threads=1)
        g = torch.Generator().manual_seed(123)
        N = world * C
        q, k, v, up = (torch.randn(B, H, N, D, generator=g, dtype=torch.float64)
                       for _ in range(4))
        blk = lambda t: t[:, :, rank * C:(rank + 1) * C].clone().requires_grad_()
        res = {}
        for causal in (False, True):
            qi, ki, vi = blk(q), blk(k), blk(v)
            out, lse = ring_attention(qi, ki, vi, causal=causal, ops=_oracle_ops(O, []),
                                      bops=_numpy_ops([]))
            (out * up[:, :, rank * C:(rank + 1) * C]).sum().backward()
            bh = B * H
            arr = lambda t: t.reshape(bh, N, D).numpy()
            w_out, w_lse = O.dense(arr(q), arr(k), arr(v), causal=causal)
            wq, wk, wv = O.backward(arr(q), arr(k), arr(v), w_out, arr(up), w_lse, world,
                                    causal=causal)
            sl = slice(rank * C, (rank + 1) * C)
            res[causal] = [float(np.abs(got.detach().reshape(bh, C, D).numpy() - want[:, sl]).max())
                           for got, want in ((out, w_out.reshape(bh, N, D)), (qi.grad, wq),
                                             (ki.grad, wk), (vi.grad, wv))]
        results[rank] = res
    finally:
        dist.destroy_process_group()


def test_ring_attention_autograd_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world,
                           join=True, start_method="spawn")
        results = dict(results)
    assert sorted(results) == list(range(world))
    for rank, res in results.items():
        for causal, errs in res.items():
            assert max(errs) <= 1e-12, (rank, causal, errs)
