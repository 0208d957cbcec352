"""The multi-device ring (long_context_ra_gb300.ring) on CPU ranks over gloo.

Each rank holds one block of a seeded sequence; the K/V blocks travel around
the ring by point-to-point send/recv while each rank folds the block it
holds.  The folds here are the fp64 oracle's (the ring's operations are
pluggable; on GPUs they are the library's kernels), so the test checks the
orchestration: every rank visits the blocks (i - t) mod P in order, each
exactly once, the exchange hands each block on intact, the causal variant
skips and masks the right blocks (contiguous and zigzag splits; under
zigzag every rank folds the same number of keys), and the merged result
equals dense attention over the whole sequence ("Ring Attention: the math", sections "The
ring schedule: passing K/V around" and "A worked numeric example")."""
import os
import socket
import types

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

B, H, C, D = 1, 2, 24, 8  # per-rank block: [B, H, C, D]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_ops(O, visits):
    from long_context_ra_gb300.ring import RingOps

    def new_state(rows, d, like):
        return types.SimpleNamespace(m=np.full(rows, -np.inf), l=np.zeros(rows),
                                     o=np.zeros((rows, d)))

    def fold(st, q, k, v, batch):
        visits.append(k.clone())
        st.m, st.l, st.o = O.fold(st.m, st.l, st.o, q.numpy(), k.numpy(), v.numpy(),
                                  dtype="f64", batch=batch)

    def diagonal(q, k, v):
        visits.append("diagonal")
        bh, c, d = q.shape[0] * q.shape[1], q.shape[2], q.shape[3]
        _, _, m, l, o = O.ring(q.reshape(bh, c, d).numpy(), k.reshape(bh, c, d).numpy(),
                               v.reshape(bh, c, d).numpy(), 1, dtype="f64", causal=True,
                               state=True)
        return types.SimpleNamespace(m=m, l=l, o=o)

    def finish(states, dtype):
        out, lse = O.merge(np.stack([s.m for s in states]), np.stack([s.l for s in states]),
                           np.stack([s.o for s in states]))
        return torch.from_numpy(out), torch.from_numpy(lse)

    return RingOps(new_state, fold, diagonal, finish)


def _sequence(world):
    g = torch.Generator().manual_seed(77 + world)
    shape = (B, H, world * C, D)
    return [torch.randn(shape, generator=g, dtype=torch.float64) * 1.2 for _ in range(3)]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    from long_context_ra_gb300.ring import ring_block, ring_forward
    from oracle import ra_oracle

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        O = ra_oracle.Oracle(threads=1)
        q, k, v = _sequence(world)
        blk = lambda t, j: t[:, :, j * C:(j + 1) * C].contiguous()
        qi, ki, vi = blk(q, rank), blk(k, rank), blk(v, rank)
        res = {}
        for causal in (False, True):
            visits = []
            out, lse = ring_forward(qi, ki, vi, ops=_oracle_ops(O, visits), causal=causal)
            # which block each fold saw, identified by its keys
            order = []
            for x in visits:
                if isinstance(x, str):
                    order.append(rank)
                    continue
                kx = x.reshape(B, H, C, D)
                order.append(next(j for j in range(world) if torch.equal(kx, blk(k, j))))
            want = [ring_block(rank, t, world) for t in range(world)]
            if causal:
                want = [j for j in want if j <= rank]
            bh = B * H
            rows = [s * world * C + rank * C + r for s in range(bh) for r in range(C)]
            w_out, w_lse = O.dense(q.reshape(bh, world * C, D).numpy(),
                                   k.reshape(bh, world * C, D).numpy(),
                                   v.reshape(bh, world * C, D).numpy(), dtype="f64",
                                   rows=np.array(rows), causal=causal)
            res[causal] = (order, want,
                           float(np.abs(out.reshape(-1, D).numpy() - w_out).max()),
                           float(np.abs(lse.reshape(-1).numpy() - w_lse).max()))
        # zigzag: rank i holds chunks i and 2P-1-i of 2P chunks of C/2 tokens
        h = C // 2
        pos = list(range(rank * h, rank * h + h)) + \
            list(range((2 * world - 1 - rank) * h, (2 * world - 1 - rank) * h + h))
        zz = lambda t: t[:, :, pos].contiguous()
        visits = []
        out, lse = ring_forward(zz(q), zz(k), zz(v), ops=_oracle_ops(O, visits), causal=True,
                                layout="zigzag")
        bh = B * H
        rows = [s * world * C + p for s in range(bh) for p in pos]
        w_out, w_lse = O.dense(q.reshape(bh, world * C, D).numpy(),
                               k.reshape(bh, world * C, D).numpy(),
                               v.reshape(bh, world * C, D).numpy(), dtype="f64",
                               rows=np.array(rows), causal=True)
        # every rank folds the same number of key rows (the point of zigzag)
        folded = sum(x.shape[1] for x in visits if not isinstance(x, str))
        res["zigzag"] = (float(np.abs(out.reshape(-1, D).numpy() - w_out).max()),
                         float(np.abs(lse.reshape(-1).numpy() - w_lse).max()), folded)
        # the caller's blocks are only read (blocks arrive in separate buffers)
        res["inputs_intact"] = bool(torch.equal(ki, blk(k, rank)) and torch.equal(vi, blk(v, rank)))
        results[rank] = res
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ring_over_gloo_equals_dense(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world,
                           join=True, start_method="spawn")
        results = dict(results)
    assert sorted(results) == list(range(world))
    folded = set()
    for rank, res in results.items():
        assert res.pop("inputs_intact"), rank
        e_out, e_lse, n = res.pop("zigzag")
        assert e_out <= 1e-12 and e_lse <= 1e-12, (rank, "zigzag", e_out, e_lse)
        folded.add(n)
        for causal, (order, want, e_out, e_lse) in res.items():
            assert order == want, (rank, causal, order, want)
            assert e_out <= 1e-12 and e_lse <= 1e-12, (rank, causal, e_out, e_lse)
    assert len(folded) == 1, folded  # the same unmasked folds on every rank


def test_ring_schedule_matches_the_pages_table():
    """(i - t) mod P, own block first, against the P = 4 golden table."""
    import json
    from pathlib import Path

    from long_context_ra_gb300.ring import ring_block, ring_neighbours

    g = json.loads((Path(__file__).parent / "golden" / "ring_schedule_p4.json").read_text())
    table = g["held"]
    for i in range(4):
        assert [ring_block(i, t, 4) for t in range(4)] == list(table[i])
    assert ring_neighbours(0, 4) == (1, 3) and ring_neighbours(3, 4) == (0, 2)
