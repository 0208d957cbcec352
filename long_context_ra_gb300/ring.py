"""Ring Attention over several devices: one rank per GPU, each holding one
block of the sequence.

The pages' ring ("Ring Attention: the math", sections "Sharding the
sequence" and "The ring schedule: passing K/V around"): with P ranks, rank i
keeps its query block Q_i for the whole computation and at step t = 0 .. P-1
folds the K/V block j = (i - t) mod P into its running state (m, l, o).  The
block it holds is sent to rank i + 1 and the next one received from rank
i - 1 while the fold runs: the send/recv is launched before the fold and
waited on after it (section "Accumulation math, step by step"; "Ring
Attention" (bembew.net), section "Performance Optimization: Overlapping
Communication and Computation").  After the last step out = o / l.

On GPUs the exchange is torch.distributed point-to-point (NCCL) into a
second, local receive buffer, so the fold kernel only ever reads this
device's memory; the fold, the causal diagonal block and the final
normalisation are the library's kernels (ra_fold, ra_forward_partial_causal,
ra_merge).  The orchestration itself is device-agnostic: `ops` supplies the
three operations, so the same loop runs on CPU ranks (gloo) with other
operations in tests.

Causal attention (section "Causal masking, load balance, and other
wrinkles") is supported for the contiguous split: a block j < i is folded
whole, block j > i is skipped (every key is later than every query of the
rank), and the rank's own block is folded under the causal mask.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Any, Callable

import torch
import torch.distributed as dist


@dataclass
class RingOps:
    """The three operations the ring needs.

    new_state(rows, d, like)            an empty state (m = -inf, l = 0, o = 0)
    fold(state, q, k, v, batch)         fold a visiting block: q [batch, rq, d],
                                        k, v [batch, kv, d]
    diagonal(q, k, v)                   the causal state of the rank's own block
                                        (q, k, v [B, H, c, d]), rows as fold's
    finish(states, dtype) -> out, lse   merge the states and normalise
    """

    new_state: Callable[[int, int, torch.Tensor], Any]
    fold: Callable[[Any, torch.Tensor, torch.Tensor, torch.Tensor, int], None]
    diagonal: Callable[[torch.Tensor, torch.Tensor, torch.Tensor], Any]
    finish: Callable[[list, torch.dtype], tuple]


def library_ops(stream=None) -> RingOps:
    """The CUDA library's kernels, on `stream` (None: the current stream)."""
    from . import new_state, ra_fold, ra_forward_partial_causal, ra_merge, ra_state_init

    def _new(rows, d, like):
        return ra_state_init(new_state(rows, d, like.device), stream=stream)

    def _fold(state, q, k, v, batch):
        ra_fold(state, q, k, v, batch=batch, stream=stream)

    def _diag(q, k, v):
        return ra_forward_partial_causal(q, k, v, 1, 1, layout="contiguous", stream=stream)[0]

    def _finish(states, dtype):
        return ra_merge(states, out_dtype=dtype, stream=stream)

    return RingOps(_new, _fold, _diag, _finish)


def ring_neighbours(rank: int, world: int) -> tuple[int, int]:
    """(send_to, recv_from) of `rank` in the ring: blocks move to rank + 1."""
    return (rank + 1) % world, (rank - 1) % world


def ring_block(rank: int, step: int, world: int) -> int:
    """The K/V block rank `rank` holds at step `step`: (rank - step) mod P."""
    return (rank - step) % world


def ring_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, group=None,
                 ops: RingOps | None = None, causal: bool = False):
    """Attention of this rank's query block over the whole sequence.

    q, k, v: this rank's block [B, H, c, d] (block i = the rank's index in
    `group`; the sequence is the blocks in rank order).  Returns out
    [B, H, c, d] (q's dtype) and lse [B, H, c] (fp32) of this block.
    Every rank must call it with blocks of the same shape."""
    if ops is None:
        ops = library_ops()
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    B, H, c, d = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v blocks must share one shape")
    bh = B * H
    send_to, recv_from = ring_neighbours(rank, world)
    if group is not None:
        send_to = dist.get_global_rank(group, send_to)
        recv_from = dist.get_global_rank(group, recv_from)

    qf = q.reshape(bh, c, d).contiguous()
    # The caller's k, v are only read: blocks arrive in two receive buffers
    # used in turn.  The one received into at step t was sent and folded at
    # step t - 1 (on GPUs the library waits for that fold before the copy).
    cur = [k.reshape(bh, c, d).contiguous(), v.reshape(bh, c, d).contiguous()]
    recv = [[torch.empty_like(cur[0]), torch.empty_like(cur[1])] for _ in range(min(world - 1, 2))]
    state = ops.new_state(bh * c, d, q)
    states = [state]
    for t in range(world):
        j = ring_block(rank, t, world)
        reqs = []
        nxt = recv[t % 2] if t + 1 < world else None
        if t + 1 < world:
            # launched before the fold, waited on after it
            p2p = [dist.P2POp(dist.isend, cur[0], send_to, group),
                   dist.P2POp(dist.isend, cur[1], send_to, group),
                   dist.P2POp(dist.irecv, nxt[0], recv_from, group),
                   dist.P2POp(dist.irecv, nxt[1], recv_from, group)]
            reqs = dist.batch_isend_irecv(p2p)
        if not causal or j < rank:
            ops.fold(state, qf, cur[0], cur[1], bh)
        elif j == rank:
            states.append(ops.diagonal(q, k, v))
        # causal and j > rank: every key of block j is after every query here
        for r in reqs:
            r.wait()
        cur = nxt
    out, lse = ops.finish(states, q.dtype)
    return out.reshape(B, H, c, d), lse.reshape(B, H, c)
