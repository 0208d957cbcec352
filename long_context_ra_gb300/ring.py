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
ra_merge; the backward's ra_backward_rowterms and ra_backward_block).  The
orchestration itself is device-agnostic: `ops` supplies the arithmetic, so
the same loops run on CPU ranks (gloo) with other operations in tests.

Causal attention (section "Causal masking, load balance, and other
wrinkles"; "Ring attention, explained", section "The causal-mask catch"):
- contiguous split: a block j < i is folded whole, block j > i is skipped
  (every key is later than every query of the rank), and the rank's own
  block is folded under the causal mask.  Rank P - 1 does P times the work
  of rank 0.
- zigzag split: the sequence is cut into 2P chunks and rank i holds chunks
  i and 2P-1-i (its block lists chunk i, then chunk 2P-1-i).  Against block
  j < i both of its chunks see chunk j whole and chunk 2P-1-j not at all;
  against j > i only its chunk 2P-1-i sees anything, and it sees the whole
  block.  Every rank then does the same work at every step.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Any, Callable

import torch
import torch.distributed as dist


@dataclass
class RingOps:
    """The operations the forward ring needs.

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


def _exchange(cur, nxt, send_to, recv_from, group):
    """Post the send of the held block and the receive of the next one."""
    p2p = [dist.P2POp(dist.isend, cur[0], send_to, group),
           dist.P2POp(dist.isend, cur[1], send_to, group),
           dist.P2POp(dist.irecv, nxt[0], recv_from, group),
           dist.P2POp(dist.irecv, nxt[1], recv_from, group)]
    return dist.batch_isend_irecv(p2p)


def _neighbours(group):
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    send_to, recv_from = ring_neighbours(rank, world)
    if group is not None:
        send_to = dist.get_global_rank(group, send_to)
        recv_from = dist.get_global_rank(group, recv_from)
    return world, rank, send_to, recv_from


def ring_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, group=None,
                 ops: RingOps | None = None, causal: bool = False,
                 layout: str = "contiguous"):
    """Attention of this rank's query block over the whole sequence.

    q, k, v: this rank's block [B, H, c, d] (block i = the rank's index in
    `group`).  layout "contiguous": the sequence is the blocks in rank
    order; "zigzag" (causal only): the block holds chunks i and 2P-1-i of
    2P chunks of c/2 tokens, in that order.  Returns out [B, H, c, d] (q's
    dtype) and lse [B, H, c] (fp32) of this block, rows in the block's
    order.  Every rank must call it with blocks of the same shape."""
    if ops is None:
        ops = library_ops()
    if layout not in ("contiguous", "zigzag"):
        raise ValueError(f"unknown layout {layout!r}")
    if layout == "zigzag":
        if not causal:
            raise ValueError("the zigzag split only matters under the causal mask")
        return _ring_forward_zigzag(q, k, v, group, ops)
    world, rank, send_to, recv_from = _neighbours(group)
    B, H, c, d = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v blocks must share one shape")
    bh = B * H

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
            reqs = _exchange(cur, nxt, send_to, recv_from, group)  # before the fold
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


def _ring_forward_zigzag(q, k, v, group, ops: RingOps):
    """The causal ring over the zigzag split (see the module docstring).

    The block's two chunks keep separate states (rows of chunk i, "lo", and
    of chunk 2P-1-i, "hi"), and blocks travel as [2 chunks, B*H, c/2, d] so
    that either chunk is a contiguous operand of the fold."""
    world, rank, send_to, recv_from = _neighbours(group)
    B, H, c, d = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v blocks must share one shape")
    if c % 2:
        raise ValueError("the zigzag split needs an even block length")
    bh, h = B * H, c // 2
    halves = lambda t: t.reshape(bh, 2, h, d).transpose(0, 1).contiguous()  # [2, bh, h, d]
    qh = halves(q)
    cur = [halves(k), halves(v)]
    recv = [[torch.empty_like(cur[0]), torch.empty_like(cur[1])] for _ in range(min(world - 1, 2))]
    st = [ops.new_state(bh * h, d, q), ops.new_state(bh * h, d, q)]  # lo, hi
    extra = [[], []]
    as4 = lambda t: t.reshape(1, bh, h, d)
    for t in range(world):
        j = ring_block(rank, t, world)
        nxt = recv[t % 2] if t + 1 < world else None
        reqs = _exchange(cur, nxt, send_to, recv_from, group) if t + 1 < world else []
        kc, vc = cur
        if j == rank:
            # own block: each chunk against itself under the mask (local
            # order is position order), and chunk 2P-1-i sees chunk i whole
            extra[0].append(ops.diagonal(as4(qh[0]), as4(kc[0]), as4(vc[0])))
            extra[1].append(ops.diagonal(as4(qh[1]), as4(kc[1]), as4(vc[1])))
            ops.fold(st[1], qh[1], kc[0], vc[0], bh)
        elif j < rank:
            # chunk j precedes both query chunks; chunk 2P-1-j follows both
            ops.fold(st[0], qh[0], kc[0], vc[0], bh)
            ops.fold(st[1], qh[1], kc[0], vc[0], bh)
        else:
            # only chunk 2P-1-i sees block j, and all of it
            ops.fold(st[1], qh[1], kc[0], vc[0], bh)
            ops.fold(st[1], qh[1], kc[1], vc[1], bh)
        for r in reqs:
            r.wait()
        cur = nxt
    outs, lses = [], []
    for x in range(2):
        o, l = ops.finish([st[x]] + extra[x], q.dtype)
        outs.append(o.reshape(bh, h, d))
        lses.append(l.reshape(bh, h))
    out = torch.stack(outs, dim=1).reshape(B, H, c, d)
    lse = torch.stack(lses, dim=1).reshape(B, H, c)
    return out, lse


@dataclass
class RingBackwardOps:
    """The operations of the ring backward.

    rowterms(out, dout, lse) -> rt          per-query terms of a block
                                            (out, dout [bh, c, d], lse [bh, c])
    block(q, k, v, dout, lse, rt, dq, dk, dv, causal)
                                            add one visiting block's gradients
                                            into the fp32 accumulators
    finish(acc, dtype) -> tensor            an accumulator in the output dtype
    """

    rowterms: Callable[[torch.Tensor, torch.Tensor, torch.Tensor], Any]
    block: Callable[..., None]
    finish: Callable[[torch.Tensor, torch.dtype], torch.Tensor]


def library_backward_ops(stream=None) -> RingBackwardOps:
    """The CUDA library's kernels (ra_backward_rowterms, ra_backward_block)."""
    from . import ra_backward_block, ra_backward_rowterms

    def _rowterms(out, dout, lse):
        return ra_backward_rowterms(out, dout, lse, stream=stream)

    def _block(q, k, v, dout, lse, rt, dq, dk, dv, causal):
        ra_backward_block(q, k, v, dout, lse, rt, dq, dk, dv, causal=causal, stream=stream)

    def _finish(acc, dtype):
        return acc.to(dtype)

    return RingBackwardOps(_rowterms, _block, _finish)


def ring_backward(q, k, v, out, dout, lse, group=None, ops: RingBackwardOps | None = None,
                  causal: bool = False, layout: str = "contiguous"):
    """Gradients (dq, dk, dv) of this rank's block for L = sum(dout * out),
    on the same ring as ring_forward (contiguous split): at step t the rank
    meets block (i - t) mod P, adds dQ of its own queries into its
    accumulator and the visiting block's dK, dV into the accumulators that
    travel with that block ("Ring attention, explained", step 6).  The K/V
    of the next block are received while the current one is processed; its
    accumulators follow once the rank's contribution is in.  After P steps
    every block is back on its rank with complete dK, dV.

    q, k, v, out, dout: this rank's block [B, H, c, d]; lse [B, H, c] (from
    ring_forward with the same causal and layout).  layout "zigzag" (causal
    only): the block holds chunks i and 2P-1-i, as in ring_forward.
    Returns dq, dk, dv [B, H, c, d] in q's dtype."""
    if ops is None:
        ops = library_backward_ops()
    if layout not in ("contiguous", "zigzag"):
        raise ValueError(f"unknown layout {layout!r}")
    if layout == "zigzag":
        if not causal:
            raise ValueError("the zigzag split only matters under the causal mask")
        return _ring_backward_zigzag(q, k, v, out, dout, lse, group, ops)
    world, rank, send_to, recv_from = _neighbours(group)
    B, H, c, d = q.shape
    for t in (k, v, out, dout):
        if t.shape != q.shape:
            raise ValueError("q, k, v, out, dout blocks must share one shape")
    bh = B * H
    q3, dout3 = q.reshape(bh, c, d).contiguous(), dout.reshape(bh, c, d).contiguous()
    lse2 = lse.reshape(bh, c).contiguous()
    rt = ops.rowterms(out.reshape(bh, c, d).contiguous(), dout3, lse2)
    # fp32 accumulators (fp64 when the blocks are fp64, as on CPU ranks)
    f32 = dict(dtype=torch.float64 if q.dtype == torch.float64 else torch.float32,
               device=q.device)
    dq = torch.zeros(bh, c, d, **f32)
    kv = [k.reshape(bh, c, d).contiguous(), v.reshape(bh, c, d).contiguous()]
    kv_recv = [[torch.empty_like(kv[0]), torch.empty_like(kv[1])]
               for _ in range(min(world - 1, 2))]
    acc = [torch.zeros(bh, c, d, **f32), torch.zeros(bh, c, d, **f32)]  # dK, dV of the held block
    acc_recv = [[torch.empty_like(acc[0]), torch.empty_like(acc[1])] for _ in range(2)]
    for t in range(world):
        j = ring_block(rank, t, world)
        kv_next = kv_recv[t % 2] if t + 1 < world else None
        reqs = _exchange(kv, kv_next, send_to, recv_from, group) if t + 1 < world else []
        if not causal or j < rank:
            ops.block(q3, kv[0], kv[1], dout3, lse2, rt, dq, acc[0], acc[1], False)
        elif j == rank:
            ops.block(q3, kv[0], kv[1], dout3, lse2, rt, dq, acc[0], acc[1], True)
        # causal and j > rank: no query here sees block j; it passes through
        if world > 1:
            # the block's accumulators follow it to the next rank (after the
            # contribution above); after P hops they are home
            acc_next = acc_recv[t % 2]
            reqs += _exchange(acc, acc_next, send_to, recv_from, group)
        for r in reqs:
            r.wait()
        if world > 1:
            acc = acc_next
        kv = kv_next
    shape = (B, H, c, d)
    return (ops.finish(dq, q.dtype).reshape(shape), ops.finish(acc[0], q.dtype).reshape(shape),
            ops.finish(acc[1], q.dtype).reshape(shape))


def _ring_backward_zigzag(q, k, v, out, dout, lse, group, ops: RingBackwardOps):
    """The causal ring backward over the zigzag split: the pieces of
    _ring_forward_zigzag, each a block step on chunks of c/2 rows, with dQ
    accumulated per query chunk and dK, dV per chunk of the visiting block
    (the two chunks travel together, [2, B*H, c/2, d])."""
    world, rank, send_to, recv_from = _neighbours(group)
    B, H, c, d = q.shape
    for t in (k, v, out, dout):
        if t.shape != q.shape:
            raise ValueError("q, k, v, out, dout blocks must share one shape")
    if c % 2:
        raise ValueError("the zigzag split needs an even block length")
    bh, h = B * H, c // 2
    halves = lambda t: t.reshape(bh, 2, h, -1).transpose(0, 1).contiguous()  # [2, bh, h, .]
    qh, gh = halves(q), halves(dout)
    lh = halves(lse.reshape(bh, c, 1)).reshape(2, bh, h)
    oh = halves(out)
    rt = [ops.rowterms(oh[x], gh[x], lh[x]) for x in range(2)]
    f32 = dict(dtype=torch.float64 if q.dtype == torch.float64 else torch.float32,
               device=q.device)
    dq = torch.zeros(2, bh, h, d, **f32)
    kv = [halves(k), halves(v)]
    kv_recv = [[torch.empty_like(kv[0]), torch.empty_like(kv[1])]
               for _ in range(min(world - 1, 2))]
    acc = [torch.zeros(2, bh, h, d, **f32), torch.zeros(2, bh, h, d, **f32)]  # dK, dV
    acc_recv = [[torch.empty_like(acc[0]), torch.empty_like(acc[1])] for _ in range(2)]

    def step(x, y, causal):
        # query chunk x of this rank against chunk y of the held block
        ops.block(qh[x], kv[0][y], kv[1][y], gh[x], lh[x], rt[x], dq[x], acc[0][y], acc[1][y],
                  causal)

    for t in range(world):
        j = ring_block(rank, t, world)
        kv_next = kv_recv[t % 2] if t + 1 < world else None
        reqs = _exchange(kv, kv_next, send_to, recv_from, group) if t + 1 < world else []
        if j == rank:
            step(0, 0, True)
            step(1, 0, False)
            step(1, 1, True)
        elif j < rank:
            step(0, 0, False)
            step(1, 0, False)
        else:
            step(1, 0, False)
            step(1, 1, False)
        if world > 1:
            acc_next = acc_recv[t % 2]
            reqs += _exchange(acc, acc_next, send_to, recv_from, group)
        for r in reqs:
            r.wait()
        if world > 1:
            acc = acc_next
        kv = kv_next
    whole = lambda a: ops.finish(a, q.dtype).transpose(0, 1).reshape(B, H, c, d)
    return whole(dq), whole(acc[0]), whole(acc[1])
