"""The multi-device ring's GPU operations (ring.library_ops: ra_state_init,
ra_fold, ra_forward_partial_causal, ra_merge) through ring_forward, on a
one-rank group: the only configuration one GPU allows (ranks on the same
GPU cannot exchange through NCCL).  The exchange itself is covered by the
gloo tests on CPU ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist

from gpu_util import check_forward
from long_context_ra_gb300.ring import ring_forward

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def O():
    from oracle import ra_oracle
    return ra_oracle.get()


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


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_one_rank_ring_on_the_gpu(O, group, causal, d):
    g = torch.Generator(device=DEV).manual_seed(50 + d)
    q, k, v = (torch.randn(1, 2, 1024, d, device=DEV, generator=g).to(torch.bfloat16)
               for _ in range(3))
    out, lse = ring_forward(q, k, v, causal=causal)
    torch.cuda.synchronize()
    check_forward(O, q, k, v, 1, out, lse, causal=causal)


def test_one_rank_zigzag_ring_on_the_gpu(O, group):
    """With one rank the zigzag block is chunks 0 and 1, the whole sequence
    in order: the result is causal attention over it."""
    g = torch.Generator(device=DEV).manual_seed(77)
    q, k, v = (torch.randn(1, 2, 1024, 128, device=DEV, generator=g).to(torch.bfloat16)
               for _ in range(3))
    out, lse = ring_forward(q, k, v, causal=True, layout="zigzag")
    torch.cuda.synchronize()
    check_forward(O, q, k, v, 1, out, lse, causal=True)
