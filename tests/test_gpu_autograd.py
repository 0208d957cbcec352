"""The autograd Functions (long_context_ra_gb300.autograd) on the GPU: a
loss's gradients through `attention` are exactly ra_backward's for the
upstream gradient of out (bf16, plain and causal), the fp32 gradients match
the oracle's backward, and `ring_attention` on a one-rank group equals
`attention` (with one rank the ring is the whole sequence)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist

import long_context_ra_gb300 as ra
from gpu_util import check_close, check_same, to_oracle
from long_context_ra_gb300.autograd import attention, ring_attention
from oracle import ra_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def O():
    return ra_oracle.get()


def leaves(shape, seed, dtype):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return [(torch.randn(shape, device=DEV, generator=g)).to(dtype).requires_grad_()
            for _ in range(3)]


@pytest.mark.parametrize("causal", [None, "zigzag"])
def test_attention_gradients_are_the_library_backward(causal):
    shape, P = (1, 2, 1024, 128), 4
    q, k, v = leaves(shape, 31, torch.bfloat16)
    up = torch.randn(shape, device=DEV, generator=torch.Generator(device=DEV).manual_seed(32))
    out, lse = attention(q, k, v, P, causal=causal)
    assert not lse.requires_grad
    (out.float() * up).sum().backward()
    with torch.no_grad():
        if causal is None:
            e_out, e_lse = ra.ra_forward(q, k, v, P)
        else:
            e_out, e_lse = ra.ra_forward_causal(q, k, v, P, layout=causal)
        e_dq, e_dk, e_dv = ra.ra_backward(q, k, v, e_out, up.to(torch.bfloat16), e_lse, P,
                                          causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(out, e_out) and torch.equal(lse, e_lse)
    assert torch.equal(q.grad, e_dq) and torch.equal(k.grad, e_dk) and torch.equal(v.grad, e_dv)
    assert ra.ra_last_device_status() == 0


def test_attention_fp32_gradients_match_the_oracle(O):
    shape, P = (1, 2, 96, 40), 3
    q, k, v = leaves(shape, 33, torch.float32)
    up = torch.randn(shape, device=DEV, generator=torch.Generator(device=DEV).manual_seed(34))
    out, lse = attention(q, k, v, P)
    (out * up).sum().backward()
    B, H, N, d = shape
    arr = lambda t: t.detach().double().reshape(B * H, N, d).cpu().numpy()
    wq, wk, wv = O.backward(to_oracle(q.detach())[0], to_oracle(k.detach())[0],
                            to_oracle(v.detach())[0], arr(out), arr(up),
                            lse.detach().double().reshape(B * H, N).cpu().numpy(), P, dtype="f32")
    for name, got, want in (("dq", q.grad, wq), ("dk", k.grad, wk), ("dv", v.grad, wv)):
        check_close(got.reshape(-1, d), want.reshape(-1, d), torch.float32,
                    f"autograd fp32 {name}", 1e-5)


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
def test_one_rank_ring_attention_equals_attention(group, causal):
    shape = (1, 2, 1024, 128)
    q, k, v = leaves(shape, 35, torch.bfloat16)
    up = torch.randn(shape, device=DEV, generator=torch.Generator(device=DEV).manual_seed(36))
    out, _ = ring_attention(q, k, v, causal=causal)
    (out.float() * up).sum().backward()
    grads = [t.grad.clone() for t in (q, k, v)]
    for t in (q, k, v):
        t.grad = None
    out2, _ = attention(q, k, v, 1, causal="contiguous" if causal else None)
    (out2.float() * up).sum().backward()
    torch.cuda.synchronize()
    check_same(out.detach().float(), out2.detach().float(), torch.bfloat16, "one-rank ring out",
               2e-2)
    for name, a, b in zip(("dq", "dk", "dv"), grads, (q.grad, k.grad, v.grad)):
        check_same(a.float(), b.float(), torch.bfloat16, f"one-rank ring {name} vs attention",
                   2e-2 * max(1.0, b.float().abs().max().item()))
    assert ra.ra_last_device_status() == 0
