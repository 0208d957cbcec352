"""Guard regions around every output buffer, checked on the host: each
output is the interior of a larger device buffer whose head and tail hold a
known pattern; after the call the pattern must be intact (no write outside
the output) and the interior must equal an unguarded call's result (no write
missing).  Covered: the striped layout's 3-D tensor maps, the causal tile
prefixes and suffixes, the split path's partial states in caller scratch,
partial states, the merge and the backward's gradients."""
import pytest
import torch

import long_context_ra_gb300 as ra

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD_BYTES = 64 * 1024
PATTERN = 0x5A


class Guarded:
    """A tensor of `shape` and `dtype` inside a buffer with guard bytes on
    both sides (the interior stays 256-byte aligned)."""

    def __init__(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        esize = torch.empty(0, dtype=dtype).element_size()
        self.body = n * esize
        self.raw = torch.full((GUARD_BYTES * 2 + self.body,), PATTERN, device=DEV,
                              dtype=torch.uint8)
        self.t = self.raw[GUARD_BYTES:GUARD_BYTES + self.body].view(dtype).view(shape)

    def intact(self) -> bool:
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.body:]
        return bool((head == PATTERN).all() and (tail == PATTERN).all())


def rnd(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(shape, device=DEV, generator=g).to(dtype)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("d", [64, 128])
def test_causal_forward_stays_inside(layout, d):
    B, H, N, P = 2, 3, 2048, 4
    q, k, v = (rnd((B, H, N, d), 900 + s) for s in range(3))
    out = Guarded((B, H, N, d), torch.bfloat16)
    lse = Guarded((B, H, N), torch.float32)
    ra.ra_forward_causal(q, k, v, P, layout=layout, out=out.t, lse=lse.t)
    ref_out, ref_lse = ra.ra_forward_causal(q, k, v, P, layout=layout)
    torch.cuda.synchronize()
    assert out.intact() and lse.intact()
    assert torch.equal(out.t, ref_out) and torch.equal(lse.t, ref_lse)
    assert ra.ra_last_device_status() == 0


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_causal_partials_stay_inside(layout):
    B, H, N, d, P, G = 1, 2, 2048, 128, 8, 4
    q, k, v = (rnd((B, H, N, d), 910 + s) for s in range(3))
    rows = B * H * N
    guards = [(Guarded((rows,), torch.float32), Guarded((rows,), torch.float32),
               Guarded((rows, d), torch.float32)) for _ in range(G)]
    parts = [ra.RaState(m.t, l.t, o.t) for m, l, o in guards]
    ra.ra_forward_partial_causal(q, k, v, P, G=G, layout=layout, partials=parts)
    ref = ra.ra_forward_partial_causal(q, k, v, P, G=G, layout=layout)
    torch.cuda.synchronize()
    for (m, l, o), p in zip(guards, ref):
        assert m.intact() and l.intact() and o.intact()
        assert torch.equal(m.t, p.m) and torch.equal(l.t, p.l) and torch.equal(o.t, p.o)
    out = Guarded((rows, d), torch.bfloat16)
    lse = Guarded((rows,), torch.float32)
    ra.ra_merge(parts, out_dtype=torch.bfloat16, out=out.t, lse=lse.t)
    torch.cuda.synchronize()
    assert out.intact() and lse.intact()
    assert ra.ra_last_device_status() == 0


@pytest.mark.parametrize("G", [2, 3, 8])
def test_split_stays_inside_its_workspace(G):
    B, H, N, d, P = 1, 3, 2048, 64, 8
    q, k, v = (rnd((B, H, N, d), 920 + s) for s in range(3))
    ws = Guarded((ra.ra_forward_split_workspace_bytes(B, H, N, d, G),), torch.uint8)
    out = Guarded((B, H, N, d), torch.bfloat16)
    lse = Guarded((B, H, N), torch.float32)
    ra.ra_forward_split(q, k, v, P, G=G, workspace=ws.t, out=out.t, lse=lse.t)
    ref_out, ref_lse = ra.ra_forward_split(q, k, v, P, G=G)
    torch.cuda.synchronize()
    assert ws.intact() and out.intact() and lse.intact()
    assert torch.equal(out.t, ref_out) and torch.equal(lse.t, ref_lse)


@pytest.mark.parametrize("causal", [None, "striped", "zigzag"])
def test_backward_stays_inside(causal):
    B, H, N, d, P = 1, 2, 2048, 128, 4
    q, k, v = (rnd((B, H, N, d), 930 + s) for s in range(3))
    if causal is None:
        out, lse = ra.ra_forward(q, k, v, P)
    else:
        out, lse = ra.ra_forward_causal(q, k, v, P, layout=causal)
    dout = rnd((B, H, N, d), 939)
    grads = [Guarded((B, H, N, d), torch.bfloat16) for _ in range(3)]
    ws = Guarded((2 * B * H * N,), torch.float32)
    L = ra._native.lib()
    ptrs = [ra._ptr(x) for x in (q, k, v, out, dout, lse)] + [ra._ptr(g.t) for g in grads] + \
        [ra._ptr(ws.t)]
    stream = ra._stream(None)
    if causal is None:
        code = L.ra_backward(*ptrs, B, H, N, d, P, ra.RA_BF16, stream)
    else:
        code = L.ra_backward_causal(*ptrs, B, H, N, d, P, ra._native.RA_LAYOUTS[causal],
                                    ra.RA_BF16, stream)
    assert code == 0
    ref = ra.ra_backward(q, k, v, out, dout, lse, P, causal=causal)
    torch.cuda.synchronize()
    for g, r in zip(grads, ref):
        assert g.intact()
        assert torch.equal(g.t, r)
    assert ws.intact()
    assert ra.ra_last_device_status() == 0
