"""fp32 (FFMA) path against the fp64 oracle, through the C ABI."""
import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch

import long_context_ra_gb300 as ra
from gpu_util import TOL_OUT, check_close, check_forward, check_same, max_err, oracle_ring
from long_context_ra_gb300 import synth
from oracle import ra_oracle

pytestmark = pytest.mark.gpu
GOLDEN = Path(__file__).resolve().parent / "golden"
DEV = "cuda"


@pytest.fixture(scope="module")
def O():
    return ra_oracle.get()


def worked_tensors():
    """The worked example of 'Ring Attention: the math' as [1, 1, 4, 1] tensors.

    d = 1 so tau = 1 and the page's scores s are the keys; every query row is
    q = [1], row 0 being the page's query (it sees block A, then B)."""
    g = json.loads((GOLDEN / "worked_example.json").read_text())
    s = g["blocks"]["A"]["s"] + g["blocks"]["B"]["s"]
    v = g["blocks"]["A"]["v"] + g["blocks"]["B"]["v"]
    q = torch.ones(1, 1, 4, 1, device=DEV)
    k = torch.tensor(s, device=DEV).reshape(1, 1, 4, 1)
    vv = torch.tensor(v, device=DEV).reshape(1, 1, 4, 1)
    return g, q, k, vv


def test_worked_example_forward(O):
    g, q, k, v = worked_tensors()
    out, lse = ra.ra_forward(q, k, v, P=2)
    torch.cuda.synchronize()
    assert abs(out[0, 0, 0, 0].item() - g["printed"]["out"]) <= g["printed_tolerance"]
    check_forward(O, q, k, v, 2, out, lse)


def test_worked_example_fold_steps():
    g, q, k, v = worked_tensors()
    tol = TOL_OUT[torch.float32]
    st = ra.ra_state_init(ra.new_state(1, 1))
    e1, e3 = math.exp(-1), math.exp(-3)
    ra.ra_fold(st, q[0, 0, :1].reshape(1, 1, 1), k[0, 0, 0:2].reshape(1, 2, 1),
               v[0, 0, 0:2].reshape(1, 2, 1))
    m, l, o = st.m.item(), st.l.item(), st.o.item()
    assert abs(m - 2.0) <= tol and abs(l - (1 + e1)) <= tol and abs(o - (e1 + 2)) <= tol
    ra.ra_fold(st, q[0, 0, :1].reshape(1, 1, 1), k[0, 0, 2:4].reshape(1, 2, 1),
               v[0, 0, 2:4].reshape(1, 2, 1))
    lB = e1 * (1 + e1) + 1 + e3
    oB = e1 * (e1 + 2) + 3 + 4 * e3
    assert abs(st.m.item() - 3.0) <= tol
    assert abs(st.l.item() - lB) <= tol and abs(st.o.item() - oB) <= tol
    out, lse = ra.ra_merge([st], out_dtype=torch.float32)
    assert abs(out.item() - g["printed"]["out"]) <= g["printed_tolerance"]
    assert abs(out.item() - oB / lB) <= tol
    assert abs(lse.item() - (3 + math.log(lB))) <= tol
    assert ra.ra_last_device_status() == 0


def test_workload1_full(O):
    w = synth.WORKLOADS[1]
    q, k, v = synth.make_inputs(w, DEV)
    out, lse = ra.ra_forward(q, k, v, P=w.P)
    eo, el = check_forward(O, q, k, v, w.P, out, lse)
    assert el <= 1e-5


@pytest.mark.parametrize("shape,P", [((2, 3, 40, 5), 4), ((1, 2, 97, 33), 1), ((1, 1, 64, 256), 8),
                                     ((1, 1, 7, 1), 7), ((3, 1, 36, 100), 6),
                                     ((1, 16, 300, 33), 3), ((1, 12, 600, 128), 5)])
def test_ragged_shapes(O, shape, P):
    g = torch.Generator(device=DEV).manual_seed(sum(shape) * 31 + P)
    q, k, v = (torch.randn(shape, device=DEV, generator=g) * 1.5 for _ in range(3))
    out, lse = ra.ra_forward(q, k, v, P=P)
    check_forward(O, q, k, v, P, out, lse)


# Shapes for the tiled fp32 kernel: ragged query tiles and K/V tiles, d in
# every width class, tiles of 64 and of 128 rows, split over clusters of 2
# and 4 CTAs or not (the last three: grids that fill the SMs with 128-row
# tiles at d = 128, 200 and 48).
TILED = [((2, 4, 1000, 100), 4), ((1, 8, 512, 256), 2), ((1, 16, 600, 33), 3),
         ((2, 8, 256, 64), 1), ((1, 12, 1024, 128), 4), ((1, 20, 1024, 128), 1),
         ((1, 40, 512, 200), 1), ((1, 16, 2048, 48), 1)]


@pytest.mark.parametrize("shape,P", TILED)
def test_tiled_shapes(O, shape, P):
    g = torch.Generator(device=DEV).manual_seed(sum(shape) * 17 + P)
    q, k, v = (torch.randn(shape, device=DEV, generator=g) * 1.5 for _ in range(3))
    out, lse = ra.ra_forward(q, k, v, P=P)
    check_forward(O, q, k, v, P, out, lse)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_tiled_causal(O, layout):
    B, H, N, d, P = 1, 8, 1024, 72, 4
    g = torch.Generator(device=DEV).manual_seed(71)
    q, k, v = (torch.randn(B, H, N, d, device=DEV, generator=g) * 1.5 for _ in range(3))
    out, lse = ra.ra_forward_causal(q, k, v, P, layout=layout)
    check_forward(O, q, k, v, P, out, lse, causal=True, layout=layout)


# Small grids run on the row kernel, whose rows are each split over up to 8
# warps (the row's chunks of 32 keys dealt round robin, the warps' states
# merged at the end).  These cases split 4 ways: the mask's early stop and
# the fold mode's incoming state under the split.
@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_small_grid_causal(O, layout):
    B, H, N, d, P = 1, 2, 256, 40, 4
    g = torch.Generator(device=DEV).manual_seed(73)
    q, k, v = (torch.randn(B, H, N, d, device=DEV, generator=g) * 1.5 for _ in range(3))
    out, lse = ra.ra_forward_causal(q, k, v, P, layout=layout)
    check_forward(O, q, k, v, P, out, lse, causal=True, layout=layout)


def test_small_grid_fold_chain(O):
    """ra_fold of 2 x 200 rows against 200-key blocks (seven chunks a row)
    in ring order, against the forward of the same tensors (the tiled
    kernel) and the oracle."""
    B, H, N, d, P = 1, 2, 800, 24, 4
    c = N // P
    g = torch.Generator(device=DEV).manual_seed(74)
    q, k, v = (torch.randn(B, H, N, d, device=DEV, generator=g) * 2 for _ in range(3))
    out_f, lse_f = ra.ra_forward(q, k, v, P=P)
    check_forward(O, q, k, v, P, out_f, lse_f)
    order = O.ring_order(P)
    for i in (0, 3):
        st = ra.ra_state_init(ra.new_state(B * H * c, d))
        qi = q[:, :, i * c:(i + 1) * c].reshape(B * H, c, d).contiguous()
        for t in range(P):
            j = int(order[i, t])
            ra.ra_fold(st, qi, k[:, :, j * c:(j + 1) * c].reshape(B * H, c, d).contiguous(),
                       v[:, :, j * c:(j + 1) * c].reshape(B * H, c, d).contiguous(), batch=B * H)
        out, lse = ra.ra_merge([st], out_dtype=torch.float32)
        check_same(out, out_f[:, :, i * c:(i + 1) * c].reshape(-1, d), torch.float32,
                   "split-row fold chain vs forward", 1e-5)
        check_same(lse, lse_f[:, :, i * c:(i + 1) * c].reshape(-1), torch.float32,
                   "split-row fold chain lse vs forward", 1e-5, relative=False)


def test_tiled_partials_and_fold_chain(O):
    """Partial states (G = 3) and a chain of ra_fold calls through the tiled
    kernel (ra_fold of 8 x 256 rows), against the oracle's segment states
    and the forward."""
    B, H, N, d, P = 1, 8, 1536, 40, 6
    c = N // P
    g = torch.Generator(device=DEV).manual_seed(72)
    q, k, v = (torch.randn(B, H, N, d, device=DEV, generator=g) for _ in range(3))
    out_f, lse_f = ra.ra_forward(q, k, v, P=P)
    check_forward(O, q, k, v, P, out_f, lse_f)
    parts = ra.ra_forward_partial(q, k, v, P=P, G=3)
    for gi in range(3):
        _, _, m, l, o = oracle_ring(O, q, k, v, P, t0=2 * gi, t1=2 * gi + 2, state=True)
        assert max_err(parts[gi].m, m) <= 1e-5
        assert np.max(np.abs(parts[gi].l.double().cpu().numpy() / l - 1)) <= 1e-5
        check_close(parts[gi].o / parts[gi].l[:, None], o / l[:, None], torch.float32,
                    f"tiled partial {gi} o/l", 1e-5)
    order = O.ring_order(P)
    i = 2
    st = ra.ra_state_init(ra.new_state(B * H * c, d))
    qi = q[:, :, i * c:(i + 1) * c].reshape(B * H, c, d).contiguous()
    for t in range(P):
        j = int(order[i, t])
        ra.ra_fold(st, qi, k[:, :, j * c:(j + 1) * c].reshape(B * H, c, d).contiguous(),
                   v[:, :, j * c:(j + 1) * c].reshape(B * H, c, d).contiguous(), batch=B * H)
    out, lse = ra.ra_merge([st], out_dtype=torch.float32)
    check_same(out, out_f[:, :, i * c:(i + 1) * c].reshape(-1, d), torch.float32,
               "tiled fold chain vs forward", 1e-5)


def test_tiled_cluster_split_partials(O):
    """A grid too small for the SMs: each 64-row query tile's walk is split
    over a cluster of CTAs whose states merge in distributed shared memory.
    Partial states (G = 2) of such a grid against the oracle's segment
    states, and their merge against the forward."""
    B, H, N, d, P = 1, 2, 2048, 64, 4
    g = torch.Generator(device=DEV).manual_seed(75)
    q, k, v = (torch.randn(B, H, N, d, device=DEV, generator=g) for _ in range(3))
    out_f, lse_f = ra.ra_forward(q, k, v, P=P)
    check_forward(O, q, k, v, P, out_f, lse_f)
    parts = ra.ra_forward_partial(q, k, v, P=P, G=2)
    for gi in range(2):
        _, _, m, l, o = oracle_ring(O, q, k, v, P, t0=2 * gi, t1=2 * gi + 2, state=True)
        assert max_err(parts[gi].m, m) <= 1e-5
        assert np.max(np.abs(parts[gi].l.double().cpu().numpy() / l - 1)) <= 1e-5
        check_close(parts[gi].o / parts[gi].l[:, None], o / l[:, None], torch.float32,
                    f"cluster-split partial {gi} o/l", 1e-5)
    out, lse = ra.ra_merge(parts, out_dtype=torch.float32)
    check_same(out, out_f.reshape(-1, d), torch.float32, "cluster-split merge vs forward", 1e-5)


def test_partial_and_merge_equal_forward(O):
    B, H, N, d, P = 1, 2, 96, 48, 6
    g = torch.Generator(device=DEV).manual_seed(5)
    q, k, v = (torch.randn(B, H, N, d, device=DEV, generator=g) for _ in range(3))
    out_f, lse_f = ra.ra_forward(q, k, v, P=P)
    for G in (1, 2, 3, 6):
        parts = ra.ra_forward_partial(q, k, v, P=P, G=G)
        out, lse = ra.ra_merge(parts, out_dtype=torch.float32)
        check_same(out, out_f.reshape(-1, d), torch.float32, f"G={G} merge vs forward out", 1e-5)
        check_same(lse, lse_f.reshape(-1), torch.float32, f"G={G} merge vs forward lse", 1e-5,
                   relative=False)
    # the partials themselves against the oracle's segment states
    parts = ra.ra_forward_partial(q, k, v, P=P, G=3)
    for gi in range(3):
        _, _, m, l, o = oracle_ring(O, q, k, v, P, t0=2 * gi, t1=2 * gi + 2, state=True)
        assert max_err(parts[gi].m, m) <= 1e-5
        rel_l = parts[gi].l.double().cpu().numpy() / l
        assert np.max(np.abs(rel_l - 1)) <= 1e-5
        norm = parts[gi].o / parts[gi].l[:, None]
        check_close(norm, o / l[:, None], torch.float32, f"partial {gi} o/l", 1e-5)


def test_fold_chain_in_ring_order_equals_forward(O):
    B, H, N, d, P = 1, 2, 60, 16, 3
    c = N // P
    g = torch.Generator(device=DEV).manual_seed(6)
    q, k, v = (torch.randn(B, H, N, d, device=DEV, generator=g) * 2 for _ in range(3))
    out_f, lse_f = ra.ra_forward(q, k, v, P=P)
    order = O.ring_order(P)
    for i in range(P):
        st = ra.ra_state_init(ra.new_state(B * H * c, d))
        qi = q[:, :, i * c:(i + 1) * c].reshape(B * H, c, d).contiguous()
        for t in range(P):
            j = int(order[i, t])
            kj = k[:, :, j * c:(j + 1) * c].reshape(B * H, c, d).contiguous()
            vj = v[:, :, j * c:(j + 1) * c].reshape(B * H, c, d).contiguous()
            ra.ra_fold(st, qi, kj, vj, batch=B * H)
        out, lse = ra.ra_merge([st], out_dtype=torch.float32)
        want = out_f[:, :, i * c:(i + 1) * c].reshape(-1, d)
        check_same(out, want, torch.float32, "fold chain vs forward", 1e-5)
        assert max_err(lse, lse_f[:, :, i * c:(i + 1) * c].reshape(-1).cpu().double().numpy()) <= 1e-5


def test_merge_empty_partials():
    rows, d = 5, 8
    a = ra.ra_state_init(ra.new_state(rows, d))
    b = ra.ra_state_init(ra.new_state(rows, d))
    out, lse = ra.ra_merge([a, b], out_dtype=torch.float32)
    assert (out == 0).all() and torch.isneginf(lse).all()


def test_empty_and_errors():
    z = torch.empty(0, 1, 4, 8, device=DEV)
    out, lse = ra.ra_forward(z, z, z, P=2)  # nothing to do
    assert out.numel() == 0
    q = torch.randn(1, 1, 6, 8, device=DEV)
    with pytest.raises(ra.RaError) as e:
        ra.ra_forward(q, q, q, P=4)
    assert e.value.code == 2
