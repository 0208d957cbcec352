"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each pin is a function ``pin_*(O)`` taking an ``oracle.ra_oracle.Oracle`` and
raising ``AssertionError`` on a miss.  ``test_oracle.py`` requires every pin to
pass on the real oracle; ``test_oracle_mutants.py`` requires every planted
mistake to fail at least one pin.

What pins what (pages cited by title and section):
  * the worked example printed in "Ring Attention: the math", section "A worked
    numeric example" (per-step m, alpha, p, l, o, out and the dense answer);
  * closed forms: two keys reduce to a logistic weight, identical keys give the
    mean of V and lse = tau q.k + ln N, a constant V is returned unchanged;
  * library routines: scipy's softmax/logsumexp over numpy matmul scores;
  * invariants stated on the pages: the ring equals dense attention, and the
    result does not depend on the number of blocks P, on the visiting order or
    on the fold granularity; shift invariance of the keys;
  * the ring schedule table for P = 4 (section "The ring schedule");
  * the merge of partial states ("Ring Attention", bembew.net, "Global
    Integration") against the ring over the whole sequence.
"""
from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np
from scipy.special import logsumexp, softmax

GOLDEN = Path(__file__).resolve().parent / "golden"
EXACT = 1e-12


def _worked():
    return json.loads((GOLDEN / "worked_example.json").read_text())


def _worked_arrays():
    """The page's one-query example as [1, 4, 1] tensors (d = 1, tau = 1)."""
    g = _worked()
    s = g["blocks"]["A"]["s"] + g["blocks"]["B"]["s"]
    v = g["blocks"]["A"]["v"] + g["blocks"]["B"]["v"]
    q = np.zeros((1, 4, 1))
    q[0, :, 0] = 1.0  # every row queries with q = [1]; row 0 is the page's query
    k = np.array(s, dtype=np.float64).reshape(1, 4, 1)  # tau = 1 for d = 1, so s = q.k
    vv = np.array(v, dtype=np.float64).reshape(1, 4, 1)
    return q, k, vv


def _rand(rng, BH, N, d, scale=1.0):
    return (rng.standard_normal((BH, N, d)) * scale,
            rng.standard_normal((BH, N, d)) * scale,
            rng.standard_normal((BH, N, d)))


def _lib_reference(q, k, v, causal=False):
    """Dense attention from numpy matmul + scipy softmax/logsumexp."""
    d = q.shape[-1]
    s = np.einsum("bnd,bmd->bnm", q, k) / math.sqrt(d)
    if causal:
        n = s.shape[-1]
        s = np.where(np.tril(np.ones((n, n), dtype=bool)), s, -np.inf)
    out = np.einsum("bnm,bmd->bnd", softmax(s, axis=-1), v)
    return out.reshape(-1, d), logsumexp(s, axis=-1).reshape(-1)


# ---------------------------------------------------------------------------
# worked example
# ---------------------------------------------------------------------------
def pin_worked_example_steps(O):
    g = _worked()
    tol = g["printed_tolerance"]
    pa, pb = g["printed"]["step_A"], g["printed"]["step_B"]
    q = np.ones((1, 1))
    kA = np.array(g["blocks"]["A"]["s"]).reshape(2, 1)
    vA = np.array(g["blocks"]["A"]["v"]).reshape(2, 1)
    kB = np.array(g["blocks"]["B"]["s"]).reshape(2, 1)
    vB = np.array(g["blocks"]["B"]["v"]).reshape(2, 1)
    m, l, o = np.array([-np.inf]), np.array([0.0]), np.zeros((1, 1))
    m, l, o = O.fold(m, l, o, q, kA, vA)
    assert abs(m[0] - pa["m"]) <= tol, ("step A m", m[0])
    assert abs(l[0] - pa["l"]) <= tol, ("step A l", l[0])
    assert abs(o[0, 0] - pa["o"]) <= tol, ("step A o", o[0, 0])
    m, l, o = O.fold(m, l, o, q, kB, vB)
    assert abs(m[0] - pb["m"]) <= tol, ("step B m", m[0])
    assert abs(l[0] - pb["l"]) <= tol, ("step B l", l[0])
    assert abs(o[0, 0] - pb["o"]) <= tol, ("step B o", o[0, 0])
    assert abs(o[0, 0] / l[0] - g["printed"]["out"]) <= tol


def pin_worked_example_exact(O):
    """The same example against its closed form (e = Euler's number)."""
    e1, e3 = math.exp(-1.0), math.exp(-3.0)
    lA, oA = 1.0 + e1, e1 * 1.0 + 2.0
    lB = e1 * lA + 1.0 + e3
    oB = e1 * oA + 3.0 + 4.0 * e3
    q, k, v = _worked_arrays()
    out, lse, m, l, o = O.ring(q, k, v, P=2, rows=[0], state=True)
    assert abs(m[0] - 3.0) <= EXACT
    assert abs(l[0] - lB) <= EXACT, (l[0], lB)
    assert abs(o[0, 0] - oB) <= EXACT, (o[0, 0], oB)
    assert abs(out[0, 0] - oB / lB) <= EXACT
    assert abs(lse[0] - (3.0 + math.log(lB))) <= EXACT


def pin_worked_example_dense_and_ring(O):
    g = _worked()
    tol = g["printed_tolerance"]
    q, k, v = _worked_arrays()
    out_d, _ = O.dense(q, k, v, rows=[0])
    out_r, _ = O.ring(q, k, v, P=2, rows=[0])
    assert abs(out_d[0, 0] - g["printed"]["dense_out"]) <= tol
    assert abs(out_r[0, 0] - g["printed"]["out"]) <= tol


def pin_worked_example_reverse_order(O):
    """Query block 1 sees block B first, then A; same answer (order independence)."""
    q, k, v = _worked_arrays()
    out0, lse0 = O.ring(q, k, v, P=2, rows=[0])
    out1, lse1, m1, l1, o1 = O.ring(q, k, v, P=2, rows=[2], state=True)
    assert abs(out1[0, 0] - out0[0, 0]) <= EXACT
    assert abs(lse1[0] - lse0[0]) <= EXACT
    # B then A: the max is found at once, A is folded with alpha = 1.
    mB, lB, oB = O.fold([-np.inf], [0.0], np.zeros((1, 1)), np.ones((1, 1)),
                        k[0, 2:4], v[0, 2:4])
    assert mB[0] == 3.0
    m2, l2, o2 = O.fold(mB, lB, oB, np.ones((1, 1)), k[0, 0:2], v[0, 0:2])
    assert m2[0] == 3.0 and abs(l2[0] - l1[0]) <= EXACT and abs(o2[0, 0] - o1[0, 0]) <= EXACT


def pin_negative_control(O):
    """Normalising each block and averaging must miss the printed answer."""
    g = _worked()
    q, k, v = _worked_arrays()
    per_block = []
    for lo in (0, 2):
        out, _ = O.ring(q[:, lo:lo + 2], k[:, lo:lo + 2], v[:, lo:lo + 2], P=1, rows=[0])
        per_block.append(out[0, 0])
    wrong = sum(per_block) / 2
    right, _ = O.ring(q, k, v, P=2, rows=[0])
    assert abs(right[0, 0] - g["printed"]["out"]) <= g["printed_tolerance"]
    assert abs(wrong - g["printed"]["out"]) > 0.1, wrong


# ---------------------------------------------------------------------------
# schedule
# ---------------------------------------------------------------------------
def pin_ring_schedule(O):
    g = json.loads((GOLDEN / "ring_schedule_p4.json").read_text())
    assert (O.ring_order(g["P"]) == np.array(g["held"])).all()
    for P in (1, 2, 3, 5, 8):
        t = O.ring_order(P)
        assert (t[:, 0] == np.arange(P)).all()  # own block first
        for row in t:
            assert sorted(row.tolist()) == list(range(P))  # every block once


# ---------------------------------------------------------------------------
# closed forms and library references
# ---------------------------------------------------------------------------
def pin_two_keys_logistic(O):
    """Two keys: out = v1 + (v2 - v1) * sigmoid(s2 - s1); lse = logaddexp(s1, s2)."""
    rng = np.random.default_rng(1)
    d = 3
    for _ in range(5):
        q = rng.standard_normal((1, 2, d))
        k = rng.standard_normal((1, 2, d))
        v = rng.standard_normal((1, 2, d))
        tau = 1.0 / math.sqrt(d)
        s1, s2 = (q[0, 0] @ k[0, 0]) * tau, (q[0, 0] @ k[0, 1]) * tau
        w = 1.0 / (1.0 + math.exp(-(s2 - s1)))
        want = v[0, 0] + (v[0, 1] - v[0, 0]) * w
        for P in (1, 2):
            out, lse = O.ring(q, k, v, P=P, rows=[0])
            assert np.abs(out[0] - want).max() <= 1e-12
            assert abs(lse[0] - np.logaddexp(s1, s2)) <= 1e-12


def pin_identical_keys(O):
    rng = np.random.default_rng(2)
    BH, N, d = 2, 12, 4
    q = rng.standard_normal((BH, N, d))
    k = np.broadcast_to(rng.standard_normal((BH, 1, d)), (BH, N, d)).copy()
    v = rng.standard_normal((BH, N, d))
    out, lse = O.ring(q, k, v, P=3)
    tau = 1.0 / math.sqrt(d)
    want_out = np.repeat(v.mean(axis=1), N, axis=0)
    want_lse = (np.einsum("bnd,bd->bn", q, k[:, 0]) * tau + math.log(N)).reshape(-1)
    assert np.abs(out - want_out).max() <= 1e-12
    assert np.abs(lse - want_lse).max() <= 1e-12


def pin_constant_v(O):
    rng = np.random.default_rng(3)
    BH, N, d = 2, 8, 5
    q, k, _ = _rand(rng, BH, N, d, 2.0)
    v0 = rng.standard_normal(d)
    v = np.broadcast_to(v0, (BH, N, d)).copy()
    out, _ = O.ring(q, k, v, P=4)
    assert np.abs(out - v0).max() <= 1e-12


def pin_dominant_key(O):
    """One key far above the rest: out is that key's v."""
    rng = np.random.default_rng(4)
    BH, N, d = 1, 8, 4
    q, k, v = _rand(rng, BH, N, d)
    q[0, :] = 0.0
    q[0, :, 0] = 1.0
    k[0, :, 0] = 0.0
    k[0, 5, 0] = 200.0 * math.sqrt(d)  # s = 200 for key 5, 0 elsewhere
    out, lse = O.ring(q, k, v, P=2)
    assert np.abs(out - v[0, 5]).max() <= 1e-12
    assert np.abs(lse - 200.0).max() <= 1e-12


def pin_library_reference(O):
    rng = np.random.default_rng(5)
    for BH, N, d, P in ((1, 16, 4, 4), (3, 12, 3, 3), (2, 10, 8, 5)):
        q, k, v = _rand(rng, BH, N, d, 1.5)
        want_out, want_lse = _lib_reference(q, k, v)
        out_d, lse_d = O.dense(q, k, v)
        out_r, lse_r = O.ring(q, k, v, P=P)
        assert np.abs(out_d - want_out).max() <= 1e-12
        assert np.abs(lse_d - want_lse).max() <= 1e-12
        assert np.abs(out_r - want_out).max() <= 1e-12
        assert np.abs(lse_r - want_lse).max() <= 1e-12


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
def pin_ring_equals_dense_all_P(O):
    rng = np.random.default_rng(6)
    BH, N, d = 2, 24, 6
    q, k, v = _rand(rng, BH, N, d, 1.5)
    out_d, lse_d = O.dense(q, k, v)
    for P in (1, 2, 3, 4, 6, 8, 12, 24):
        out, lse = O.ring(q, k, v, P=P)
        assert np.abs(out - out_d).max() <= 1e-12, P
        assert np.abs(lse - lse_d).max() <= 1e-12, P


def pin_order_and_tile_invariance(O):
    rng = np.random.default_rng(7)
    BH, N, d, P = 1, 32, 4, 4
    q, k, v = _rand(rng, BH, N, d, 2.0)
    base, base_lse = O.ring(q, k, v, P=P)
    for _ in range(4):
        order = np.stack([rng.permutation(P) for _ in range(P)])
        out, lse = O.ring(q, k, v, P=P, order=order)
        assert np.abs(out - base).max() <= 1e-12
        assert np.abs(lse - base_lse).max() <= 1e-12
    for tile in (1, 3, 8):
        out, lse = O.ring(q, k, v, P=P, tile=tile)
        assert np.abs(out - base).max() <= 1e-12
        assert np.abs(lse - base_lse).max() <= 1e-12


def pin_brute_force_all_orders(O):
    """Every visiting order (all permutations per query block), P <= 3, tiny N."""
    import itertools

    rng = np.random.default_rng(8)
    BH, N, d = 1, 6, 2
    q, k, v = _rand(rng, BH, N, d, 2.0)
    want_out, want_lse = _lib_reference(q, k, v)
    for P in (1, 2, 3):
        perms = list(itertools.permutations(range(P)))
        for combo in itertools.product(perms, repeat=P):
            order = np.array(combo)
            out, lse = O.ring(q, k, v, P=P, order=order)
            assert np.abs(out - want_out).max() <= 1e-12
            assert np.abs(lse - want_lse).max() <= 1e-12


def pin_key_shift(O):
    """Adding u to every key leaves out unchanged and adds tau q.u to lse."""
    rng = np.random.default_rng(9)
    BH, N, d = 2, 16, 4
    q, k, v = _rand(rng, BH, N, d)
    u = rng.standard_normal(d) * 3.0
    out0, lse0 = O.ring(q, k, v, P=4)
    out1, lse1 = O.ring(q, k + u, v, P=4)
    assert np.abs(out1 - out0).max() <= 1e-12
    want = lse0 + (q @ u).reshape(-1) / math.sqrt(d)
    assert np.abs(lse1 - want).max() <= 1e-11


def pin_merge(O):
    rng = np.random.default_rng(10)
    BH, N, d, P = 2, 16, 4, 4
    q, k, v = _rand(rng, BH, N, d, 2.0)
    out_full, lse_full, m_f, l_f, o_f = O.ring(q, k, v, P=P, state=True)
    for G in (1, 2, 4):
        seg = P // G
        ms, ls, os_ = [], [], []
        for g in range(G):
            _, _, m, l, o = O.ring(q, k, v, P=P, t0=g * seg, t1=(g + 1) * seg, state=True)
            ms.append(m), ls.append(l), os_.append(o)
        out, lse = O.merge(np.stack(ms), np.stack(ls), np.stack(os_))
        assert np.abs(out - out_full).max() <= 1e-12, G
        assert np.abs(lse - lse_full).max() <= 1e-12, G
        # commutative: reversed partial order
        out_r, lse_r = O.merge(np.stack(ms[::-1]), np.stack(ls[::-1]), np.stack(os_[::-1]))
        assert np.abs(out_r - out_full).max() <= 1e-12
    # one partial: identity; an empty partial (m = -inf, l = 0) changes nothing
    out1, lse1, m1, l1, o1 = O.merge(m_f[None], l_f[None], o_f[None], state=True)
    assert np.abs(out1 - out_full).max() <= 1e-12
    assert np.array_equal(m1, m_f) and np.abs(l1 - l_f).max() <= 1e-12
    empty_m = np.full_like(m_f, -np.inf)
    out2, lse2 = O.merge(np.stack([m_f, empty_m]), np.stack([l_f, 0 * l_f]),
                         np.stack([o_f, 0 * o_f]))
    assert np.abs(out2 - out_full).max() <= 1e-12
    # all empty: out = 0, lse = -inf
    out3, lse3 = O.merge(empty_m[None], 0 * l_f[None], 0 * o_f[None])
    assert (out3 == 0).all() and np.isneginf(lse3).all()


def pin_fold_chain_equals_ring(O):
    """Folding blocks one call at a time in ring order reproduces the ring."""
    rng = np.random.default_rng(11)
    BH, N, d, P = 2, 12, 3, 3
    c = N // P
    q, k, v = _rand(rng, BH, N, d, 2.0)
    out_r, lse_r, m_r, l_r, o_r = O.ring(q, k, v, P=P, state=True)
    order = O.ring_order(P)
    for i in range(P):
        rows = np.concatenate([np.arange(b * N + i * c, b * N + (i + 1) * c) for b in range(BH)])
        m = np.full(BH * c, -np.inf)
        l = np.zeros(BH * c)
        o = np.zeros((BH * c, d))
        qi = q[:, i * c:(i + 1) * c]
        for t in range(P):
            j = order[i, t]
            m, l, o = O.fold(m, l, o, qi, k[:, j * c:(j + 1) * c], v[:, j * c:(j + 1) * c],
                             batch=BH)
        assert np.abs(m - m_r[rows]).max() <= 1e-12
        assert np.abs(l - l_r[rows]).max() <= 1e-12
        assert np.abs(o - o_r[rows]).max() <= 1e-12


def pin_bf16_inputs_exact(O):
    """bf16 bit patterns are read exactly: same result as their f64 values."""
    rng = np.random.default_rng(12)
    BH, N, d = 1, 8, 4
    x = rng.standard_normal((3, BH, N, d)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16
    vals = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    o16, l16 = O.ring(bits[0], bits[1], bits[2], P=2, dtype="bf16")
    o64, l64 = O.ring(vals[0], vals[1], vals[2], P=2, dtype="f64")
    assert np.array_equal(o16, o64) and np.array_equal(l16, l64)
    o32, l32 = O.ring(vals[0].astype(np.float32), vals[1].astype(np.float32),
                      vals[2].astype(np.float32), P=2, dtype="f32")
    assert np.array_equal(o32, o64) and np.array_equal(l32, l64)


def pin_row_subset(O):
    rng = np.random.default_rng(13)
    BH, N, d = 3, 16, 4
    q, k, v = _rand(rng, BH, N, d)
    out, lse = O.ring(q, k, v, P=4)
    rows = np.array([0, 5, 17, 47, 31])
    out_s, lse_s = O.ring(q, k, v, P=4, rows=rows)
    assert np.array_equal(out_s, out[rows]) and np.array_equal(lse_s, lse[rows])
    outd, lsed = O.dense(q, k, v, rows=rows)
    assert np.abs(outd - out[rows]).max() <= 1e-12


# ---------------------------------------------------------------------------
# causal mask and layouts ("Ring attention, explained", "The causal-mask
# catch"; "Ring Attention: the math", "Causal masking, load balance, and other
# wrinkles")
# ---------------------------------------------------------------------------
LAYOUTS = ("contiguous", "zigzag", "striped")


def pin_layout_tables(O):
    g = json.loads((GOLDEN / "layouts_p4_c4.json").read_text())
    for name in LAYOUTS:
        assert (O.layout_positions(name, g["P"], g["c"]) == np.array(g[name])).all(), name
    for name in LAYOUTS:  # every layout is a permutation of the positions
        for P, c in ((3, 6), (8, 4), (5, 2)):
            pos = O.layout_positions(name, P, c)
            assert sorted(pos.ravel().tolist()) == list(range(P * c))


def pin_zigzag_balances_causal_work(O):
    """Visible (query, key) pairs per device: equal under zigzag, within c of
    each other under striped, growing with the device under contiguous."""
    P, c = 8, 6
    work = {}
    for name in LAYOUTS:
        pos = O.layout_positions(name, P, c)
        work[name] = [int(sum(p + 1 for p in pos[j])) for j in range(P)]  # keys 0..p
    assert len(set(work["zigzag"])) == 1
    assert max(work["striped"]) - min(work["striped"]) == c * (P - 1)
    assert all(a < b for a, b in zip(work["contiguous"], work["contiguous"][1:]))
    assert sum(work["zigzag"]) == sum(work["contiguous"]) == P * c * (P * c + 1) // 2


def pin_causal_library_reference(O):
    rng = np.random.default_rng(20)
    for BH, N, d, P in ((1, 16, 4, 4), (2, 24, 3, 6), (1, 12, 5, 2)):
        q, k, v = _rand(rng, BH, N, d, 1.5)
        want_out, want_lse = _lib_reference(q, k, v, causal=True)
        out_d, lse_d = O.dense(q, k, v, causal=True)
        assert np.abs(out_d - want_out).max() <= 1e-12
        assert np.abs(lse_d - want_lse).max() <= 1e-12
        for layout in LAYOUTS:
            for PP in (1, P):
                out, lse = O.ring(q, k, v, P=PP, causal=True, layout=layout)
                assert np.abs(out - want_out).max() <= 1e-12, (layout, PP)
                assert np.abs(lse - want_lse).max() <= 1e-12, (layout, PP)


def pin_causal_first_token(O):
    """Position 0 sees only itself: out = v_0, lse = tau q_0 . k_0."""
    rng = np.random.default_rng(21)
    BH, N, d = 2, 8, 4
    q, k, v = _rand(rng, BH, N, d, 2.0)
    for layout in LAYOUTS:
        out, lse = O.ring(q, k, v, P=4, causal=True, layout=layout, rows=[0, N])
        for b, r in enumerate((0, N)):
            assert np.abs(out[b] - v[b, 0]).max() <= 1e-12
            assert abs(lse[b] - q[b, 0] @ k[b, 0] / math.sqrt(d)) <= 1e-12


def pin_causal_identical_keys(O):
    """Identical keys: position n averages v_0..v_n; lse = tau q.k + ln(n + 1)."""
    rng = np.random.default_rng(22)
    BH, N, d = 1, 12, 3
    q = rng.standard_normal((BH, N, d))
    k = np.broadcast_to(rng.standard_normal((BH, 1, d)), (BH, N, d)).copy()
    v = rng.standard_normal((BH, N, d))
    want = np.cumsum(v[0], axis=0) / np.arange(1, N + 1)[:, None]
    want_lse = q[0] @ k[0, 0] / math.sqrt(d) + np.log(np.arange(1, N + 1))
    for layout in LAYOUTS:
        out, lse = O.ring(q, k, v, P=3 if layout != "zigzag" else 2, causal=True, layout=layout)
        assert np.abs(out - want).max() <= 1e-12, layout
        assert np.abs(lse - want_lse).max() <= 1e-12, layout


def pin_causal_segments_merge(O):
    """Ring segments under the mask (some fully masked, hence empty) merge back
    to the whole causal ring."""
    rng = np.random.default_rng(23)
    BH, N, d, P = 1, 16, 4, 4
    q, k, v = _rand(rng, BH, N, d, 2.0)
    for layout in LAYOUTS:
        full_out, full_lse = O.ring(q, k, v, P=P, causal=True, layout=layout)
        ms, ls, os_ = [], [], []
        for g in range(P):
            _, _, m, l, o = O.ring(q, k, v, P=P, t0=g, t1=g + 1, causal=True, layout=layout,
                                   state=True)
            ms.append(m), ls.append(l), os_.append(o)
        assert np.isneginf(np.stack(ms)).any()  # some segments see only future keys
        out, lse = O.merge(np.stack(ms), np.stack(ls), np.stack(os_))
        assert np.abs(out - full_out).max() <= 1e-12
        assert np.abs(lse - full_lse).max() <= 1e-12


# ---------------------------------------------------------------------------
# backward ("Ring attention, explained", step 6: the same ring, with the K/V
# blocks carrying their gradient accumulators)
# ---------------------------------------------------------------------------
def _loss(O, q, k, v, dout, causal):
    out, _ = O.dense(q, k, v, causal=causal)
    return float((out.reshape(dout.shape) * dout).sum())


def pin_backward_finite_differences(O):
    """Every gradient against central differences of the forward oracle."""
    rng = np.random.default_rng(30)
    BH, N, d = 2, 12, 3
    eps = 1e-5
    for causal, layout, P in ((False, "contiguous", 3), (True, "zigzag", 2), (True, "striped", 4)):
        q, k, v = _rand(rng, BH, N, d, 1.5)
        dout = rng.standard_normal((BH, N, d))
        out, lse = O.dense(q, k, v, causal=causal)
        grads = O.backward(q, k, v, out.reshape(BH, N, d), dout, lse.reshape(BH, N), P=P,
                           causal=causal, layout=layout)
        for which, (x, g) in enumerate(zip((q, k, v), grads)):
            for _ in range(6):
                idx = tuple(int(rng.integers(0, s)) for s in x.shape)
                xp, xm = x.copy(), x.copy()
                xp[idx] += eps
                xm[idx] -= eps
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[which], args_m[which] = xp, xm
                fd = (_loss(O, *args_p, dout, causal) - _loss(O, *args_m, dout, causal)) / (2 * eps)
                assert abs(g[idx] - fd) <= 1e-7 * max(1.0, abs(fd)), (which, idx, g[idx], fd)


def pin_backward_ring_order_invariance(O):
    """Gradients do not depend on P or on the layout (the ring only reorders)."""
    rng = np.random.default_rng(31)
    BH, N, d = 1, 16, 4
    q, k, v = _rand(rng, BH, N, d, 1.5)
    dout = rng.standard_normal((BH, N, d))
    for causal in (False, True):
        out, lse = O.dense(q, k, v, causal=causal)
        base = O.backward(q, k, v, out.reshape(BH, N, d), dout, lse.reshape(BH, N), P=1,
                          causal=causal)
        for layout, P in (("contiguous", 4), ("zigzag", 2), ("striped", 8)):
            g = O.backward(q, k, v, out.reshape(BH, N, d), dout, lse.reshape(BH, N), P=P,
                           causal=causal, layout=layout)
            for a, b in zip(base, g):
                assert np.abs(a - b).max() <= 1e-12


def pin_backward_identical_keys_dv(O):
    """Identical keys give uniform weights 1/N, so dV_j = mean_i dO_i."""
    rng = np.random.default_rng(32)
    BH, N, d = 1, 10, 3
    q = rng.standard_normal((BH, N, d))
    k = np.broadcast_to(rng.standard_normal((BH, 1, d)), (BH, N, d)).copy()
    v = rng.standard_normal((BH, N, d))
    dout = rng.standard_normal((BH, N, d))
    out, lse = O.dense(q, k, v)
    _, _, dv = O.backward(q, k, v, out.reshape(BH, N, d), dout, lse.reshape(BH, N), P=2)
    assert np.abs(dv - dout.mean(axis=1, keepdims=True)).max() <= 1e-12


def pin_backward_rows_match_full(O):
    """The per-row backward used on sampled rows equals the full backward."""
    rng = np.random.default_rng(33)
    BH, N, d = 2, 10, 3
    q, k, v = _rand(rng, BH, N, d, 1.5)
    dout = rng.standard_normal((BH, N, d))
    out, lse = O.dense(q, k, v)
    out = out.reshape(BH, N, d)
    dq, dk, dv = O.backward(q, k, v, out, dout, lse.reshape(BH, N), P=2)
    rows = np.array([0, 7, 13, 19])
    rq, rk, rv = O.backward_rows(q, k, v, out, dout, lse, rows, rows[::-1])
    assert np.abs(rq - dq.reshape(-1, d)[rows]).max() <= 1e-12
    assert np.abs(rk - dk.reshape(-1, d)[rows[::-1]]).max() <= 1e-12
    assert np.abs(rv - dv.reshape(-1, d)[rows[::-1]]).max() <= 1e-12
    # causal
    out, lse = O.dense(q, k, v, causal=True)
    out = out.reshape(BH, N, d)
    dq, dk, dv = O.backward(q, k, v, out, dout, lse.reshape(BH, N), P=2, causal=True)
    rq, rk, rv = O.backward_rows(q, k, v, out, dout, lse, rows, rows, causal=True)
    assert np.abs(rq - dq.reshape(-1, d)[rows]).max() <= 1e-12
    assert np.abs(rk - dk.reshape(-1, d)[rows]).max() <= 1e-12
    assert np.abs(rv - dv.reshape(-1, d)[rows]).max() <= 1e-12


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
