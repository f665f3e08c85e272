"""Pins that tie the fp64 oracle to something other than itself.

Each ``check_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the pages or the mathematics fix:

* hand-worked cases stored in ``tests/golden/hand_worked.json``, each citing
  the passage it applies;
* the naive materialised computation written with numpy library routines
  (similarity grid by einsum, masked max/argmax by ``np.max``/``np.argmax``,
  sum by ``np.sum``) -- the reference path the colpali PR describes as
  "einsum + amax + sum" -- including the top-2 gap;
* exact widening of f16 and bf16 storage, against numpy's and torch's own
  conversions;
* invariants: document- and query-token permutation, positive scaling,
  deleting masked tokens, cross-layout consistency;
* a closed form: when D holds every unit-norm query token among other
  unit-norm tokens the score is the number of valid query tokens
  (Cauchy-Schwarz), with the argmax on the copies;
* central finite differences of the forward for the backward.

The same checks run against deliberately broken copies of the oracle in
``test_oracle_mutants.py``, to show that each plausible mistake fails at
least one of them.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _arr(x, dtype=np.float64):
    return None if x is None else np.asarray(x, dtype=dtype)


# ---------------------------------------------------------------- goldens --

def check_golden_cases(orc):
    for c in _golden_cases():
        layout = c.get("layout", "allpairs")
        Q, D = _arr(c["Q"]), _arr(c["D"])
        qm = _arr(c["qmask"], np.uint8)
        dm = _arr(c["dmask"], np.uint8)
        fwd = getattr(orc, f"{layout}_fwd")
        bwd = getattr(orc, f"{layout}_bwd")
        s, am, _ = fwd(Q, D, qm, dm)
        assert np.array_equal(s, _arr(c["scores"])), (c["name"], s)
        assert np.array_equal(am, np.asarray(c["argmax"], np.int32)), (c["name"], am)
        gQ, gD = bwd(Q, D, _arr(c["grad_out"]), am)
        assert np.array_equal(gQ, _arr(c["gQ"])), (c["name"], "gQ", gQ)
        assert np.array_equal(gD, _arr(c["gD"])), (c["name"], "gD", gD)


# ------------------------------------------------- numpy naive reference --

def naive_allpairs(Q, D, qm, dm):
    """Materialise the [Nq,Nd,Lq,Ld] grid, mask, max, sum (library routines)."""
    S = np.einsum("qik,djk->qdij", Q, D)
    if dm is not None:
        S = np.where(dm[None, :, None, :].astype(bool), S, -np.inf)
    Ld = D.shape[1]
    if Ld == 0:
        best = np.full(S.shape[:3], -np.inf)
        arg = np.full(S.shape[:3], -1)
        gap = np.full(S.shape[:3], np.nan)
    else:
        best = S.max(axis=3)
        arg = S.argmax(axis=3)  # first occurrence: lowest index on ties
        top2 = np.sort(S, axis=3)[..., -2] if Ld > 1 else np.full(best.shape, -np.inf)
        with np.errstate(invalid="ignore"):
            gap = best - top2
    qvalid = np.ones(Q.shape[:2], bool) if qm is None else qm.astype(bool)
    empty = np.zeros(D.shape[0], bool) if dm is None else ~dm.astype(bool).any(axis=1)
    if Ld == 0:
        empty[:] = True
    terms = np.where(qvalid[:, None, :], best, 0.0)
    scores = np.sum(terms, axis=2)
    scores[:, empty] = -1e9
    dead = ~qvalid[:, None, :] | empty[None, :, None]
    arg = np.where(dead, -1, arg).astype(np.int32)
    gap = np.where(dead, np.nan, gap)
    return scores, arg, gap


def _random_inputs(rng, Nq, Nd, Lq, Ld, dim, p_mask=0.3, p_empty=0.2):
    Q = rng.standard_normal((Nq, Lq, dim))
    D = rng.standard_normal((Nd, Ld, dim))
    qm = (rng.random((Nq, Lq)) > p_mask).astype(np.uint8)
    dm = (rng.random((Nd, Ld)) > p_mask).astype(np.uint8)
    dm[rng.random(Nd) < p_empty] = 0
    return Q, D, qm, dm


def check_naive_reference(orc):
    rng = np.random.default_rng(1234)
    shapes = [(3, 4, 5, 7, 6), (1, 1, 1, 1, 1), (2, 5, 3, 17, 4), (4, 3, 8, 9, 16), (2, 2, 4, 0, 3)]
    for (Nq, Nd, Lq, Ld, dim) in shapes:
        for masks in (True, False):
            Q, D, qm, dm = _random_inputs(rng, Nq, Nd, Lq, Ld, dim)
            if not masks:
                qm = dm = None
            s, am, gap = orc.allpairs_fwd(Q, D, qm, dm)
            s_ref, am_ref, gap_ref = naive_allpairs(Q, D, qm, dm)
            np.testing.assert_allclose(s, s_ref, rtol=1e-12, atol=1e-12)
            assert np.array_equal(am, am_ref)
            np.testing.assert_allclose(gap, gap_ref, rtol=1e-12, atol=1e-12, equal_nan=True)


def check_naive_reference_storage_dtypes(orc):
    """f16 / bf16 / f32 storage is widened exactly: same result as the
    library's own widening followed by the fp64 naive reference."""
    rng = np.random.default_rng(99)
    Q, D, qm, dm = _random_inputs(rng, 3, 4, 6, 11, 8)
    for tdt, tag in ((torch.float16, "f16"), (torch.bfloat16, "bf16"), (torch.float32, "f32")):
        Qt = torch.from_numpy(Q).to(tdt)
        Dt = torch.from_numpy(D).to(tdt)
        if tag == "bf16":
            Qs = Qt.view(torch.int16).numpy().view(np.uint16)
            Ds = Dt.view(torch.int16).numpy().view(np.uint16)
        else:
            Qs, Ds = Qt.numpy(), Dt.numpy()
        s, am, _ = orc.allpairs_fwd(Qs, Ds, qm, dm, dtype=tag)
        s_ref, am_ref, _ = naive_allpairs(Qt.double().numpy(), Dt.double().numpy(), qm, dm)
        np.testing.assert_allclose(s, s_ref, rtol=1e-12, atol=1e-12)
        assert np.array_equal(am, am_ref)


def check_f16_special_values(orc):
    """Subnormal, normal and extreme f16 values widen exactly (numpy's astype)."""
    bits = np.array([0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x8001, 0xC000, 0x3555],
                    dtype=np.uint16)
    vals = bits.view(np.float16)
    n = len(vals)
    Q = np.zeros((1, n, n), np.float16)
    D = np.zeros((1, 1, n), np.float16)
    D[0, 0, :] = np.float16(1.0)
    for i in range(n):
        Q[0, i, i] = vals[i]
    s, am, _ = orc.allpairs_fwd(Q, D)
    assert s[0, 0] == float(np.sum(vals.astype(np.float64)))
    # and each single value on its own
    for i in range(n):
        s1, _, _ = orc.allpairs_fwd(Q[:, i:i + 1], D)
        assert s1[0, 0] == float(vals[i].astype(np.float64)), (hex(bits[i]), s1)


# ------------------------------------------------------------- invariants --

def check_doc_permutation(orc):
    rng = np.random.default_rng(7)
    Q, D, qm, dm = _random_inputs(rng, 3, 4, 5, 9, 6, p_empty=0.0)
    s, am, _ = orc.allpairs_fwd(Q, D, qm, dm)
    perm = rng.permutation(9)
    s2, am2, _ = orc.allpairs_fwd(Q, D[:, perm], qm, dm[:, perm])
    np.testing.assert_allclose(s2, s, rtol=0, atol=0)
    mapped = np.where(am2 >= 0, perm[np.maximum(am2, 0)], -1)
    assert np.array_equal(mapped, am)


def check_query_permutation(orc):
    rng = np.random.default_rng(8)
    # integer-valued inputs keep every partial sum exact
    Q = rng.integers(-4, 5, (2, 6, 5)).astype(np.float64)
    D = rng.integers(-4, 5, (3, 7, 5)).astype(np.float64)
    qm = (rng.random((2, 6)) > 0.3).astype(np.uint8)
    s, am, _ = orc.allpairs_fwd(Q, D, qm, None)
    perm = rng.permutation(6)
    s2, am2, _ = orc.allpairs_fwd(Q[:, perm], D, qm[:, perm], None)
    assert np.array_equal(s2, s)
    assert np.array_equal(am2, am[:, :, perm])


def check_positive_scaling(orc):
    rng = np.random.default_rng(9)
    Q, D, qm, dm = _random_inputs(rng, 2, 3, 4, 5, 6)
    s, am, _ = orc.allpairs_fwd(Q, D, qm, dm)
    for c in (0.25, 4.0):
        s2, am2, _ = orc.allpairs_fwd(c * Q, D, qm, dm)
        expect = np.where(s == -1e9, -1e9, c * s)
        np.testing.assert_allclose(s2, expect, rtol=1e-13)
        assert np.array_equal(am2, am)


def check_delete_equals_mask(orc):
    rng = np.random.default_rng(10)
    Q, D, qm, dm = _random_inputs(rng, 2, 3, 5, 8, 4, p_empty=0.0)
    dm[:, 0] = 1  # keep every document non-empty
    s, am, _ = orc.allpairs_fwd(Q, D, qm, dm)
    for q in range(2):
        for d in range(3):
            keep_j = np.flatnonzero(dm[d])
            keep_i = np.flatnonzero(qm[q])
            s1, am1, _ = orc.allpairs_fwd(Q[q:q + 1, keep_i], D[d:d + 1, keep_j])
            np.testing.assert_allclose(s1[0, 0], s[q, d], rtol=1e-13, atol=1e-13)
            assert np.array_equal(keep_j[am1[0, 0]], am[q, d, keep_i])


def check_cross_layout(orc):
    rng = np.random.default_rng(11)
    B, N, Lq, Ld, dim = 3, 4, 5, 7, 6
    Q = rng.standard_normal((B, Lq, dim))
    Dk = rng.standard_normal((B, N, Ld, dim))
    qm = (rng.random((B, Lq)) > 0.3).astype(np.uint8)
    dmk = (rng.random((B, N, Ld)) > 0.3).astype(np.uint8)
    dmk[0, 1] = 0
    # kd[b, n] == all-pairs(Q[b], D[b, n])
    sk, amk, _ = orc.kd_fwd(Q, Dk, qm, dmk)
    for b in range(B):
        sa, ama, _ = orc.allpairs_fwd(Q[b:b + 1], Dk[b], qm[b:b + 1], dmk[b])
        assert np.array_equal(sk[b], sa[0])
        assert np.array_equal(amk[b], ama[0])
    # pairwise[b] == all-pairs diagonal
    Dp = Dk[:, 0]
    dmp = dmk[:, 0]
    sp, amp, _ = orc.pairwise_fwd(Q, Dp, qm, dmp)
    sa, ama, _ = orc.allpairs_fwd(Q, Dp, qm, dmp)
    assert np.array_equal(sp, np.diagonal(sa))
    assert np.array_equal(amp, np.stack([ama[b, b] for b in range(B)]))
    # and the backward of each layout equals the all-pairs backward restricted
    # to the same pairs (zero upstream gradient elsewhere)
    g = rng.standard_normal(B)
    gQp, gDp = orc.pairwise_bwd(Q, Dp, g, amp)
    gfull = np.diag(g)
    gQa, gDa = orc.allpairs_bwd(Q, Dp, gfull, ama)
    np.testing.assert_allclose(gQp, gQa, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(gDp, gDa, rtol=1e-13, atol=1e-13)
    gk = rng.standard_normal((B, N))
    gQk, gDk = orc.kd_bwd(Q, Dk, gk, amk)
    for b in range(B):
        gQa, gDa = orc.allpairs_bwd(Q[b:b + 1], Dk[b], gk[b:b + 1], amk[b:b + 1])
        np.testing.assert_allclose(gQk[b], gQa[0], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(gDk[b], gDa, rtol=1e-13, atol=1e-13)


def check_closed_form_unit_copies(orc):
    """D holds every valid unit-norm Q_i among other unit-norm tokens:
    each max is Q_i.Q_i = 1 (Cauchy-Schwarz), so the score is the number of
    valid query tokens and the argmax points at the copy."""
    rng = np.random.default_rng(12)
    Lq, Ld, dim = 6, 20, 8
    Q = rng.standard_normal((1, Lq, dim))
    Q /= np.linalg.norm(Q, axis=-1, keepdims=True)
    D = rng.standard_normal((1, Ld, dim))
    D /= np.linalg.norm(D, axis=-1, keepdims=True)
    slots = rng.permutation(Ld)[:Lq]
    D[0, slots] = Q[0]
    qm = np.array([[1, 1, 0, 1, 1, 1]], np.uint8)
    s, am, _ = orc.allpairs_fwd(Q, D, qm, None)
    assert abs(s[0, 0] - qm.sum()) < 1e-12, s
    valid = qm[0].astype(bool)
    assert np.array_equal(am[0, 0][valid], slots[valid])


def check_degenerate_lengths(orc):
    rng = np.random.default_rng(13)
    Q = rng.standard_normal((2, 3, 4))
    D = rng.standard_normal((3, 5, 4))
    # Lq = 0: non-empty documents score 0, empty ones -1e9
    dm = np.ones((3, 5), np.uint8)
    dm[1] = 0
    s, am, _ = orc.allpairs_fwd(Q[:, :0], D, None, dm)
    assert np.array_equal(s, np.array([[0.0, -1e9, 0.0]] * 2))
    assert am.shape == (2, 3, 0)
    # Ld = 0: every document is empty
    s, am, _ = orc.allpairs_fwd(Q, D[:, :0], None, None)
    assert np.all(s == -1e9) and np.all(am == -1)


# -------------------------------------------------- finite differences --

def _loss(orc, Q, D, qm, dm, g):
    s, _, _ = orc.allpairs_fwd(Q, D, qm, dm)
    live = s != -1e9
    return float(np.sum(np.where(live, g * s, 0.0)))


def check_finite_difference_gradients(orc):
    """Central differences at h = 1e-5 on a case whose top-2 gaps all exceed
    1e-3: the score is linear around such a point, so the difference quotient
    equals the gradient up to rounding."""
    rng = np.random.default_rng(14)
    for _ in range(20):
        Q, D, qm, dm = _random_inputs(rng, 2, 3, 3, 4, 3, p_empty=0.0)
        dm[:, 0] = 1
        dm[2] = 0  # one empty document: its upstream gradient must be ignored
        _, am, gap = orc.allpairs_fwd(Q, D, qm, dm)
        finite = gap[~np.isnan(gap)]
        if finite.size and finite.min() > 1e-3:
            break
    else:  # pragma: no cover - the seed above finds a case quickly
        raise AssertionError("no well-separated case found")
    g = rng.standard_normal((2, 3))
    gQ, gD = orc.allpairs_bwd(Q, D, g, am)
    h = 1e-5
    for X, G in ((Q, gQ), (D, gD)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            old = X[idx]
            X[idx] = old + h
            fp = _loss(orc, Q, D, qm, dm, g)
            X[idx] = old - h
            fm = _loss(orc, Q, D, qm, dm, g)
            X[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(G, num, rtol=1e-6, atol=1e-7)


# ---------------------------------------------------- cross-entropy head --

def check_ce_golden(orc):
    """The hand-worked cases of tests/golden/ce_hand_worked.json."""
    with open(os.path.join(os.path.dirname(__file__), "golden", "ce_hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        loss, row_loss, grad = orc.ce_rows(np.array(c["scores"]), np.array(c["target"]), c["scale"])
        np.testing.assert_allclose(loss, c["loss"], rtol=1e-14, atol=1e-15, err_msg=c["name"])
        np.testing.assert_allclose(row_loss, c["row_loss"], rtol=1e-14, atol=1e-15, err_msg=c["name"])
        np.testing.assert_allclose(grad, c["grad"], rtol=1e-14, atol=1e-15, err_msg=c["name"])


def check_ce_invariants(orc):
    """Shift invariance per row, gradient rows summing to zero with the only
    negative entry at the target, the scale acting on the logits, and equal
    logits giving log(cols)."""
    rng = np.random.default_rng(21)
    S = rng.standard_normal((6, 9)) * 3
    t = rng.integers(0, 9, size=6)
    loss, rl, g = orc.ce_rows(S, t)
    loss2, rl2, g2 = orc.ce_rows(S + rng.standard_normal((6, 1)) * 50, t)
    np.testing.assert_allclose(rl2, rl, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g2, g, rtol=1e-9, atol=1e-13)
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-15)
    for r in range(6):
        assert g[r, t[r]] < 0 and np.all(np.delete(g[r], t[r]) > 0)
    assert np.isclose(loss, rl.mean(), rtol=1e-15)
    # scale 2 on S is scale 1 on 2S for the loss; the gradient picks up the factor
    l3, rl3, g3 = orc.ce_rows(S, t, 2.0)
    l4, rl4, g4 = orc.ce_rows(2 * S, t, 1.0)
    np.testing.assert_allclose(rl3, rl4, rtol=1e-13)
    np.testing.assert_allclose(g3, 2 * g4, rtol=1e-12, atol=1e-15)
    # equal logits
    l5, rl5, g5 = orc.ce_rows(np.full((3, 7), 0.25), np.array([0, 3, 6]))
    np.testing.assert_allclose(rl5, np.log(7.0), rtol=1e-15)


def check_ce_finite_difference(orc):
    """Central differences of the mean loss with respect to every score."""
    rng = np.random.default_rng(22)
    S = rng.standard_normal((4, 5))
    t = np.array([0, 4, 2, 1])
    _, _, g = orc.ce_rows(S, t, 1.7)
    h = 1e-6
    num = np.zeros_like(S)
    for idx in np.ndindex(S.shape):
        old = S[idx]
        S[idx] = old + h
        fp = orc.ce_rows(S, t, 1.7)[0]
        S[idx] = old - h
        fm = orc.ce_rows(S, t, 1.7)[0]
        S[idx] = old
        num[idx] = (fp - fm) / (2 * h)
    np.testing.assert_allclose(g, num, rtol=1e-7, atol=1e-9)


ALL_CHECKS = [
    check_golden_cases,
    check_naive_reference,
    check_naive_reference_storage_dtypes,
    check_f16_special_values,
    check_doc_permutation,
    check_query_permutation,
    check_positive_scaling,
    check_delete_equals_mask,
    check_cross_layout,
    check_closed_form_unit_copies,
    check_degenerate_lengths,
    check_finite_difference_gradients,
    check_ce_golden,
    check_ce_invariants,
    check_ce_finite_difference,
]
