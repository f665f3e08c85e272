"""Comparison rules between the CUDA library and the fp64 oracle.

* Scores and gradients: normwise relative error max|x - r| / max|r| over the
  entries that are not the empty-document sentinel, at most 2e-3 for
  fp16/bf16 inputs and 1e-5 for fp32 inputs.  Sentinel entries (-1e9) must
  match bit for bit.
* argmax: -1 exactly where the oracle has -1; the oracle's index exactly
  wherever the oracle's top-2 gap exceeds 1e-2; elsewhere any index whose
  oracle similarity is within 1e-4 of the maximum and that is a valid
  (unmasked) document token -- several answers are correct there.
"""
from __future__ import annotations

import numpy as np
import torch

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}
GAP_EXACT = 1e-2
NEAR_TIE = 1e-4
EMPTY = -1e9


def normwise_rel_err(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    denom = np.max(np.abs(ref)) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    if denom == 0.0:
        return float(np.max(np.abs(x)))
    return float(np.max(np.abs(x - ref)) / denom)


def assert_scores_close(gpu_scores, orc_scores, dtype: str, what="scores"):
    g = np.asarray(gpu_scores, np.float64)
    r = np.asarray(orc_scores, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    empty = r == EMPTY
    assert np.array_equal(g[empty], r[empty]), f"{what}: empty-document sentinel mismatch"
    assert np.all(g[~empty] != EMPTY), f"{what}: sentinel where the oracle has a score"
    err = normwise_rel_err(g[~empty], r[~empty])
    assert err <= TOL[dtype], f"{what}: normwise relative error {err:.3g} > {TOL[dtype]:g}"
    return err


def assert_grad_close(gpu, orc, dtype: str, what):
    err = normwise_rel_err(gpu, orc)
    assert err <= TOL[dtype], f"{what}: normwise relative error {err:.3g} > {TOL[dtype]:g}"
    return err


def widen(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def assert_argmax_valid(am_gpu, am_orc, gap, Qw, Dw, query_of, doc_of, dmask=None):
    """am_* [P, Lq]; gap [P, Lq]; Qw [nQ, Lq, dim] and Dw [nD, Ld, dim] fp64;
    query_of/doc_of map a pair index to its query / document."""
    am_gpu = np.asarray(am_gpu).reshape(am_orc.shape)
    dead = am_orc < 0
    assert np.array_equal(am_gpu[dead], am_orc[dead]), "argmax: -1 entries differ"
    live = ~dead
    sure = live & (gap > GAP_EXACT)
    bad = sure & (am_gpu != am_orc)
    assert not bad.any(), f"argmax differs where the top-2 gap > {GAP_EXACT}: {np.argwhere(bad)[:5]}"
    near = live & ~sure & (am_gpu != am_orc)
    for p, i in np.argwhere(near):
        a = int(am_gpu[p, i])
        Ld = Dw.shape[1]
        assert 0 <= a < Ld, f"argmax out of range at {(p, i)}: {a}"
        d = doc_of(p)
        if dmask is not None:
            assert dmask[d, a], f"argmax on a masked token at {(p, i)}"
        q = query_of(p)
        s_gpu = float(Qw[q, i] @ Dw[d, a])
        s_best = float(Qw[q, i] @ Dw[d, am_orc[p, i]])
        assert s_gpu >= s_best - NEAR_TIE, f"argmax at {(p, i)} is not a near-tie"
    return int(near.sum())
