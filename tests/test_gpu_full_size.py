"""CUDA library vs fp64 oracle at the full workload sizes (GPU).

Inputs are drawn on the device by the seeded generators and copied to the
host for the oracle.  Where the oracle finishes in seconds it runs on every
pair (in-batch, per-query candidates, reranking); on the large all-pairs
inference workload it scores every query against a seeded subset of 256
documents.  Gradients are checked on sampled query and document rows by
running the oracle backward on the sub-problem that owns them, with the
oracle's own argmax fed to the GPU backward.
"""
import numpy as np
import pytest
import torch

import gpu_harness
import oracle
import parity
from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300.workloads import ce_grad_rows, generate, to_numpy

pytestmark = pytest.mark.gpu


def _gpu_scores_argmax(h, inp):
    Q, D = inp.Q.contiguous(), inp.D.contiguous()
    shape = inp.workload.score_shape
    scores = torch.empty(shape, dtype=torch.float32, device=Q.device)
    am = torch.empty((*shape, h.Lq), dtype=torch.int32, device=Q.device)
    getattr(binding, f"lik_maxsim_{h.kind}_fwd")(Q, D, inp.qmask, inp.dmask, scores, am)
    binding.lik_check_device_error()
    return scores, am


_ORACLE_FWD = {}


def _oracle_fwd(name, h):
    """The oracle's forward of a full workload (computed once per run)."""
    if name not in _ORACLE_FWD:
        _ORACLE_FWD[name] = h.oracle_fwd()
    return _ORACLE_FWD[name]


def _check_full_forward(name):
    inp = generate(name, device="cuda")
    h = gpu_harness.Layout(inp)
    s_g, am_g = _gpu_scores_argmax(h, inp)
    s_o, am_o, gap = _oracle_fwd(name, h)
    tag = inp.workload.dtype
    parity.assert_scores_close(s_g.cpu().numpy(), s_o, tag)
    Qw = parity.widen(inp.Q)
    Dw = parity.widen(inp.D).reshape(h.nD, h.Ld, h.dim)
    dm = inp.dmask.cpu().numpy().reshape(h.nD, h.Ld)
    parity.assert_argmax_valid(am_g.cpu().numpy().reshape(h.n_pairs, h.Lq),
                               am_o.reshape(h.n_pairs, h.Lq), gap.reshape(h.n_pairs, h.Lq),
                               Qw, Dw, h.query_of, h.doc_of, dm)
    return inp, h, s_o, am_o


def test_inbatch_b128_bf16_full():
    inp, h, s_o, am_o = _check_full_forward("inbatch_b128_bf16")
    g = ce_grad_rows(torch.from_numpy(s_o), inp.ce_target.cpu()).numpy()
    g32 = g.astype(np.float32)
    gQ_g, gD_g = h.gpu_bwd(g32, am_o)
    Qn, tag = to_numpy(inp.Q)
    Dn, _ = to_numpy(inp.D)
    orc = oracle.get()
    rng = np.random.default_rng(0)
    for q in rng.choice(h.nQ, 6, replace=False):
        gQ_o, _ = orc.allpairs_bwd(Qn[q:q + 1], Dn, g32[q:q + 1].astype(np.float64),
                                   am_o[q:q + 1], dtype=tag)
        parity.assert_grad_close(gQ_g[q], gQ_o[0], "bf16", f"grad_Q[{q}]")
    for d in rng.choice(h.nD, 6, replace=False):
        _, gD_o = orc.allpairs_bwd(Qn, Dn[d:d + 1], g32[:, d:d + 1].astype(np.float64),
                                   am_o[:, d:d + 1], dtype=tag)
        parity.assert_grad_close(gD_g[d], gD_o[0], "bf16", f"grad_D[{d}]")


def test_kd_b256_n17_bf16_full():
    inp, h, s_o, am_o = _check_full_forward("kd_b256_n17_bf16")
    # the planted positive (candidate 0) scores highest for most queries
    assert np.mean(np.argmax(s_o, axis=1) == 0) > 0.9
    g = ce_grad_rows(torch.from_numpy(s_o), inp.ce_target.cpu()).numpy()
    g32 = g.astype(np.float32)
    gQ_g, gD_g = h.gpu_bwd(g32, am_o)
    Qn, tag = to_numpy(inp.Q)
    Dn, _ = to_numpy(inp.D)
    orc = oracle.get()
    rng = np.random.default_rng(1)
    for b in rng.choice(h.nQ, 8, replace=False):
        gQ_o, gD_o = orc.kd_bwd(Qn[b:b + 1], Dn[b:b + 1], g32[b:b + 1].astype(np.float64),
                                am_o[b:b + 1], dtype=tag)
        parity.assert_grad_close(gQ_g[b], gQ_o[0], "bf16", f"grad_Q[{b}]")
        parity.assert_grad_close(gD_g[b], gD_o[0], "bf16", f"grad_D[{b}]")
    # rows no argmax points at are exactly zero
    hit = np.zeros((h.nD, h.Ld), bool)
    pairs, toks = np.nonzero(am_o.reshape(h.n_pairs, h.Lq) >= 0)
    hit[pairs, am_o.reshape(h.n_pairs, h.Lq)[pairs, toks]] = True
    row_max = np.abs(gD_g.reshape(h.nD, h.Ld, h.dim)).max(axis=2)
    assert not np.any(row_max[~hit])


@pytest.mark.parametrize("name", ["inbatch_b128_bf16", "kd_b256_n17_bf16"])
def test_one_call_step_full(name):
    """The one-call training step in the launch configuration bench.py times
    (the forward, the loss head and both fp32 gradients; in-batch, grad_D
    zero-filled by the forward), at full size.  Scores, argmax, loss and score
    gradient against the oracle; sampled gradient rows against the oracle
    backward run on the step's own argmax (each entry checked to be a valid
    maximum first) with the oracle's score gradient."""
    inp = generate(name, device="cuda")
    h = gpu_harness.Layout(inp)
    rows = h.nQ
    cols = h.n_pairs // rows
    dev = inp.Q.device
    target = inp.ce_target.to(device=dev, dtype=torch.int32).contiguous()
    scores = torch.empty(rows, cols, device=dev)
    am = torch.empty(rows, cols, h.Lq, dtype=torch.int32, device=dev)
    loss = torch.empty(1, device=dev)
    rl = torch.empty(rows, device=dev)
    gs = torch.empty(rows, cols, device=dev)
    gQ = torch.full(inp.Q.shape, float("nan"), device=dev)
    gD = torch.full(inp.D.shape, float("nan"), device=dev)
    getattr(binding, f"lik_maxsim_{h.kind}_ce_step")(inp.Q, inp.D, inp.qmask, inp.dmask, target, scores, am, loss,
                                                     rl, gs, gQ, gD)
    binding.lik_check_device_error()
    s_o, am_o, gap = _oracle_fwd(name, h)
    tag = inp.workload.dtype
    parity.assert_scores_close(scores.cpu().numpy(), s_o.reshape(rows, cols), tag)
    am_g = am.cpu().numpy().reshape(h.n_pairs, h.Lq)
    Qw = parity.widen(inp.Q)
    Dw = parity.widen(inp.D).reshape(h.nD, h.Ld, h.dim)
    dm = inp.dmask.cpu().numpy().reshape(h.nD, h.Ld)
    parity.assert_argmax_valid(am_g, am_o.reshape(h.n_pairs, h.Lq), gap.reshape(h.n_pairs, h.Lq), Qw, Dw,
                               h.query_of, h.doc_of, dm)
    loss_o, rl_o, gs_o = oracle.get().ce_rows(s_o.reshape(rows, cols), target.cpu().numpy(), 1.0)
    assert abs(loss.item() - loss_o) <= parity.TOL[tag] * max(abs(loss_o), 1.0)
    assert parity.normwise_rel_err(rl.cpu().numpy(), rl_o) <= parity.TOL[tag]
    assert parity.normwise_rel_err(gs.cpu().numpy(), gs_o) <= parity.TOL[tag]
    gQ_g, gD_g = gQ.cpu().numpy(), gD.cpu().numpy()
    assert np.isfinite(gQ_g).all() and np.isfinite(gD_g).all(), "a gradient element was not written"
    am_g = am_g.reshape(rows, cols, h.Lq)
    Qn, _ = to_numpy(inp.Q)
    Dn, _ = to_numpy(inp.D)
    orc = oracle.get()
    rng = np.random.default_rng(3)
    # the GPU's score gradient carries the bf16 bar; the backward is linear in it
    tol = 2 * parity.TOL[tag]
    if h.kind == "allpairs":
        for q in rng.choice(rows, 6, replace=False):
            gQ_o, _ = orc.allpairs_bwd(Qn[q:q + 1], Dn, gs_o[q:q + 1], am_g[q:q + 1], dtype=tag)
            assert parity.normwise_rel_err(gQ_g[q], gQ_o[0]) <= tol, f"grad_Q[{q}]"
        for d in rng.choice(h.nD, 6, replace=False):
            _, gD_o = orc.allpairs_bwd(Qn, Dn[d:d + 1], gs_o[:, d:d + 1], am_g[:, d:d + 1], dtype=tag)
            assert parity.normwise_rel_err(gD_g[d], gD_o[0]) <= tol, f"grad_D[{d}]"
    else:
        for b in rng.choice(rows, 8, replace=False):
            gQ_o, gD_o = orc.kd_bwd(Qn[b:b + 1], Dn[b:b + 1], gs_o[b:b + 1], am_g[b:b + 1], dtype=tag)
            assert parity.normwise_rel_err(gQ_g[b], gQ_o[0]) <= tol, f"grad_Q[{b}]"
            assert parity.normwise_rel_err(gD_g[b], gD_o[0]) <= tol, f"grad_D[{b}]"


def test_rerank_b512_ld8192_f16_full():
    _check_full_forward("rerank_b512_ld8192_f16")


def test_allpairs_q128_d4096_bf16_subset():
    """All 128 queries against a seeded subset of 256 of the 4096 documents
    (32 of them from the 410 shortened ones, the rest from the full ones):
    scores and argmax of the full-size launch against the oracle on that
    subset, 32768 pairs (about 1.1 TFLOP of fp64 oracle work)."""
    inp = generate("allpairs_q128_d4096_bf16", device="cuda")
    h = gpu_harness.Layout(inp)
    s_g, am_g = _gpu_scores_argmax(h, inp)
    s_g, am_g = s_g.cpu().numpy(), am_g.cpu().numpy()
    short = torch.nonzero(~inp.dmask[:, -1]).flatten().cpu().numpy()
    full = np.setdiff1d(np.arange(h.nD), short)
    assert len(short) == 410
    rng = np.random.default_rng(2)
    docs = np.sort(np.concatenate([rng.choice(short, 32, replace=False), rng.choice(full, 224, replace=False)]))
    Qn, tag = to_numpy(inp.Q)
    Dn, _ = to_numpy(inp.D[torch.as_tensor(docs, device=inp.D.device)])
    qm = inp.qmask.cpu().numpy()
    dm = inp.dmask.cpu().numpy()[docs]
    s_o, am_o, gap = oracle.get().allpairs_fwd(Qn, Dn, qm, dm, dtype=tag)
    parity.assert_scores_close(s_g[:, docs], s_o, "bf16")
    n = len(docs)
    Qw = parity.widen(inp.Q)
    Dw = parity.widen(inp.D[torch.as_tensor(docs, device=inp.D.device)])
    parity.assert_argmax_valid(am_g[:, docs].reshape(-1, h.Lq), am_o.reshape(-1, h.Lq), gap.reshape(-1, h.Lq),
                               Qw, Dw, lambda p: p // n, lambda p: p % n, dm)
