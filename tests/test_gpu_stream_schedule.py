"""Streaming forward (pairwise, kd) with documents cut between CTAs (GPU).

The streaming kernel spreads the tiles of all pairs evenly over the CTAs, so a
long document may be split between several CTAs; each piece leaves its
per-query-token (max, argmax) in a workspace and the last piece to finish
merges them.  These cases force cuts: a few pairs with long documents (each
spread over dozens of CTAs), mixes of empty, one-tile and long documents, no
document mask (every tile visited), more CTAs than tiles, and exact ties whose
two tokens fall in different pieces.  The oracle is the same fp64 triple loop
as everywhere else; exact ties go to the lowest token index.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gpu_harness
import parity
from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300.workloads import random_case

pytestmark = pytest.mark.gpu

CUT_CASES = [
    # layout, nq, nd (N for kd), Lq, Ld, dim, dtype, p_doc_empty, min_dlen
    ("pairwise", 2, 2, 32, 20000, 128, "bf16", 0.0, 15000),   # 2 documents over every CTA
    ("pairwise", 5, 5, 17, 3000, 64, "f16", 0.2, 1),
    ("pairwise", 1, 1, 32, 300, 128, "bf16", 0.0, 300),       # fewer tiles (3) than CTAs
    ("kd", 3, 5, 32, 2500, 128, "bf16", 0.3, 1),
    ("kd", 40, 3, 8, 130, 32, "bf16", 0.3, 1),                # many one- and two-tile pairs
    ("kd", 2, 2, 32, 9000, 256, "f16", 0.25, 1),
]


@pytest.mark.parametrize("case", CUT_CASES, ids=lambda c: "-".join(map(str, c[:7])))
def test_cut_documents_match_oracle(case):
    layout, nq, nd, lq, ld, dim, dtype, p_empty, min_dlen = case
    inp = random_case(layout, nq, nd, lq, ld, dim, dtype, seed=ld + nq, p_doc_empty=p_empty,
                      min_dlen=min_dlen)
    gpu_harness.Layout(inp).check_forward()


@pytest.mark.parametrize("layout,nq,nd,ld", [("pairwise", 3, 3, 5000), ("kd", 2, 4, 1100)])
def test_cut_documents_without_document_mask(layout, nq, nd, ld):
    inp = random_case(layout, nq, nd, 32, ld, 128, "bf16", seed=11)
    inp = dataclasses.replace(inp, dmask=None)
    gpu_harness.Layout(inp).check_forward()


def _tied_case(layout, nq, nd, ld, half, seed):
    """Documents whose tokens [half, 2*half) repeat tokens [0, half) exactly,
    all valid, so every query token's maximum is reached twice."""
    inp = random_case(layout, nq, nd, 32, ld, 128, "bf16", seed=seed, p_query_tail=0.0)
    D = inp.D.clone()
    D[..., half:2 * half, :] = D[..., :half, :]
    dmask = torch.zeros_like(inp.dmask)
    dmask[..., :2 * half] = True
    return dataclasses.replace(inp, D=D, dmask=dmask)


@pytest.mark.parametrize("layout,nq,nd,ld,half", [
    ("pairwise", 2, 2, 12000, 6000),   # the two copies 6000 tokens apart: other pieces, other lanes
    ("pairwise", 3, 3, 700, 300),
    ("kd", 2, 3, 600, 256),            # same TMEM lane, other tiles
])
def test_exact_ties_across_pieces_take_the_lowest_index(layout, nq, nd, ld, half):
    inp = _tied_case(layout, nq, nd, ld, half, seed=half)
    h = gpu_harness.Layout(inp)
    s_o, am_o, _ = h.oracle_fwd()
    s_g, am_g = h.gpu_fwd()
    parity.assert_scores_close(s_g, s_o, "bf16")
    am_o = am_o.reshape(h.n_pairs, h.Lq)
    am_g = am_g.reshape(h.n_pairs, h.Lq)
    assert (am_o < half).all()  # the oracle takes the first copy
    # where the best token of the first half leads the runner-up of the first
    # half by more than the argmax bar, the answer is unique up to the copy
    Qw = parity.widen(inp.Q)
    Dw = parity.widen(inp.D).reshape(h.nD, h.Ld, h.dim)[:, :half]
    for p in range(h.n_pairs):
        sims = Qw[h.query_of(p)] @ Dw[h.doc_of(p)].T
        top2 = np.sort(sims, axis=1)[:, -2:]
        sure = (top2[:, 1] - top2[:, 0]) > parity.GAP_EXACT
        assert np.array_equal(am_g[p][sure], am_o[p][sure]), f"pair {p}: {am_g[p][sure]} vs {am_o[p][sure]}"


def test_repeat_calls_are_bitwise_identical():
    inp = random_case("pairwise", 4, 4, 32, 9000, 128, "f16", seed=5)
    h = gpu_harness.Layout(inp)
    s1, a1 = h.gpu_fwd()
    s2, a2 = h.gpu_fwd()
    assert np.array_equal(s1, s2) and np.array_equal(a1, a2)


def test_cut_documents_on_two_streams_at_once():
    """Two streaming calls in flight together each get their own workspace."""
    layouts = [gpu_harness.Layout(random_case("pairwise", 3, 3, 32, 8000, 128, "bf16", seed=21)),
               gpu_harness.Layout(random_case("kd", 2, 3, 32, 4000, 128, "bf16", seed=22))]
    alone = [h.gpu_fwd() for h in layouts]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    bufs = []
    for h in layouts:
        shape = h.inp.workload.score_shape
        bufs.append((torch.empty(shape, device="cuda"),
                     torch.empty((*shape, h.Lq), dtype=torch.int32, device="cuda"), *h.gpu_inputs()))
    torch.cuda.synchronize()
    for _ in range(4):
        for h, st, (s, am, Q, D, qm, dm) in zip(layouts, streams, bufs):
            with torch.cuda.stream(st):
                getattr(binding, f"lik_maxsim_{h.kind}_fwd")(Q, D, qm, dm, s, am, stream=st)
    torch.cuda.synchronize()
    binding.lik_check_device_error()
    for (s_a, am_a), (s, am, *_rest) in zip(alone, bufs):
        assert np.array_equal(s.cpu().numpy(), s_a)
        assert np.array_equal(am.cpu().numpy(), am_a)


@pytest.mark.parametrize("layout,nq,nd,ld", [("pairwise", 10, 10, 1030), ("pairwise", 6, 6, 5000),
                                             ("kd", 2, 5, 1031)])
def test_scattered_document_masks(layout, nq, nd, ld):
    """Masks that are not prefixes: Bernoulli tokens, a document valid only at
    its first token, only at its last, at one token in the middle, and empty
    (rows of odd length start at every alignment, so the plan's scan meets
    every head and tail case)."""
    inp = random_case(layout, nq, nd, 32, ld, 128, "bf16", seed=ld + 7)
    g = torch.Generator().manual_seed(ld)
    dm = (torch.rand(inp.dmask.shape, generator=g) < 0.3)
    flat = dm.view(-1, ld)
    special = [lambda r: r.zero_().__setitem__(0, True), lambda r: r.zero_().__setitem__(ld - 1, True),
               lambda r: r.zero_().__setitem__(ld // 2, True), lambda r: r.zero_()]
    for k, f in enumerate(special):
        f(flat[k])
    gpu_harness.Layout(dataclasses.replace(inp, dmask=dm)).check_forward()


def test_more_than_256_groups_of_pairs():
    """Over 8192 pairs: the range search reads the per-group unit sums in
    several passes."""
    inp = random_case("kd", 300, 31, 16, 40, 64, "bf16", seed=31, p_doc_empty=0.1)
    assert inp.D.shape[0] * inp.D.shape[1] > 32 * 256
    gpu_harness.Layout(inp).check_forward()


def test_fewer_units_than_ctas():
    """Long padded rows with short documents: every pair has one unit, so
    there are fewer units than CTAs and some CTAs get nothing."""
    inp = random_case("pairwise", 100, 100, 32, 1000, 128, "bf16", seed=41, p_doc_empty=0.1)
    dm = inp.dmask.clone()
    dm[:, 64:] = False
    gpu_harness.Layout(dataclasses.replace(inp, dmask=dm)).check_forward()
