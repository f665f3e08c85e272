"""Backward that recomputes the argmax (GPU): the argmax-free training forward.

lik_maxsim_*_bwd_recompute re-runs the forward into a workspace and then runs
the backward.  The workspace must hold exactly the argmax the forward writes
(the kernels are deterministic), the gradients must equal the stored-argmax
backward's, and the oracle's: the inputs come from ``separated_case``, whose
argmax is unique, so the recomputed argmax must be the oracle's and the
gradients are compared with the oracle's on every run.
"""
import zlib

import numpy as np
import pytest
import torch

import gpu_harness
import parity
from late_interaction_retrieval_gb300 import binding, layers
from late_interaction_retrieval_gb300.workloads import random_case, separated_case

pytestmark = pytest.mark.gpu

CASES = [
    ("allpairs", 5, 7, 32, 257, 128, "bf16"),
    ("allpairs", 3, 4, 8, 64, 64, "f32"),
    ("pairwise", 6, 0, 32, 700, 128, "f16"),
    ("kd", 3, 5, 32, 260, 128, "bf16"),
    ("kd", 2, 3, 6, 40, 64, "f32"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_recompute_matches_stored_argmax(case):
    layout, nq, nd, lq, ld, dim, dtype = case
    inp = separated_case(layout, nq, nd, lq, ld, dim, dtype, seed=zlib.crc32(repr(case).encode()) % 10_000,
                         p_doc_empty=0.15)
    h = gpu_harness.Layout(inp)
    s_o, am_o, _ = h.oracle_fwd_separated()
    _, am_gpu = h.gpu_fwd()
    g = inp.grad_out.cpu().numpy().astype(np.float64)
    gQ_ref, gD_ref = h.gpu_bwd(g, am_gpu)

    Q, D, qm, dm = h.gpu_inputs()
    shape = inp.workload.score_shape
    ws = torch.full((*shape, lq), -7, dtype=torch.int32, device="cuda")
    gQ = torch.full(Q.shape, float("nan"), device="cuda")
    gD = torch.full(D.shape, float("nan"), device="cuda")
    gg = torch.as_tensor(g, dtype=torch.float32, device="cuda").reshape(shape)
    getattr(binding, f"lik_maxsim_{layout}_bwd_recompute")(Q, D, qm, dm, gg, ws, gQ, gD)
    binding.lik_check_device_error()
    assert np.array_equal(ws.cpu().numpy(), am_gpu)
    assert np.array_equal(gQ.cpu().numpy(), gQ_ref)       # fixed summation order
    assert parity.normwise_rel_err(gD.cpu().numpy(), gD_ref) <= 1e-6  # fp32 atomics, any order
    assert np.array_equal(ws.cpu().numpy().reshape(am_o.shape), am_o), "recomputed argmax is not the oracle's"
    gQ_o, gD_o = h.oracle_bwd(np.asarray(g, np.float32).astype(np.float64), am_o)
    parity.assert_grad_close(gQ.cpu().numpy(), gQ_o, dtype, "grad_Q")
    parity.assert_grad_close(gD.cpu().numpy(), gD_o, dtype, "grad_D")


@pytest.mark.parametrize("layout", ["allpairs", "pairwise", "kd"])
def test_recompute_degenerate_lengths(layout):
    for lq, ld in ((0, 9), (5, 0)):
        inp = random_case(layout, 3, 2, lq, ld, 32, "bf16", seed=lq + 3 * ld)
        h = gpu_harness.Layout(inp)
        Q, D, qm, dm = h.gpu_inputs()
        shape = inp.workload.score_shape
        ws = torch.empty((*shape, lq), dtype=torch.int32, device="cuda")
        gQ = torch.full(Q.shape, float("nan"), device="cuda")
        gD = torch.full(D.shape, float("nan"), device="cuda")
        gg = torch.ones(shape, device="cuda")
        getattr(binding, f"lik_maxsim_{layout}_bwd_recompute")(Q, D, qm, dm, gg, ws, gQ, gD)
        binding.lik_check_device_error()
        assert torch.all(gQ == 0) and torch.all(gD == 0)


@pytest.mark.parametrize("layout", ["allpairs", "kd"])
def test_recompute_layers_match_default(layout):
    inp = random_case(layout, 4, 5, 32, 150, 128, "bf16", seed=31)
    h = gpu_harness.Layout(inp)
    Q, D, qm, dm = h.gpu_inputs()
    fn = layers.maxsim if layout == "allpairs" else layers.maxsim_kd
    grads = []
    for recompute in (False, True):
        q = Q.clone().requires_grad_(True)
        d = D.clone().requires_grad_(True)
        s = fn(q, d, qm, dm, recompute=recompute)
        s.backward(inp.grad_out.cuda())
        grads.append((s.detach(), q.grad.float(), d.grad.float()))
    (s0, q0, d0), (s1, q1, d1) = grads
    assert torch.equal(s0, s1)
    # the default path writes bf16 gradients directly; the recompute path casts fp32 ones
    assert parity.normwise_rel_err(q1.cpu().numpy(), q0.cpu().numpy()) <= 2.0 ** -7
    assert parity.normwise_rel_err(d1.cpu().numpy(), d0.cpu().numpy()) <= 2.0 ** -7
