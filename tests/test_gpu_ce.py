"""Cross-entropy loss head (GPU) against the fp64 oracle.

lik_ce_rows computes the mean softmax cross-entropy over score rows in fp32;
its scores are given to both sides, so the fp32 bar (1e-5) applies.  The
one-call steps (forward, loss, backward) start from embeddings: their scores
carry the input dtype's error, so the loss and the score gradient are held to
the fp16/bf16 bar.  Their inputs come from ``separated_case`` (a unique
argmax), so the step's own argmax must be the oracle's and the Q/D gradients
are compared with the oracle's on every run.
"""
import numpy as np
import pytest
import torch

import gpu_harness
import oracle
import parity
from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300.workloads import separated_case

pytestmark = pytest.mark.gpu


def _ce_gpu(S, t, scale, with_grad=True):
    dev = "cuda"
    s = torch.as_tensor(S, dtype=torch.float32, device=dev).contiguous()
    tt = torch.as_tensor(t, dtype=torch.int32, device=dev).contiguous()
    loss = torch.full((1,), float("nan"), device=dev)
    rl = torch.full((S.shape[0],), float("nan"), device=dev)
    g = torch.full(S.shape, float("nan"), device=dev) if with_grad else None
    binding.lik_ce_rows(s, tt, loss, rl, g, scale=scale)
    torch.cuda.synchronize()
    return loss.item(), rl.cpu().numpy(), None if g is None else g.cpu().numpy()


@pytest.mark.parametrize("rows,cols,scale", [(5, 7, 1.0), (128, 128, 1.0), (256, 17, 2.5), (3, 4096, 0.7),
                                             (1, 1, 1.0)])
def test_ce_rows_matches_oracle(rows, cols, scale):
    rng = np.random.default_rng(rows * 1000 + cols)
    S = (rng.standard_normal((rows, cols)) * 4).astype(np.float32)
    if cols > 2:
        S[rng.random((rows, cols)) < 0.1] = -1e9  # empty documents
    t = rng.integers(0, cols, size=rows).astype(np.int32)
    if rows > 2:
        t[1] = cols + 3  # a row left out
    loss_o, rl_o, g_o = oracle.get().ce_rows(S.astype(np.float64), t, scale)
    loss_g, rl_g, g_g = _ce_gpu(S, t, scale)
    assert abs(loss_g - loss_o) <= 1e-5 * max(abs(loss_o), 1.0)
    assert parity.normwise_rel_err(rl_g, rl_o) <= 1e-5
    assert parity.normwise_rel_err(g_g, g_o) <= 1e-5
    # the mean is summed in a fixed order
    assert _ce_gpu(S, t, scale)[0] == loss_g


def test_ce_rows_without_gradient_and_empty():
    S = np.zeros((0, 4), np.float32)
    loss, rl, _ = _ce_gpu(S, np.zeros(0, np.int32), 1.0, with_grad=False)
    assert loss == 0.0 and rl.shape == (0,)
    S = np.array([[0.5, 0.5]], np.float32)
    loss, rl, _ = _ce_gpu(S, np.array([1], np.int32), 1.0, with_grad=False)
    assert abs(loss - np.log(2)) < 1e-6


@pytest.mark.parametrize("grads", ["f32", "input"])
@pytest.mark.parametrize("layout,nq,nd,lq,ld,dim", [("allpairs", 6, 6, 32, 260, 128), ("allpairs", 9, 9, 16, 300, 64),
                                                    ("kd", 4, 5, 32, 200, 128),
                                                    # 4096 score rows: the most the one-launch backward takes,
                                                    # its loss block summing all of them
                                                    ("kd", 4096, 2, 4, 24, 64),
                                                    # more than 4096 score rows: the head in two backward launches
                                                    ("kd", 4100, 2, 4, 24, 64)])
def test_ce_step_matches_oracle(layout, nq, nd, lq, ld, dim, grads):
    inp = separated_case(layout, nq, nd, lq, ld, dim, "bf16", seed=nq * 7 + nd, p_doc_empty=0.0)
    h = gpu_harness.Layout(inp)
    rows, cols = (nq, nd)
    target = np.arange(rows, dtype=np.int32) % cols if layout == "allpairs" else np.zeros(rows, np.int32)
    # oracle: forward, loss, backward on its own scores and argmax
    s_o, am_o, _ = h.oracle_fwd_separated()
    scale = 1.5
    loss_o, rl_o, gs_o = oracle.get().ce_rows(s_o.reshape(rows, cols), target, scale)
    gQ_o, gD_o = h.oracle_bwd(gs_o.reshape(-1), am_o)
    # GPU: one call
    Q, D, qm, dm = h.gpu_inputs()
    dev = "cuda"
    scores = torch.empty(rows, cols, device=dev)
    am = torch.empty(rows, cols, lq, dtype=torch.int32, device=dev)
    loss = torch.empty(1, device=dev)
    rl = torch.empty(rows, device=dev)
    gs = torch.empty(rows, cols, device=dev)
    gdt = Q.dtype if grads == "input" else torch.float32
    gQ = torch.empty(Q.shape, dtype=gdt, device=dev)
    gD = torch.empty(D.shape, dtype=gdt, device=dev)
    tt = torch.as_tensor(target, device=dev)
    getattr(binding, f"lik_maxsim_{layout}_ce_step")(Q, D, qm, dm, tt, scores, am, loss, rl, gs, gQ, gD, scale=scale)
    binding.lik_check_device_error()
    parity.assert_scores_close(scores.cpu().numpy(), s_o.reshape(rows, cols), "bf16")
    assert abs(loss.item() - loss_o) <= parity.TOL["bf16"] * max(abs(loss_o), 1.0)
    assert parity.normwise_rel_err(gs.cpu().numpy(), gs_o) <= parity.TOL["bf16"]
    assert np.array_equal(am.cpu().numpy().reshape(am_o.shape), am_o), "argmax differs on separated inputs"
    extra = 2.0 ** -8 if grads == "input" else 0.0
    # the GPU's score gradient carries the bf16 bar; the backward is linear in it
    tol = 2 * parity.TOL["bf16"] + extra
    assert parity.normwise_rel_err(gQ.float().cpu().numpy(), gQ_o) <= tol
    assert parity.normwise_rel_err(gD.float().cpu().numpy(), gD_o) <= tol


@pytest.mark.parametrize("grads", ["f32", "input"])
@pytest.mark.parametrize("layout,nq,nd,lq,ld,dim,dtype", [("allpairs", 6, 6, 32, 260, 128, "bf16"),
                                                          ("kd", 4, 5, 32, 200, 128, "bf16"),
                                                          ("allpairs", 5, 9, 20, 100, 64, "bf16"),
                                                          ("allpairs", 4, 7, 16, 90, 64, "f32"),
                                                          ("kd", 3, 6, 12, 70, 32, "f16")])
def test_ce_step_head_inside_backward(layout, nq, nd, lq, ld, dim, dtype, grads):
    """With both gradients requested, the one-call step computes the loss head
    inside the backward: with fp32 gradients in its one launch (the score
    gradient in the blocks that use it, the row losses and their mean in one
    more block), with gradients in the inputs' dtype in the grad_Q launch (the
    mean in the grad_D launch).  Its loss, row losses and score
    gradient must agree with the separate head (lik_ce_rows) on the step's own
    scores, the loss must be bit-identical from call to call (fixed summation
    order), and the steps without grad_Q or without grad_D (separate head) must
    give the same loss and gradients."""
    inp = separated_case(layout, nq, nd, lq, ld, dim, dtype, seed=nq * 13 + nd, p_doc_empty=0.0)
    h = gpu_harness.Layout(inp)
    rows, cols = nq, nd
    target = np.arange(rows, dtype=np.int32) % cols if layout == "allpairs" else np.zeros(rows, np.int32)
    target[0] = cols + 1  # a row left out of the loss
    Q, D, qm, dm = h.gpu_inputs()
    dev = "cuda"
    gdt = Q.dtype if grads == "input" else torch.float32
    tt = torch.as_tensor(target, device=dev)
    step = getattr(binding, f"lik_maxsim_{layout}_ce_step")

    def run(with_q=True, with_d=True):
        out = dict(scores=torch.empty(rows, cols, device=dev), am=torch.empty(rows, cols, lq, dtype=torch.int32, device=dev),
                   loss=torch.empty(1, device=dev), rl=torch.empty(rows, device=dev), gs=torch.empty(rows, cols, device=dev),
                   gQ=torch.empty(Q.shape, dtype=gdt, device=dev) if with_q else None,
                   gD=torch.empty(D.shape, dtype=gdt, device=dev) if with_d else None)
        step(Q, D, qm, dm, tt, out["scores"], out["am"], out["loss"], out["rl"], out["gs"], out["gQ"], out["gD"],
             scale=1.3)
        binding.lik_check_device_error()
        return out

    a, b, c, d = run(), run(), run(with_q=False), run(with_d=False)
    assert a["loss"].item() == b["loss"].item()
    loss = torch.empty(1, device=dev)
    rl = torch.empty(rows, device=dev)
    gs = torch.empty(rows, cols, device=dev)
    binding.lik_ce_rows(a["scores"], tt, loss, rl, gs, scale=1.3)
    torch.cuda.synchronize()
    assert abs(a["loss"].item() - loss.item()) <= 1e-6 * max(1.0, abs(loss.item()))
    assert parity.normwise_rel_err(a["rl"].cpu().numpy(), rl.cpu().numpy()) <= 1e-6
    assert parity.normwise_rel_err(a["gs"].cpu().numpy(), gs.cpu().numpy()) <= 1e-6
    assert float(a["rl"][0]) == 0.0 and torch.all(a["gs"][0] == 0)
    # the separate-head paths (no grad_Q, or no grad_D) give the same loss and gradients
    assert parity.normwise_rel_err(c["gD"].float().cpu().numpy(), a["gD"].float().cpu().numpy()) <= 1e-5
    assert parity.normwise_rel_err(d["gQ"].float().cpu().numpy(), a["gQ"].float().cpu().numpy()) <= 1e-5
    for other in (c, d):
        assert abs(other["loss"].item() - a["loss"].item()) <= 1e-6 * max(1.0, abs(a["loss"].item()))


def test_one_call_step_repeats_bit_for_bit():
    """Repeated one-call steps on the same inputs: scores, argmax, loss, row
    losses, score gradient and grad_Q are bit-identical (fixed summation
    orders); grad_D, whose hits arrive as fp32 atomic additions, agrees to
    rounding."""
    inp = separated_case("allpairs", 12, 12, 32, 420, 128, "bf16", seed=5, p_doc_empty=0.1)
    h = gpu_harness.Layout(inp)
    Q, D, qm, dm = h.gpu_inputs()
    dev = "cuda"
    rows = cols = 12
    tt = torch.arange(rows, dtype=torch.int32, device=dev)

    def run():
        out = dict(scores=torch.empty(rows, cols, device=dev),
                   am=torch.empty(rows, cols, 32, dtype=torch.int32, device=dev),
                   loss=torch.empty(1, device=dev), rl=torch.empty(rows, device=dev),
                   gs=torch.empty(rows, cols, device=dev), gQ=torch.empty(Q.shape, device=dev),
                   gD=torch.empty(D.shape, device=dev))
        binding.lik_maxsim_allpairs_ce_step(Q, D, qm, dm, tt, out["scores"], out["am"], out["loss"], out["rl"],
                                            out["gs"], out["gQ"], out["gD"])
        binding.lik_check_device_error()
        return out

    a = run()
    for _ in range(2):
        b = run()
        for k in ("scores", "am", "loss", "rl", "gs", "gQ"):
            assert torch.equal(a[k], b[k]), k
        assert parity.normwise_rel_err(b["gD"].cpu().numpy(), a["gD"].cpu().numpy()) <= 1e-6
