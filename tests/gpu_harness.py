"""Run one workload through the CUDA library (C ABI via the binding) and the
fp64 oracle, and compare them with the rules in ``parity.py``.

Inputs always come from the seeded generators; the oracle never receives a
value the CUDA library produced.  The backward is checked on the oracle's own
argmax, fed to both sides.  Where the GPU computes its own argmax inside a
call (autograd layers, recompute, loss-head steps), the inputs come from
``separated_case``: their argmax is unique, the GPU's must equal the
oracle's exactly, and the gradients are compared with the oracle's on every
run, with no condition.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import parity
from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300.workloads import Inputs, to_numpy


def _np_mask(m):
    return None if m is None else m.detach().cpu().numpy().astype(np.uint8)


class Layout:
    """Index maps and calls of one layout."""

    def __init__(self, inp: Inputs):
        self.inp = inp
        w = inp.workload
        self.kind = w.layout
        Q, D = inp.Q, inp.D
        self.nQ, self.Lq, self.dim = Q.shape
        if self.kind == "kd":
            self.B, self.N, self.Ld = D.shape[0], D.shape[1], D.shape[2]
            self.nD = self.B * self.N
            self.ppq = self.N
        else:
            self.nD, self.Ld = D.shape[0], D.shape[1]
            self.ppq = self.nD if self.kind == "allpairs" else 1
        self.n_pairs = self.nQ * self.ppq

    def query_of(self, p):
        return p // self.ppq

    def doc_of(self, p):
        return p % self.nD if self.kind == "allpairs" else p

    # ---- oracle ---------------------------------------------------------
    def oracle_fwd(self):
        Qn, tag = to_numpy(self.inp.Q)
        Dn, _ = to_numpy(self.inp.D)
        qm, dm = _np_mask(self.inp.qmask), _np_mask(self.inp.dmask)
        return getattr(oracle.get(), f"{self.kind}_fwd")(Qn, Dn, qm, dm, dtype=tag)

    def oracle_fwd_separated(self):
        """The oracle forward of inputs drawn by ``separated_case``, after
        checking what such inputs promise: every valid query token of a
        non-empty document has a best similarity more than GAP_EXACT above
        its second best.  The argmax is then unique, so the GPU must return
        exactly the oracle's and both backwards run on the same indices."""
        s, am, gap = self.oracle_fwd()
        live = am >= 0
        assert live.any(), "separated inputs with no live query token"
        assert float(gap[live].min()) > parity.GAP_EXACT, "inputs are not separated"
        return s, am, gap

    def oracle_bwd(self, grad_out, argmax):
        Qn, tag = to_numpy(self.inp.Q)
        Dn, _ = to_numpy(self.inp.D)
        return getattr(oracle.get(), f"{self.kind}_bwd")(Qn, Dn, grad_out, argmax, dtype=tag)

    # ---- GPU --------------------------------------------------------------
    def gpu_inputs(self, device="cuda"):
        i = self.inp
        mv = lambda t: None if t is None else t.to(device).contiguous()  # noqa: E731
        return mv(i.Q), mv(i.D), mv(i.qmask), mv(i.dmask)

    def gpu_fwd(self, with_argmax=True, device="cuda"):
        Q, D, qm, dm = self.gpu_inputs(device)
        shape = self.inp.workload.score_shape
        scores = torch.empty(shape, dtype=torch.float32, device=device)
        am = (torch.full((*shape, self.Lq), -7, dtype=torch.int32, device=device)
              if with_argmax else None)
        getattr(binding, f"lik_maxsim_{self.kind}_fwd")(Q, D, qm, dm, scores, am)
        binding.lik_check_device_error()
        return scores.cpu().numpy(), None if am is None else am.cpu().numpy()

    def gpu_bwd(self, grad_out, argmax, device="cuda", with_q=True, with_d=True):
        """fp32 gradients from the plain backward entry point (both in one
        call by default; a gradient not asked for comes back as None)."""
        Q, D, _, _ = self.gpu_inputs(device)
        g = torch.as_tensor(np.ascontiguousarray(grad_out), dtype=torch.float32).to(device)
        am = torch.as_tensor(np.ascontiguousarray(argmax), dtype=torch.int32).to(device)
        shape = self.inp.workload.score_shape
        g = g.reshape(shape)
        am = am.reshape(*shape, self.Lq)
        gQ = torch.full(Q.shape, float("nan"), dtype=torch.float32, device=device) if with_q else None
        gD = torch.full(D.shape, float("nan"), dtype=torch.float32, device=device) if with_d else None
        getattr(binding, f"lik_maxsim_{self.kind}_bwd")(Q, D, g, am, gQ, gD)
        binding.lik_check_device_error()
        return (None if gQ is None else gQ.cpu().numpy()), (None if gD is None else gD.cpu().numpy())

    def gpu_bwd_same_dtype(self, grad_out, argmax, device="cuda"):
        """Gradients from the entry points that write them in the inputs' dtype
        (outputs start as NaN, so an element the kernels skip shows up)."""
        Q, D, _, _ = self.gpu_inputs(device)
        g = torch.as_tensor(np.ascontiguousarray(grad_out), dtype=torch.float32).to(device)
        am = torch.as_tensor(np.ascontiguousarray(argmax), dtype=torch.int32).to(device)
        shape = self.inp.workload.score_shape
        g = g.reshape(shape)
        am = am.reshape(*shape, self.Lq)
        gQ = torch.full(Q.shape, float("nan"), dtype=Q.dtype, device=device)
        gD = torch.full(D.shape, float("nan"), dtype=D.dtype, device=device)
        getattr(binding, f"lik_maxsim_{self.kind}_bwd_same_dtype")(Q, D, g, am, gQ, gD)
        binding.lik_check_device_error()
        return gQ.float().cpu().numpy(), gD.float().cpu().numpy()

    # ---- comparisons ------------------------------------------------------
    def check_forward(self):
        s_o, am_o, gap = self.oracle_fwd()
        s_g, am_g = self.gpu_fwd()
        tag = self.inp.workload.dtype
        err = parity.assert_scores_close(s_g, s_o, tag)
        Qw = parity.widen(self.inp.Q)
        Dw = parity.widen(self.inp.D).reshape(self.nD, self.Ld, self.dim)
        dm = None if self.inp.dmask is None else self.inp.dmask.cpu().numpy().reshape(self.nD, self.Ld)
        near = parity.assert_argmax_valid(am_g.reshape(self.n_pairs, self.Lq),
                                          am_o.reshape(self.n_pairs, self.Lq),
                                          gap.reshape(self.n_pairs, self.Lq), Qw, Dw,
                                          self.query_of, self.doc_of, dm)
        # scores without the argmax output must be the same computation
        s_g2, _ = self.gpu_fwd(with_argmax=False)
        assert np.array_equal(s_g, s_g2), "scores depend on whether argmax is requested"
        return dict(score_err=err, near_ties=near, s_oracle=s_o, am_oracle=am_o, am_gpu=am_g)

    def check_backward(self, grad_out=None, am_oracle=None):
        if am_oracle is None:
            _, am_oracle, _ = self.oracle_fwd()
        if grad_out is None:
            grad_out = self.inp.grad_out.cpu().numpy().astype(np.float64)
        # both sides get the same fp32 upstream gradient
        g32 = np.asarray(grad_out, np.float32).astype(np.float64)
        gQ_o, gD_o = self.oracle_bwd(g32, am_oracle)
        gQ_g, gD_g = self.gpu_bwd(g32, am_oracle)
        tag = self.inp.workload.dtype
        eq = parity.assert_grad_close(gQ_g, gQ_o, tag, "grad_Q")
        ed = parity.assert_grad_close(gD_g, gD_o, tag, "grad_D")
        return dict(grad_q_err=eq, grad_d_err=ed)

    def check_backward_single(self, am_oracle):
        """Each gradient requested alone (one launch each, not the launch that
        writes both) against the oracle."""
        g32 = np.asarray(self.inp.grad_out.cpu().numpy(), np.float32).astype(np.float64)
        gQ_o, gD_o = self.oracle_bwd(g32, am_oracle)
        tag = self.inp.workload.dtype
        gQ_g, none_d = self.gpu_bwd(g32, am_oracle, with_d=False)
        none_q, gD_g = self.gpu_bwd(g32, am_oracle, with_q=False)
        assert none_d is None and none_q is None
        return dict(grad_q_err=parity.assert_grad_close(gQ_g, gQ_o, tag, "grad_Q"),
                    grad_d_err=parity.assert_grad_close(gD_g, gD_o, tag, "grad_D"))

    def check_backward_same_dtype(self, am_oracle):
        """Same-dtype gradients against the oracle: the bar plus one rounding to
        the output type (2^-8 relative for bf16, 2^-11 for fp16)."""
        g32 = np.asarray(self.inp.grad_out.cpu().numpy(), np.float32).astype(np.float64)
        gQ_o, gD_o = self.oracle_bwd(g32, am_oracle)
        gQ_g, gD_g = self.gpu_bwd_same_dtype(g32, am_oracle)
        tag = self.inp.workload.dtype
        tol = parity.TOL[tag] + {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 0.0}[tag]
        out = {}
        for got, ref, name in ((gQ_g, gQ_o, "grad_Q"), (gD_g, gD_o, "grad_D")):
            assert np.isfinite(got).all(), f"{name}: an element was not written"
            err = parity.normwise_rel_err(got, ref)
            assert err <= tol, f"{name}: normwise relative error {err:.3g} > {tol:.3g}"
            out[name] = err
        return out
