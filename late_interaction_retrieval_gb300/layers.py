"""Autograd layers over liblik: MaxSim, MaxSimPairwise, MaxSimKD.

Call shapes follow the Late Interaction Kernels README ("Scoring interface"
table) and, for the per-query candidate layout, the colpali PR "Add support
for late-interaction-kernels (LIK)" (Design section):

  MaxSim          Q [Nq, Lq, dim], D [Nd, Ld, dim]     -> [Nq, Nd]
  MaxSimPairwise  Q [B, Lq, dim],  D [B, Ld, dim]      -> [B]
  MaxSimKD        Q [B, Lq, dim],  D [B, N, Ld, dim]   -> [B, N]

Masks are bool, True = valid, or None.  Scores are fp32.  The forward saves
only the int32 argmax [pairs, Lq] (linear in the number of pairs; no
[pairs, Lq, Ld] similarity grid exists anywhere).  For fp16/bf16 inputs with
dim % 8 == 0 and dim <= 256 the backward asks liblik for gradients in the
input dtype directly (summed in fp32, rounded once); otherwise it asks for
fp32 gradients and casts them.  This module only allocates tensors and calls
the binding.  With recompute=True the forward saves no argmax: the
backward re-runs the forward into a transient workspace.
"""
from __future__ import annotations

import torch

from . import binding


def _contig(t):
    return None if t is None else t.contiguous()


def _score_shape(kind, Q, D):
    if kind == "allpairs":
        return (Q.shape[0], D.shape[0])
    if kind == "pairwise":
        return (Q.shape[0],)
    return (Q.shape[0], D.shape[1])


class _MaxSimFn(torch.autograd.Function):
    """MaxSim of layout `kind`.  With `recompute`, the forward keeps only the
    scores (and the inputs it already needs); the backward re-runs the
    forward into a transient argmax workspace (lik_maxsim_*_bwd_recompute)."""

    @staticmethod
    def forward(ctx, kind, recompute, Q, D, qmask, dmask):
        Q, D, qmask, dmask = Q.contiguous(), D.contiguous(), _contig(qmask), _contig(dmask)
        Lq = Q.shape[1]
        shape = _score_shape(kind, Q, D)
        scores = torch.empty(shape, dtype=torch.float32, device=Q.device)
        need = ctx.needs_input_grad[2] or ctx.needs_input_grad[3]
        argmax = (torch.empty((*shape, Lq), dtype=torch.int32, device=Q.device)
                  if need and not recompute else None)
        getattr(binding, f"lik_maxsim_{kind}_fwd")(Q, D, qmask, dmask, scores, argmax)
        ctx.kind, ctx.recompute = kind, recompute
        if recompute:
            ctx.save_for_backward(Q, D, qmask, dmask)
        else:
            ctx.save_for_backward(Q, D, argmax)
        return scores

    @staticmethod
    def backward(ctx, g):
        kind = ctx.kind
        g = g.contiguous().float()
        want_q, want_d = ctx.needs_input_grad[2], ctx.needs_input_grad[3]
        if ctx.recompute:
            Q, D, qmask, dmask = ctx.saved_tensors
            ws = torch.empty((*_score_shape(kind, Q, D), Q.shape[1]), dtype=torch.int32, device=Q.device)
            gQ = torch.empty(Q.shape, dtype=torch.float32, device=Q.device) if want_q else None
            gD = torch.empty(D.shape, dtype=torch.float32, device=D.device) if want_d else None
            getattr(binding, f"lik_maxsim_{kind}_bwd_recompute")(Q, D, qmask, dmask, g, ws, gQ, gD)
        else:
            Q, D, argmax = ctx.saved_tensors
            same = Q.dtype != torch.float32 and Q.shape[-1] % 8 == 0 and Q.shape[-1] <= 256
            gdt = Q.dtype if same else torch.float32
            gQ = torch.empty(Q.shape, dtype=gdt, device=Q.device) if want_q else None
            gD = torch.empty(D.shape, dtype=gdt, device=D.device) if want_d else None
            getattr(binding, f"lik_maxsim_{kind}_bwd" + ("_same_dtype" if same else ""))(Q, D, g, argmax, gQ, gD)
        return (None, None, None if gQ is None else gQ.to(Q.dtype), None if gD is None else gD.to(D.dtype),
                None, None)


def maxsim(Q, D, qmask=None, dmask=None, recompute=False):
    """All-pairs MaxSim scores [Nq, Nd] (fp32), differentiable in Q and D.
    recompute=True keeps no argmax between forward and backward."""
    return _MaxSimFn.apply("allpairs", recompute, Q, D, qmask, dmask)


def maxsim_pairwise(Q, D, qmask=None, dmask=None, recompute=False):
    """Pairwise MaxSim scores [B] (fp32), differentiable in Q and D."""
    return _MaxSimFn.apply("pairwise", recompute, Q, D, qmask, dmask)


def maxsim_kd(Q, D, qmask=None, dmask=None, recompute=False):
    """Per-query candidate MaxSim scores [B, N] (fp32), differentiable in Q and D."""
    return _MaxSimFn.apply("kd", recompute, Q, D, qmask, dmask)


class MaxSim(torch.nn.Module):
    def __init__(self, recompute: bool = False):
        super().__init__()
        self.recompute = recompute

    def forward(self, Q, D, qmask=None, dmask=None):
        return maxsim(Q, D, qmask, dmask, self.recompute)


class MaxSimPairwise(torch.nn.Module):
    def __init__(self, recompute: bool = False):
        super().__init__()
        self.recompute = recompute

    def forward(self, Q, D, qmask=None, dmask=None):
        return maxsim_pairwise(Q, D, qmask, dmask, self.recompute)


class MaxSimKD(torch.nn.Module):
    def __init__(self, recompute: bool = False):
        super().__init__()
        self.recompute = recompute

    def forward(self, Q, D, qmask=None, dmask=None):
        return maxsim_kd(Q, D, qmask, dmask, self.recompute)
