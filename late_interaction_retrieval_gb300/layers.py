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
the binding.
"""
from __future__ import annotations

import torch

from . import binding


def _contig(t):
    return None if t is None else t.contiguous()


def _backward(kind, ctx, g):
    """Gradients of Q and D for layout `kind` from the saved argmax."""
    Q, D, argmax = ctx.saved_tensors
    same = Q.dtype != torch.float32 and Q.shape[-1] % 8 == 0 and Q.shape[-1] <= 256
    gdt = Q.dtype if same else torch.float32
    gQ = torch.empty(Q.shape, dtype=gdt, device=Q.device) if ctx.needs_input_grad[0] else None
    gD = torch.empty(D.shape, dtype=gdt, device=D.device) if ctx.needs_input_grad[1] else None
    fn = getattr(binding, f"lik_maxsim_{kind}_bwd" + ("_same_dtype" if same else ""))
    fn(Q, D, g.contiguous().float(), argmax, gQ, gD)
    return (None if gQ is None else gQ.to(Q.dtype), None if gD is None else gD.to(D.dtype), None, None)


class _MaxSimFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Q, D, qmask, dmask):
        Q, D, qmask, dmask = Q.contiguous(), D.contiguous(), _contig(qmask), _contig(dmask)
        Nq, Lq, _ = Q.shape
        Nd = D.shape[0]
        scores = torch.empty((Nq, Nd), dtype=torch.float32, device=Q.device)
        need = ctx.needs_input_grad[0] or ctx.needs_input_grad[1]
        argmax = torch.empty((Nq, Nd, Lq), dtype=torch.int32, device=Q.device) if need else None
        binding.lik_maxsim_allpairs_fwd(Q, D, qmask, dmask, scores, argmax)
        ctx.save_for_backward(Q, D, argmax)
        return scores

    @staticmethod
    def backward(ctx, g):
        return _backward("allpairs", ctx, g)


class _MaxSimPairwiseFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Q, D, qmask, dmask):
        Q, D, qmask, dmask = Q.contiguous(), D.contiguous(), _contig(qmask), _contig(dmask)
        B, Lq, _ = Q.shape
        scores = torch.empty((B,), dtype=torch.float32, device=Q.device)
        need = ctx.needs_input_grad[0] or ctx.needs_input_grad[1]
        argmax = torch.empty((B, Lq), dtype=torch.int32, device=Q.device) if need else None
        binding.lik_maxsim_pairwise_fwd(Q, D, qmask, dmask, scores, argmax)
        ctx.save_for_backward(Q, D, argmax)
        return scores

    @staticmethod
    def backward(ctx, g):
        return _backward("pairwise", ctx, g)


class _MaxSimKDFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Q, D, qmask, dmask):
        Q, D, qmask, dmask = Q.contiguous(), D.contiguous(), _contig(qmask), _contig(dmask)
        B, Lq, _ = Q.shape
        N = D.shape[1]
        scores = torch.empty((B, N), dtype=torch.float32, device=Q.device)
        need = ctx.needs_input_grad[0] or ctx.needs_input_grad[1]
        argmax = torch.empty((B, N, Lq), dtype=torch.int32, device=Q.device) if need else None
        binding.lik_maxsim_kd_fwd(Q, D, qmask, dmask, scores, argmax)
        ctx.save_for_backward(Q, D, argmax)
        return scores

    @staticmethod
    def backward(ctx, g):
        return _backward("kd", ctx, g)


def maxsim(Q, D, qmask=None, dmask=None):
    """All-pairs MaxSim scores [Nq, Nd] (fp32), differentiable in Q and D."""
    return _MaxSimFn.apply(Q, D, qmask, dmask)


def maxsim_pairwise(Q, D, qmask=None, dmask=None):
    """Pairwise MaxSim scores [B] (fp32), differentiable in Q and D."""
    return _MaxSimPairwiseFn.apply(Q, D, qmask, dmask)


def maxsim_kd(Q, D, qmask=None, dmask=None):
    """Per-query candidate MaxSim scores [B, N] (fp32), differentiable in Q and D."""
    return _MaxSimKDFn.apply(Q, D, qmask, dmask)


class MaxSim(torch.nn.Module):
    def forward(self, Q, D, qmask=None, dmask=None):
        return maxsim(Q, D, qmask, dmask)


class MaxSimPairwise(torch.nn.Module):
    def forward(self, Q, D, qmask=None, dmask=None):
        return maxsim_pairwise(Q, D, qmask, dmask)


class MaxSimKD(torch.nn.Module):
    def forward(self, Q, D, qmask=None, dmask=None):
        return maxsim_kd(Q, D, qmask, dmask)
