"""Seeded synthetic inputs for the MaxSim operator.

This module only draws inputs: it holds none of the operator's arithmetic, so
both the CUDA library's tests and the fp64 oracle can take their inputs from
it.  Every recipe follows the same rules:

* token embeddings are i.i.d. N(0, 1) per element, each token L2-normalised
  in fp32, then cast (round-to-nearest-even) to the workload dtype; the
  operator itself never normalises (Late Interaction Kernels README,
  "Scoring interface": the layers use raw dot products);
* draws come from one seeded ``torch.Generator`` in the order Q, D, lengths,
  planted positives, masks, grad_out;
* a "length" is a number of valid leading tokens; the tail after it is masked
  (bool mask, True = valid, as in the README's "Scoring interface").

The named configurations stand in for the workloads the pages measure on
(in-batch ColPali/ColQwen2 training at B=128 with 128x1024-scale grids, loss
heads at Lq=32 / Ld=1030 with 16 negatives, long-document reranking with
Ld >= 8k); the datasets and models themselves are not used.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

# Tokens generated per randn call.  Fixed, so that a recipe's draws do not
# depend on the size of the tensor being produced.
_CHUNK_TOKENS = 1 << 15


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and recipe of one named workload."""

    name: str
    layout: str  # "allpairs" | "pairwise" | "kd"
    nq: int  # Nq (all-pairs) or B (pairwise, kd)
    nd: int  # Nd (all-pairs), B (pairwise) or N candidates per query (kd)
    lq: int
    ld: int
    dim: int
    dtype: str
    seed: int
    backward: bool
    description: str

    @property
    def q_shape(self):
        return (self.nq, self.lq, self.dim)

    @property
    def d_shape(self):
        if self.layout == "kd":
            return (self.nq, self.nd, self.ld, self.dim)
        return (self.nd, self.ld, self.dim)

    @property
    def score_shape(self):
        if self.layout == "allpairs":
            return (self.nq, self.nd)
        if self.layout == "pairwise":
            return (self.nq,)
        return (self.nq, self.nd)

    @property
    def n_pairs(self) -> int:
        if self.layout == "pairwise":
            return self.nq
        return self.nq * self.nd

    @property
    def counted_flops(self) -> int:
        """2 * pairs * Lq * Ld * dim on padded lengths (the headline count)."""
        return 2 * self.n_pairs * self.lq * self.ld * self.dim


WORKLOADS = {
    "tiny_allpairs_f32": Workload(
        "tiny_allpairs_f32", "allpairs", 4, 8, 32, 180, 128, "f32", 0, True,
        "tiny all-pairs fwd+bwd, fp32: Q[4,32,128] x D[8,180,128]; doc tokens "
        ">=150 masked, doc 7 fully masked, query 3 tokens >=28 masked; "
        "grad_out ~ N(0,1)"),
    "inbatch_b128_bf16": Workload(
        "inbatch_b128_bf16", "allpairs", 128, 128, 32, 1030, 128, "bf16", 1, True,
        "in-batch contrastive all-pairs fwd+bwd, bf16: Q[128,32,128] x "
        "D[128,1030,128]; doc lengths U[700,1030]; grad_out from row-wise "
        "cross-entropy with the diagonal as target"),
    "inbatch_b128_f32": Workload(
        "inbatch_b128_f32", "allpairs", 128, 128, 32, 1030, 128, "f32", 5, True,
        "in-batch contrastive all-pairs fwd+bwd, fp32 inputs: the in-batch recipe "
        "(Q[128,32,128] x D[128,1030,128], doc lengths U[700,1030], cross-entropy "
        "score gradient) without rounding the tokens to 16 bits"),
    "kd_b256_n17_bf16": Workload(
        "kd_b256_n17_bf16", "kd", 256, 17, 32, 1030, 128, "bf16", 2, True,
        "per-query candidates fwd+bwd, bf16: Q[256,32,128] x D[256,17,1030,128]; "
        "candidate 0 holds 8 noisy copies of query tokens; doc lengths "
        "U[512,1030]; grad_out from cross-entropy over the 17 candidates"),
    "rerank_b512_ld8192_f16": Workload(
        "rerank_b512_ld8192_f16", "pairwise", 512, 512, 32, 8192, 128, "f16", 3, False,
        "long-document pairwise reranking fwd, fp16: Q[512,32,128] x "
        "D[512,8192,128]; doc lengths U[4096,8192]; query lengths U[16,32]"),
    "allpairs_q128_d4096_bf16": Workload(
        "allpairs_q128_d4096_bf16", "allpairs", 128, 4096, 128, 1024, 128, "bf16", 4, False,
        "large all-pairs inference fwd, bf16: Q[128,128,128] x D[4096,1024,128]; "
        "410 docs (seeded permutation) have lengths U[256,1024], the rest are full"),
}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def tokens(gen: torch.Generator, shape, dtype: str, device="cpu") -> torch.Tensor:
    """i.i.d. Gaussian tokens, each L2-normalised in fp32, cast to ``dtype``."""
    shape = tuple(shape)
    dim = shape[-1]
    n = math.prod(shape[:-1])
    out = torch.empty((n, dim), dtype=DTYPES[dtype], device=device)
    for s in range(0, n, _CHUNK_TOKENS):
        e = min(n, s + _CHUNK_TOKENS)
        x = torch.randn((e - s, dim), generator=gen, device=device, dtype=torch.float32)
        out[s:e] = (x / x.norm(dim=-1, keepdim=True)).to(out.dtype)
    return out.view(shape)


def lengths(gen: torch.Generator, n: int, lo: int, hi: int, device="cpu") -> torch.Tensor:
    """n integers drawn uniformly from [lo, hi] inclusive (int64)."""
    return torch.randint(lo, hi + 1, (n,), generator=gen, device=device)


def prefix_mask(lens: torch.Tensor, L: int) -> torch.Tensor:
    """Bool mask [n, L]: True for the first lens[r] tokens of row r."""
    return torch.arange(L, device=lens.device)[None, :] < lens[:, None]


def ce_grad_rows(scores: torch.Tensor, target: torch.Tensor) -> torch.Tensor:
    """d(mean cross-entropy)/d(scores) for logits ``scores`` [R, C], temperature 1.

    This is the loss head of the training workloads (not part of the MaxSim
    operator): (softmax(scores) - onehot(target)) / R, computed in fp64.
    """
    s = scores.to(torch.float64)
    p = torch.softmax(s, dim=-1)
    p[torch.arange(s.shape[0], device=s.device), target] -= 1.0
    return p / s.shape[0]


@dataclasses.dataclass
class Inputs:
    """One draw of a workload.  Masks are bool; grad_out is fp32 or None.

    ``grad_out`` is None for the cross-entropy workloads, whose upstream
    gradient depends on the scores: call :func:`ce_grad_rows` on scores
    computed by whoever runs the workload (the oracle in tests).
    """

    workload: Workload
    Q: torch.Tensor
    D: torch.Tensor
    qmask: Optional[torch.Tensor]
    dmask: Optional[torch.Tensor]
    grad_out: Optional[torch.Tensor]
    ce_target: Optional[torch.Tensor]


def generate(name: str, device="cpu") -> Inputs:
    """Draw the named workload on ``device`` with its own seed."""
    w = WORKLOADS[name]
    gen = generator(w.seed, device)
    Q = tokens(gen, w.q_shape, w.dtype, device)
    D = tokens(gen, w.d_shape, w.dtype, device)
    grad_out = ce_target = None

    if name == "tiny_allpairs_f32":
        dmask = torch.ones((w.nd, w.ld), dtype=torch.bool, device=device)
        dmask[:, 150:] = False
        dmask[7, :] = False
        qmask = torch.ones((w.nq, w.lq), dtype=torch.bool, device=device)
        qmask[3, 28:] = False
        grad_out = torch.randn(w.score_shape, generator=gen, device=device, dtype=torch.float32)
    elif name in ("inbatch_b128_bf16", "inbatch_b128_f32"):
        dlen = lengths(gen, w.nd, 700, 1030, device)
        dmask = prefix_mask(dlen, w.ld)
        qmask = torch.ones((w.nq, w.lq), dtype=torch.bool, device=device)
        ce_target = torch.arange(w.nq, device=device)
    elif name == "kd_b256_n17_bf16":
        dlen = lengths(gen, w.nq * w.nd, 512, 1030, device).view(w.nq, w.nd)
        _plant_positives(gen, Q, D, dlen[:, 0], n_plant=8, noise_std=0.1)
        dmask = prefix_mask(dlen.reshape(-1), w.ld).view(w.nq, w.nd, w.ld)
        qmask = torch.ones((w.nq, w.lq), dtype=torch.bool, device=device)
        ce_target = torch.zeros(w.nq, dtype=torch.long, device=device)
    elif name == "rerank_b512_ld8192_f16":
        dlen = lengths(gen, w.nq, 4096, 8192, device)
        qlen = lengths(gen, w.nq, 16, 32, device)
        dmask = prefix_mask(dlen, w.ld)
        qmask = prefix_mask(qlen, w.lq)
    elif name == "allpairs_q128_d4096_bf16":
        short = torch.randperm(w.nd, generator=gen, device=device)[:410]
        dlen = torch.full((w.nd,), w.ld, dtype=torch.long, device=device)
        dlen[short] = lengths(gen, 410, 256, 1024, device)
        dmask = prefix_mask(dlen, w.ld)
        qmask = torch.ones((w.nq, w.lq), dtype=torch.bool, device=device)
    else:  # pragma: no cover - WORKLOADS and this switch list the same names
        raise KeyError(name)
    return Inputs(w, Q, D, qmask, dmask, grad_out, ce_target)


def _plant_positives(gen, Q, D, pos_len, n_plant: int, noise_std: float):
    """Make candidate 0 of every query a positive.

    ``n_plant`` distinct valid positions of D[b, 0] are overwritten by copies
    of ``n_plant`` distinct query tokens Q[b, i] plus N(0, noise_std^2) noise,
    renormalised in fp32 and cast back to the storage dtype.
    """
    B, Lq, dim = Q.shape
    device = Q.device
    for b in range(B):
        L = int(pos_len[b])
        pos = torch.randperm(L, generator=gen, device=device)[:n_plant]
        src = torch.randperm(Lq, generator=gen, device=device)[:n_plant]
        noise = noise_std * torch.randn((len(pos), dim), generator=gen, device=device)
        x = Q[b, src].to(torch.float32) + noise
        D[b, 0, pos] = (x / x.norm(dim=-1, keepdim=True)).to(D.dtype)


def random_case(layout: str, nq: int, nd: int, lq: int, ld: int, dim: int, dtype: str,
                seed: int, device="cpu", p_doc_empty=0.0, p_query_tail=0.5,
                min_dlen=1) -> Inputs:
    """A small random case for sweeps: random prefix lengths, optional empty docs.

    ``nd`` is Nd (all-pairs), ignored for pairwise (B = nq), or N (kd).
    Each document keeps a random prefix of at least ``min_dlen`` tokens
    (or none, with probability ``p_doc_empty``); each query keeps a random
    prefix with probability ``p_query_tail`` and is full otherwise.
    grad_out ~ N(0, 1).
    """
    w = Workload(f"random_{layout}", layout, nq, nd if layout != "pairwise" else nq,
                 lq, ld, dim, dtype, seed, True, "random sweep case")
    gen = generator(seed, device)
    Q = tokens(gen, w.q_shape, dtype, device)
    D = tokens(gen, w.d_shape, dtype, device)
    n_docs = math.prod(w.d_shape[:-2])
    lo = min(max(min_dlen, 0), ld)
    dlen = lengths(gen, n_docs, lo, ld, device) if ld > 0 else torch.zeros(n_docs, dtype=torch.long)
    empty = torch.rand(n_docs, generator=gen, device=device) < p_doc_empty
    dlen = torch.where(empty, torch.zeros_like(dlen), dlen)
    qlen = lengths(gen, nq, 0, lq, device) if lq > 0 else torch.zeros(nq, dtype=torch.long)
    tail = torch.rand(nq, generator=gen, device=device) < p_query_tail
    qlen = torch.where(tail, qlen, torch.full_like(qlen, lq))
    dmask = prefix_mask(dlen, ld).view(*w.d_shape[:-2], ld)
    qmask = prefix_mask(qlen, lq)
    grad_out = torch.randn(w.score_shape, generator=gen, device=device, dtype=torch.float32)
    return Inputs(w, Q, D, qmask, dmask, grad_out, None)


def separated_case(layout: str, nq: int, nd: int, lq: int, ld: int, dim: int, dtype: str,
                   seed: int, device="cpu", p_doc_empty=0.0, p_query_tail=0.5,
                   background=0.25) -> Inputs:
    """A random case in which every query token has one clear best document token.

    Drawn as :func:`random_case` (every non-empty document long enough to hold
    the copies below), then, with a second generator seeded from ``seed``:
    every document token is scaled by ``background``, and for every pair
    (q, d) of the layout each token Q[q, i] gets a copy Q[q, i] * s,
    s ~ U[0.6, 1.0], at its own random valid position of document d.  The
    copy's similarity is s * |Q[q, i]|^2 >= 0.6 (tokens are unit-norm), while
    every other valid token of d is a background token or a scaled copy of
    another token, whose similarity is a cosine of two independent random
    directions (standard deviation 1/sqrt(dim)).  With dim >= 64 the best and
    second-best similarities are then far apart (> 1e-2) for every valid
    query token, which a test must still check on its own inputs; the argmax
    of such inputs is unique and the same in any accumulation order.
    """
    per_doc = nq if layout == "allpairs" else 1
    if lq * per_doc > ld:
        raise ValueError("documents are too short for one copy per query token")
    inp = random_case(layout, nq, nd, lq, ld, dim, dtype, seed, device, p_doc_empty, p_query_tail,
                      min_dlen=lq * per_doc)
    gen = generator(seed + 7919, device)
    n_docs = math.prod(inp.workload.d_shape[:-2])
    D = inp.D.reshape(n_docs, ld, dim).to(torch.float32) * background
    dlen = inp.dmask.reshape(n_docs, ld).sum(dim=1)
    Qf = inp.Q.to(torch.float32)
    for doc in range(n_docs):
        L = int(dlen[doc])
        if L == 0:
            continue
        if layout == "allpairs":
            src = Qf.reshape(nq * lq, dim)
        elif layout == "kd":
            src = Qf[doc // nd]
        else:
            src = Qf[doc]
        pos = torch.randperm(L, generator=gen, device=device)[:src.shape[0]]
        s = 0.6 + 0.4 * torch.rand(src.shape[0], generator=gen, device=device)
        D[doc, pos] = src * s[:, None]
    inp.D = D.to(inp.D.dtype).reshape(inp.workload.d_shape).contiguous()
    return inp


def to_numpy(t: torch.Tensor):
    """(array, dtype tag) in the form the oracle accepts; bf16 as uint16 bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16"), "bf16"
    if t.dtype == torch.float16:
        return t.numpy(), "f16"
    if t.dtype == torch.float32:
        return t.numpy(), "f32"
    if t.dtype == torch.float64:
        return t.numpy(), "f64"
    raise TypeError(t.dtype)
