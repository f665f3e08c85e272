"""Seeded random shapes across every layout and dtype (GPU) against the oracle,
and concurrent calls on two streams.

The fuzz draws layout, dtype, embedding size (multiples of 16 for the
tensor-core kernels, and others for the FFMA kernel), query and document
lengths around every tile edge, batch sizes and mask densities, and checks
the forward and the backward (on the oracle's argmax) with the usual rules.
"""
import numpy as np
import pytest
import torch

import gpu_harness
from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300.workloads import random_case

pytestmark = pytest.mark.gpu


def _draw(rng):
    layout = ["allpairs", "pairwise", "kd"][rng.integers(3)]
    dtype = ["bf16", "f16", "f32"][rng.integers(3)]
    dim = int(rng.choice([16, 32, 48, 64, 80, 96, 128, 144, 192, 256, 8, 24, 40, 100]))
    lq = int(rng.choice([1, 2, 7, 16, 31, 32, 33, 48, 64, 100, 128]))
    ld = int(rng.choice([1, 15, 16, 17, 63, 64, 127, 128, 129, 200, 255, 256, 257, 511, 600]))
    nq = int(rng.integers(1, 7))
    nd = int(rng.integers(1, 9))
    return layout, nq, nd, lq, ld, dim, dtype


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_against_oracle(seed):
    rng = np.random.default_rng(1000 + seed)
    layout, nq, nd, lq, ld, dim, dtype = _draw(rng)
    inp = random_case(layout, nq, nd, lq, ld, dim, dtype, seed=seed, p_doc_empty=float(rng.uniform(0, 0.3)),
                      p_query_tail=float(rng.uniform(0, 1)))
    h = gpu_harness.Layout(inp)
    f = h.check_forward()
    h.check_backward(am_oracle=f["am_oracle"])


def test_two_streams_at_once():
    """Different workloads enqueued on two streams together give the results
    each gives alone."""
    cases = [random_case("allpairs", 6, 40, 32, 400, 128, "bf16", seed=7, p_doc_empty=0.1),
             random_case("kd", 8, 9, 32, 300, 128, "bf16", seed=8, p_doc_empty=0.1)]
    layouts = [gpu_harness.Layout(c) for c in cases]
    alone = [h.gpu_fwd() for h in layouts]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for h, st in zip(layouts, streams):
        Q, D, qm, dm = h.gpu_inputs()
        shape = h.inp.workload.score_shape
        outs.append((torch.empty(shape, device="cuda"),
                     torch.empty((*shape, h.Lq), dtype=torch.int32, device="cuda"), Q, D, qm, dm))
    torch.cuda.synchronize()
    for _ in range(3):
        for h, st, (s, am, Q, D, qm, dm) in zip(layouts, streams, outs):
            with torch.cuda.stream(st):
                getattr(binding, f"lik_maxsim_{h.kind}_fwd")(Q, D, qm, dm, s, am, stream=st)
    torch.cuda.synchronize()
    binding.lik_check_device_error()
    for (s_a, am_a), (s, am, *_rest) in zip(alone, outs):
        assert np.array_equal(s.cpu().numpy(), s_a)
        assert np.array_equal(am.cpu().numpy(), am_a)
