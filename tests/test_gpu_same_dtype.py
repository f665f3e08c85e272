"""Backward with gradients in the inputs' dtype (GPU) against the fp64 oracle.

The `_bwd_same_dtype` entry points sum every gradient element in fp32 and
round it to fp16/bf16 once; grad_D rows are written exactly once (zeros
included).  The bar is the fp16/bf16 tolerance plus that one rounding.
Shapes reach both grad_D kernels: the per-document streaming kernel
(pairwise and kd with Lq <= 32) and the document-owner kernel (all-pairs,
and any layout with Lq > 32), including more than 4096 query tokens per
document (several bucketing rounds).
"""
import zlib

import numpy as np
import pytest
import torch

import gpu_harness
from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300.workloads import random_case

pytestmark = pytest.mark.gpu

CASES = [
    # layout,     nq, nd, lq,  ld,  dim
    ("allpairs",   3,  5, 32,  180, 128),
    ("allpairs",   9,  4, 32, 1030, 128),
    ("allpairs", 150,  3, 32,  200,  64),   # 4800 hits per document: two rounds
    ("allpairs",  40,  2, 128, 130, 128),   # 5120 hits per document, Lq = 128
    ("allpairs",   2,  3, 100,  33, 256),
    ("allpairs",   4,  2,  5,   40,  96),
    ("pairwise",   7,  0, 32,  700, 128),
    ("pairwise",   5,  0, 48,  300, 128),   # Lq > 32: document-owner kernel
    ("pairwise",   3,  0, 17,   31,   8),
    ("kd",         3,  5, 32,  260, 128),
    ("kd",         2, 17, 32, 1030, 128),
    ("kd",         3,  4, 33,  200,  64),   # Lq > 32
    ("kd",         2,  3,  8,   77, 256),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_same_dtype_backward_matches_oracle(case, dtype):
    layout, nq, nd, lq, ld, dim = case
    inp = random_case(layout, nq, nd, lq, ld, dim, dtype, seed=zlib.crc32(repr(case).encode()) % 10_000,
                      p_doc_empty=0.15)
    h = gpu_harness.Layout(inp)
    f = h.check_forward()
    h.check_backward_same_dtype(am_oracle=f["am_oracle"])


@pytest.mark.parametrize("layout", ["allpairs", "pairwise", "kd"])
def test_same_dtype_degenerate_lengths(layout):
    for lq, ld in ((0, 9), (5, 0), (1, 1)):
        inp = random_case(layout, 3, 2, lq, ld, 64, "bf16", seed=lq * 10 + ld, p_doc_empty=0.3)
        h = gpu_harness.Layout(inp)
        f = h.check_forward()
        h.check_backward_same_dtype(am_oracle=f["am_oracle"])


def test_fp32_inputs_take_the_fp32_path():
    inp = random_case("kd", 2, 3, 20, 50, 64, "f32", seed=5)
    h = gpu_harness.Layout(inp)
    _, am, _ = h.oracle_fwd()
    g = inp.grad_out.cpu().numpy().astype(np.float64)
    a = h.gpu_bwd(g, am)
    b = h.gpu_bwd_same_dtype(g, am)
    # the same kernels; grad_D's fp32 atomics may add in another order
    for x, y in zip(a, b):
        assert np.abs(x - y).max() <= 1e-6 * max(np.abs(x).max(), 1e-30)


def test_unsupported_dim_is_rejected():
    Q = torch.randn(2, 4, 20, device="cuda").bfloat16()
    D = torch.randn(3, 5, 20, device="cuda").bfloat16()
    am = torch.zeros(2, 3, 4, dtype=torch.int32, device="cuda")
    g = torch.ones(2, 3, device="cuda")
    with pytest.raises(binding.LIKError) as ei:
        binding.lik_maxsim_allpairs_bwd_same_dtype(Q, D, g, am, torch.empty_like(Q), torch.empty_like(D))
    assert ei.value.status_name == "LIK_ERR_UNSUPPORTED"


@pytest.mark.parametrize("layout", ["allpairs", "kd"])
def test_out_of_range_argmax_is_flagged(layout):
    """An argmax >= Ld is skipped by both grad_D kernels and reported."""
    Q = torch.randn(2, 4, 16, device="cuda").bfloat16()
    if layout == "allpairs":
        D = torch.randn(3, 5, 16, device="cuda").bfloat16()
        am = torch.zeros(2, 3, 4, dtype=torch.int32, device="cuda")
        am[1, 2, 3] = 5
        g = torch.ones(2, 3, device="cuda")
        fn = binding.lik_maxsim_allpairs_bwd_same_dtype
    else:
        D = torch.randn(2, 3, 5, 16, device="cuda").bfloat16()
        am = torch.zeros(2, 3, 4, dtype=torch.int32, device="cuda")
        am[1, 2, 3] = 7
        g = torch.ones(2, 3, device="cuda")
        fn = binding.lik_maxsim_kd_bwd_same_dtype
    fn(Q, D, g, am, torch.empty_like(Q), torch.empty_like(D))
    with pytest.raises(binding.LIKError) as ei:
        binding.lik_check_device_error()
    assert ei.value.status_name == "LIK_ERR_INVALID_ARG"
    binding.lik_check_device_error()
