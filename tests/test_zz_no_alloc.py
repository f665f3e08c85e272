"""The all-pairs recompute backward with the library's built-in workspace.

lik_maxsim_allpairs_bwd_recompute_noalloc is for callers that cannot
allocate device memory (a memory manager that owns the whole device, a loop
that cannot pay for cudaMalloc): its argmax workspace is an array built into
the library instead of a caller's buffer.  It must give the same gradients
as lik_maxsim_allpairs_bwd_recompute with a caller-allocated workspace, also
on a second call right after the first (the array keeps the previous call's
contents), and refuse sizes beyond the array.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import gpu_harness
import parity
from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300.workloads import random_case

pytestmark = pytest.mark.gpu


def _reference(h, g):
    Q, D, qm, dm = h.gpu_inputs()
    shape = h.inp.workload.score_shape
    ws = torch.empty((*shape, h.Lq), dtype=torch.int32, device="cuda")
    gQ = torch.empty(Q.shape, device="cuda")
    gD = torch.empty(D.shape, device="cuda")
    binding.lik_maxsim_allpairs_bwd_recompute(Q, D, qm, dm, g, ws, gQ, gD)
    return gQ, gD


def _no_alloc(h, g):
    Q, D, qm, dm = h.gpu_inputs()
    gQ = torch.full(Q.shape, float("nan"), device="cuda")
    gD = torch.full(D.shape, float("nan"), device="cuda")
    binding.lik_maxsim_allpairs_bwd_recompute_noalloc(Q, D, qm, dm, g, gQ, gD)
    return gQ, gD


def test_no_alloc_matches_workspace_version_twice_in_a_row():
    cases = [random_case("allpairs", 6, 9, 32, 300, 128, "bf16", seed=41, p_doc_empty=0.2),
             random_case("allpairs", 4, 5, 16, 700, 64, "f16", seed=42, p_doc_empty=0.2)]
    for inp in cases:  # the second call finds the first call's argmax in the array
        h = gpu_harness.Layout(inp)
        g = inp.grad_out.to("cuda").float().contiguous()
        gQ_ref, gD_ref = _reference(h, g)
        gQ, gD = _no_alloc(h, g)
        binding.lik_check_device_error()
        tag = inp.workload.dtype
        assert torch.isfinite(gQ).all() and torch.isfinite(gD).all()
        assert parity.normwise_rel_err(gQ.cpu().numpy(), gQ_ref.cpu().numpy()) <= parity.TOL[tag]
        assert parity.normwise_rel_err(gD.cpu().numpy(), gD_ref.cpu().numpy()) <= parity.TOL[tag]


def test_no_alloc_refuses_sizes_beyond_its_workspace():
    Q = torch.randn(64, 32, 16, device="cuda").bfloat16()
    D = torch.randn(1025, 4, 16, device="cuda").bfloat16()  # 64 * 1025 * 32 > 2**21
    g = torch.zeros(64, 1025, device="cuda")
    with pytest.raises(binding.LIKError) as ei:
        binding.lik_maxsim_allpairs_bwd_recompute_noalloc(Q, D, None, None, g, torch.empty(Q.shape, device="cuda"),
                                                          torch.empty(D.shape, device="cuda"))
    assert ei.value.status_name == "LIK_ERR_UNSUPPORTED"
