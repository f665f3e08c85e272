"""The all-pairs recompute backward with the library's built-in workspace.

lik_maxsim_allpairs_bwd_recompute_noalloc is for callers that cannot
allocate device memory (a memory manager that owns the whole device, a loop
that cannot pay for cudaMalloc): its argmax workspace is an array built into
the library instead of a caller's buffer.  It must give the same gradients
as lik_maxsim_allpairs_bwd_recompute with a caller-allocated workspace, also
on a second call right after the first (the array keeps the previous call's
contents), and the oracle's gradients; it must take no device memory of its
own per call, and refuse sizes beyond the array.  This file is collected
last.
"""
import numpy as np
import pytest
import torch

import gpu_harness
import parity
from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300.workloads import separated_case

pytestmark = pytest.mark.gpu

# bf16 with query masks, fp16, and fp32 (the FFMA path), each with empty
# documents; inputs with a unique argmax so the oracle's gradients apply
CASES = [
    ("bf16", 6, 9, 32, 300, 128, 0.5),
    ("f16", 4, 5, 16, 700, 64, 0.0),
    ("f32", 3, 4, 8, 64, 64, 0.5),
]


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


def test_no_alloc_matches_workspace_version_and_oracle_twice_in_a_row():
    for dtype, nq, nd, lq, ld, dim, p_tail in CASES:
        inp = separated_case("allpairs", nq, nd, lq, ld, dim, dtype, seed=41 + nq, p_doc_empty=0.2,
                             p_query_tail=p_tail)
        h = gpu_harness.Layout(inp)
        _, am_o, _ = h.oracle_fwd_separated()
        gQ_o, gD_o = h.oracle_bwd(inp.grad_out.numpy().astype(np.float64), am_o)
        g = inp.grad_out.to("cuda").float().contiguous()
        gQ_ref, gD_ref = _reference(h, g)
        # two calls in a row: the second finds the first call's argmax in the array
        for _ in range(2):
            gQ, gD = _no_alloc(h, g)
            binding.lik_check_device_error()
            assert torch.isfinite(gQ).all() and torch.isfinite(gD).all()
            for got, ref, orc, name in ((gQ, gQ_ref, gQ_o, "grad_Q"), (gD, gD_ref, gD_o, "grad_D")):
                got = got.cpu().numpy()
                assert parity.normwise_rel_err(got, ref.cpu().numpy()) <= parity.TOL[dtype], (dtype, name)
                parity.assert_grad_close(got, orc, dtype, f"{dtype} {name}")


def test_no_alloc_takes_no_device_memory_per_call():
    inp = separated_case("allpairs", 6, 9, 32, 300, 128, "bf16", seed=47, p_doc_empty=0.2)
    h = gpu_harness.Layout(inp)
    Q, D, qm, dm = h.gpu_inputs()
    g = inp.grad_out.to("cuda").float().contiguous()
    gQ = torch.empty(Q.shape, device="cuda")
    gD = torch.empty(D.shape, device="cuda")
    binding.lik_maxsim_allpairs_bwd_recompute_noalloc(Q, D, qm, dm, g, gQ, gD)  # first call: set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch_bytes0 = torch.cuda.memory_allocated()
    for _ in range(3):
        binding.lik_maxsim_allpairs_bwd_recompute_noalloc(Q, D, qm, dm, g, gQ, gD)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert torch.cuda.memory_allocated() == torch_bytes0
    binding.lik_check_device_error()


def test_no_alloc_refuses_sizes_beyond_its_workspace():
    Q = torch.randn(64, 32, 16, device="cuda").bfloat16()
    D = torch.randn(1025, 4, 16, device="cuda").bfloat16()  # 64 * 1025 * 32 > 2**21
    g = torch.zeros(64, 1025, device="cuda")
    with pytest.raises(binding.LIKError) as ei:
        binding.lik_maxsim_allpairs_bwd_recompute_noalloc(Q, D, None, None, g, torch.empty(Q.shape, device="cuda"),
                                                          torch.empty(D.shape, device="cuda"))
    assert ei.value.status_name == "LIK_ERR_UNSUPPORTED"
