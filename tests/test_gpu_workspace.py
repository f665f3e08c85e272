"""Pairwise and kd forward with a caller-provided workspace (GPU).

lik_maxsim_{pairwise,kd}_fwd_ws take the streaming forward's schedule
workspace from the caller (its size from the _fwd_workspace_bytes query), so
a caller that manages all device memory can use these layouts.  Their results
must be bit-identical to the plain entry points' (which take the workspace
from the library's pool), match the oracle, survive a workspace full of
garbage, and take no device memory of their own.
"""
import numpy as np
import pytest
import torch

import gpu_harness
import parity
from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300.workloads import random_case

pytestmark = pytest.mark.gpu

CASES = [
    # layout,     nq, nd, lq,   ld,  dim, dtype
    ("pairwise",   7,  0, 32,  700, 128, "bf16"),
    ("pairwise",   4,  0, 20, 9000, 128, "f16"),   # few long documents: cut between CTAs
    ("kd",         3,  5, 32,  260, 128, "bf16"),
    ("kd",         2, 17, 32, 1030,  64, "f16"),
]


def _run(h, workspace=None, pooled=False, masks=True):
    Q, D, qm, dm = h.gpu_inputs()
    if not masks:
        qm = dm = None
    shape = h.inp.workload.score_shape
    s = torch.full(shape, float("nan"), device="cuda")
    am = torch.full((*shape, h.Lq), -7, dtype=torch.int32, device="cuda")
    if pooled:
        getattr(binding, f"lik_maxsim_{h.kind}_fwd")(Q, D, qm, dm, s, am)
    else:
        getattr(binding, f"lik_maxsim_{h.kind}_fwd_ws")(Q, D, qm, dm, s, am, workspace)
    binding.lik_check_device_error()
    return s.cpu().numpy(), am.cpu().numpy()


@pytest.mark.parametrize("masks", [True, False], ids=["masks", "no-masks"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_caller_workspace_matches_pooled_and_oracle(case, masks):
    layout, nq, nd, lq, ld, dim, dtype = case
    inp = random_case(layout, nq, nd, lq, ld, dim, dtype, seed=nq * 31 + ld, p_doc_empty=0.15)
    if not masks:
        inp.qmask = inp.dmask = None
    h = gpu_harness.Layout(inp)
    Q, D, _, dm = h.gpu_inputs()
    nbytes = getattr(binding, f"lik_maxsim_{layout}_fwd_workspace_bytes")(Q, D, has_dmask=masks)
    assert nbytes > 0
    ws = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")  # contents must not matter
    s_ws, am_ws = _run(h, ws, masks=masks)
    s_pool, am_pool = _run(h, pooled=True, masks=masks)
    assert np.array_equal(s_ws, s_pool) and np.array_equal(am_ws, am_pool)
    s_o, am_o, gap = h.oracle_fwd()
    parity.assert_scores_close(s_ws, s_o, dtype)
    if masks:
        assert nbytes >= getattr(binding, f"lik_maxsim_{layout}_fwd_workspace_bytes")(Q, D, has_dmask=False)


def test_caller_workspace_takes_no_device_memory():
    inp = random_case("kd", 4, 9, 32, 1030, 128, "bf16", seed=5, p_doc_empty=0.1)
    h = gpu_harness.Layout(inp)
    Q, D, qm, dm = h.gpu_inputs()
    nbytes = binding.lik_maxsim_kd_fwd_workspace_bytes(Q, D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.empty(4, 9, device="cuda")
    am = torch.empty(4, 9, 32, dtype=torch.int32, device="cuda")
    binding.lik_maxsim_kd_fwd_ws(Q, D, qm, dm, s, am, ws)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch_bytes0 = torch.cuda.memory_allocated()
    for _ in range(3):
        binding.lik_maxsim_kd_fwd_ws(Q, D, qm, dm, s, am, ws)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == torch_bytes0
    binding.lik_check_device_error()


def test_caller_workspace_errors():
    inp = random_case("pairwise", 5, 0, 32, 300, 128, "bf16", seed=3)
    h = gpu_harness.Layout(inp)
    Q, D, qm, dm = h.gpu_inputs()
    s = torch.empty(5, device="cuda")
    nbytes = binding.lik_maxsim_pairwise_fwd_workspace_bytes(Q, D)
    for ws in (None, torch.empty(nbytes - 16, dtype=torch.uint8, device="cuda")):
        with pytest.raises(binding.LIKError) as ei:
            binding.lik_maxsim_pairwise_fwd_ws(Q, D, qm, dm, s, None, ws)
        assert ei.value.status_name == "LIK_ERR_INVALID_ARG"
    big = torch.empty(nbytes + 32, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.LIKError) as ei:  # 16-byte alignment
        lib = binding.load()
        st = lib.lik_maxsim_pairwise_fwd_ws(Q.data_ptr(), D.data_ptr(), 2, 5, 32, 300, 128, qm.data_ptr(),
                                            dm.data_ptr(), s.data_ptr(), None, big.data_ptr() + 8, nbytes,
                                            torch.cuda.current_stream().cuda_stream)
        binding._check(st)
    assert ei.value.status_name == "LIK_ERR_INVALID_ARG"
    # fp32 inputs take the FFMA forward, which needs no workspace
    Qf, Df = Q.float(), D.float()
    assert binding.lik_maxsim_pairwise_fwd_workspace_bytes(Qf, Df) == 0
    binding.lik_maxsim_pairwise_fwd_ws(Qf, Df, qm, dm, s, None, None)
    binding.lik_check_device_error()
