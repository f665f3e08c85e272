"""CUDA library vs fp64 oracle on small seeded cases (GPU).

Shapes are chosen to span several tiles of every kernel and to end on ragged
tails: query counts around the 128-row tensor-core tile, document lengths
around the 32/128/256-token tiles, empty documents, masked query tokens.
"""
import json
import os
import zlib

import numpy as np
import pytest
import torch

import gpu_harness
import parity
from late_interaction_retrieval_gb300 import binding, layers
from late_interaction_retrieval_gb300.workloads import Inputs, Workload, generate, random_case, separated_case

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")
TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


# ------------------------------------------------------------ workloads --

def test_tiny_allpairs_f32_fwd_bwd():
    inp = generate("tiny_allpairs_f32")
    h = gpu_harness.Layout(inp)
    f = h.check_forward()
    assert (f["s_oracle"][:, 7] == -1e9).all()  # the fully masked document
    h.check_backward(am_oracle=f["am_oracle"])


# --------------------------------------------------------- hand-worked --

def _golden_inputs(case, dtype):
    layout = case.get("layout", "allpairs")
    dt = TORCH_DT[dtype]
    Q = torch.tensor(case["Q"], dtype=torch.float64).to(dt)
    D = torch.tensor(case["D"], dtype=torch.float64).to(dt)
    qm = None if case["qmask"] is None else torch.tensor(case["qmask"], dtype=torch.bool)
    dm = None if case["dmask"] is None else torch.tensor(case["dmask"], dtype=torch.bool)
    g = torch.tensor(case["grad_out"], dtype=torch.float32)
    nq, lq, dim = Q.shape
    if layout == "kd":
        nd, ld = D.shape[1], D.shape[2]
    else:
        nd, ld = D.shape[0], D.shape[1]
    w = Workload(case["name"], layout, nq, nd, lq, ld, dim, dtype, 0, True, "golden")
    return Inputs(w, Q, D, qm, dm, g, None)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_golden_cases_exact(dtype):
    """Small integers are exact in every dtype: the GPU must reproduce the
    hand-worked values bit for bit."""
    for case in json.load(open(GOLDEN))["cases"]:
        h = gpu_harness.Layout(_golden_inputs(case, dtype))
        s, am = h.gpu_fwd()
        assert np.array_equal(s, np.asarray(case["scores"], np.float32)), (case["name"], s)
        assert np.array_equal(am, np.asarray(case["argmax"], np.int32)), (case["name"], am)
        gQ, gD = h.gpu_bwd(np.asarray(case["grad_out"]), np.asarray(case["argmax"]))
        assert np.array_equal(gQ, np.asarray(case["gQ"], np.float32)), (case["name"], gQ)
        assert np.array_equal(gD, np.asarray(case["gD"], np.float32)), (case["name"], gD)


# ------------------------------------------------------- random sweeps --

SWEEP = [
    # layout,     nq, nd, lq,  ld,   dim
    ("allpairs",   3,  5, 32,  180,  128),
    ("allpairs",   5,  7, 33,  257,  128),
    ("allpairs",   9,  4, 32, 1030,  128),
    ("allpairs",   2,  3, 128, 300,  128),
    ("allpairs",   5,  4, 64,  230,  128),  # two 64-token queries per row block
    ("allpairs",  17,  3,  8,   64,   64),
    ("allpairs",   3,  6, 100,  33,  256),
    ("allpairs",   3,  4, 32,  300,  256),  # 80-column tiles: the widest with two D stages at dim 256
    ("kd",         2,  3, 16,  150,  256),  # streaming forward does not fit at dim 256: SIMT forward
    ("allpairs",   2,  2,  7,   31,   16),
    ("allpairs",   2,  3,  5,   40,   96),
    ("allpairs",   4, 400, 32, 300,  128),  # 160-column tiles, 3 accumulators, several per CTA
    ("allpairs",   1, 700, 128, 140, 128),  # 144-column tiles, many per CTA
    ("allpairs", 150,  3, 32,  200,   64),  # 4800 query tokens reach each document in the backward
    ("allpairs",  40,  2, 128, 130,  128),  # 5120 of them, at Lq = 128
    ("pairwise",   7,  0, 32,  700,  128),
    ("pairwise",   4,  0, 20, 2100,  128),
    ("pairwise",   3,  0, 128, 129,   64),
    ("pairwise",   5,  0, 48,  300,  128),
    ("kd",         3,  4, 33,  200,   64),
    ("kd",         3,  5, 32,  260,  128),
    ("kd",         2, 17, 32, 1030,  128),
    ("kd",         4,  3, 16,   77,   32),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("case", SWEEP, ids=lambda c: "-".join(map(str, c)))
def test_random_sweep(case, dtype):
    layout, nq, nd, lq, ld, dim = case
    inp = random_case(layout, nq, nd, lq, ld, dim, dtype, seed=zlib.crc32(repr(case).encode()) % 10_000,
                      p_doc_empty=0.15)
    h = gpu_harness.Layout(inp)
    f = h.check_forward()
    h.check_backward(am_oracle=f["am_oracle"])


SINGLE_GRAD_CASES = [
    # layout,     nq, nd, lq,  ld,  dim
    ("allpairs",   5,  7, 33,  257, 128),
    ("allpairs",   3,  4, 32,  300, 256),
    ("allpairs",   4,  3, 20,   90,  72),
    ("kd",         3,  5, 32,  260, 128),
    ("pairwise",   4,  0, 20,  700,  16),
    ("allpairs",   3,  5, 16,   70,   8),  # one 8-element vector per row: most threads idle
    ("allpairs",   2,  3, 24,   90, 136),  # dim 136: four vectors per thread, the last partial
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", SINGLE_GRAD_CASES, ids=lambda c: "-".join(map(str, c)))
def test_single_gradient_calls(case, dtype):
    """grad_Q alone and grad_D alone (their own launches) against the oracle;
    the sweep above takes both in the one launch that writes the two."""
    layout, nq, nd, lq, ld, dim = case
    inp = random_case(layout, nq, nd, lq, ld, dim, dtype, seed=zlib.crc32(repr(case).encode()) % 10_000,
                      p_doc_empty=0.15)
    h = gpu_harness.Layout(inp)
    f = h.check_forward()
    h.check_backward_single(am_oracle=f["am_oracle"])
    h.check_backward(am_oracle=f["am_oracle"])


F32_TC_CASES = [
    # layout,     nq, nd, lq,  ld,  dim   (fp32 inputs on the split-TF32 tensor-core kernel)
    ("allpairs",   3,  4,  1,   65,   8),  # one K step, one query token
    ("allpairs",   5,  3, 127, 130,  24),  # Lq = 127: one query per row block, a partial atom
    ("allpairs",   2,  5, 128,  64,  40),
    ("allpairs",   9,  6, 33,  200, 120),  # 3 queries per row block, 4 atoms (the last partial)
    ("allpairs",  37,  3, 16,  129, 128),  # 8 queries per row block, a partial last row block
    ("allpairs",   1, 300, 32,  70, 128),  # many documents per work unit
    ("pairwise",   6,  0, 128, 500,  64),
    ("kd",         3,  7, 20,  333,  96),
    ("allpairs",   2,  3, 129,  40,  64),  # Lq > 128: the FFMA kernel
]


@pytest.mark.parametrize("case", F32_TC_CASES, ids=lambda c: "-".join(map(str, c)))
def test_f32_tensor_core_shapes(case):
    """fp32 inputs at the bar of 1e-5 through the split-TF32 tensor-core
    forward: embedding sizes from one K step to 128, query lengths up to 128,
    partial row blocks and atoms, empty documents, all three layouts."""
    layout, nq, nd, lq, ld, dim = case
    inp = random_case(layout, nq, nd, lq, ld, dim, "f32", seed=zlib.crc32(repr(case).encode()) % 10_000,
                      p_doc_empty=0.15)
    h = gpu_harness.Layout(inp)
    f = h.check_forward()
    h.check_backward(am_oracle=f["am_oracle"])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_odd_dims_simt(dtype):
    """Embedding sizes that are not multiples of 16 still compute exactly."""
    for dim in (1, 3, 100):
        inp = random_case("allpairs", 3, 4, 6, 45, dim, dtype, seed=dim)
        h = gpu_harness.Layout(inp)
        f = h.check_forward()
        h.check_backward(am_oracle=f["am_oracle"])


# ----------------------------------------------------------- edge cases --

@pytest.mark.parametrize("layout", ["allpairs", "pairwise", "kd"])
def test_degenerate_lengths(layout):
    for lq, ld in ((0, 9), (5, 0), (1, 1), (0, 0)):
        inp = random_case(layout, 3, 2, lq, ld, 64, "bf16", seed=lq * 10 + ld, p_doc_empty=0.3)
        h = gpu_harness.Layout(inp)
        f = h.check_forward()
        h.check_backward(am_oracle=f["am_oracle"])


def test_no_masks_and_all_empty():
    inp = random_case("allpairs", 4, 5, 32, 200, 128, "bf16", seed=5)
    inp.qmask = None
    inp.dmask = None
    gpu_harness.Layout(inp).check_forward()
    inp = random_case("allpairs", 4, 5, 32, 200, 128, "bf16", seed=6, p_doc_empty=1.0)
    s, am = gpu_harness.Layout(inp).gpu_fwd()
    assert (s == -1e9).all() and (am == -1).all()


def test_exact_ties_resolve_low():
    """Duplicated document tokens: the lowest index wins, as in the oracle."""
    inp = random_case("allpairs", 2, 3, 32, 300, 128, "bf16", seed=8, p_doc_empty=0.0)
    inp.dmask = None
    D = inp.D.clone()
    D[:, 200:] = D[:, 100:200]  # every token >= 200 repeats an earlier one
    inp.D = D
    h = gpu_harness.Layout(inp)
    f = h.check_forward()
    assert (f["am_gpu"] < 200).all()


def test_zero_padding_differs_from_mask():
    """All valid similarities negative: a masked token must not act as 0."""
    Q = torch.zeros(1, 1, 16)
    Q[0, 0, 0] = 1.0
    D = torch.zeros(1, 40, 16)
    D[0, :, 0] = -torch.arange(1, 41, dtype=torch.float32) / 64
    dm = torch.ones(1, 40, dtype=torch.bool)
    dm[0, 0] = False  # mask the best (-1/64); zero tokens would win if padding counted
    w = Workload("neg", "allpairs", 1, 1, 1, 40, 16, "bf16", 0, True, "neg")
    inp = Inputs(w, Q.to(torch.bfloat16), D.to(torch.bfloat16), None, dm, torch.ones(1, 1), None)
    s, am = gpu_harness.Layout(inp).gpu_fwd()
    assert s[0, 0] == np.float32(-2 / 64) and am[0, 0, 0] == 1


# -------------------------------------------------------- autograd path --

@pytest.mark.parametrize("layout", ["allpairs", "pairwise", "kd"])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_autograd_layers(layout, dtype):
    """Forward and backward through the autograd layers against the oracle,
    on inputs whose argmax is unique (the GPU's own argmax must then be the
    oracle's), with the gradients compared on every run."""
    ld = 150 if layout != "allpairs" else 160
    inp = separated_case(layout, 4, 5, 32, ld, 128, dtype, seed=21, p_doc_empty=0.2)
    h = gpu_harness.Layout(inp)
    s_o, am_o, _ = h.oracle_fwd_separated()
    Q, D, qm, dm = h.gpu_inputs()
    Q.requires_grad_(True)
    D.requires_grad_(True)
    layer = {"allpairs": layers.MaxSim, "pairwise": layers.MaxSimPairwise, "kd": layers.MaxSimKD}[layout]
    scores = layer()(Q, D, qm, dm)
    g = inp.grad_out.cuda()
    scores.backward(g)
    parity.assert_scores_close(scores.detach().cpu().numpy(), s_o, dtype)
    _, am_g = h.gpu_fwd()
    assert np.array_equal(am_g.reshape(am_o.shape), am_o), "argmax differs on separated inputs"
    gQ_o, gD_o = h.oracle_bwd(inp.grad_out.numpy().astype(np.float64), am_o)
    # the layer hands autograd gradients in the input dtype: one extra
    # rounding to 16 bits costs up to 2^-8 (bf16) / 2^-11 (fp16) relative on
    # top of the kernel's bar
    extra = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 0.0}[dtype]
    for got, ref, name in ((Q.grad, gQ_o, "grad_Q"), (D.grad, gD_o, "grad_D")):
        err = parity.normwise_rel_err(got.float().cpu().numpy(), ref)
        assert err <= parity.TOL[dtype] + extra, (name, err)
    assert Q.grad.dtype == Q.dtype and D.grad.dtype == D.dtype


def test_pairwise_and_kd_layers_match_allpairs():
    inp = random_case("kd", 3, 4, 32, 90, 128, "bf16", seed=22)
    Q, D = inp.Q.cuda(), inp.D.cuda()
    qm, dm = inp.qmask.cuda(), inp.dmask.cuda()
    kd = layers.MaxSimKD()(Q, D, qm, dm)
    pw = layers.MaxSimPairwise()(Q, D[:, 0].contiguous(), qm, dm[:, 0].contiguous())
    for b in range(3):
        ap = layers.MaxSim()(Q[b:b + 1], D[b], qm[b:b + 1], dm[b])
        torch.testing.assert_close(kd[b], ap[0], rtol=1e-5, atol=1e-5)
        torch.testing.assert_close(pw[b], ap[0, 0], rtol=1e-5, atol=1e-5)


# ----------------------------------------------------------- host errors --

def test_host_pointer_rejected():
    lib = binding.load()
    Q = torch.zeros(2, 4, 16, dtype=torch.bfloat16)  # host memory
    D = torch.zeros(3, 5, 16, dtype=torch.bfloat16)
    s = torch.zeros(2, 3, device="cuda")
    st = lib.lik_maxsim_allpairs_fwd(Q.data_ptr(), D.data_ptr(), 2, 2, 3, 4, 5, 16, None, None,
                                     s.data_ptr(), None, None)
    assert st == 1 and "device memory" in lib.lik_last_error_message().decode()


def test_misaligned_rejected():
    lib = binding.load()
    Q = torch.zeros(2 * 4 * 16 + 1, dtype=torch.bfloat16, device="cuda")
    D = torch.zeros(3 * 5 * 16, dtype=torch.bfloat16, device="cuda")
    s = torch.zeros(2, 3, device="cuda")
    st = lib.lik_maxsim_allpairs_fwd(Q.data_ptr() + 2, D.data_ptr(), 2, 2, 3, 4, 5, 16, None, None,
                                     s.data_ptr(), None, None)
    assert st == 1 and "aligned" in lib.lik_last_error_message().decode()


def test_binding_checks_shapes():
    Q = torch.zeros(2, 4, 16, dtype=torch.bfloat16, device="cuda")
    D = torch.zeros(3, 5, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        binding.lik_maxsim_allpairs_fwd(Q, D, None, None, torch.zeros(3, 2, device="cuda"))
    with pytest.raises(ValueError):
        binding.lik_maxsim_allpairs_fwd(Q, D.float(), None, None, torch.zeros(2, 3, device="cuda"))


def test_out_of_range_argmax_is_flagged_not_followed():
    """A saved argmax the forward could not have written (>= Ld) is skipped
    by the kernels (no memory access) and reported by lik_check_device_error."""
    Q = torch.randn(2, 4, 16, device="cuda").bfloat16()
    D = torch.randn(3, 5, 16, device="cuda").bfloat16()
    am = torch.zeros(2, 3, 4, dtype=torch.int32, device="cuda")
    am[1, 2, 3] = 5
    g = torch.ones(2, 3, device="cuda")
    gQ = torch.empty(2, 4, 16, device="cuda")
    gD = torch.empty(3, 5, 16, device="cuda")
    binding.lik_maxsim_allpairs_bwd(Q, D, g, am, gQ, gD)
    with pytest.raises(binding.LIKError) as ei:
        binding.lik_check_device_error()
    assert ei.value.status_name == "LIK_ERR_INVALID_ARG"
    binding.lik_check_device_error()  # the word was cleared


def test_side_stream():
    inp = random_case("allpairs", 3, 4, 32, 100, 128, "bf16", seed=30)
    h = gpu_harness.Layout(inp)
    Q, D, qm, dm = h.gpu_inputs()
    s_ref = torch.empty(3, 4, device="cuda")
    binding.lik_maxsim_allpairs_fwd(Q, D, qm, dm, s_ref)
    st = torch.cuda.Stream()
    s = torch.empty(3, 4, device="cuda")
    with torch.cuda.stream(st):
        binding.lik_maxsim_allpairs_fwd(Q, D, qm, dm, s)
    st.synchronize()
    assert torch.equal(s, s_ref)
