"""Peak device memory of a training step through the autograd layers (GPU).

The extra memory over the inputs is exactly the outputs the step needs: the
scores, the saved argmax (or, with recompute, the backward's argmax
workspace) and the gradients.  It is linear in the pairs, and no
[pairs, Lq, Ld] similarity grid is ever allocated (the colpali PR "Add support
for late-interaction-kernels (LIK)", Results: the fused backward allocates
only the input gradients).  liblik allocates nothing of its own on these
paths, so torch's allocator statistics see every byte.
"""
import pytest
import torch

from late_interaction_retrieval_gb300 import layers
from late_interaction_retrieval_gb300.workloads import generate

pytestmark = pytest.mark.gpu

SLACK = 4 << 20  # allocator rounding


def _peak_extra(fn):
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    fn()
    torch.cuda.synchronize()
    return torch.cuda.max_memory_allocated() - base


@pytest.mark.parametrize("recompute", [False, True], ids=["saved-argmax", "recompute"])
def test_inbatch_step_extra_memory_is_outputs_only(recompute):
    inp = generate("inbatch_b128_bf16", device="cuda")
    Q = inp.Q.detach().requires_grad_()
    D = inp.D.detach().requires_grad_()
    nq, lq, _ = Q.shape
    nd, ld, _ = D.shape
    g = torch.randn(nq, nd, device="cuda")

    def step():
        layers.maxsim(Q, D, inp.qmask, inp.dmask, recompute=recompute).backward(g)

    peak = _peak_extra(step)
    scores, argmax = nq * nd * 4, nq * nd * lq * 4
    grads16 = (Q.numel() + D.numel()) * 2
    if recompute:
        # the argmax workspace and fp32 gradients live only inside the backward,
        # next to their bf16 casts
        expected = scores + argmax + 2 * grads16 + grads16
    else:
        # the forward saves the argmax; the backward writes bf16 gradients directly
        expected = scores + argmax + grads16
    grid = nq * nd * lq * ld * 4
    assert peak <= expected + SLACK, (peak, expected)
    assert peak < grid / 20, (peak, grid)
    assert Q.grad is not None and D.grad is not None
