"""A bounded device wait that runs out reaches the caller as LIK_ERR_TIMEOUT (GPU).

Every mbarrier wait of the tensor-core kernels is bounded; when one runs out
the kernel sets the library's error word and stops.  In a healthy run no
wait runs out, so lik_selftest_bounded_wait makes one do so safely (one
thread, the same bounded wait with a 1 ms limit, an mbarrier that nothing
arrives at).  The status must come back through lik_check_device_error, be
cleared by it, and leave the context usable for the next call.
"""
import numpy as np
import pytest

import gpu_harness
import parity
from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300.workloads import random_case

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_is_reported_then_cleared():
    binding.lik_check_device_error()  # nothing pending
    binding.lik_selftest_bounded_wait(1000)
    with pytest.raises(binding.LIKError) as ei:
        binding.lik_check_device_error()
    assert ei.value.status_name == "LIK_ERR_TIMEOUT"
    binding.lik_check_device_error()  # the word was cleared
    # the context is still usable: a forward right after matches the oracle
    inp = random_case("allpairs", 3, 4, 32, 200, 128, "bf16", seed=77, p_doc_empty=0.2)
    h = gpu_harness.Layout(inp)
    s_g, _ = h.gpu_fwd()
    s_o, _, _ = h.oracle_fwd()
    parity.assert_scores_close(s_g, s_o, "bf16")
    assert np.isfinite(s_g).all()
