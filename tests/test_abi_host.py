"""liblik loads, exports every entry point of include/lik.h, and rejects bad
arguments on the host before touching a GPU (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

from late_interaction_retrieval_gb300 import binding
from late_interaction_retrieval_gb300 import build as lik_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lik.h")


def declared_entry_points():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lik_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    path = lik_build.build()
    return binding.load(path)


def test_header_declares_the_abi():
    names = declared_entry_points()
    for n in ("lik_maxsim_allpairs_fwd", "lik_maxsim_allpairs_bwd", "lik_maxsim_pairwise_fwd",
              "lik_maxsim_pairwise_bwd", "lik_maxsim_kd_fwd", "lik_maxsim_kd_bwd",
              "lik_status_string", "lik_check_device_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), f"{name} declared in lik.h but not exported"
        assert name in binding.SIGNATURES, f"{name} has no binding signature"


def test_exports_are_c_symbols():
    out = os.popen(f"nm -D --defined-only {lik_build.LIB_PATH}").read()
    for name in declared_entry_points():
        assert re.search(rf"\bT {name}$", out, re.M), f"{name} is not an exported C symbol"


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert lib.lik_status_string(code).decode() == name
    assert lib.lik_status_string(99).decode() == "LIK_ERR_UNKNOWN_STATUS"
    assert lib.lik_version().decode().count(".") == 2


# Calls below return before any CUDA call: argument errors are found first.
NULL = None


def _fwd(lib, dtype=2, Nq=2, Nd=3, Lq=4, Ld=5, dim=128):
    return lib.lik_maxsim_allpairs_fwd(NULL, NULL, dtype, Nq, Nd, Lq, Ld, dim,
                                       NULL, NULL, NULL, NULL, NULL)


def test_invalid_dtype(lib):
    assert _fwd(lib, dtype=7) == 1
    assert "dtype" in lib.lik_last_error_message().decode()


@pytest.mark.parametrize("field", ["Nq", "Nd", "Lq", "Ld"])
def test_negative_sizes(lib, field):
    kw = {field: -1}
    assert _fwd(lib, **kw) == 1


def test_dim_limits(lib):
    assert _fwd(lib, dim=0) == 1
    assert _fwd(lib, dim=1025) == 2
    assert _fwd(lib, Lq=4097) == 2


def test_zero_pairs_is_a_noop(lib):
    assert _fwd(lib, Nq=0) == 0
    assert _fwd(lib, Nd=0) == 0
    assert lib.lik_maxsim_pairwise_fwd(NULL, NULL, 0, 0, 4, 5, 8, NULL, NULL, NULL, NULL, NULL) == 0
    assert lib.lik_maxsim_kd_fwd(NULL, NULL, 0, 3, 0, 4, 5, 8, NULL, NULL, NULL, NULL, NULL) == 0


def test_message_cleared_on_next_call(lib):
    assert _fwd(lib, dtype=7) == 1
    assert lib.lik_last_error_message().decode() != ""
    assert _fwd(lib, Nq=0) == 0
    assert lib.lik_last_error_message().decode() == ""


def test_selftest_timeout_range(lib):
    assert lib.lik_selftest_bounded_wait(0, NULL) == 1
    assert lib.lik_selftest_bounded_wait(1000001, NULL) == 1
    assert "timeout_us" in lib.lik_last_error_message().decode()


def test_workspace_query_rejects_bad_arguments(lib):
    assert lib.lik_maxsim_pairwise_fwd_workspace_bytes(2, 4, 32, 100, 128, 1, NULL) == 1
    import ctypes
    out = ctypes.c_size_t(7)
    assert lib.lik_maxsim_kd_fwd_workspace_bytes(2, -1, 3, 32, 100, 128, 1, ctypes.byref(out)) == 1
    assert out.value == 0
    assert lib.lik_maxsim_kd_fwd_workspace_bytes(2, 0, 3, 32, 100, 128, 1, ctypes.byref(out)) == 0
    assert out.value == 0
