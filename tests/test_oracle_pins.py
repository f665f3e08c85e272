"""The oracle against its pins (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)


def test_thread_control(orc):
    n = orc.num_threads()
    assert n >= 1
    orc.set_num_threads(1)
    assert orc.num_threads() == 1
    orc.set_num_threads(n)
    assert orc.num_threads() == n
