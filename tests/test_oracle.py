"""The float64 oracle against its pins (closed forms, invariants, library cross-checks)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_invalid_problem_rejected(orc):
    from synth.workloads import custom
    p = custom("bad", 2, 2, 1, 64, [4, 4], "f16")
    p.cu[1] = 9  # cu no longer monotone
    with pytest.raises(ValueError):
        orc.attention(p)
    p = custom("bad2", 1, 3, 2, 64, [4], "f16")  # 3 query heads on 2 KV heads
    with pytest.raises(ValueError):
        orc.attention(p)
