"""The committed oracle passes every pin in tests/pins.py."""
import pytest

import oracle
from tests import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(orc, check):
    check(orc)


def test_oracle_uses_threads(orc):
    assert orc.num_threads() >= 1
