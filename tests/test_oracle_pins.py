"""The CPU oracle against the pages' worked examples, closed forms, an
independent brute force, torch SDPA and structural identities."""
import pytest

import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle_lib, check):
    check(oracle_lib.default())
