"""The CPU oracle against its pins (no GPU).  See oracle_checks.py for what
each check compares the oracle with."""
import pytest

import oracle_checks as C


@pytest.mark.parametrize("check", C.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check, olib):
    check(olib)
