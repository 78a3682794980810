"""The oracle against its pins (see oracle_checks.py for what pins what)."""
import pytest

import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda f: f.__name__[len("check_"):])
def test_oracle_pin(orc, check):
    check(orc)
