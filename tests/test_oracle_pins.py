"""The float64 oracle against its pins (CPU only)."""
import pytest

import oracle
from tests import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle.cosa_oracle)
