"""The oracle against the pages' worked examples, brute force and exact arithmetic."""

import pytest

import oracle_checks as C


@pytest.mark.parametrize("check", C.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()
