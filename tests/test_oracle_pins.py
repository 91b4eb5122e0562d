"""The CPU oracle against hand-worked examples, library routines, brute-force
float64 evaluation and invariants (no GPU)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def test_layer_stages_consistent():
    P.check_layer_consistency()
