"""The oracle against its pins (CPU only)."""
import pytest

import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def test_two_worker_hand_brute_force():
    pins.check_two_worker_hand("brute_force")


def test_brute_vs_method_more_seeds():
    pins.check_brute_vs_method(seeds=range(6, 14))
