"""The CPU oracle against closed forms, exact arithmetic, numpy and invariants."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(oracle_mod, pin):
    pin(oracle_mod.default())


def test_bad_arguments_rejected(oracle_mod):
    import ctypes
    lib = oracle_mod.default()._lib
    # lda < K
    rc = lib.oracle_sgemm(2, 2, 3, 1.0, None, 2, None, 2, 0.0, None, 2, None, None, None, 2, 1)
    assert rc == 1
    # negative M
    rc = lib.oracle_sgemm(-1, 2, 3, 1.0, None, 3, None, 2, 0.0, None, 2, None, None, None, 2, 1)
    assert rc == 1
    del ctypes


def test_error_ratio_semantics(oracle_mod):
    import numpy as np
    ref = np.array([1.0, 0.0, 2.0])
    den = np.array([1.0, 0.0, 4.0])
    assert oracle_mod.error_ratio(np.array([1.5, 0.0, 2.0]), ref, den) == 0.5
    assert oracle_mod.error_ratio(np.array([1.0, 1e-30, 2.0]), ref, den) == float("inf")
    assert oracle_mod.error_ratio(np.array([np.nan, 0.0, 2.0]), ref, den) == float("inf")
