"""The CPU oracle against facts outside itself (CPU only)."""
import numpy as np
import pytest

import oracle_pins


def test_dense_matrix_is_sylvester():
    oracle_pins.pin_dense_is_sylvester()


@pytest.mark.parametrize("pin", oracle_pins.ORACLE_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_lib, pin):
    pin(oracle_lib)


def test_threads_split_whole_vectors(oracle_lib):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 1 << 11))
    one = oracle_lib.fwt(x, normalize=True, nthreads=1)
    many = oracle_lib.fwt(x, normalize=True, nthreads=4)
    assert np.array_equal(one, many)
    xi = rng.integers(-8, 9, size=(5, 1 << 10), dtype=np.int32)
    assert np.array_equal(oracle_lib.fwt(xi, False, 1), oracle_lib.fwt(xi, False, 3))


def test_empty_batch_and_n0(oracle_lib):
    assert oracle_lib.fwt(np.zeros((0, 8)), normalize=True).shape == (0, 8)
    x = np.array([[2.5], [-1.0]])
    assert np.array_equal(oracle_lib.fwt(x, normalize=True), x)


def test_int_normalise_rejected(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.fwt(np.zeros((1, 4), np.int32), normalize=True)


def test_nonfinite_propagation(oracle_lib):
    # IEEE: an inf input reaches every output with its Walsh sign; inf - inf is NaN.
    x = np.zeros((1, 8))
    x[0, 3] = np.inf
    y = oracle_lib.fwt(x, normalize=False)[0]
    k = np.arange(8)
    assert np.array_equal(y, np.where(oracle_pins._popc_parity(k & 3) == 1, -np.inf, np.inf))
    x[0, 5] = np.inf
    y = oracle_lib.fwt(x, normalize=False)[0]
    both = oracle_pins._popc_parity(k & 3) != oracle_pins._popc_parity(k & 5)
    assert np.all(np.isnan(y[both])) and np.all(np.isinf(y[~both]))
