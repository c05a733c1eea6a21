"""The oracle's gradient against finite differences, identities, closed
forms and a chunk-level derivation (``tests/pins_bwd.py``); every planted
mistake in ``tests/mutants_bwd.py`` must fail at least one pin.  CPU only.
"""
import numpy as np
import pytest

from tests import mutants_bwd, pins_bwd


@pytest.fixture(scope="module")
def fwd(oracle_lib):
    return lambda q, k, v, beta, S0: oracle_lib.forward(q, k, v, beta, S0, nthreads=2)


@pytest.fixture(scope="module")
def grad(oracle_lib):
    return lambda q, k, v, beta, dO, S0, dS_T: oracle_lib.backward(
        q, k, v, beta, dO, S0, dS_T, nthreads=2)


@pytest.mark.parametrize("name", sorted(pins_bwd.ALL_BWD_PINS))
def test_oracle_gradient_satisfies_pin(grad, fwd, name):
    err = pins_bwd.ALL_BWD_PINS[name](grad, fwd)
    assert err <= 1.0, f"pin {name}: {err:.3e} of its bound"


def _fails_some_pin(grad, fwd):
    failed = []
    for name, pin in pins_bwd.ALL_BWD_PINS.items():
        try:
            err = pin(grad, fwd)
        except Exception:  # a shape error counts as a failure
            err = np.inf
        if not err <= 1.0:
            failed.append(name)
    return failed


@pytest.mark.parametrize("name", sorted(mutants_bwd.ALL_BWD_MUTANTS))
def test_planted_gradient_mistake_is_caught(fwd, name):
    assert _fails_some_pin(mutants_bwd.ALL_BWD_MUTANTS[name], fwd), \
        f"planted mistake {name} passed every gradient pin"


def test_correct_reverse_loop_passes_every_pin(fwd):
    """Control for the mutation test: the unbroken numpy reverse loop passes."""
    assert _fails_some_pin(mutants_bwd.reverse_loop, fwd) == []


def test_oracle_gradient_threads_and_optional_arguments(oracle_lib):
    q, k, v, beta, S0, dO, dS_T = pins_bwd.random_grad_case(36, B=2, H=3, T=17, dk=4, dv=6)
    g1 = oracle_lib.backward(q, k, v, beta, dO, S0, dS_T, nthreads=1)
    g4 = oracle_lib.backward(q, k, v, beta, dO, S0, dS_T, nthreads=4)
    assert all(np.array_equal(a, b) for a, b in zip(g1, g4))
    # None means zeros, for the initial state and for the final-state gradient
    z = oracle_lib.backward(q, k, v, beta, dO, None, None, nthreads=2)
    zz = oracle_lib.backward(q, k, v, beta, dO, np.zeros_like(S0), np.zeros_like(dS_T), nthreads=2)
    assert all(np.array_equal(a, b) for a, b in zip(z, zz))


def test_oracle_gradient_empty_sequence(oracle_lib):
    q = np.zeros((1, 2, 0, 3))
    v = np.zeros((1, 2, 0, 4))
    dS_T = np.arange(24, dtype=np.float64).reshape(1, 2, 3, 4)
    dq, dk, dv, db, dS0 = oracle_lib.backward(q, q, v, np.zeros((1, 2, 0)), v, None, dS_T)
    assert dq.shape == (1, 2, 0, 3) and db.shape == (1, 2, 0)
    assert np.array_equal(dS0, dS_T)
