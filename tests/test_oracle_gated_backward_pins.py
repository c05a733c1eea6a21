"""The oracle's Gated DeltaNet gradient against finite differences, the plain
gradient at zero decay, a one-token closed form and a chunk-level derivation
(``tests/pins_gated_bwd.py``); a correct numpy reverse pass passes every pin
and each planted mistake fails at least one.  CPU only.
"""
import numpy as np
import pytest

from tests import pins_gated_bwd as P


@pytest.fixture(scope="module")
def fwd(oracle_lib):
    return lambda q, k, v, beta, g, S0: oracle_lib.forward_gated(q, k, v, beta, g, S0, nthreads=2)


@pytest.fixture(scope="module")
def grad(oracle_lib):
    return lambda q, k, v, beta, g, dO, S0, dS_T: oracle_lib.backward_gated(
        q, k, v, beta, g, dO, S0, dS_T, nthreads=2)


@pytest.fixture(scope="module")
def plain_grad(oracle_lib):
    return lambda q, k, v, beta, dO, S0, dS_T: oracle_lib.backward(
        q, k, v, beta, dO, S0, dS_T, nthreads=2)


def _run(pin, grad, fwd, plain_grad):
    if pin is P.pin_zero_decay:
        return pin(grad, fwd, plain_grad)
    return pin(grad, fwd)


@pytest.mark.parametrize("name", sorted(P.ALL_GATED_BWD_PINS))
def test_oracle_gated_gradient_satisfies_pin(grad, fwd, plain_grad, name):
    err = _run(P.ALL_GATED_BWD_PINS[name], grad, fwd, plain_grad)
    assert err <= 1.0, f"pin {name}: {err:.3e} of its bound"


def _numpy_grad(mistake):
    return lambda q, k, v, beta, g, dO, S0, dS_T: P.reverse_loop_gated(
        q, k, v, beta, g, dO, S0, dS_T, mistake)


@pytest.mark.parametrize("name", sorted(P.ALL_GATED_BWD_PINS))
def test_correct_numpy_reverse_pass_satisfies_pin(fwd, plain_grad, name):
    err = _run(P.ALL_GATED_BWD_PINS[name], _numpy_grad(None), fwd, plain_grad)
    assert err <= 1.0, f"pin {name}: {err:.3e} of its bound"


@pytest.mark.parametrize("mistake", P.GATED_BWD_MISTAKES)
def test_planted_mistake_fails_a_pin(fwd, plain_grad, mistake):
    failed = []
    for name, pin in P.ALL_GATED_BWD_PINS.items():
        try:
            err = _run(pin, _numpy_grad(mistake), fwd, plain_grad)
        except Exception:  # a shape error counts as a failure
            err = np.inf
        if not err <= 1.0:
            failed.append(name)
    assert failed, f"mistake {mistake} passes every pin"
