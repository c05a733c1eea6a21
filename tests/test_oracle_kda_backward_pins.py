"""The oracle's KDA gradient against finite differences, the gated gradient
on equal channels, a one-token closed form and a chunk-level derivation
(``tests/pins_kda_bwd.py``); a correct numpy reverse pass passes every pin
and each planted mistake fails at least one.  CPU only.
"""
import numpy as np
import pytest

from tests import pins_kda_bwd as P


@pytest.fixture(scope="module")
def fwd(oracle_lib):
    return lambda q, k, v, beta, g, S0: oracle_lib.forward_kda(q, k, v, beta, g, S0, nthreads=2)


@pytest.fixture(scope="module")
def grad(oracle_lib):
    return lambda q, k, v, beta, g, dO, S0, dS_T: oracle_lib.backward_kda(
        q, k, v, beta, g, dO, S0, dS_T, nthreads=2)


@pytest.fixture(scope="module")
def gated_grad(oracle_lib):
    return lambda q, k, v, beta, g, dO, S0, dS_T: oracle_lib.backward_gated(
        q, k, v, beta, g, dO, S0, dS_T, nthreads=2)


@pytest.mark.parametrize("name", sorted(P.ALL_KDA_BWD_PINS))
def test_oracle_kda_gradient_satisfies_pin(grad, fwd, gated_grad, name):
    err = P.ALL_KDA_BWD_PINS[name](grad, fwd, gated_grad)
    assert err <= 1.0, f"pin {name}: {err:.3e} of its bound"


def _numpy_grad(mistake):
    return lambda q, k, v, beta, g, dO, S0, dS_T: P.reverse_loop_kda(
        q, k, v, beta, g, dO, S0, dS_T, mistake)


@pytest.mark.parametrize("name", sorted(P.ALL_KDA_BWD_PINS))
def test_correct_numpy_reverse_pass_satisfies_pin(fwd, gated_grad, name):
    err = P.ALL_KDA_BWD_PINS[name](_numpy_grad(None), fwd, gated_grad)
    assert err <= 1.0, f"pin {name}: {err:.3e} of its bound"


@pytest.mark.parametrize("mistake", P.KDA_BWD_MISTAKES)
def test_planted_mistake_fails_a_pin(fwd, gated_grad, mistake):
    failed = []
    for name, pin in P.ALL_KDA_BWD_PINS.items():
        try:
            err = pin(_numpy_grad(mistake), fwd, gated_grad)
        except Exception:  # a shape error counts as a failure
            err = np.inf
        if not err <= 1.0:
            failed.append(name)
    assert failed, f"mistake {mistake} passes every pin"
