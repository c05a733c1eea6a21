"""The oracle's Gated DeltaNet against zero-decay reduction, closed forms,
the normalised-state identity, the pages' product form and a chunk-level
derivation (``tests/pins_gated.py``); every planted mistake must fail at
least one pin.  CPU only.
"""
import numpy as np
import pytest

from tests import pins_gated


@pytest.fixture(scope="module")
def plain(oracle_lib):
    return lambda q, k, v, beta, S0: oracle_lib.forward(q, k, v, beta, S0, nthreads=2)


@pytest.fixture(scope="module")
def gated(oracle_lib):
    return lambda q, k, v, beta, g, S0: oracle_lib.forward_gated(q, k, v, beta, g, S0, nthreads=2)


@pytest.mark.parametrize("name", sorted(pins_gated.ALL_GATED_PINS))
def test_oracle_gated_satisfies_pin(gated, plain, name):
    err = pins_gated.ALL_GATED_PINS[name](gated, plain)
    assert err <= 1.0, f"pin {name}: {err:.3e} of its bound"


def _fails_some_pin(run, plain):
    failed = []
    for name, pin in pins_gated.ALL_GATED_PINS.items():
        try:
            err = pin(run, plain)
        except Exception:
            err = np.inf
        if not err <= 1.0:
            failed.append(name)
    return failed


@pytest.mark.parametrize("slip", pins_gated.GATED_SLIPS)
def test_planted_gated_mistake_is_caught(plain, slip):
    run = lambda q, k, v, beta, g, S0: pins_gated.gated_loop(q, k, v, beta, g, S0, slip=slip)
    assert _fails_some_pin(run, plain), f"planted mistake {slip} passed every pin"


def test_correct_gated_loop_passes_every_pin(plain):
    assert _fails_some_pin(pins_gated.gated_loop, plain) == []


def test_gated_decode_step_matches_one_token(oracle_lib):
    q, k, v, beta, g, S0 = pins_gated.random_gated_case(46, T=1)
    o1, S1 = oracle_lib.forward_gated(q, k, v, beta, g, S0)
    o2, S2 = oracle_lib.recurrent_step_gated(q[:, :, 0], k[:, :, 0], v[:, :, 0], beta[:, :, 0],
                                             g[:, :, 0], S0)
    assert np.array_equal(o1[:, :, 0], o2) and np.array_equal(S1, S2)
