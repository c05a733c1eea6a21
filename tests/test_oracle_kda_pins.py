"""The oracle's KDA against the gated and plain oracles, closed forms, the
pages' DPLR form and a chunk-level derivation (``tests/pins_kda.py``); every
planted mistake must fail at least one pin.  CPU only.
"""
import numpy as np
import pytest

from tests import pins_kda


@pytest.fixture(scope="module")
def refs(oracle_lib):
    plain = lambda q, k, v, beta, S0: oracle_lib.forward(q, k, v, beta, S0, nthreads=2)
    gated = lambda q, k, v, beta, g, S0: oracle_lib.forward_gated(q, k, v, beta, g, S0, nthreads=2)
    return plain, gated


@pytest.fixture(scope="module")
def kda(oracle_lib):
    return lambda q, k, v, beta, g, S0: oracle_lib.forward_kda(q, k, v, beta, g, S0, nthreads=2)


@pytest.mark.parametrize("name", sorted(pins_kda.ALL_KDA_PINS))
def test_oracle_kda_satisfies_pin(kda, refs, name):
    err = pins_kda.ALL_KDA_PINS[name](kda, *refs)
    assert err <= 1.0, f"pin {name}: {err:.3e} of its bound"


def _fails_some_pin(run, refs):
    failed = []
    for name, pin in pins_kda.ALL_KDA_PINS.items():
        try:
            err = pin(run, *refs)
        except Exception:
            err = np.inf
        if not err <= 1.0:
            failed.append(name)
    return failed


@pytest.mark.parametrize("slip", pins_kda.KDA_SLIPS)
def test_planted_kda_mistake_is_caught(refs, slip):
    run = lambda q, k, v, beta, g, S0: pins_kda.kda_loop(q, k, v, beta, g, S0, slip=slip)
    assert _fails_some_pin(run, refs), f"planted mistake {slip} passed every pin"


def test_correct_kda_loop_passes_every_pin(refs):
    assert _fails_some_pin(pins_kda.kda_loop, refs) == []


def test_kda_decode_step_matches_one_token(oracle_lib):
    q, k, v, beta, g, S0 = pins_kda.random_kda_case(65, T=1)
    o1, S1 = oracle_lib.forward_kda(q, k, v, beta, g, S0)
    o2, S2 = oracle_lib.recurrent_step_kda(q[:, :, 0], k[:, :, 0], v[:, :, 0], beta[:, :, 0],
                                           g[:, :, 0], S0)
    assert np.array_equal(o1[:, :, 0], o2) and np.array_equal(S1, S2)
