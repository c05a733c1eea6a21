"""The fp64 oracle against what the pages and the mathematics fix.

Every pin in ``tests/pins.py`` is an independent statement (another form of
the update, an invariant, a closed form or a brute-force expansion).  The
oracle must satisfy all of them to fp64 rounding, and every planted mistake
in ``tests/mutants.py`` must fail at least one.  CPU only.
"""
import numpy as np
import pytest

from tests import mutants, pins


def _oracle_run(oracle_lib):
    def run(q, k, v, beta, S0):
        return oracle_lib.forward(q, k, v, beta, S0, nthreads=2)
    return run


@pytest.mark.parametrize("name", sorted(pins.ALL_PINS))
def test_oracle_satisfies_pin(oracle_lib, name):
    err = pins.ALL_PINS[name](_oracle_run(oracle_lib))
    assert err <= pins.PIN_TOL, f"pin {name}: max error {err:.3e}"


def _fails_some_pin(run):
    failed = []
    for name, pin in pins.ALL_PINS.items():
        try:
            err = pin(run)
        except Exception:  # a shape error counts as a failure
            err = np.inf
        if not err <= pins.PIN_TOL:
            failed.append(name)
    return failed


@pytest.mark.parametrize("name", sorted(mutants.ALL_MUTANTS))
def test_planted_mistake_is_caught(name):
    failed = _fails_some_pin(mutants.ALL_MUTANTS[name])
    assert failed, f"planted mistake {name} passed every pin"


def test_correct_restatement_passes_every_pin():
    """Control for the mutation test: the unbroken numpy loop passes."""
    def correct(q, k, v, beta, S0):
        def step(S, qt, kt, vt, bt, kprev):
            S = S + np.outer(bt * (vt - S @ kt), kt)
            return S, S @ qt
        return mutants._loop(q, k, v, beta, S0, step)
    assert _fails_some_pin(correct) == []


def test_oracle_threads_do_not_change_results(oracle_lib):
    q, k, v, beta, S0 = pins.random_case(21, B=3, H=5, T=33, dk=6, dv=4)
    o1, S1 = oracle_lib.forward(q, k, v, beta, S0, nthreads=1)
    o4, S4 = oracle_lib.forward(q, k, v, beta, S0, nthreads=4)
    assert np.array_equal(o1, o4) and np.array_equal(S1, S4)


def test_oracle_empty_sequence(oracle_lib):
    q, k, v, beta, S0 = pins.random_case(22, T=0)
    o, S = oracle_lib.forward(q, k, v, beta, S0)
    assert o.shape == (2, 2, 0, 7) and np.array_equal(S, S0)


def test_oracle_decode_step_matches_one_token(oracle_lib):
    q, k, v, beta, S0 = pins.random_case(23, T=1)
    o, S = oracle_lib.recurrent_step(q[:, :, 0], k[:, :, 0], v[:, :, 0],
                                     beta[:, :, 0], S0)
    o_ref, S_ref = oracle_lib.forward(q, k, v, beta, S0)
    assert np.array_equal(o, o_ref[:, :, 0]) and np.array_equal(S, S_ref)


def test_oracle_recall_workload_closed_form(oracle_lib):
    """The recall workload's expected output is the stored value of each
    re-queried key; bf16 rounding of the keys keeps the match approximate."""
    import workloads
    inp, expect = workloads.workload_inputs("recall_bf16", B=1, H=2, T=256)
    o, _ = oracle_lib.forward(inp.q, inp.k, inp.v, inp.beta, None)
    from tests.conftest import rel_l2
    assert rel_l2(o, expect) < 1e-2


def test_oracle_varlen_is_independent_sequences(oracle_lib):
    """Packed sequences equal the same sequences run as a padded batch (each
    from its own state; padding tokens have beta = 0 and k = 0, which is
    exactly neutral), which the pinned forward computes."""
    r = np.random.default_rng(51)
    lens = [0, 1, 17, 64, 65, 30]
    cu = np.concatenate([[0], np.cumsum(lens)])
    H, dk, dv, T = 2, 5, 7, int(cu[-1])
    q = r.standard_normal((H, T, dk))
    k = r.standard_normal((H, T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((H, T, dv))
    beta = r.uniform(0.1, 1.0, (H, T))
    S0 = r.standard_normal((len(lens), H, dk, dv))
    o, S_T = oracle_lib.forward_varlen(q, k, v, beta, cu, S0)
    L = max(lens)
    pad = lambda x, n, w: np.concatenate([x, np.zeros(x.shape[:1] + (L - n,) + x.shape[2:])], 1)
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        ln = b - a
        ob, Sb = oracle_lib.forward(pad(q[:, a:b], ln, dk)[None], pad(k[:, a:b], ln, dk)[None],
                                    pad(v[:, a:b], ln, dv)[None], pad(beta[:, a:b], ln, 1)[None],
                                    S0[n][None])
        assert np.allclose(o[:, a:b], ob[0, :, :ln], rtol=0, atol=1e-12)
        assert np.allclose(S_T[n], Sb[0], rtol=0, atol=1e-12)
