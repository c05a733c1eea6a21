"""The oracle's input preparation (optional q/k L2 normalisation and the query
scale) against closed forms and invariants.  CPU only.

The preparation is the l2norm helper of the Gated DeltaNet PyTorch code on
"DeltaNet 引入 Delta Rule" (garden.houmin.site/infra/delta-net): a row x
becomes x / sqrt(sum x^2 + eps), eps = 1e-6, and the queries are divided by
the square root of the head dimension; the KDA read of "Kimi Delta
Attention" (fr.news.hada.io/topic?id=31925) scales q by d_k^{-1/2}.

Each pin takes the preparation as a function ``prep(q, k, scale, l2norm,
eps) -> (q', k')`` and returns True when it holds.  The oracle must pass
every pin, and each planted mistake below (a plausible slip in writing the
preparation, planted in a numpy copy on the CPU) must fail at least one.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _rows(*rows):
    return np.array(rows, dtype=np.float64)


def pin_pythagorean_rows(prep):
    """Rows whose norms are integers normalise to exact fractions:
    (3,4,0) -> /5, (2,3,6) -> /7, (1,4,8) -> /9."""
    x = _rows([3, 4, 0], [2, 3, 6], [1, 4, 8])
    qn, kn = prep(x, x, 1.0, True, 0.0)
    want = np.array([[float(Fraction(int(c), n)) for c in row]
                     for row, n in zip(x, [5, 7, 9])])
    return np.max(np.abs(qn - want)) < 1e-15 and np.max(np.abs(kn - want)) < 1e-15


def pin_scale_on_normalised_queries_only(prep):
    """63 (2,3,6)/7 = (18,27,54) and 63 (1,4,8)/9 = (7,28,56); keys unscaled."""
    x = _rows([2, 3, 6], [1, 4, 8])
    qs, ks = prep(x, x, 63.0, True, 0.0)
    return (np.max(np.abs(qs - _rows([18, 27, 54], [7, 28, 56]))) < 1e-12
            and np.max(np.abs(ks - _rows([2 / 7, 3 / 7, 6 / 7], [1 / 9, 4 / 9, 8 / 9]))) < 1e-15)


def pin_eps_inside_the_root(prep):
    """sum x^2 = 3e-6 and eps = 1e-6: the denominator is sqrt(4e-6) = 2e-3."""
    x = _rows([1e-3, 1e-3, 1e-3])
    qn, _ = prep(x, x, 1.0, True, 1e-6)
    return np.max(np.abs(qn - 0.5)) < 1e-12


def pin_zero_rows_stay_zero(prep):
    x = np.zeros((2, 3, 8))
    qn, kn = prep(x, x, 0.125, True, 1e-6)
    return bool(np.all(qn == 0) and np.all(kn == 0))


def pin_scale_alone(prep):
    """Without the normalisation the keys come back unchanged and the
    queries are multiplied by the scale (a power of two: exactly)."""
    r = np.random.default_rng(0)
    q, k = r.standard_normal((2, 3, 5, 16)), r.standard_normal((2, 3, 5, 16))
    qs, ks = prep(q, k, 0.25, False, 1e-6)
    return bool(np.array_equal(ks, k) and np.array_equal(qs, q * 0.25))


def pin_unit_rows_along_the_last_axis(prep):
    """Every row (last axis) has norm 1 (eps = 0), is a positive multiple of
    its input, and is unchanged by rescaling the input."""
    r = np.random.default_rng(1)
    x = r.standard_normal((3, 4, 7, 32))
    y, _ = prep(x, x, 1.0, True, 0.0)
    y5, _ = prep(5.0 * x, x, 1.0, True, 0.0)
    cos = np.sum(x * y, axis=-1) / np.linalg.norm(x, axis=-1)
    return (np.max(np.abs(np.linalg.norm(y, axis=-1) - 1.0)) < 1e-14
            and np.max(np.abs(cos - 1.0)) < 1e-14 and np.max(np.abs(y5 - y)) < 1e-14)


def pin_scale_scales_the_outputs_not_the_state(prep, s=128 ** -0.5):
    """The read is linear in q and q never enters the state: preparing with
    scale s multiplies every output of the (pinned) recurrence by s and
    leaves S_T as it was."""
    r = np.random.default_rng(2)
    B, H, T, d = 1, 2, 19, 8
    q, k = r.standard_normal((B, H, T, d)), r.standard_normal((B, H, T, d))
    v = r.standard_normal((B, H, T, d))
    beta = r.uniform(0, 1, (B, H, T))
    S0 = r.standard_normal((B, H, d, d))
    q1, k1 = prep(q, k, 1.0, True, 1e-6)
    qs, ks = prep(q, k, s, True, 1e-6)
    o1, S1 = oracle.forward(q1, k1, v, beta, S0, nthreads=1)
    os_, Ss = oracle.forward(qs, ks, v, beta, S0, nthreads=1)
    return (np.max(np.abs(os_ - s * o1)) < 1e-12 * max(1.0, np.max(np.abs(o1)))
            and np.array_equal(Ss, S1))


PINS = {f.__name__[4:]: f for f in (
    pin_pythagorean_rows, pin_scale_on_normalised_queries_only, pin_eps_inside_the_root,
    pin_zero_rows_stay_zero, pin_scale_alone, pin_unit_rows_along_the_last_axis,
    pin_scale_scales_the_outputs_not_the_state)}


def _oracle_prep(q, k, scale, l2norm, eps):
    return oracle.prepare_qk(q, k, scale=scale, l2norm=l2norm, eps=eps)


# ---- planted mistakes (numpy copies of the preparation, each with one slip) ----

def _mutant(norm, scale_k=False, scale_first=False):
    def prep(q, k, scale, l2norm, eps):
        q, k = np.asarray(q, np.float64), np.asarray(k, np.float64)
        if scale_first:
            q = q * scale
        if l2norm:
            q, k = norm(q, eps), norm(k, eps)
        if not scale_first:
            q = q * scale
        if scale_k:
            k = k * scale
        return q, k
    return prep


def _right(x, eps):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


MUTANTS = {
    "eps_outside_the_root": _mutant(
        lambda x, eps: x / (np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) + eps)),
    "no_square_root": _mutant(lambda x, eps: x / (np.sum(x * x, axis=-1, keepdims=True) + eps)),
    "norm_over_the_wrong_axis": _mutant(
        lambda x, eps: x / np.sqrt(np.sum(x * x, axis=-2, keepdims=True) + eps)),
    "keys_scaled_too": _mutant(_right, scale_k=True),
    "scale_before_the_norm": _mutant(_right, scale_first=True),
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_oracle_satisfies_pin(oracle_lib, name):
    assert PINS[name](_oracle_prep), name


def test_a_correct_numpy_preparation_passes_every_pin():
    right = _mutant(_right)
    assert [n for n, pin in PINS.items() if not pin(right)] == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle_lib, name):
    failed = []
    for pin_name, pin in PINS.items():
        try:
            ok = pin(MUTANTS[name])
        except Exception:  # a shape error counts as a failure
            ok = False
        if not ok:
            failed.append(pin_name)
    assert failed, f"mutant {name} passes every pin"
