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
The preparation's gradient (``oracle.prepare_qk_backward``) is held the same
way to central finite differences of the forward and to closed forms.
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


# ---- the preparation's gradient (oracle.prepare_qk_backward) ------------------
#
# Each pin takes the gradient as ``bwd(q, k, d_q, d_k, scale, l2norm, eps)``.
# The central pin differentiates the (pinned) forward preparation numerically,
# so it shares nothing with the gradient's own code.

def _oracle_bwd(q, k, d_q, d_k, scale, l2norm, eps):
    return oracle.prepare_qk_backward(q, k, d_q, d_k, scale=scale, l2norm=l2norm, eps=eps)


def bpin_finite_differences(bwd):
    """<d_q, dq'/dx . e> by central differences of the forward preparation,
    every input coordinate of a few rows, against the analytic gradient."""
    r = np.random.default_rng(3)
    q, k = r.standard_normal((2, 3, 6)), r.standard_normal((2, 3, 6))
    dq, dk = r.standard_normal(q.shape), r.standard_normal(k.shape)
    s, eps, h = 0.375, 1e-3, 1e-6
    gq, gk = bwd(q, k, dq, dk, s, True, eps)
    num_q, num_k = np.zeros_like(q), np.zeros_like(k)
    for idx in np.ndindex(q.shape):
        for x, num, is_q in ((q, num_q, True), (k, num_k, False)):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = (xp, k) if is_q else (q, xp)
            args_m = (xm, k) if is_q else (q, xm)
            yp = oracle.prepare_qk(*args_p, scale=s, l2norm=True, eps=eps)
            ym = oracle.prepare_qk(*args_m, scale=s, l2norm=True, eps=eps)
            num[idx] = (np.sum(dq * (yp[0] - ym[0])) + np.sum(dk * (yp[1] - ym[1]))) / (2 * h)
    return np.max(np.abs(gq - num_q)) < 1e-7 and np.max(np.abs(gk - num_k)) < 1e-7


def bpin_gradient_orthogonal_to_the_row(bwd):
    """With eps = 0 the output does not change along x itself, so x . dx = 0."""
    r = np.random.default_rng(4)
    x, g = r.standard_normal((5, 32)), r.standard_normal((5, 32))
    gq, _ = bwd(x, x, g, g, 2.0, True, 0.0)
    return np.max(np.abs(np.sum(gq * x, axis=-1))) < 1e-13


def bpin_scale_only(bwd):
    """Without the normalisation: dq = scale dq', dk = dk'."""
    r = np.random.default_rng(5)
    x, g = r.standard_normal((4, 16)), r.standard_normal((4, 16))
    gq, gk = bwd(x, x, g, g, 0.25, False, 1e-6)
    return bool(np.array_equal(gq, 0.25 * g) and np.array_equal(gk, g))


def bpin_zero_row(bwd):
    """At x = 0 the map is x scale / sqrt(eps): dx = scale dy / sqrt(eps)."""
    g = np.arange(1.0, 9.0).reshape(1, 8)
    gq, gk = bwd(np.zeros((1, 8)), np.zeros((1, 8)), g, g, 3.0, True, 0.25)
    return np.max(np.abs(gq - 6.0 * g)) < 1e-14 and np.max(np.abs(gk - 2.0 * g)) < 1e-14


def bpin_inverse_scaling_in_x(bwd):
    """With eps = 0 the output is invariant to x -> c x, so dx scales as 1/c."""
    r = np.random.default_rng(6)
    x, g = r.standard_normal((3, 8)), r.standard_normal((3, 8))
    g1, _ = bwd(x, x, g, g, 1.0, True, 0.0)
    g4, _ = bwd(4.0 * x, x, g, g, 1.0, True, 0.0)
    return np.max(np.abs(g4 - g1 / 4.0)) < 1e-14


BPINS = {f.__name__[5:]: f for f in (
    bpin_finite_differences, bpin_gradient_orthogonal_to_the_row, bpin_scale_only,
    bpin_zero_row, bpin_inverse_scaling_in_x)}


def _bwd_mutant(slip):
    def bwd(q, k, d_q, d_k, scale, l2norm, eps):
        def one(x, g, s):
            x, g = np.asarray(x, np.float64), np.asarray(g, np.float64)
            if not l2norm:
                return (1.0 if slip == "scale_dropped" else s) * g
            n2 = np.sum(x * x, axis=-1, keepdims=True) + eps
            n = np.sqrt(n2)
            xg = np.sum(x * g, axis=-1, keepdims=True)
            if slip == "missing_1_over_n2":
                return s / n * (g - x * xg)
            if slip == "wrong_sign":
                return s / n * (g + x * xg / n2)
            if slip == "scale_dropped":
                return 1.0 / n * (g - x * xg / n2)
            return s / n * (g - x * xg / n2)
        kscale = scale if slip == "keys_scaled" else 1.0
        return one(q, d_q, scale), one(k, d_k, kscale)
    return bwd


BMUTANTS = {name: _bwd_mutant(name) for name in
            ("missing_1_over_n2", "wrong_sign", "scale_dropped", "keys_scaled")}


@pytest.mark.parametrize("name", sorted(BPINS))
def test_oracle_gradient_satisfies_pin(oracle_lib, name):
    assert BPINS[name](_oracle_bwd), name


def test_a_correct_numpy_gradient_passes_every_pin(oracle_lib):
    right = _bwd_mutant("none")
    assert [n for n, pin in BPINS.items() if not pin(right)] == []


@pytest.mark.parametrize("name", sorted(BMUTANTS))
def test_planted_gradient_mistake_is_caught(oracle_lib, name):
    failed = [n for n, pin in BPINS.items() if not pin(BMUTANTS[name])]
    assert failed, f"mutant {name} passes every pin"
