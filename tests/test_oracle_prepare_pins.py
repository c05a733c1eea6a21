"""The oracle's input preparation (optional q/k L2 normalisation and the query
scale) against closed forms and invariants.  CPU only.

The preparation is the l2norm helper of the Gated DeltaNet PyTorch code on
"DeltaNet 引入 Delta Rule" (garden.houmin.site/infra/delta-net): a row x
becomes x / sqrt(sum x^2 + eps), eps = 1e-6, and the queries are divided by
the square root of the head dimension; the KDA read of "Kimi Delta
Attention" (fr.news.hada.io/topic?id=31925) scales q by d_k^{-1/2}.  The
pins below fail for an eps outside the square root, a missing square root,
a scale applied to k or before the normalisation, and a norm over the wrong
axis.
"""
from fractions import Fraction

import numpy as np
import pytest


def _rows(*rows):
    return np.array(rows, dtype=np.float64)


def test_pythagorean_rows_normalise_to_exact_fractions(oracle_lib):
    # rows whose norms are integers: (3,4,0) -> 5, (2,3,6) -> 7, (1,4,8) -> 9
    x = _rows([3, 4, 0], [2, 3, 6], [1, 4, 8])
    norms = [5, 7, 9]
    qn, kn = oracle_lib.prepare_qk(x, x, l2norm=True, eps=0.0)
    want = np.array([[float(Fraction(int(c), n)) for c in row]
                     for row, n in zip(x, norms)])
    assert np.max(np.abs(qn - want)) < 1e-15
    assert np.max(np.abs(kn - want)) < 1e-15


def test_scale_multiplies_the_normalised_queries_only(oracle_lib):
    x = _rows([2, 3, 6], [1, 4, 8])
    qs, ks = oracle_lib.prepare_qk(x, x, scale=63.0, l2norm=True, eps=0.0)
    # 63 * (2,3,6)/7 = (18,27,54); 63 * (1,4,8)/9 = (7,28,56)
    assert np.max(np.abs(qs - _rows([18, 27, 54], [7, 28, 56]))) < 1e-12
    assert np.max(np.abs(ks - _rows([2 / 7, 3 / 7, 6 / 7], [1 / 9, 4 / 9, 8 / 9]))) < 1e-15


def test_eps_sits_inside_the_square_root(oracle_lib):
    # sum x^2 = 3e-6; with eps = 1e-6 the denominator is sqrt(4e-6) = 2e-3
    x = _rows([1e-3, 1e-3, 1e-3])
    qn, _ = oracle_lib.prepare_qk(x, x, l2norm=True, eps=1e-6)
    assert np.max(np.abs(qn - 0.5)) < 1e-12


def test_zero_rows_stay_zero(oracle_lib):
    x = np.zeros((2, 3, 8))
    qn, kn = oracle_lib.prepare_qk(x, x, scale=0.125, l2norm=True)
    assert np.all(qn == 0) and np.all(kn == 0)


def test_scale_alone_leaves_the_keys_untouched(oracle_lib):
    r = np.random.default_rng(0)
    q, k = r.standard_normal((2, 3, 5, 16)), r.standard_normal((2, 3, 5, 16))
    qs, ks = oracle_lib.prepare_qk(q, k, scale=0.25)
    assert np.array_equal(ks, k)
    assert np.array_equal(qs, q * 0.25)   # a power of two: exact


def test_rows_have_unit_norm_and_keep_their_direction(oracle_lib):
    """Normalised over the last axis: every row has norm 1 (eps = 0), is a
    positive multiple of its input, and is unchanged by rescaling the input."""
    r = np.random.default_rng(1)
    x = r.standard_normal((3, 4, 7, 32))
    y, _ = oracle_lib.prepare_qk(x, x, l2norm=True, eps=0.0)
    assert np.max(np.abs(np.linalg.norm(y, axis=-1) - 1.0)) < 1e-14
    cos = np.sum(x * y, axis=-1) / np.linalg.norm(x, axis=-1)
    assert np.max(np.abs(cos - 1.0)) < 1e-14
    y5, _ = oracle_lib.prepare_qk(5.0 * x, x, l2norm=True, eps=0.0)
    assert np.max(np.abs(y5 - y)) < 1e-14


@pytest.mark.parametrize("s", [0.5, 128 ** -0.5])
def test_query_scale_scales_the_outputs_not_the_state(oracle_lib, s):
    """The read is linear in q and q never enters the state, so preparing
    with scale s multiplies every output by s and leaves S_T as it was."""
    r = np.random.default_rng(2)
    B, H, T, d = 1, 2, 19, 8
    q, k = r.standard_normal((B, H, T, d)), r.standard_normal((B, H, T, d))
    v = r.standard_normal((B, H, T, d))
    beta = r.uniform(0, 1, (B, H, T))
    S0 = r.standard_normal((B, H, d, d))
    q1, k1 = oracle_lib.prepare_qk(q, k, l2norm=True)
    qs, ks = oracle_lib.prepare_qk(q, k, scale=s, l2norm=True)
    o1, S1 = oracle_lib.forward(q1, k1, v, beta, S0, nthreads=1)
    os_, Ss = oracle_lib.forward(qs, ks, v, beta, S0, nthreads=1)
    assert np.max(np.abs(os_ - s * o1)) < 1e-12 * max(1.0, np.max(np.abs(o1)))
    assert np.array_equal(Ss, S1)
