"""The autograd wrapper's host logic on the CPU.

``DeltaRule`` only wires library calls together: the query scale before the
forward, the state recomputing backward, the scale's chain rule on d_q.
Here the three library calls are replaced by fakes backed by the fp64
oracle (the library itself needs a GPU), so the wiring is checked without
one: the gradients must be the oracle's for s q, with d_q multiplied by s.
"""
import numpy as np
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import oracle


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a))


@pytest.fixture
def fakes(monkeypatch):
    calls = []

    def qk_prepare(q, k, scale=1.0, l2norm=True, eps=1e-6, inplace=False):
        assert not l2norm
        calls.append(("qk_prepare", inplace))
        if inplace:
            q.mul_(scale)
            return q, k
        return q * scale, k

    def chunk_fwd(q, k, v, beta, initial_state=None, output_final_state=True, **_):
        calls.append(("chunk_fwd",))
        o, S = oracle.forward(q, k, v, beta, initial_state, nthreads=1)
        return _t(o), _t(S)

    def chunk_bwd(q, k, v, beta, d_o, initial_state=None, d_final_state=None, **_):
        calls.append(("chunk_bwd",))
        return tuple(_t(g) for g in oracle.backward(q, k, v, beta, d_o, initial_state,
                                                    d_final_state, nthreads=1))

    monkeypatch.setattr(dn, "qk_prepare", qk_prepare)
    monkeypatch.setattr(dn, "chunk_fwd", chunk_fwd)
    monkeypatch.setattr(dn, "chunk_bwd", chunk_bwd)
    return calls


def _inputs(seed=0, B=1, H=2, T=21, d=8):
    r = np.random.default_rng(seed)
    q, k = r.standard_normal((B, H, T, d)), r.standard_normal((B, H, T, d))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((B, H, T, d))
    beta = r.uniform(0, 1, (B, H, T))
    S0 = 0.1 * r.standard_normal((B, H, d, d))
    d_o = r.standard_normal((B, H, T, d))
    # the wrapper hands the state gradient on in fp32, the library's state type
    d_S = r.standard_normal((B, H, d, d)).astype(np.float32).astype(np.float64)
    return q, k, v, beta, S0, d_o, d_S


@pytest.mark.parametrize("scale", [None, 0.25, 8 ** -0.5])
def test_scale_chain_rule(fakes, scale):
    q, k, v, beta, S0, d_o, d_S = _inputs()
    leaves = [_t(x).requires_grad_() for x in (q, k, v, beta, S0)]
    o, S_T = dn.DeltaRule.apply(*leaves, scale)
    torch.autograd.backward([o, S_T], [_t(d_o), _t(d_S)])
    s = 1.0 if scale is None else scale
    o_ref, S_ref = oracle.forward(s * q, k, v, beta, S0, nthreads=1)
    assert np.allclose(o.detach().numpy(), o_ref, rtol=0, atol=1e-12)
    assert np.allclose(S_T.detach().numpy(), S_ref, rtol=0, atol=1e-12)
    ref = list(oracle.backward(s * q, k, v, beta, d_o, S0, d_S, nthreads=1))
    ref[0] = ref[0] * s
    for leaf, want in zip(leaves, ref):
        assert np.allclose(leaf.grad.numpy(), want, rtol=0, atol=1e-12)
    prep = [c for c in fakes if c[0] == "qk_prepare"]
    # one preparation before the forward and one in place on d_q, only with a scale
    assert prep == ([] if scale is None else [("qk_prepare", False), ("qk_prepare", True)])


def test_scaled_gradient_matches_finite_differences_of_the_scaled_forward(fakes):
    """The q gradient of <d_o, o(s q)> by central differences on a few
    coordinates: the wrapper's d_q = s * (gradient at s q)."""
    q, k, v, beta, S0, d_o, _ = _inputs(seed=1, T=9, d=4)
    s, h = 0.3, 1e-6
    leaf = _t(q).requires_grad_()
    o, _ = dn.DeltaRule.apply(leaf, _t(k), _t(v), _t(beta), _t(S0), s)
    o.backward(_t(d_o))
    for idx in [(0, 0, 0, 0), (0, 1, 4, 2), (0, 0, 8, 3)]:
        qp, qm = q.copy(), q.copy()
        qp[idx] += h
        qm[idx] -= h
        fp = np.sum(d_o * oracle.forward(s * qp, k, v, beta, S0, nthreads=1)[0])
        fm = np.sum(d_o * oracle.forward(s * qm, k, v, beta, S0, nthreads=1)[0])
        assert abs(leaf.grad[idx].item() - (fp - fm) / (2 * h)) < 1e-7
