"""The autograd wrapper's host logic on the CPU.

``DeltaRule`` only wires library calls together: the forward (with the q/k
preparation inside its kernels), the state-recomputing backward on the
prepared q and k, and the preparation's gradient after it.  Here the library
calls are replaced by fakes backed by the fp64 oracle (the library itself
needs a GPU), so the wiring is checked without one: the gradients must be
the oracle's for the prepared inputs, carried back through the oracle's
gradient of the preparation, and must match finite differences of the whole
prepared forward.
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

    def chunk_fwd(q, k, v, beta, initial_state=None, output_final_state=True, scale=None,
                  qk_l2norm=False, **_):
        calls.append(("chunk_fwd", scale, bool(qk_l2norm)))
        qp, kp = oracle.prepare_qk(q, k, 1.0 if scale is None else scale, bool(qk_l2norm))
        o, S = oracle.forward(qp, kp, v, beta, initial_state, nthreads=1)
        return _t(o), _t(S)

    def qk_prepare(q, k, scale=1.0, l2norm=True, eps=1e-6, inplace=False):
        calls.append(("qk_prepare", scale, bool(l2norm)))
        qp, kp = oracle.prepare_qk(q, k, scale, l2norm, eps)
        return _t(qp), _t(kp)

    def qk_prepare_bwd(q, k, d_q_out, d_k_out, scale=1.0, l2norm=True, eps=1e-6):
        calls.append(("qk_prepare_bwd", scale, bool(l2norm)))
        gq, gk = oracle.prepare_qk_backward(q, k, d_q_out, d_k_out, scale, l2norm, eps)
        return _t(gq), (_t(gk) if l2norm else d_k_out)

    def chunk_bwd(q, k, v, beta, d_o, initial_state=None, d_final_state=None, **_):
        calls.append(("chunk_bwd",))
        return tuple(_t(g) for g in oracle.backward(q, k, v, beta, d_o, initial_state,
                                                    d_final_state, nthreads=1))

    monkeypatch.setattr(dn, "qk_prepare", qk_prepare)
    monkeypatch.setattr(dn, "qk_prepare_bwd", qk_prepare_bwd)
    monkeypatch.setattr(dn, "chunk_fwd", chunk_fwd)
    monkeypatch.setattr(dn, "chunk_bwd", chunk_bwd)
    return calls


def _inputs(seed=0, B=1, H=2, T=21, d=8, raw=False):
    r = np.random.default_rng(seed)
    q, k = r.standard_normal((B, H, T, d)), r.standard_normal((B, H, T, d))
    if not raw:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((B, H, T, d))
    beta = r.uniform(0, 1, (B, H, T))
    S0 = 0.1 * r.standard_normal((B, H, d, d))
    d_o = r.standard_normal((B, H, T, d))
    # the wrapper hands the state gradient on in fp32, the library's state type
    d_S = r.standard_normal((B, H, d, d)).astype(np.float32).astype(np.float64)
    return q, k, v, beta, S0, d_o, d_S


@pytest.mark.parametrize("scale,l2norm", [(None, False), (0.25, False), (8 ** -0.5, False),
                                          (None, True), (8 ** -0.5, True)])
def test_chain_rule_through_the_preparation(fakes, scale, l2norm):
    q, k, v, beta, S0, d_o, d_S = _inputs(raw=l2norm)
    leaves = [_t(x).requires_grad_() for x in (q, k, v, beta, S0)]
    o, S_T = dn.DeltaRule.apply(*leaves, scale, l2norm)
    torch.autograd.backward([o, S_T], [_t(d_o), _t(d_S)])
    s = 1.0 if scale is None else scale
    qp, kp = oracle.prepare_qk(q, k, s, l2norm)
    o_ref, S_ref = oracle.forward(qp, kp, v, beta, S0, nthreads=1)
    assert np.allclose(o.detach().numpy(), o_ref, rtol=0, atol=1e-12)
    assert np.allclose(S_T.detach().numpy(), S_ref, rtol=0, atol=1e-12)
    ref = list(oracle.backward(qp, kp, v, beta, d_o, S0, d_S, nthreads=1))
    ref[0], gk = oracle.prepare_qk_backward(q, k, ref[0], ref[1], s, l2norm)
    if l2norm:
        ref[1] = gk
    for leaf, want in zip(leaves, ref):
        assert np.allclose(leaf.grad.numpy(), want, rtol=0, atol=1e-12)
    prepared = scale is not None or l2norm
    names = [c[0] for c in fakes]
    assert names == (["chunk_fwd", "qk_prepare", "chunk_bwd", "qk_prepare_bwd"] if prepared
                     else ["chunk_fwd", "chunk_bwd"])


@pytest.mark.parametrize("l2norm", [False, True])
def test_gradient_matches_finite_differences_of_the_prepared_forward(fakes, l2norm):
    """q and k gradients of <d_o, o(prepare(q, k))> by central differences on
    a few coordinates of the raw inputs."""
    q, k, v, beta, S0, d_o, _ = _inputs(seed=1, T=9, d=4, raw=l2norm)
    s, h = 0.3, 1e-6
    lq, lk = _t(q).requires_grad_(), _t(k).requires_grad_()
    o, _ = dn.DeltaRule.apply(lq, lk, _t(v), _t(beta), _t(S0), s, l2norm)
    o.backward(_t(d_o))

    def loss(qx, kx):
        qp, kp = oracle.prepare_qk(qx, kx, s, l2norm)
        return np.sum(d_o * oracle.forward(qp, kp, v, beta, S0, nthreads=1)[0])

    for leaf, which in ((lq, 0), (lk, 1)):
        for idx in [(0, 0, 0, 0), (0, 1, 4, 2), (0, 0, 8, 3)]:
            xp = [q.copy(), k.copy()]
            xm = [q.copy(), k.copy()]
            xp[which][idx] += h
            xm[which][idx] -= h
            fd = (loss(*xp) - loss(*xm)) / (2 * h)
            assert abs(leaf.grad[idx].item() - fd) < 1e-7, (which, idx)


@pytest.fixture
def gated_fakes(monkeypatch):
    calls = []

    def chunk_fwd_gated(q, k, v, beta, g, initial_state=None, output_final_state=True,
                        scale=None, qk_l2norm=False, **_):
        calls.append("chunk_fwd_gated")
        qp, kp = oracle.prepare_qk(q, k, 1.0 if scale is None else scale, bool(qk_l2norm))
        o, S = oracle.forward_gated(qp, kp, v, beta, g, initial_state, nthreads=1)
        return _t(o), _t(S)

    def qk_prepare(q, k, scale=1.0, l2norm=True, eps=1e-6, inplace=False):
        calls.append("qk_prepare")
        qp, kp = oracle.prepare_qk(q, k, scale, l2norm, eps)
        return _t(qp), _t(kp)

    def qk_prepare_bwd(q, k, d_q_out, d_k_out, scale=1.0, l2norm=True, eps=1e-6):
        calls.append("qk_prepare_bwd")
        gq, gk = oracle.prepare_qk_backward(q, k, d_q_out, d_k_out, scale, l2norm, eps)
        return _t(gq), (_t(gk) if l2norm else d_k_out)

    def chunk_bwd_gated(q, k, v, beta, g, d_o, initial_state=None, d_final_state=None, **_):
        calls.append("chunk_bwd_gated")
        return tuple(_t(x) for x in oracle.backward_gated(q, k, v, beta, g, d_o, initial_state,
                                                          d_final_state, nthreads=1))

    monkeypatch.setattr(dn, "qk_prepare", qk_prepare)
    monkeypatch.setattr(dn, "qk_prepare_bwd", qk_prepare_bwd)
    monkeypatch.setattr(dn, "chunk_fwd_gated", chunk_fwd_gated)
    monkeypatch.setattr(dn, "chunk_bwd_gated", chunk_bwd_gated)
    return calls


@pytest.mark.parametrize("scale,l2norm", [(None, False), (8 ** -0.5, True)])
def test_gated_wrapper_wires_the_gate_gradient(gated_fakes, scale, l2norm):
    """GatedDeltaRule: g gets the gated backward's d_g, the other leaves the
    gated gradients for the prepared q and k carried back through the
    preparation's gradient, and the decay is checked against a central
    difference of the whole prepared forward."""
    q, k, v, beta, S0, d_o, d_S = _inputs(seed=2, raw=l2norm)
    g = np.log(np.random.default_rng(5).uniform(0.5, 1.0, beta.shape))
    leaves = [_t(x).requires_grad_() for x in (q, k, v, beta, g, S0)]
    o, S_T = dn.GatedDeltaRule.apply(*leaves, scale, l2norm)
    torch.autograd.backward([o, S_T], [_t(d_o), _t(d_S)])
    s = 1.0 if scale is None else scale
    qp, kp = oracle.prepare_qk(q, k, s, l2norm)
    ref = list(oracle.backward_gated(qp, kp, v, beta, g, d_o, S0, d_S, nthreads=1))
    prepared = scale is not None or l2norm
    if prepared:
        ref[0], gk = oracle.prepare_qk_backward(q, k, ref[0], ref[1], s, l2norm)
        if l2norm:
            ref[1] = gk
    for leaf, want in zip(leaves, ref):
        assert np.allclose(leaf.grad.numpy(), want, rtol=0, atol=1e-12)
    assert gated_fakes == (["chunk_fwd_gated", "qk_prepare", "chunk_bwd_gated",
                            "qk_prepare_bwd"] if prepared else
                           ["chunk_fwd_gated", "chunk_bwd_gated"])

    def loss(gx):
        o2, S2 = oracle.forward_gated(qp, kp, v, beta, gx, S0, nthreads=1)
        return np.sum(d_o * o2) + np.sum(d_S * S2)

    h = 1e-6
    for idx in [(0, 0, 0), (0, 1, 7), (0, 0, 20)]:
        gp, gm = g.copy(), g.copy()
        gp[idx] += h
        gm[idx] -= h
        fd = (loss(gp) - loss(gm)) / (2 * h)
        assert abs(leaves[4].grad[idx].item() - fd) < 1e-6 * max(1.0, abs(fd)), idx
