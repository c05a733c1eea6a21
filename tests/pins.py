"""Independent checks ("pins") of a delta-rule implementation.

Each pin takes ``run(q, k, v, beta, S0) -> (o, S_T)`` with the library's
layouts (q, k ``[B,H,T,dk]``, v ``[B,H,T,dv]``, beta ``[B,H,T]``, state
``[B,H,dk,dv]`` = the pages' dv x dk state transposed) and checks it against
something other than the recurrence itself: an algebraically different form
of the update, an invariant, a closed form, or a brute-force expansion.
Each pin returns the largest error it saw; the tests hold it below a bound.

The same pins are run against deliberately broken implementations (planted
mistakes) to show that every plausible mistake fails at least one of them.
Dimensions are chosen with dk != dv so that a transposed state cannot pass.
"""
from __future__ import annotations

import json
from pathlib import Path

import numpy as np
import scipy.linalg
import torch

GOLDEN = Path(__file__).resolve().parent / "golden"


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def random_case(seed, B=2, H=2, T=12, dk=5, dv=7, beta_hi=1.0, s0=True):
    r = _rng(seed)
    q = _unit(r.standard_normal((B, H, T, dk)))
    k = _unit(r.standard_normal((B, H, T, dk)))
    v = r.standard_normal((B, H, T, dv))
    beta = r.uniform(0.05, beta_hi, size=(B, H, T))
    S0 = r.standard_normal((B, H, dk, dv)) * 0.5 if s0 else None
    return q, k, v, beta, S0


def _err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return np.inf
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def _math_state(S_mem):
    """[.., dk, dv] memory layout -> the pages' dv x dk state."""
    return np.swapaxes(S_mem, -1, -2)


# ---------------------------------------------------------------------------
# P1: alternative forms of one update.
# ---------------------------------------------------------------------------
def pin_householder_form(run, seed=1, beta_hi=2.0):
    """S_t = S_{t-1}(I - beta k k^T) + beta v k^T, o_t = S_t q_t as explicit
    matrix products ("DeltaNet 引入 Delta Rule", last line of the derivation;
    also the DeltaNetAttention docstring).  beta up to 2 covers the
    negative-eigenvalue variant."""
    q, k, v, beta, S0 = random_case(seed, beta_hi=beta_hi)
    o, S = run(q, k, v, beta, S0)
    B, H, T, dk = q.shape
    worst = 0.0
    for b in range(B):
        for h in range(H):
            Sm = _math_state(S0[b, h]).copy()
            for t in range(T):
                kt, vt, qt, bt = k[b, h, t], v[b, h, t], q[b, h, t], beta[b, h, t]
                Sm = Sm @ (np.eye(dk) - bt * np.outer(kt, kt)) + bt * np.outer(vt, kt)
                worst = max(worst, _err(o[b, h, t], Sm @ qt))
            worst = max(worst, _err(S[b, h], Sm.T))
    return worst


def pin_blended_form(run, seed=2):
    """v_old = S k, v_new = beta v + (1 - beta) v_old,
    S <- S - v_old k^T + v_new k^T ("DeltaNet 引入 Delta Rule", the
    old-value / new-value equations)."""
    q, k, v, beta, S0 = random_case(seed)
    o, S = run(q, k, v, beta, S0)
    B, H, T, dk = q.shape
    worst = 0.0
    for b in range(B):
        for h in range(H):
            Sm = _math_state(S0[b, h]).copy()
            for t in range(T):
                kt, vt, qt, bt = k[b, h, t], v[b, h, t], q[b, h, t], beta[b, h, t]
                v_old = Sm @ kt
                v_new = bt * vt + (1.0 - bt) * v_old
                Sm = Sm - np.outer(v_old, kt) + np.outer(v_new, kt)
                worst = max(worst, _err(o[b, h, t], Sm @ qt))
            worst = max(worst, _err(S[b, h], Sm.T))
    return worst


def pin_gradient_step(run, seed=3):
    """One step equals one gradient-descent step of size beta on
    1/2 ||S k - v||^2 from S_{t-1} ("Dérivation par perte de reconstruction",
    fr.news.hada.io/topic?id=31925).  The gradient comes from autograd."""
    q, k, v, beta, S0 = random_case(seed, T=1)
    o, S = run(q, k, v, beta, S0)
    B, H = q.shape[:2]
    worst = 0.0
    for b in range(B):
        for h in range(H):
            Sm = torch.tensor(_math_state(S0[b, h]).copy(), dtype=torch.float64,
                              requires_grad=True)
            kt = torch.tensor(k[b, h, 0])
            vt = torch.tensor(v[b, h, 0])
            loss = 0.5 * torch.sum((Sm @ kt - vt) ** 2)
            (grad,) = torch.autograd.grad(loss, Sm)
            S1 = (Sm - float(beta[b, h, 0]) * grad).detach().numpy()
            worst = max(worst, _err(S[b, h], S1.T))
            worst = max(worst, _err(o[b, h, 0], S1 @ q[b, h, 0]))
    return worst


# ---------------------------------------------------------------------------
# P2-P4: invariants and special cases.
# ---------------------------------------------------------------------------
def pin_reconstruction(run, seed=4):
    """S_t k_t = (1 - beta_t) S_{t-1} k_t + beta_t v_t, and = v_t when
    beta_t = 1 (the immediate read-back in "DeltaNet : écrire l'erreur de
    prédiction plutôt que la valeur").  Uses the implementation's own states
    after t-1 and t tokens."""
    q, k, v, beta, S0 = random_case(seed, T=8)
    beta[..., 3] = 1.0
    worst = 0.0
    _, S_prev = run(q[:, :, :0], k[:, :, :0], v[:, :, :0], beta[:, :, :0], S0)
    worst = max(worst, _err(S_prev, S0))
    for t in range(q.shape[2]):
        _, S_t = run(q[:, :, :t + 1], k[:, :, :t + 1], v[:, :, :t + 1],
                     beta[:, :, :t + 1], S0)
        kt = k[:, :, t]
        bt = beta[:, :, t][..., None]
        lhs = np.einsum("bhij,bhi->bhj", S_t, kt)
        rhs = (1.0 - bt) * np.einsum("bhij,bhi->bhj", S_prev, kt) + bt * v[:, :, t]
        worst = max(worst, _err(lhs, rhs))
        if t == 3:
            worst = max(worst, _err(lhs, v[:, :, t]))
        S_prev = S_t
    return worst


def pin_beta_zero(run, seed=5):
    """beta = 0 leaves the state unchanged (the special cases listed after the
    old/new-value equations, "DeltaNet 引入 Delta Rule",
    garden.houmin.site/infra/delta-net), so o_t = S_0 q_t."""
    q, k, v, beta, S0 = random_case(seed)
    beta[:] = 0.0
    o, S = run(q, k, v, beta, S0)
    expect_o = np.einsum("bhij,bhti->bhtj", S0, q)
    return max(_err(S, S0), _err(o, expect_o))


def pin_transition_eigen(run, seed=6):
    """With v = 0 one step applies I - beta k k^T: eigenvalue 1 - beta on k,
    1 on every direction orthogonal to k ("Transition d'état structurée",
    fr.news.hada.io/topic?id=31925)."""
    q, k, v, beta, S0 = random_case(seed, T=1, beta_hi=2.0)
    v[:] = 0.0
    _, S = run(q, k, v, beta, S0)
    r = _rng(seed + 100)
    worst = 0.0
    B, H, _, dk = q.shape
    for b in range(B):
        for h in range(H):
            kt = k[b, h, 0]
            Sm0, Sm1 = _math_state(S0[b, h]), _math_state(S[b, h])
            worst = max(worst, _err(Sm1 @ kt, (1.0 - beta[b, h, 0]) * (Sm0 @ kt)))
            x = r.standard_normal(dk)
            x -= (x @ kt) * kt
            worst = max(worst, _err(Sm1 @ x, Sm0 @ x))
    return worst


# ---------------------------------------------------------------------------
# P6-P9: closed forms.
# ---------------------------------------------------------------------------
def _orthonormal_rows(r, n, d):
    a = r.standard_normal((d, d))
    qm, _ = np.linalg.qr(a)
    return qm[:n]


def pin_exact_recall(run, seed=7):
    """Orthonormal keys written with beta = 1, then read back with beta = 0:
    every read returns the stored value exactly.  At beta = 1 a write replaces
    the old value (special cases after the old/new-value equations in
    "DeltaNet 引入 Delta Rule"), and with orthonormal keys a write leaves every
    other key's value untouched (locality of the update in "DeltaNet : écrire
    l'erreur de prédiction plutôt que la valeur")."""
    r = _rng(seed)
    B, H, d, n_write, n_read = 2, 2, 6, 6, 10
    T = n_write + n_read
    dv = 4
    q = np.zeros((B, H, T, d)); k = np.zeros_like(q)
    v = r.standard_normal((B, H, T, dv)); beta = np.zeros((B, H, T))
    expect = np.zeros((B, H, T, dv))
    for b in range(B):
        for h in range(H):
            basis = _orthonormal_rows(r, d, d)
            order = np.concatenate([np.arange(n_write),
                                    r.integers(0, n_write, n_read)])
            k[b, h] = basis[order]
            q[b, h] = basis[order]
            beta[b, h, :n_write] = 1.0
            expect[b, h] = v[b, h, order]
    o, _ = run(q, k, v, beta, np.zeros((B, H, d, dv)))
    return _err(o, expect)


def pin_linear_attention(run, seed=8):
    """Mutually orthogonal unit keys with beta = 1 on first writes and a zero
    initial state: every prediction S_{t-1} k_t is zero, so the delta rule is
    plain linear attention, O = (Q K^T . M) V with M causal including the
    diagonal, and S_T = sum_t v_t k_t^T (the linear-attention forms of
    "Linear Attention", garden.houmin.site/infra/delta-net)."""
    r = _rng(seed)
    B, H, T, dk, dv = 2, 3, 7, 9, 5
    k = np.stack([np.stack([_orthonormal_rows(r, T, dk) for _ in range(H)])
                  for _ in range(B)])
    q = r.standard_normal((B, H, T, dk))
    v = r.standard_normal((B, H, T, dv))
    beta = np.ones((B, H, T))
    o, S = run(q, k, v, beta, np.zeros((B, H, dk, dv)))
    M = np.tril(np.ones((T, T)))
    expect_o = np.einsum("bhts,bhsj->bhtj", np.einsum("bhti,bhsi->bhts", q, k) * M, v)
    expect_S = np.einsum("bhti,bhtj->bhij", k, v)
    return max(_err(o, expect_o), _err(S, expect_S))


def pin_householder_product(run, seed=9):
    """Brute-force expansion over explicit dk x dk transition matrices,
    H_t = I - beta_t k_t k_t^T (the Householder-product view, section 3 of
    paperlayer.ai/abs/2406.06484v6):
        S_t = S_0 H_1 ... H_t + sum_{s<=t} beta_s v_s k_s^T H_{s+1} ... H_t
    for every prefix t <= 8."""
    q, k, v, beta, S0 = random_case(seed, T=8, beta_hi=2.0)
    o, S = run(q, k, v, beta, S0)
    B, H, T, dk = q.shape
    worst = 0.0
    for b in range(B):
        for h in range(H):
            Hs = [np.eye(dk) - beta[b, h, t] * np.outer(k[b, h, t], k[b, h, t])
                  for t in range(T)]
            for t in range(T):
                St = _math_state(S0[b, h]).copy()
                for s in range(t + 1):
                    St = St @ Hs[s]
                for s in range(t + 1):
                    term = beta[b, h, s] * np.outer(v[b, h, s], k[b, h, s])
                    for u in range(s + 1, t + 1):
                        term = term @ Hs[u]
                    St = St + term
                worst = max(worst, _err(o[b, h, t], St @ q[b, h, t]))
                if t == T - 1:
                    worst = max(worst, _err(S[b, h], St.T))
    return worst


def pin_parallel_form(run, seed=10, T=96):
    """Fully parallel form with a zero initial state (the "DeltaNet" row of
    the closing table of garden.houmin.site/infra/delta-net, with beta
    restored):  O = (Q K^T . M)(I + tril(diag(beta) K K^T, -1))^{-1} diag(beta) V,
    solved densely in fp64."""
    q, k, v, beta, _ = random_case(seed, B=1, H=2, T=T, dk=16, dv=12)
    B, H = q.shape[:2]
    o, _ = run(q, k, v, beta, np.zeros((B, H, 16, 12)))
    worst = 0.0
    M = np.tril(np.ones((T, T)))
    for b in range(B):
        for h in range(H):
            K, Q, V, bt = k[b, h], q[b, h], v[b, h], beta[b, h]
            L = np.tril(bt[:, None] * (K @ K.T), -1)
            U = scipy.linalg.solve_triangular(np.eye(T) + L, bt[:, None] * V,
                                              lower=True, unit_diagonal=True)
            worst = max(worst, _err(o[b, h], ((Q @ K.T) * M) @ U))
    return worst


# ---------------------------------------------------------------------------
# P10: the chunkwise (UT / WY) restatement the CUDA path evaluates.
# ---------------------------------------------------------------------------
def chunkwise_reference(q, k, v, beta, S0, C):
    """Chunkwise evaluation, test-side, in fp64 (chunk algebra of "Chunkwise
    KDA : réorganiser la récurrence en multiplications matricielles" with no
    decay, i.e. D = I; the UT transform of appendix B.2 of
    paperlayer.ai/abs/2406.06484v6).  Per chunk, with state S stored [dk][dv]:
        A  = tril(diag(beta) K K^T, -1)      T = (I + A)^{-1} diag(beta)
        W  = T K,   U = T V,   U' = U - W S
        O  = Q S + (Q K^T . M) U'            S <- S + K^T U'
    A ragged tail chunk is simply shorter."""
    B, H, Tn, dk = q.shape
    dv = v.shape[3]
    o = np.zeros((B, H, Tn, dv))
    S_out = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else S0[b, h].copy()
            for c0 in range(0, Tn, C):
                sl = slice(c0, min(c0 + C, Tn))
                K, Q, V, bt = k[b, h, sl], q[b, h, sl], v[b, h, sl], beta[b, h, sl]
                n = K.shape[0]
                A = np.tril(bt[:, None] * (K @ K.T), -1)
                Tm = scipy.linalg.solve_triangular(np.eye(n) + A, np.diag(bt),
                                                   lower=True, unit_diagonal=True)
                W, U = Tm @ K, Tm @ V
                Up = U - W @ S
                o[b, h, sl] = Q @ S + np.tril(Q @ K.T) @ Up
                S = S + K.T @ Up
            S_out[b, h] = S
    return o, S_out


def pin_chunkwise(run, seed=11):
    """The chunkwise restatement at C in {1, 3, 16, 64, T} (C = 1 is the
    recurrent form and C = T the fully parallel one, "Chunkwise Parallel
    Form" in section 2 of paperlayer.ai/abs/2406.06484v6), with a carried
    initial state and a ragged last chunk, agrees with ``run``."""
    q, k, v, beta, S0 = random_case(seed, B=1, H=2, T=200, dk=8, dv=6)
    o, S = run(q, k, v, beta, S0)
    worst = 0.0
    for C in (1, 3, 16, 64, 200):
        oc, Sc = chunkwise_reference(q, k, v, beta, S0, C)
        worst = max(worst, _err(o, oc), _err(S, Sc))
    return worst


def pin_carried_state(run, seed=12):
    """Running T1 tokens, then T2 more from the returned state, equals one run
    over T1 + T2 tokens (the initial_state / output_final_state hand-off of
    fla/layers/delta_net.py, DeltaNet.forward)."""
    q, k, v, beta, S0 = random_case(seed, T=20)
    o, S = run(q, k, v, beta, S0)
    o1, S1 = run(q[:, :, :13], k[:, :, :13], v[:, :, :13], beta[:, :, :13], S0)
    o2, S2 = run(q[:, :, 13:], k[:, :, 13:], v[:, :, 13:], beta[:, :, 13:], S1)
    return max(_err(o, np.concatenate([o1, o2], axis=2)), _err(S, S2))


def pin_golden(run):
    """Hand-worked examples stored in tests/golden (derivations included)."""
    worst = 0.0
    for path in sorted(GOLDEN.glob("hand_*.json")):
        case = json.loads(path.read_text())
        f = lambda key: np.asarray(case[key], dtype=np.float64)[None, None]
        S0 = f("S0_mem") if "S0_mem" in case else None
        if S0 is None:
            S0 = np.zeros((1, 1, len(case["k"][0]), len(case["v"][0])))
        o, S = run(f("q"), f("k"), f("v"), f("beta"), S0)
        worst = max(worst, _err(o, f("o")), _err(S, f("S_T_mem")))
    return worst


ALL_PINS = {
    "householder_form": pin_householder_form,
    "blended_form": pin_blended_form,
    "gradient_step": pin_gradient_step,
    "reconstruction": pin_reconstruction,
    "beta_zero": pin_beta_zero,
    "transition_eigen": pin_transition_eigen,
    "exact_recall": pin_exact_recall,
    "linear_attention": pin_linear_attention,
    "householder_product": pin_householder_product,
    "parallel_form": pin_parallel_form,
    "chunkwise": pin_chunkwise,
    "carried_state": pin_carried_state,
    "golden": pin_golden,
}

# fp64 throughout: every pin holds to rounding.
PIN_TOL = 1e-10
