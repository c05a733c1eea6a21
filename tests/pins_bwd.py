"""Independent checks ("pins") of the delta-rule gradient.

A gradient implementation is ``grad(q, k, v, beta, dO, S0, dS_T) ->
(dq, dk, dv, dbeta, dS0)``: the gradients of L = <dO, o> + <dS_T, S_T> where
(o, S_T) is the recurrence's forward (library layouts, state [dk][dv]).  Each
pin checks it against something other than the reverse recurrence itself:

- central finite differences of the (separately pinned) forward oracle;
- two homogeneity identities: o is linear in q, and (o, S_T) are jointly
  linear in (v, S0), so Euler's theorem fixes <q, dq> and <v, dv> + <S0, dS0>;
- closed forms at beta = 0, where the state never changes;
- a chunk-level derivation (``chunkwise_backward``) that reaches the same
  numbers through matrices of whole chunks, the form the GPU kernels use.

Each pin returns its largest relative error divided by the bound that pin
allows (so a passing pin returns at most 1).  Dimensions use dk != dv so a
transposed state cannot pass.
"""
from __future__ import annotations

import numpy as np

from tests.pins import _unit

FD_BOUND = 1e-6      # central differences with h = 1e-6 are good to ~1e-9 here
EXACT_BOUND = 1e-10  # identities that hold to fp64 rounding
CHUNK_BOUND = 1e-9   # fp64 solves of the chunk systems


def random_grad_case(seed, B=1, H=2, T=6, dk=3, dv=4, beta_hi=2.0):
    r = np.random.default_rng(seed)
    q = _unit(r.standard_normal((B, H, T, dk)))
    k = _unit(r.standard_normal((B, H, T, dk)))
    v = r.standard_normal((B, H, T, dv))
    beta = r.uniform(0.05, beta_hi, size=(B, H, T))
    S0 = r.standard_normal((B, H, dk, dv)) * 0.5
    dO = r.standard_normal((B, H, T, dv))
    dS_T = r.standard_normal((B, H, dk, dv))
    return q, k, v, beta, S0, dO, dS_T


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return np.inf
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)) / max(1.0, float(np.max(np.abs(b)))))


def _loss(fwd, q, k, v, beta, S0, dO, dS_T):
    o, S = fwd(q, k, v, beta, S0)
    return float(np.sum(o * dO) + np.sum(S * dS_T))


def pin_finite_differences(grad, fwd, seed=31, h=1e-6):
    """Every gradient entry against a central difference of the forward."""
    q, k, v, beta, S0, dO, dS_T = random_grad_case(seed)
    g = grad(q, k, v, beta, dO, S0, dS_T)
    args = [q, k, v, beta, S0]
    worst = 0.0
    for a_i in range(5):
        fd = np.zeros_like(args[a_i])
        for idx in np.ndindex(args[a_i].shape):
            plus = [x.copy() for x in args]
            minus = [x.copy() for x in args]
            plus[a_i][idx] += h
            minus[a_i][idx] -= h
            fd[idx] = (_loss(fwd, *plus, dO, dS_T) - _loss(fwd, *minus, dO, dS_T)) / (2 * h)
        worst = max(worst, _rel(g[a_i], fd) / FD_BOUND)
    return worst


def pin_query_homogeneity(grad, fwd, seed=32):
    """o is linear in q and S_T does not depend on it: <q, dq> = <dO, o>."""
    q, k, v, beta, S0, dO, dS_T = random_grad_case(seed, B=2, H=2, T=40, dk=6, dv=5)
    dq = grad(q, k, v, beta, dO, S0, dS_T)[0]
    o, _ = fwd(q, k, v, beta, S0)
    lhs, rhs = float(np.sum(q * dq)), float(np.sum(dO * o))
    return abs(lhs - rhs) / max(1.0, abs(rhs)) / EXACT_BOUND


def pin_value_homogeneity(grad, fwd, seed=33):
    """(o, S_T) are jointly linear in (v, S0):
    <v, dv> + <S0, dS0> = <dO, o> + <dS_T, S_T>."""
    q, k, v, beta, S0, dO, dS_T = random_grad_case(seed, B=2, H=2, T=40, dk=6, dv=5)
    _, _, dv_, _, dS0 = grad(q, k, v, beta, dO, S0, dS_T)
    o, S = fwd(q, k, v, beta, S0)
    lhs = float(np.sum(v * dv_) + np.sum(S0 * dS0))
    rhs = float(np.sum(dO * o) + np.sum(dS_T * S))
    return abs(lhs - rhs) / max(1.0, abs(rhs)) / EXACT_BOUND


def pin_beta_zero(grad, fwd, seed=34):
    """beta = 0: the state stays S0, so o_t = S0^T q_t (stored layout) and
    dq_t = S0 dO_t, dk = dv = 0, dS0 = dS_T + sum_t q_t dO_t^T, and the
    strength gradient is the error the write would have corrected, seen
    through G_t = dS_T + sum_{s >= t} q_s dO_s^T."""
    q, k, v, beta, S0, dO, dS_T = random_grad_case(seed, T=9)
    beta = np.zeros_like(beta)
    dq, dk, dv_, db, dS0 = grad(q, k, v, beta, dO, S0, dS_T)
    e_dq = np.einsum("bhij,bhtj->bhti", S0, dO)
    e_dS0 = dS_T + np.einsum("bhti,bhtj->bhij", q, dO)
    tail = np.flip(np.cumsum(np.flip(np.einsum("bhti,bhtj->bhtij", q, dO), 2), 2), 2)
    G = dS_T[:, :, None] + tail                                   # G_t, [B,H,T,dk,dv]
    du = np.einsum("bhtij,bhti->bhtj", G, k)
    err = v - np.einsum("bhij,bhti->bhtj", S0, k)
    e_db = np.sum(du * err, axis=-1)
    return max(_rel(dq, e_dq), _rel(dk, np.zeros_like(dk)), _rel(dv_, np.zeros_like(dv_)),
               _rel(dS0, e_dS0), _rel(db, e_db)) / EXACT_BOUND


def chunkwise_backward(q, k, v, beta, dO, S0, dS_T, C):
    """Gradients through whole-chunk matrices (fp64), one (b, h) at a time.

    Forward per chunk (rows K, Q, V, strengths beta; incoming state S):
        A = tril(diag(beta) K K^T, -1),  X = (I + A)^{-1},  Tm = X diag(beta)
        R = V - K S,  U' = Tm R,  P = tril(Q K^T),  O = Q S + P U',
        S_next = S + K^T U'
    Backward per chunk, last to first, with G = dL/dS_next:
        dU' = P^T dO + K G,   dV = dR = Tm^T dU',   dP = tril(dO U'^T)
        dQ = dO S^T + dP K,   dK = dP^T Q + U' G^T - dV S^T
        dTm = dU' R^T,  dbeta_j = sum_i X_ij dTm_ij,  dX = dTm diag(beta)
        dA = strict_tril(-X^T dX X^T),  dbeta_i += sum_j dA_ij (K K^T)_ij
        dK += diag(beta) dA K + (diag(beta) dA)^T K
        dL/dS = G + Q^T dO - K^T dV
    """
    B, H, T, dk = q.shape
    dv = v.shape[3]
    out = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(beta),
           np.zeros((B, H, dk, dv))]
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            starts = list(range(0, T, C))
            S_at = []
            for t0 in starts:
                sl = slice(t0, min(T, t0 + C))
                K, V, bt = k[b, h, sl], v[b, h, sl], beta[b, h, sl]
                n = K.shape[0]
                A = np.tril(bt[:, None] * (K @ K.T), -1)
                Tm = np.linalg.solve(np.eye(n) + A, np.diag(bt))
                S_at.append(S)
                S = S + K.T @ (Tm @ (V - K @ S))
            G = np.zeros((dk, dv)) if dS_T is None else np.array(dS_T[b, h], dtype=np.float64)
            for t0, S in reversed(list(zip(starts, S_at))):
                sl = slice(t0, min(T, t0 + C))
                K, Q, V, bt, dOc = k[b, h, sl], q[b, h, sl], v[b, h, sl], beta[b, h, sl], dO[b, h, sl]
                n = K.shape[0]
                KK = K @ K.T
                A = np.tril(bt[:, None] * KK, -1)
                X = np.linalg.inv(np.eye(n) + A)
                Tm = X * bt[None, :]
                R = V - K @ S
                U = Tm @ R
                P = np.tril(Q @ K.T)
                dU = P.T @ dOc + K @ G
                dV = Tm.T @ dU
                dP = np.tril(dOc @ U.T)
                dQ = dOc @ S.T + dP @ K
                dK = dP.T @ Q + U @ G.T - dV @ S.T
                dTm = dU @ R.T
                db = np.sum(X * dTm, axis=0)
                dX = dTm * bt[None, :]
                dA = np.tril(-X.T @ dX @ X.T, -1)
                db = db + np.sum(dA * KK, axis=1)
                dAb = bt[:, None] * dA
                dK = dK + dAb @ K + dAb.T @ K
                out[0][b, h, sl], out[1][b, h, sl], out[2][b, h, sl], out[3][b, h, sl] = dQ, dK, dV, db
                G = G + Q.T @ dOc - K.T @ dV
            out[4][b, h] = G
    return tuple(out)


def pin_chunkwise(grad, fwd, seed=35):
    """The chunk-level derivation at C = 1 (token by token), C = 16 with a
    ragged last chunk, and C = T (one chunk) gives the same gradients."""
    q, k, v, beta, S0, dO, dS_T = random_grad_case(seed, B=1, H=2, T=37, dk=6, dv=5)
    g = grad(q, k, v, beta, dO, S0, dS_T)
    worst = 0.0
    for C in (1, 16, 37):
        ref = chunkwise_backward(q, k, v, beta, dO, S0, dS_T, C)
        worst = max(worst, max(_rel(a, b) for a, b in zip(g, ref)))
    return worst / CHUNK_BOUND


ALL_BWD_PINS = {
    "finite_differences": pin_finite_differences,
    "query_homogeneity": pin_query_homogeneity,
    "value_homogeneity": pin_value_homogeneity,
    "beta_zero": pin_beta_zero,
    "chunkwise": pin_chunkwise,
}
