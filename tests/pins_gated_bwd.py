"""Independent checks ("pins") of the Gated DeltaNet gradient.

A gradient implementation is ``grad(q, k, v, beta, g, dO, S0, dS_T) ->
(dq, dk, dv, dbeta, dg, dS0)``: the gradients of L = <dO, o> + <dS_T, S_T>
where (o, S_T) is the gated forward (library layouts, state [dk][dv], g the
log keep rate [B, H, T]).  Each pin checks it against something other than
the reverse recurrence itself:

- central finite differences of the (separately pinned) gated forward oracle,
  for all six inputs;
- zero decay (g = 0) is the plain delta rule: the first five gradients equal
  the (separately pinned) plain gradient oracle's;
- one token: S_1 = alpha (I - beta k k^T) S0 + beta k v^T (stored layout), so
  dL/dg is alpha times L's decay-dependent part, in closed form;
- a whole-chunk derivation (``chunkwise_gated_backward``) at C = 1, 16
  (ragged) and T: the algebra a chunkwise kernel follows, with the decay
  entering as ratios exp(G_i - G_j) and the keep factors gamma_i = exp(G_i),
  Gamma = gamma_last of each chunk.

Each pin returns its largest relative error divided by the bound it allows
(a passing pin returns at most 1).  Dimensions use dk != dv.
"""
from __future__ import annotations

import numpy as np

from tests.pins import _unit
from tests.pins_bwd import _rel

FD_BOUND = 1e-6
EXACT_BOUND = 1e-10
CHUNK_BOUND = 1e-9


def random_gated_grad_case(seed, B=1, H=2, T=6, dk=3, dv=4, g_lo=-1.0):
    r = np.random.default_rng(seed)
    q = _unit(r.standard_normal((B, H, T, dk)))
    k = _unit(r.standard_normal((B, H, T, dk)))
    v = r.standard_normal((B, H, T, dv))
    beta = r.uniform(0.05, 1.5, size=(B, H, T))
    g = r.uniform(g_lo, 0.0, size=(B, H, T))
    S0 = r.standard_normal((B, H, dk, dv)) * 0.5
    dO = r.standard_normal((B, H, T, dv))
    dS_T = r.standard_normal((B, H, dk, dv))
    return q, k, v, beta, g, S0, dO, dS_T


def _loss(fwd, q, k, v, beta, g, S0, dO, dS_T):
    o, S = fwd(q, k, v, beta, g, S0)
    return float(np.sum(o * dO) + np.sum(S * dS_T))


def pin_finite_differences(grad, fwd, seed=41, h=1e-6):
    """Every gradient entry, g's included, against a central difference."""
    q, k, v, beta, g, S0, dO, dS_T = random_gated_grad_case(seed)
    got = grad(q, k, v, beta, g, dO, S0, dS_T)
    args = [q, k, v, beta, g, S0]
    worst = 0.0
    for a_i, want_i in zip(range(6), (0, 1, 2, 3, 4, 5)):
        fd = np.zeros_like(args[a_i])
        for idx in np.ndindex(args[a_i].shape):
            plus = [x.copy() for x in args]
            minus = [x.copy() for x in args]
            plus[a_i][idx] += h
            minus[a_i][idx] -= h
            fd[idx] = (_loss(fwd, *plus, dO, dS_T) - _loss(fwd, *minus, dO, dS_T)) / (2 * h)
        worst = max(worst, _rel(got[want_i], fd) / FD_BOUND)
    return worst


def pin_zero_decay(grad, fwd, plain_grad, seed=42):
    """g = 0 keeps every state: the plain rule's gradients."""
    q, k, v, beta, g, S0, dO, dS_T = random_gated_grad_case(seed, B=2, H=2, T=23, dk=5, dv=4)
    g = np.zeros_like(g)
    got = grad(q, k, v, beta, g, dO, S0, dS_T)
    ref = plain_grad(q, k, v, beta, dO, S0, dS_T)
    return max(_rel(a, b) for a, b in zip(got[:4] + got[5:], ref)) / EXACT_BOUND


def pin_one_token(grad, fwd, seed=43):
    """T = 1: S_1 = alpha M + beta k v^T with M = (I - beta k k^T) S0 and
    o = S_1^T q (stored layout), so dL/dg = alpha (<dO, M^T q> + <dS_T, M>)."""
    q, k, v, beta, g, S0, dO, dS_T = random_gated_grad_case(seed, B=2, H=3, T=1, dk=4, dv=3)
    got = grad(q, k, v, beta, g, dO, S0, dS_T)
    kk = k[:, :, 0]
    M = S0 - beta[:, :, 0, None, None] * np.einsum("bhi,bhj,bhjv->bhiv", kk, kk, S0)
    alpha = np.exp(g[:, :, 0])
    want = alpha * (np.einsum("bhv,bhiv,bhi->bh", dO[:, :, 0], M, q[:, :, 0])
                    + np.einsum("bhiv,bhiv->bh", dS_T, M))
    return _rel(got[4][:, :, 0], want) / EXACT_BOUND


def chunkwise_gated_backward(q, k, v, beta, g, dO, S0, dS_T, C):
    """Gradients through whole-chunk matrices (fp64), one (b, h) at a time.

    Per chunk, with G_i the log decay accumulated from the chunk start through
    token i, gamma = exp(G), Gamma = gamma of the chunk's last token and
    D_ij = exp(G_i - G_j):
        A = tril(diag(beta) (K K^T o D), -1),  X = (I + A)^{-1},  Tm = X diag(beta)
        R = V - diag(gamma) K S,  U' = Tm R,  P = tril(Q K^T o D)
        O = diag(gamma) Q S + P U',   S_next = Gamma S + (diag(Gamma / gamma) K)^T U'
    Backward, last chunk first, with G_end = dL/dS_next:
        dU' = P^T dO + diag(Gamma / gamma) K G_end,  dV = dR = Tm^T dU'
        dP = tril(dO U'^T),  dTm = dU' R^T,  dA = strict_tril(-X^T dTm diag(beta) X^T)
        dQ = diag(gamma) dO S^T + (dP o D) K
        dK = (dP o D)^T Q - diag(gamma) dV S^T + diag(Gamma / gamma) U' G_end^T + Z K,
             Z = diag(beta) (dA o D) + (diag(beta) (dA o D))^T
        dbeta_j = sum_i X_ij dTm_ij + sum_l dA_jl (K K^T o D)_jl
        dG_i = sum_j (dA_ij A_ij - dA_ji A_ji) + sum_j (dP_ij P_ij - dP_ji P_ji)
               - gamma_i dV_i . (K S)_i + gamma_i dO_i . (Q S)_i
               - (Gamma / gamma_i) (K G_end)_i . U'_i  + [i last] <G_end, S_next>
        dg_t = sum_{i >= t} dG_i (within the chunk)
        dL/dS = Gamma G_end + (diag(gamma) Q)^T dO - (diag(gamma) K)^T dV
    """
    B, H, T, dk = q.shape
    dv = v.shape[3]
    out = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(beta),
           np.zeros_like(g), np.zeros((B, H, dk, dv))]
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            starts = list(range(0, T, C))
            S_at = []
            for t0 in starts:
                sl = slice(t0, min(T, t0 + C))
                K, V, bt, gl = k[b, h, sl], v[b, h, sl], beta[b, h, sl], np.cumsum(g[b, h, sl])
                n = K.shape[0]
                gam, D = np.exp(gl), np.exp(gl[:, None] - gl[None, :])
                A = np.tril(bt[:, None] * (K @ K.T) * D, -1)
                Tm = np.linalg.solve(np.eye(n) + A, np.diag(bt))
                S_at.append(S)
                U = Tm @ (V - gam[:, None] * (K @ S))
                S = gam[-1] * S + (K * (gam[-1] / gam)[:, None]).T @ U
            G = np.zeros((dk, dv)) if dS_T is None else np.array(dS_T[b, h], dtype=np.float64)
            for t0, S in reversed(list(zip(starts, S_at))):
                sl = slice(t0, min(T, t0 + C))
                K, Q, V = k[b, h, sl], q[b, h, sl], v[b, h, sl]
                bt, dOc, gl = beta[b, h, sl], dO[b, h, sl], np.cumsum(g[b, h, sl])
                n = K.shape[0]
                gam, D = np.exp(gl), np.exp(gl[:, None] - gl[None, :])
                Gam, r = gam[-1], gam[-1] / gam
                KKD = (K @ K.T) * D
                A = np.tril(bt[:, None] * KKD, -1)
                X = np.linalg.inv(np.eye(n) + A)
                Tm = X * bt[None, :]
                KS, QS, KG = K @ S, Q @ S, K @ G
                R = V - gam[:, None] * KS
                U = Tm @ R
                P = np.tril((Q @ K.T) * D)
                S_next = Gam * S + (K * r[:, None]).T @ U
                dU = P.T @ dOc + r[:, None] * KG
                dV = Tm.T @ dU
                dP = np.tril(dOc @ U.T)
                dQ = gam[:, None] * (dOc @ S.T) + (dP * D) @ K
                dK = (dP * D).T @ Q - gam[:, None] * (dV @ S.T) + r[:, None] * (U @ G.T)
                dTm = dU @ R.T
                db = np.sum(X * dTm, axis=0)
                dA = np.tril(-X.T @ (dTm * bt[None, :]) @ X.T, -1)
                db = db + np.sum(dA * KKD, axis=1)
                Zh = bt[:, None] * dA * D
                dK = dK + (Zh + Zh.T) @ K
                dG = (np.sum(dA * A, axis=1) - np.sum(dA * A, axis=0)
                      + np.sum(dP * P, axis=1) - np.sum(dP * P, axis=0)
                      - gam * np.sum(dV * KS, axis=1) + gam * np.sum(dOc * QS, axis=1)
                      - r * np.sum(KG * U, axis=1))
                dG[-1] += np.sum(G * S_next)
                out[0][b, h, sl], out[1][b, h, sl], out[2][b, h, sl] = dQ, dK, dV
                out[3][b, h, sl] = db
                out[4][b, h, sl] = np.flip(np.cumsum(np.flip(dG)))
                G = Gam * G + (gam[:, None] * Q).T @ dOc - (gam[:, None] * K).T @ dV
            out[5][b, h] = G
    return tuple(out)


def pin_chunkwise(grad, fwd, seed=44):
    """The chunk-level derivation at C = 1, C = 16 with a ragged last chunk,
    and C = T gives the same six gradients."""
    q, k, v, beta, g, S0, dO, dS_T = random_gated_grad_case(seed, B=1, H=2, T=37, dk=6, dv=5)
    got = grad(q, k, v, beta, g, dO, S0, dS_T)
    worst = 0.0
    for C in (1, 16, 37):
        ref = chunkwise_gated_backward(q, k, v, beta, g, dO, S0, dS_T, C)
        worst = max(worst, max(_rel(a, b) for a, b in zip(got, ref)))
    return worst / CHUNK_BOUND


def reverse_loop_gated(q, k, v, beta, g, dO, S0, dS_T, mistake=None):
    """A numpy statement of the token-level reverse pass, for planting
    mistakes (``mistake`` names one; None is the correct pass)."""
    B, H, T, dk = q.shape
    dv = v.shape[3]
    out = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(beta),
           np.zeros_like(g), np.zeros((B, H, dk, dv))]
    for b in range(B):
        for h in range(H):
            S = [np.zeros((dk, dv)) if S0 is None else np.array(S0[b, h], dtype=np.float64)]
            for t in range(T):
                a = np.exp(g[b, h, t])
                kt = k[b, h, t]
                e = v[b, h, t] - (a * S[-1]).T @ kt
                S.append(a * S[-1] + beta[b, h, t] * np.outer(kt, e))
            G = np.zeros((dk, dv)) if dS_T is None else np.array(dS_T[b, h], dtype=np.float64)
            for t in reversed(range(T)):
                a, bt = np.exp(g[b, h, t]), beta[b, h, t]
                kt, qt, d = k[b, h, t], q[b, h, t], dO[b, h, t]
                G = G + np.outer(qt, d)
                out[0][b, h, t] = S[t + 1] @ d
                St = a * S[t] if mistake != "predict_without_decay" else S[t]
                e = v[b, h, t] - St.T @ kt
                du = G.T @ kt
                out[2][b, h, t] = bt * du
                out[3][b, h, t] = du @ e
                out[1][b, h, t] = G @ (bt * e) - bt * (St @ du)
                G = G - bt * np.outer(kt, du)
                da = np.sum(G * S[t])
                out[4][b, h, t] = a * da if mistake != "dg_without_alpha" else da
                if mistake != "state_gradient_not_decayed":
                    G = a * G
            out[5][b, h] = G
    return tuple(out)


GATED_BWD_MISTAKES = ("predict_without_decay", "dg_without_alpha", "state_gradient_not_decayed")

ALL_GATED_BWD_PINS = {
    "finite_differences": pin_finite_differences,
    "zero_decay": pin_zero_decay,
    "one_token": pin_one_token,
    "chunkwise": pin_chunkwise,
}
