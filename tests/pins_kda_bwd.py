"""Independent checks ("pins") of the KDA gradient.

A gradient implementation is ``grad(q, k, v, beta, g, dO, S0, dS_T) ->
(dq, dk, dv, dbeta, dg, dS0)``: the gradients of L = <dO, o> + <dS_T, S_T>
where (o, S_T) is the KDA forward (library layouts, state [dk][dv], g the
per-key-channel log keep rates [B, H, T, dk]).  Each pin checks it against
something other than the reverse recurrence itself:

- central finite differences of the (separately pinned) KDA forward oracle,
  for all six inputs, every channel of g included;
- equal channels: a rate shared by every key channel is Gated DeltaNet, so
  the first four gradients and dS0 equal the (separately pinned) gated
  gradient's and the channels of dg sum to the gated dg;
- one token: S_1 = M diag(alpha) S0 + beta k v^T with M = I - beta k k^T
  (stored layout), so dL/dg_i = alpha_i sum_j (M G_1)_ij S0_ij with
  G_1 = q dO^T + dS_T, in closed form;
- a whole-chunk derivation (``chunkwise_kda_backward``) at C = 1, 16
  (ragged) and T: the algebra a chunkwise kernel follows, with the decay
  ratios exp(G_t[c] - G_s[c]) inside the channel sums.

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


def random_kda_grad_case(seed, B=1, H=2, T=6, dk=3, dv=4, g_lo=-1.0):
    r = np.random.default_rng(seed)
    q = _unit(r.standard_normal((B, H, T, dk)))
    k = _unit(r.standard_normal((B, H, T, dk)))
    v = r.standard_normal((B, H, T, dv))
    beta = r.uniform(0.05, 1.5, size=(B, H, T))
    g = r.uniform(g_lo, 0.0, size=(B, H, T, dk))
    S0 = r.standard_normal((B, H, dk, dv)) * 0.5
    dO = r.standard_normal((B, H, T, dv))
    dS_T = r.standard_normal((B, H, dk, dv))
    return q, k, v, beta, g, S0, dO, dS_T


def _loss(fwd, q, k, v, beta, g, S0, dO, dS_T):
    o, S = fwd(q, k, v, beta, g, S0)
    return float(np.sum(o * dO) + np.sum(S * dS_T))


def pin_finite_differences(grad, fwd, gated_grad=None, seed=51, h=1e-6):
    """Every gradient entry, each channel of g included, against a central
    difference."""
    q, k, v, beta, g, S0, dO, dS_T = random_kda_grad_case(seed)
    got = grad(q, k, v, beta, g, dO, S0, dS_T)
    args = [q, k, v, beta, g, S0]
    worst = 0.0
    for a_i in range(6):
        fd = np.zeros_like(args[a_i])
        for idx in np.ndindex(args[a_i].shape):
            plus = [x.copy() for x in args]
            minus = [x.copy() for x in args]
            plus[a_i][idx] += h
            minus[a_i][idx] -= h
            fd[idx] = (_loss(fwd, *plus, dO, dS_T) - _loss(fwd, *minus, dO, dS_T)) / (2 * h)
        worst = max(worst, _rel(got[a_i], fd) / FD_BOUND)
    return worst


def pin_equal_channels(grad, fwd, gated_grad, seed=52):
    """One rate on every key channel is Gated DeltaNet: the gated gradients,
    with dg's channels summing to the gated dg."""
    q, k, v, beta, g, S0, dO, dS_T = random_kda_grad_case(seed, B=2, H=2, T=23, dk=5, dv=4)
    g1 = g[..., 0]
    gk = np.repeat(g1[..., None], q.shape[-1], axis=-1)
    got = grad(q, k, v, beta, gk, dO, S0, dS_T)
    ref = gated_grad(q, k, v, beta, g1, dO, S0, dS_T)
    worst = max(_rel(a, b) for a, b in zip(got[:4] + got[5:], ref[:4] + ref[5:]))
    worst = max(worst, _rel(got[4].sum(axis=-1), ref[4]))
    return worst / EXACT_BOUND


def pin_one_token(grad, fwd, gated_grad=None, seed=53):
    """T = 1: dL/dg_i = alpha_i sum_j (M G_1)_ij S0_ij, M = I - beta k k^T,
    G_1 = q dO^T + dS_T (the state gradient after the read)."""
    q, k, v, beta, g, S0, dO, dS_T = random_kda_grad_case(seed, B=2, H=3, T=1, dk=4, dv=3)
    got = grad(q, k, v, beta, g, dO, S0, dS_T)
    kk, qq, d = k[:, :, 0], q[:, :, 0], dO[:, :, 0]
    eye = np.eye(kk.shape[-1])
    M = eye - beta[:, :, 0, None, None] * np.einsum("bhi,bhj->bhij", kk, kk)
    G1 = np.einsum("bhi,bhv->bhiv", qq, d) + dS_T
    want = np.exp(g[:, :, 0]) * np.einsum("bhij,bhjv,bhiv->bhi", M, G1, S0)
    return _rel(got[4][:, :, 0], want) / EXACT_BOUND


def chunkwise_kda_backward(q, k, v, beta, g, dO, S0, dS_T, C):
    """Gradients through whole-chunk matrices (fp64), one (b, h) at a time.

    Per chunk, with G_t[c] the log decay of key channel c accumulated from
    the chunk start through token t, gamma = exp(G) (per token and channel),
    Gamma = gamma of the chunk's last token, f = Gamma / gamma and the ratios
    D[t, s, c] = exp(G_t[c] - G_s[c]):
        A2[t, s] = sum_c k_t[c] k_s[c] D[t, s, c],  A = tril(diag(beta) A2, -1)
        P[t, s]  = sum_c q_t[c] k_s[c] D[t, s, c]   (s <= t)
        X = (I + A)^{-1},  Tm = X diag(beta)
        R = V - (K o gamma) S,  U' = Tm R,  O = (Q o gamma) S + P U'
        S_next = diag(Gamma) S + (K o f)^T U'
    Backward, last chunk first, with G_end = dL/dS_next:
        dU' = P^T dO + (K o f) G_end,  dV = Tm^T dU'
        dP = tril(dO U'^T),  dTm = dU' R^T,  dA = strict_tril(-X^T dTm diag(beta) X^T),
        dA2 = diag(beta) dA
        dQ_P[t, c] = sum_s dP[t, s] k_s[c] D[t, s, c]
        dK_P[s, c] = sum_t dP[t, s] q_t[c] D[t, s, c]
        dK_r[t, c] = sum_s dA2[t, s] k_s[c] D[t, s, c],  dK_c[s, c] = sum_t dA2[t, s] k_t[c] D[t, s, c]
        dQ = gamma o (dO S^T) + dQ_P
        dK = -gamma o (dV S^T) + f o (U' G_end^T) + dK_P + dK_r + dK_c
        dbeta_j = sum_i X_ij dTm_ij + sum_s dA[j, s] A2[j, s]
        dG = q o (gamma o (dO S^T) + dQ_P) + k o (-gamma o (dV S^T) + dK_r)
             - k o (f o (U' G_end^T) + dK_P + dK_c),
             plus, on the last token, sum_j G_end[c, j] S_next[c, j] per channel
        dg_t = sum_{i >= t} dG_i (within the chunk, per channel)
        dL/dS = diag(Gamma) G_end + (Q o gamma)^T dO - (K o gamma)^T dV
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
                K, V, bt = k[b, h, sl], v[b, h, sl], beta[b, h, sl]
                gl = np.cumsum(g[b, h, sl], axis=0)
                n = K.shape[0]
                gam = np.exp(gl)
                D = np.exp(gl[:, None, :] - gl[None, :, :])
                A = np.tril(bt[:, None] * np.einsum("tc,sc,tsc->ts", K, K, D), -1)
                Tm = np.linalg.solve(np.eye(n) + A, np.diag(bt))
                S_at.append(S)
                U = Tm @ (V - (K * gam) @ S)
                S = gam[-1][:, None] * S + (K * (gam[-1] / gam)).T @ U
            G = np.zeros((dk, dv)) if dS_T is None else np.array(dS_T[b, h], dtype=np.float64)
            for t0, S in reversed(list(zip(starts, S_at))):
                sl = slice(t0, min(T, t0 + C))
                K, Q, V = k[b, h, sl], q[b, h, sl], v[b, h, sl]
                bt, dOc = beta[b, h, sl], dO[b, h, sl]
                gl = np.cumsum(g[b, h, sl], axis=0)
                n = K.shape[0]
                gam = np.exp(gl)
                Gam, f = gam[-1], gam[-1] / gam
                D = np.exp(gl[:, None, :] - gl[None, :, :])
                A2 = np.einsum("tc,sc,tsc->ts", K, K, D)
                A = np.tril(bt[:, None] * A2, -1)
                X = np.linalg.inv(np.eye(n) + A)
                Tm = X * bt[None, :]
                R = V - (K * gam) @ S
                U = Tm @ R
                P = np.tril(np.einsum("tc,sc,tsc->ts", Q, K, D))
                S_next = Gam[:, None] * S + (K * f).T @ U
                dU = P.T @ dOc + (K * f) @ G
                dV = Tm.T @ dU
                dP = np.tril(dOc @ U.T)
                dTm = dU @ R.T
                dA = np.tril(-X.T @ (dTm * bt[None, :]) @ X.T, -1)
                dA2 = bt[:, None] * dA
                dQ_P = np.einsum("ts,sc,tsc->tc", dP, K, D)
                dK_P = np.einsum("ts,tc,tsc->sc", dP, Q, D)
                dK_r = np.einsum("ts,sc,tsc->tc", dA2, K, D)
                dK_c = np.einsum("ts,tc,tsc->sc", dA2, K, D)
                dQ_S = gam * (dOc @ S.T)
                dK_S = -gam * (dV @ S.T)
                dK_G = f * (U @ G.T)
                dQ = dQ_S + dQ_P
                dK = dK_S + dK_G + dK_P + dK_r + dK_c
                db = np.sum(X * dTm, axis=0) + np.sum(dA * A2, axis=1)
                dG = Q * dQ + K * (dK_S + dK_r) - K * (dK_G + dK_P + dK_c)
                dG[-1] += np.sum(G * S_next, axis=1)
                out[0][b, h, sl], out[1][b, h, sl], out[2][b, h, sl] = dQ, dK, dV
                out[3][b, h, sl] = db
                out[4][b, h, sl] = np.flip(np.cumsum(np.flip(dG, axis=0), axis=0), axis=0)
                G = Gam[:, None] * G + (Q * gam).T @ dOc - (K * gam).T @ dV
            out[5][b, h] = G
    return tuple(out)


def pin_chunkwise(grad, fwd, gated_grad=None, seed=54):
    """The chunk-level derivation at C = 1, C = 16 with a ragged last chunk,
    and C = T gives the same six gradients."""
    q, k, v, beta, g, S0, dO, dS_T = random_kda_grad_case(seed, B=1, H=2, T=37, dk=6, dv=5)
    got = grad(q, k, v, beta, g, dO, S0, dS_T)
    worst = 0.0
    for C in (1, 16, 37):
        ref = chunkwise_kda_backward(q, k, v, beta, g, dO, S0, dS_T, C)
        worst = max(worst, max(_rel(a, b) for a, b in zip(got, ref)))
    return worst / CHUNK_BOUND


def reverse_loop_kda(q, k, v, beta, g, dO, S0, dS_T, mistake=None):
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
                a = np.exp(g[b, h, t])[:, None]
                kt = k[b, h, t]
                e = v[b, h, t] - (a * S[-1]).T @ kt
                S.append(a * S[-1] + beta[b, h, t] * np.outer(kt, e))
            G = np.zeros((dk, dv)) if dS_T is None else np.array(dS_T[b, h], dtype=np.float64)
            for t in reversed(range(T)):
                a, bt = np.exp(g[b, h, t])[:, None], beta[b, h, t]
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
                da = np.sum(G * S[t], axis=1)
                if mistake == "dg_channel_sum":
                    da = np.full(dk, np.sum(G * S[t]))
                out[4][b, h, t] = a[:, 0] * da if mistake != "dg_without_alpha" else da
                if mistake != "state_gradient_not_decayed":
                    G = a * G
            out[5][b, h] = G
    return tuple(out)


KDA_BWD_MISTAKES = ("predict_without_decay", "dg_without_alpha", "state_gradient_not_decayed",
                    "dg_channel_sum")

ALL_KDA_BWD_PINS = {
    "finite_differences": pin_finite_differences,
    "equal_channels": pin_equal_channels,
    "one_token": pin_one_token,
    "chunkwise": pin_chunkwise,
}
