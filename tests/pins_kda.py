"""Independent checks ("pins") of a Kimi Delta Attention (KDA) implementation.

An implementation is ``run(q, k, v, beta, g, S0) -> (o, S_T)`` with the
library's layouts (state ``[dk][dv]``) and ``g`` the per-key-channel log keep
rates ``[B, H, T, dk]``.  Each pin checks it against a statement that does
not reuse its code:

- equal channels (g_t[i] the same for every i) is Gated DeltaNet, and zero
  decay the plain delta rule (both pinned oracles);
- beta = 0 leaves only the per-channel decay: closed forms;
- the pages' diagonal-plus-low-rank form S_t = S_{t-1} D_t (I - beta_t k_t
  k_t^T) + beta_t v_t k_t^T with explicit matrices;
- a whole-chunk derivation (``chunkwise_kda``), the algebra the GPU kernel
  uses, at C = 1, 16 (ragged) and T.

Each pin returns its largest error divided by its bound.  dk != dv.
"""
from __future__ import annotations

import numpy as np

from tests.pins import _unit

EXACT_BOUND = 1e-11
CHUNK_BOUND = 1e-9


def random_kda_case(seed, B=2, H=2, T=24, dk=5, dv=7, beta_hi=1.0, g_lo=-0.4):
    r = np.random.default_rng(seed)
    q = _unit(r.standard_normal((B, H, T, dk)))
    k = _unit(r.standard_normal((B, H, T, dk)))
    v = r.standard_normal((B, H, T, dv))
    beta = r.uniform(0.05, beta_hi, size=(B, H, T))
    g = r.uniform(g_lo, 0.0, size=(B, H, T, dk))
    S0 = r.standard_normal((B, H, dk, dv)) * 0.5
    return q, k, v, beta, g, S0


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return np.inf
    return float(np.max(np.abs(a - b)) / max(1.0, float(np.max(np.abs(b))))) if a.size else 0.0


def pin_equal_channels(run, plain, gated, seed=61):
    q, k, v, beta, g, S0 = random_kda_case(seed)
    gs = g[..., 0]
    o, S = run(q, k, v, beta, np.repeat(gs[..., None], q.shape[-1], -1), S0)
    o_ref, S_ref = gated(q, k, v, beta, gs, S0)
    o2, S2 = run(q, k, v, beta, np.zeros_like(g), S0)
    o2_ref, S2_ref = plain(q, k, v, beta, S0)
    return max(_rel(o, o_ref), _rel(S, S_ref), _rel(o2, o2_ref), _rel(S2, S2_ref)) / EXACT_BOUND


def pin_beta_zero(run, plain, gated, seed=62):
    q, k, v, beta, g, S0 = random_kda_case(seed)
    o, S = run(q, k, v, np.zeros_like(beta), g, S0)
    gam = np.exp(np.cumsum(g, axis=2))                         # [B,H,T,dk]
    S_t = gam[..., None] * S0[:, :, None]                      # [B,H,T,dk,dv]
    o_ref = np.einsum("bhtij,bhti->bhtj", S_t, q)
    return max(_rel(o, o_ref), _rel(S, S_t[:, :, -1])) / EXACT_BOUND


def pin_dplr_form(run, plain, gated, seed=63):
    q, k, v, beta, g, S0 = random_kda_case(seed, beta_hi=2.0)
    o, S = run(q, k, v, beta, g, S0)
    B, H, T, dk = q.shape
    o_ref, S_ref = np.zeros_like(o), np.zeros_like(S)
    for b in range(B):
        for h in range(H):
            Sm = S0[b, h].T.copy()                              # the pages' dv x dk state
            for t in range(T):
                kt = k[b, h, t]
                A = np.diag(np.exp(g[b, h, t])) @ (np.eye(dk) - beta[b, h, t] * np.outer(kt, kt))
                Sm = Sm @ A + beta[b, h, t] * np.outer(v[b, h, t], kt)
                o_ref[b, h, t] = Sm @ q[b, h, t]
            S_ref[b, h] = Sm.T
    return max(_rel(o, o_ref), _rel(S, S_ref)) / EXACT_BOUND


def chunkwise_kda(q, k, v, beta, g, S0, C):
    """KDA through whole-chunk matrices (fp64).  Per chunk, with G_t[d] the
    cumulative log decay of key channel d from the chunk start (token t
    included) and S stored [dk][dv]:
        A[i][j] = beta_i sum_d k_i[d] k_j[d] exp(G_i[d] - G_j[d])     (j < i)
        P[i][j] = sum_d q_i[d] k_j[d] exp(G_i[d] - G_j[d])            (j <= i)
        E = (I + A)^{-1} diag(beta) (V - (K . exp G) S)
        O = (Q . exp G) S + P E
        S <- diag(exp G_C) S + (K . exp(G_C - G))^T E
    Every exponent is <= 0.
    """
    B, H, T, dk = q.shape
    dv = v.shape[3]
    o = np.zeros((B, H, T, dv))
    S_out = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            for t0 in range(0, T, C):
                sl = slice(t0, min(T, t0 + C))
                K, Q, V, bt = k[b, h, sl], q[b, h, sl], v[b, h, sl], beta[b, h, sl]
                n = K.shape[0]
                G = np.cumsum(g[b, h, sl], axis=0)              # [n, dk]
                ratio = np.exp(G[:, None, :] - G[None, :, :])   # [i, j, d]
                A = np.tril(bt[:, None] * np.einsum("id,jd,ijd->ij", K, K, ratio), -1)
                P = np.tril(np.einsum("id,jd,ijd->ij", Q, K, ratio))
                E = np.linalg.solve(np.eye(n) + A, bt[:, None] * (V - (K * np.exp(G)) @ S))
                o[b, h, sl] = (Q * np.exp(G)) @ S + P @ E
                S = np.exp(G[-1])[:, None] * S + (K * np.exp(G[-1] - G)).T @ E
            S_out[b, h] = S
    return o, S_out


def pin_chunkwise(run, plain, gated, seed=64):
    q, k, v, beta, g, S0 = random_kda_case(seed, B=1, T=37, beta_hi=2.0)
    o, S = run(q, k, v, beta, g, S0)
    worst = 0.0
    for C in (1, 16, 37):
        o_ref, S_ref = chunkwise_kda(q, k, v, beta, g, S0, C)
        worst = max(worst, _rel(o, o_ref), _rel(S, S_ref))
    return worst / CHUNK_BOUND


ALL_KDA_PINS = {
    "equal_channels": pin_equal_channels,
    "beta_zero": pin_beta_zero,
    "dplr_form": pin_dplr_form,
    "chunkwise": pin_chunkwise,
}


def kda_loop(q, k, v, beta, g, S0, slip=None):
    """A plain numpy statement of KDA (math orientation); ``slip`` switches on
    one planted mistake."""
    B, H, T, dk = q.shape
    dv = v.shape[3]
    o, S_out = np.zeros((B, H, T, dv)), np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            Sm = np.zeros((dv, dk)) if S0 is None else np.array(S0[b, h]).T.copy()
            for t in range(T):
                kt, qt, vt, bt = k[b, h, t], q[b, h, t], v[b, h, t], beta[b, h, t]
                gt = g[b, h, t - 1] if (slip == "previous_token_decay" and t > 0) else g[b, h, t]
                a = np.exp(gt)
                if slip == "decay_after_predict":
                    p = Sm @ kt
                    Sm = Sm * a[None, :]
                elif slip == "decay_on_value_channels":  # rates cycled over the dv rows
                    Sm = Sm * np.resize(a, Sm.shape[0])[:, None]
                    p = Sm @ kt
                else:
                    Sm = Sm * a[None, :]
                    p = Sm @ kt
                Sm = Sm + np.outer(bt * (vt - p), kt)
                o[b, h, t] = Sm @ qt
            S_out[b, h] = Sm.T
    return o, S_out


KDA_SLIPS = ("decay_after_predict", "decay_on_value_channels", "previous_token_decay")
