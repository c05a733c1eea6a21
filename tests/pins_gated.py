"""Independent checks ("pins") of a Gated DeltaNet implementation.

An implementation is ``run(q, k, v, beta, g, S0) -> (o, S_T)`` with the
library's layouts (state ``[dk][dv]``) and ``g`` the log keep rate
``[B, H, T]``.  Each pin checks it against a statement that does not reuse
its code:

- zero decay (g = 0) is the plain delta rule (the pinned forward oracle);
- beta = 0 leaves only the decay: closed forms for o and S_T;
- the normalised-state identity: with Gamma_t = exp(sum_{s<=t} g_s), the
  state S_t / Gamma_t follows the plain delta rule with values v_t / Gamma_t,
  so the gated outputs are Gamma_t times plain outputs (run by the plain
  oracle on rescaled inputs);
- the pages' product form S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T)
  + beta_t v_t k_t^T with explicit matrices;
- a whole-chunk derivation (``chunkwise_gated``), the algebra the GPU kernel
  uses, at C = 1, 16 (ragged) and T.

Each pin returns its largest error divided by its bound (a passing pin
returns at most 1).  Dimensions use dk != dv.
"""
from __future__ import annotations

import numpy as np

from tests.pins import _unit

EXACT_BOUND = 1e-11
CHUNK_BOUND = 1e-9


def random_gated_case(seed, B=2, H=2, T=24, dk=5, dv=7, beta_hi=1.0, g_lo=-0.3):
    r = np.random.default_rng(seed)
    q = _unit(r.standard_normal((B, H, T, dk)))
    k = _unit(r.standard_normal((B, H, T, dk)))
    v = r.standard_normal((B, H, T, dv))
    beta = r.uniform(0.05, beta_hi, size=(B, H, T))
    g = r.uniform(g_lo, 0.0, size=(B, H, T))
    S0 = r.standard_normal((B, H, dk, dv)) * 0.5
    return q, k, v, beta, g, S0


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return np.inf
    return float(np.max(np.abs(a - b)) / max(1.0, float(np.max(np.abs(b))))) if a.size else 0.0


def pin_zero_decay(run, plain, seed=41):
    q, k, v, beta, g, S0 = random_gated_case(seed)
    o, S = run(q, k, v, beta, np.zeros_like(g), S0)
    o_ref, S_ref = plain(q, k, v, beta, S0)
    return max(_rel(o, o_ref), _rel(S, S_ref)) / EXACT_BOUND


def pin_beta_zero(run, plain, seed=42):
    q, k, v, beta, g, S0 = random_gated_case(seed)
    o, S = run(q, k, v, np.zeros_like(beta), g, S0)
    gam = np.exp(np.cumsum(g, axis=-1))                       # Gamma_t
    o_ref = gam[..., None] * np.einsum("bhij,bhti->bhtj", S0, q)
    S_ref = gam[..., -1, None, None] * S0
    return max(_rel(o, o_ref), _rel(S, S_ref)) / EXACT_BOUND


def pin_normalised_state(run, plain, seed=43):
    q, k, v, beta, g, S0 = random_gated_case(seed, T=20, g_lo=-0.2)
    o, S = run(q, k, v, beta, g, S0)
    gam = np.exp(np.cumsum(g, axis=-1))
    o_hat, S_hat = plain(q, k, v / gam[..., None], beta, S0)
    o_ref = gam[..., None] * o_hat
    S_ref = gam[..., -1, None, None] * S_hat
    return max(_rel(o, o_ref), _rel(S, S_ref)) / CHUNK_BOUND


def pin_product_form(run, plain, seed=44):
    q, k, v, beta, g, S0 = random_gated_case(seed, beta_hi=2.0)
    o, S = run(q, k, v, beta, g, S0)
    B, H, T, dk = q.shape
    o_ref = np.zeros_like(o)
    S_ref = np.zeros_like(S)
    for b in range(B):
        for h in range(H):
            Sm = S0[b, h].T.copy()                              # the pages' dv x dk state
            for t in range(T):
                kt = k[b, h, t]
                Sm = (np.exp(g[b, h, t]) * Sm @ (np.eye(dk) - beta[b, h, t] * np.outer(kt, kt))
                      + beta[b, h, t] * np.outer(v[b, h, t], kt))
                o_ref[b, h, t] = Sm @ q[b, h, t]
            S_ref[b, h] = Sm.T
    return max(_rel(o, o_ref), _rel(S, S_ref)) / EXACT_BOUND


def chunkwise_gated(q, k, v, beta, g, S0, C):
    """Gated delta rule through whole-chunk matrices (fp64).  Per chunk, with
    G_t the cumulative log decay from the chunk start and S stored [dk][dv]:
        A = tril(diag(beta) (K K^T . exp(G_i - G_j)), -1),  T = (I + A)^{-1} diag(beta)
        E = T (V - diag(exp G) K S)                             (the true errors)
        O = diag(exp G) Q S + (Q K^T . M . exp(G_i - G_j)) E    (M causal, diagonal in)
        S <- exp(G_C) S + K^T diag(exp(G_C - G_s)) E
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
                G = np.cumsum(g[b, h, sl])
                ratio = np.exp(G[:, None] - G[None, :])
                A = np.tril(bt[:, None] * (K @ K.T) * ratio, -1)
                Tm = np.linalg.solve(np.eye(n) + A, np.diag(bt))
                E = Tm @ (V - np.exp(G)[:, None] * (K @ S))
                o[b, h, sl] = np.exp(G)[:, None] * (Q @ S) + (np.tril(Q @ K.T) * ratio) @ E
                S = np.exp(G[-1]) * S + K.T @ (np.exp(G[-1] - G)[:, None] * E)
            S_out[b, h] = S
    return o, S_out


def pin_chunkwise(run, plain, seed=45):
    q, k, v, beta, g, S0 = random_gated_case(seed, B=1, T=37, beta_hi=2.0)
    o, S = run(q, k, v, beta, g, S0)
    worst = 0.0
    for C in (1, 16, 37):
        o_ref, S_ref = chunkwise_gated(q, k, v, beta, g, S0, C)
        worst = max(worst, _rel(o, o_ref), _rel(S, S_ref))
    return worst / CHUNK_BOUND


ALL_GATED_PINS = {
    "zero_decay": pin_zero_decay,
    "beta_zero": pin_beta_zero,
    "normalised_state": pin_normalised_state,
    "product_form": pin_product_form,
    "chunkwise": pin_chunkwise,
}


def gated_loop(q, k, v, beta, g, S0, slip=None):
    """A plain numpy statement of the gated recurrence; ``slip`` switches on
    one planted mistake (tests/test_oracle_gated_pins.py)."""
    B, H, T, dk = q.shape
    dv = v.shape[3]
    o = np.zeros((B, H, T, dv))
    S_out = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            Sm = np.zeros((dv, dk)) if S0 is None else np.array(S0[b, h]).T.copy()
            for t in range(T):
                kt, qt, vt, bt = k[b, h, t], q[b, h, t], v[b, h, t], beta[b, h, t]
                gt = g[b, h, t - 1] if (slip == "previous_token_gate" and t > 0) else g[b, h, t]
                alpha = gt if slip == "gate_not_exponentiated" else np.exp(gt)
                if slip == "predict_before_forget":
                    p = Sm @ kt
                    Sm = alpha * Sm
                elif slip == "forget_after_write":
                    p = Sm @ kt
                else:
                    Sm = alpha * Sm
                    p = Sm @ kt
                Sm = Sm + np.outer(bt * (vt - p), kt)
                if slip == "forget_after_write":
                    Sm = alpha * Sm
                o[b, h, t] = Sm @ qt
            S_out[b, h] = Sm.T
    return o, S_out


GATED_SLIPS = ("predict_before_forget", "forget_after_write", "gate_not_exponentiated",
               "previous_token_gate")
