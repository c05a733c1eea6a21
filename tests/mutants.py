"""Deliberately broken restatements of the recurrence (planted mistakes).

Each mutant reproduces one plausible slip in writing the oracle.  The pin
tests require every mutant to fail at least one pin, which shows the pins
would catch that slip in the real oracle.  These run on the CPU only.
"""
import numpy as np


def _loop(q, k, v, beta, S0, step):
    B, H, T, dk = q.shape
    dv = v.shape[3]
    o = np.zeros((B, H, T, dv))
    S = np.zeros((B, H, dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    Sm = np.swapaxes(S, -1, -2).copy()          # the pages' dv x dk state
    for b in range(B):
        for h in range(H):
            for t in range(T):
                Sm[b, h], o[b, h, t] = step(Sm[b, h], q[b, h, t], k[b, h, t],
                                            v[b, h, t], beta[b, h, t],
                                            k[b, h, t - 1] if t else k[b, h, t])
    return o, np.swapaxes(Sm, -1, -2).copy()


def read_before_write(q, k, v, beta, S0):
    def step(S, qt, kt, vt, bt, kprev):
        o = S @ qt
        return S + np.outer(bt * (vt - S @ kt), kt), o
    return _loop(q, k, v, beta, S0, step)


def flipped_error_sign(q, k, v, beta, S0):
    def step(S, qt, kt, vt, bt, kprev):
        S = S + np.outer(bt * (S @ kt - vt), kt)
        return S, S @ qt
    return _loop(q, k, v, beta, S0, step)


def dropped_beta(q, k, v, beta, S0):
    def step(S, qt, kt, vt, bt, kprev):
        S = S + np.outer(vt - S @ kt, kt)
        return S, S @ qt
    return _loop(q, k, v, beta, S0, step)


def beta_on_value_only(q, k, v, beta, S0):
    def step(S, qt, kt, vt, bt, kprev):
        S = S + np.outer(bt * vt - S @ kt, kt)
        return S, S @ qt
    return _loop(q, k, v, beta, S0, step)


def hadamard_transition(q, k, v, beta, S0):
    """The elementwise slip: S * (1 - beta k k^T) instead of a matrix product."""
    def step(S, qt, kt, vt, bt, kprev):
        S = S * (1.0 - bt * np.outer(np.ones(S.shape[0]), kt * kt)) + bt * np.outer(vt, kt)
        return S, S @ qt
    return _loop(q, k, v, beta, S0, step)


def transposed_state(q, k, v, beta, S0):
    """Treats the stored [dk][dv] array as the dv x dk state without
    transposing (only shape-compatible when dk == dv)."""
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if dk != dv:
        raise ValueError("shape mismatch")
    o = np.zeros((B, H, T, dv))
    S = np.zeros((B, H, dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                kt, vt, qt, bt = k[b, h, t], v[b, h, t], q[b, h, t], beta[b, h, t]
                S[b, h] = S[b, h] + np.outer(bt * (vt - S[b, h] @ kt), kt)
                o[b, h, t] = S[b, h] @ qt
    return o, S


def stale_key(q, k, v, beta, S0):
    """Predicts with the previous token's key."""
    def step(S, qt, kt, vt, bt, kprev):
        S = S + np.outer(bt * (vt - S @ kprev), kt)
        return S, S @ qt
    return _loop(q, k, v, beta, S0, step)


def query_for_prediction(q, k, v, beta, S0):
    def step(S, qt, kt, vt, bt, kprev):
        S = S + np.outer(bt * (vt - S @ qt), kt)
        return S, S @ qt
    return _loop(q, k, v, beta, S0, step)


def ignores_initial_state(q, k, v, beta, S0):
    return _loop(q, k, v, beta, None, lambda S, qt, kt, vt, bt, kp: (
        S + np.outer(bt * (vt - S @ kt), kt),
        (S + np.outer(bt * (vt - S @ kt), kt)) @ qt))


def one_minus_beta(q, k, v, beta, S0):
    """Uses 1 - beta as the write strength."""
    def step(S, qt, kt, vt, bt, kprev):
        S = S + np.outer((1.0 - bt) * (vt - S @ kt), kt)
        return S, S @ qt
    return _loop(q, k, v, beta, S0, step)


ALL_MUTANTS = {
    "read_before_write": read_before_write,
    "flipped_error_sign": flipped_error_sign,
    "dropped_beta": dropped_beta,
    "beta_on_value_only": beta_on_value_only,
    "hadamard_transition": hadamard_transition,
    "transposed_state": transposed_state,
    "stale_key": stale_key,
    "query_for_prediction": query_for_prediction,
    "ignores_initial_state": ignores_initial_state,
    "one_minus_beta": one_minus_beta,
}
