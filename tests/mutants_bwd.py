"""Deliberately broken restatements of the gradient (planted mistakes).

``reverse_loop`` is a plain numpy statement of the reverse pass through the
token recurrence; each mutant switches on one plausible slip in it.  The
gradient pins must catch every mutant.  CPU only.
"""
import numpy as np


def reverse_loop(q, k, v, beta, dO, S0, dS_T, slip=None):
    B, H, T, dk = q.shape
    dv = v.shape[3]
    dq, dkk, dvv, db = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(beta)
    dS0 = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = [np.zeros((dk, dv)) if S0 is None else np.array(S0[b, h], dtype=np.float64)]
            for t in range(T):  # stored layout: S[i, j], o_t = S^T q_t
                kt = k[b, h, t]
                e = v[b, h, t] - S[-1].T @ kt
                S.append(S[-1] + beta[b, h, t] * np.outer(kt, e))
            G = np.zeros((dk, dv)) if dS_T is None else np.array(dS_T[b, h], dtype=np.float64)
            for t in reversed(range(T)):
                kt, qt, dOt, bt = k[b, h, t], q[b, h, t], dO[b, h, t], beta[b, h, t]
                Sp, St = S[t], S[t + 1]
                G = G + np.outer(qt, dOt)
                dq[b, h, t] = (Sp if slip == "dq_from_old_state" else St) @ dOt
                du = G.T @ kt
                e = v[b, h, t] - (St if slip == "error_from_new_state" else Sp).T @ kt
                dvv[b, h, t] = du if slip == "dv_without_beta" else bt * du
                db[b, h, t] = du @ (bt * e if slip == "dbeta_from_write" else e)
                part = G @ (bt * e)
                if slip != "dropped_prediction_term":
                    part = part - bt * (Sp @ du)
                dkk[b, h, t] = part
                if slip == "state_adjoint_sign":
                    G = G + bt * np.outer(kt, du)
                elif slip != "state_adjoint_skipped":
                    G = G - bt * np.outer(kt, du)
            dS0[b, h] = G
    return dq, dkk, dvv, db, dS0


SLIPS = ("dq_from_old_state", "error_from_new_state", "dv_without_beta", "dbeta_from_write",
         "dropped_prediction_term", "state_adjoint_sign", "state_adjoint_skipped")

ALL_BWD_MUTANTS = {
    s: (lambda s_: (lambda q, k, v, beta, dO, S0, dS_T:
                    reverse_loop(q, k, v, beta, dO, S0, dS_T, slip=s_)))(s)
    for s in SLIPS
}
