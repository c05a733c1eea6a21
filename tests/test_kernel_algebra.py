"""The regroupings the tensor-core kernels compute, pinned to the oracle.

CPU only, fp64.  Each test walks a sequence chunk by chunk using exactly the
products and operand blocks a kernel forms (not the kernel's code: numpy
matrices in the same arrangement) and compares the result with the oracle's
token-by-token recurrence, at a chunk length of 16 over 37 tokens (two full
chunks and a ragged one) and dk != dv, so that a dropped term, a sign, a
transposed block or a misplaced decay factor fails:

- the forward scan: D1 = [PT; Tm] V - ([[PT, -I]; [Tm, 0]] [K; Q]) S, the
  chunk group's one MMA chain and the D1 MMAs' negated operand;
- the gated scan: the same with the decay-scaled blocks
  [[PT E, -E]; [Tm E, 0]] (E = diag(exp G)), the keep factor exp(G_C) on the
  state and exp(G_C - G_s) on U';
- the backward chain: dV = PT^T dO + (K^T Tm)^T G, G <- G + Q^T dO - K^T dV,
  reading the forward's [PT; Tm] transposed; and its KDA form, with the
  forward's decayed operands (K o f in the chunk group's tile, Q o gamma and
  K o gamma in the update) and the keep factors exp G_L on G's key rows,
  which the gated backward also takes with one rate on every channel;
- KDA on CUDA cores: the per-channel ratio as exp(G_i[d]) exp(-G_j[d]).
- the per-chunk gradients in feature-lane form (the layout a tcgen05
  gradient kernel takes), dP and dTm as diagonal blocks of one product.
- the independence of the value columns (plain, gated, KDA), which lets a
  scan split dv across CTAs with no exchange.
- a sequence split through augmented state columns ([v | 0] from [0 | I]),
  and the same as two packed-sequence calls plus a scan over segments.
"""
import numpy as np
import pytest

import oracle
from tests.pins import _unit

C = 16


def _case(seed, T=37, dk=5, dv=7, gate=False, kda=False):
    r = np.random.default_rng(seed)
    q = _unit(r.standard_normal((1, 1, T, dk)))
    k = _unit(r.standard_normal((1, 1, T, dk)))
    v = r.standard_normal((1, 1, T, dv))
    beta = r.uniform(0.05, 1.5, size=(1, 1, T))
    S0 = r.standard_normal((1, 1, dk, dv)) * 0.5
    g = None
    if gate:
        g = np.log(r.uniform(0.5, 1.0, size=(1, 1, T)))
    if kda:
        g = np.log(r.uniform(0.5, 1.0, size=(1, 1, T, dk)))
    return q, k, v, beta, S0, g


def _chunk_tiles(K, Q, bt, ratio=None):
    """[PT; Tm] as the prepare pass forms it (ratio: in-chunk decay)."""
    n = K.shape[0]
    KK, QK = K @ K.T, Q @ K.T
    if ratio is not None:
        KK, QK = KK * ratio, QK * ratio
    A = np.tril(bt[:, None] * KK, -1)
    Tm = np.linalg.solve(np.eye(n) + A, np.diag(bt))
    P = np.tril(QK)
    return P @ Tm, Tm


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(1.0, float(np.max(np.abs(b)))))


def test_forward_scan_regrouping():
    q, k, v, beta, S0, _ = _case(1)
    K_, Q_, V_, b_ = k[0, 0], q[0, 0], v[0, 0], beta[0, 0]
    S = S0[0, 0].copy()
    o = np.zeros_like(V_)
    for t0 in range(0, K_.shape[0], C):
        sl = slice(t0, t0 + C)
        K, Q, V, bt = K_[sl], Q_[sl], V_[sl], b_[sl]
        n = K.shape[0]
        PT, Tm = _chunk_tiles(K, Q, bt)
        left = np.vstack([PT, Tm])                                    # [PT; Tm]
        Ablk = np.block([[PT, -np.eye(n)], [Tm, np.zeros((n, n))]])   # the chain's A
        negQW = Ablk @ np.vstack([K, Q])                              # [-Q'; W]
        D1 = left @ V - negQW @ S                                     # negated B operand
        o[sl] = D1[:n]
        S = S + K.T @ D1[n:]                                          # S += K^T U'
    o_ref, S_ref = oracle.forward(q, k, v, beta, S0)
    assert _rel(o, o_ref[0, 0]) < 1e-10
    assert _rel(S, S_ref[0, 0]) < 1e-10


def test_gated_scan_regrouping():
    q, k, v, beta, S0, g = _case(2, gate=True)
    K_, Q_, V_, b_, g_ = k[0, 0], q[0, 0], v[0, 0], beta[0, 0], g[0, 0]
    S = S0[0, 0].copy()
    o = np.zeros_like(V_)
    for t0 in range(0, K_.shape[0], C):
        sl = slice(t0, t0 + C)
        K, Q, V, bt = K_[sl], Q_[sl], V_[sl], b_[sl]
        n = K.shape[0]
        G = np.cumsum(g_[sl])
        ratio = np.exp(np.minimum(G[:, None] - G[None, :], 0.0))
        PT, Tm = _chunk_tiles(K, Q, bt, ratio)
        E = np.diag(np.exp(G))
        Ablk = np.block([[PT @ E, -E], [Tm @ E, np.zeros((n, n))]])
        negQW = Ablk @ np.vstack([K, Q])
        D1 = np.vstack([PT, Tm]) @ V - negQW @ S
        o[sl] = D1[:n]
        dec = np.exp(G[-1] - G)
        S = np.exp(G[-1]) * S + K.T @ (dec[:, None] * D1[n:])
    o_ref, S_ref = oracle.forward_gated(q, k, v, beta, g, S0)
    assert _rel(o, o_ref[0, 0]) < 1e-10
    assert _rel(S, S_ref[0, 0]) < 1e-10


def test_backward_chain_regrouping():
    """The chain's dV and state gradients; the oracle's d_v and d_S0."""
    q, k, v, beta, S0, _ = _case(3)
    r = np.random.default_rng(33)
    dO = r.standard_normal(v.shape)
    dS_T = r.standard_normal(S0.shape)
    K_, Q_, V_, b_, dO_ = k[0, 0], q[0, 0], v[0, 0], beta[0, 0], dO[0, 0]
    T = K_.shape[0]
    starts = list(range(0, T, C))
    tiles = [_chunk_tiles(K_[t0:t0 + C], Q_[t0:t0 + C], b_[t0:t0 + C]) for t0 in starts]
    G = dS_T[0, 0].copy()
    dV = np.zeros_like(V_)
    for t0, (PT, Tm) in reversed(list(zip(starts, tiles))):
        sl = slice(t0, t0 + C)
        K, Q, D = K_[sl], Q_[sl], dO_[sl]
        B2 = K.T @ Tm                       # the chunk group's tile (dk x tokens)
        dVc = PT.T @ D + B2.T @ G           # dV^T = dO^T PT + G^T (K^T Tm)
        dV[sl] = dVc
        G = G + Q.T @ D - K.T @ dVc         # G^T += dO^T Q - dV^T K
    ref = oracle.backward(q, k, v, beta, dO, S0, dS_T)
    assert _rel(dV, ref[2][0, 0]) < 1e-9
    assert _rel(G, ref[4][0, 0]) < 1e-9


@pytest.mark.parametrize("equal_channels", [False, True], ids=["kda", "gated"])
def test_kda_backward_chain_regrouping(equal_channels):
    """The tcgen05 KDA chain: dV = PT^T dO + ((K o f)^T Tm)^T G and
    G <- diag(exp G_L) G + (Q o gamma)^T dO - (K o gamma)^T dV, with [PT; Tm]
    carrying the per-channel ratios; the oracle's d_v and d_S0 (KDA, and with
    one rate on every key channel the gated oracle's)."""
    q, k, v, beta, S0, g = _case(5, kda=True)
    if equal_channels:
        g = np.repeat(g[..., :1], g.shape[-1], axis=-1)
    r = np.random.default_rng(55)
    dO = r.standard_normal(v.shape)
    dS_T = r.standard_normal(S0.shape)
    K_, Q_, b_, dO_, g_ = k[0, 0], q[0, 0], beta[0, 0], dO[0, 0], g[0, 0]
    T = K_.shape[0]
    G = dS_T[0, 0].copy()
    dV = np.zeros_like(v[0, 0])
    for t0 in reversed(range(0, T, C)):
        sl = slice(t0, t0 + C)
        K, Q, D, bt = K_[sl], Q_[sl], dO_[sl], b_[sl]
        Gc = np.cumsum(g_[sl], axis=0)                   # per-channel log decay from the chunk start
        n = K.shape[0]
        ratio = np.exp(Gc[:, None, :] - Gc[None, :, :])  # exp(G_t[c] - G_s[c])
        A = np.tril(bt[:, None] * np.einsum("tc,sc,tsc->ts", K, K, ratio), -1)
        Tm = np.linalg.solve(np.eye(n) + A, np.diag(bt))
        PT = np.tril(np.einsum("tc,sc,tsc->ts", Q, K, ratio)) @ Tm
        gam, eL = np.exp(Gc), np.exp(Gc[-1])
        Kh, Kp, Qp = K * (eL / gam), K * gam, Q * gam    # the forward's decayed operands
        dVc = PT.T @ D + (Kh.T @ Tm).T @ G               # dV^T = dO^T PT + G^T (K^T Tm)
        dV[sl] = dVc
        G = eL[:, None] * G + Qp.T @ D - Kp.T @ dVc      # keep on G's key rows, then the update
    if equal_channels:
        ref = oracle.backward_gated(q, k, v, beta, g[..., 0], dO, S0, dS_T)
    else:
        ref = oracle.backward_kda(q, k, v, beta, g, dO, S0, dS_T)
    assert _rel(dV, ref[2][0, 0]) < 1e-9
    assert _rel(G, ref[5][0, 0]) < 1e-9


@pytest.mark.parametrize("scale", [1.0, 40.0], ids=["mild", "strong"])
def test_kda_separable_ratio(scale):
    """A and P from K exp(G), Q exp(G) and K exp(-G), against the per-entry
    ratio inside the sums, and the whole KDA chunk walk against the oracle
    (strong: G reaches about -40 per channel inside a chunk, still normal)."""
    q, k, v, beta, S0, g = _case(4, kda=True)
    g = g * scale
    K_, Q_, V_, b_, g_ = k[0, 0], q[0, 0], v[0, 0], beta[0, 0], g[0, 0]
    S = S0[0, 0].copy()
    o = np.zeros_like(V_)
    for t0 in range(0, K_.shape[0], C):
        sl = slice(t0, t0 + C)
        K, Q, V, bt = K_[sl], Q_[sl], V_[sl], b_[sl]
        n = K.shape[0]
        Gk = np.cumsum(g_[sl], axis=0)                      # [n][dk]
        Kp, Km, Qp = K * np.exp(Gk), K * np.exp(-Gk), Q * np.exp(Gk)
        A_sep, P_sep = Kp @ Km.T, Qp @ Km.T
        ratio = np.exp(np.minimum(Gk[:, None, :] - Gk[None, :, :], 0.0))
        A_dir = np.einsum("id,jd,ijd->ij", K, K, ratio)
        mask = np.tril(np.ones((n, n)), -1).astype(bool)
        assert np.allclose(A_sep[mask], A_dir[mask], rtol=1e-9, atol=1e-12)
        A = np.tril(bt[:, None] * A_sep, -1)
        P = np.tril(P_sep)
        Tm = np.linalg.solve(np.eye(n) + A, np.diag(bt))
        U = Tm @ (V - Kp @ S)
        o[sl] = Qp @ S + P @ U
        eC = np.exp(Gk[-1])
        S = eC[:, None] * S + (Km * eC).T @ U
    o_ref, S_ref = oracle.forward_kda(q, k, v, beta, g, S0)
    assert _rel(o, o_ref[0, 0]) < 1e-9
    assert _rel(S, S_ref[0, 0]) < 1e-9


def test_gradient_kernel_feature_lane_plan():
    """The per-chunk gradients in the feature-lane form a tcgen05 gradient
    kernel would use (every product with a 128-wide feature dimension as M):
    R^T = V^T - S^T K^T, U'^T = R^T Tm^T, dU'^T = dO^T P + G^T K^T,
    dV^T = dU'^T Tm, dP and dTm as the diagonal blocks of one product
    [dO; dU'] [U'; R]^T, dQ^T = S dO^T + K^T dP^T and
    dK^T = Q^T dP + G U'^T - S dV^T + K^T Z; against the oracle's gradient."""
    q, k, v, beta, S0, _ = _case(5)
    r = np.random.default_rng(55)
    dO = r.standard_normal(v.shape)
    dS_T = r.standard_normal(S0.shape)
    K_, Q_, V_, b_, dO_ = k[0, 0], q[0, 0], v[0, 0], beta[0, 0], dO[0, 0]
    T = K_.shape[0]
    starts = list(range(0, T, C))
    S_at, S = [], S0[0, 0].copy()
    for t0 in starts:  # the states at chunk starts (the recompute)
        sl = slice(t0, t0 + C)
        _, Tm = _chunk_tiles(K_[sl], Q_[sl], b_[sl])
        S_at.append(S)
        S = S + K_[sl].T @ (Tm @ (V_[sl] - K_[sl] @ S))
    G_end, G = [None] * len(starts), dS_T[0, 0].copy()
    for i in reversed(range(len(starts))):  # the chain: G at every chunk end
        sl = slice(starts[i], starts[i] + C)
        PT, Tm = _chunk_tiles(K_[sl], Q_[sl], b_[sl])
        G_end[i] = G
        dVc = PT.T @ dO_[sl] + (K_[sl].T @ Tm).T @ G
        G = G + Q_[sl].T @ dO_[sl] - K_[sl].T @ dVc
    dq, dk, dv, db = (np.zeros_like(Q_), np.zeros_like(K_), np.zeros_like(V_),
                      np.zeros_like(b_))
    for i, t0 in enumerate(starts):
        sl = slice(t0, t0 + C)
        K, Q, V, D, bt, S, G = K_[sl], Q_[sl], V_[sl], dO_[sl], b_[sl], S_at[i], G_end[i]
        n = K.shape[0]
        KK = K @ K.T
        X = np.linalg.inv(np.eye(n) + np.tril(bt[:, None] * KK, -1))
        Tm = X * bt[None, :]
        P = np.tril(Q @ K.T)
        Rt = V.T - S.T @ K.T                       # dv x n
        Ut = Rt @ Tm.T                             # U'^T
        dUt = D.T @ P + G.T @ K.T                  # dU'^T
        dVt = dUt @ Tm                             # dV^T
        D5 = np.vstack([D, dUt.T]) @ np.vstack([Ut.T, Rt.T]).T
        dP = np.tril(D5[:n, :n])
        dTm = D5[n:, n:]
        M1 = (dTm * bt[None, :]) @ X.T
        dA = np.tril(-X.T @ M1, -1)
        Z = bt[:, None] * dA + (bt[:, None] * dA).T
        dQt = S @ D.T + K.T @ dP.T                 # dk x n
        dKt = Q.T @ dP + G @ Ut - S @ dVt + K.T @ Z
        dq[sl], dk[sl], dv[sl] = dQt.T, dKt.T, dVt.T
        db[sl] = np.sum(X * dTm, axis=0) + np.sum(dA * KK, axis=1)
    ref = oracle.backward(q, k, v, beta, dO, S0, dS_T)
    for got, want in zip((dq, dk, dv, db), ref[:4]):
        assert _rel(got, want[0, 0]) < 1e-9


@pytest.mark.parametrize("form", ["plain", "gated", "kda"])
def test_value_columns_are_independent(form):
    """Column j of the state, of U' and of the output depends only on column
    j of v and of S0, so a scan may split the value dimension across CTAs
    with no exchange: the oracle run on a column slice of v and S0 gives
    that slice of the full run's o and S_T, exactly."""
    q, k, v, beta, S0, g = _case(6, dv=9, gate=form == "gated", kda=form == "kda")
    run = {"plain": lambda vv, SS: oracle.forward(q, k, vv, beta, SS),
           "gated": lambda vv, SS: oracle.forward_gated(q, k, vv, beta, g, SS),
           "kda": lambda vv, SS: oracle.forward_kda(q, k, vv, beta, g, SS)}[form]
    o, S = run(v, S0)
    for cols in (slice(0, 4), slice(4, 9), slice(2, 3)):
        o_c, S_c = run(np.ascontiguousarray(v[..., cols]), np.ascontiguousarray(S0[..., cols]))
        assert np.array_equal(o_c, o[..., cols])
        assert np.array_equal(S_c, S[..., cols])


@pytest.mark.parametrize("form", ["plain", "gated", "kda"])
def test_sequence_split_through_augmented_columns(form):
    """A sequence cut into segments, each run from its own start with no
    knowledge of the others, then joined by a short scan over segments.

    The state is linear in the initial state, S_t = A_t S_start + B_t (A_t
    the product of the transitions so far, decay included).  Running a
    segment with value columns [v | 0] from the initial state [0 | I] gives,
    column by column (the columns are independent): o_zero and B in the
    first dv columns, and in the last dk columns the transformed queries
    q~_t = A_t^T q_t (outputs) and A (final state).  Then per segment
    o = o_zero + q~ S_start and S_end = A S_start + B."""
    q, k, v, beta, S0, g = _case(7, T=41, gate=form == "gated", kda=form == "kda")
    dk, dv = q.shape[-1], v.shape[-1]

    def run(sl, vv, SS):
        if form == "plain":
            return oracle.forward(q[..., sl, :], k[..., sl, :], vv, beta[..., sl], SS)
        gg = g[..., sl, :] if form == "kda" else g[..., sl]
        f = oracle.forward_kda if form == "kda" else oracle.forward_gated
        return f(q[..., sl, :], k[..., sl, :], vv, beta[..., sl], gg, SS)

    o_full, S_full = run(slice(None), v, S0)
    S_start = S0[0, 0]
    outs = []
    for a, b in ((0, 13), (13, 29), (29, 41)):
        sl = slice(a, b)
        v_aug = np.concatenate([v[..., sl, :], np.zeros((1, 1, b - a, dk))], axis=-1)
        S_aug = np.concatenate([np.zeros((1, 1, dk, dv)), np.eye(dk)[None, None]], axis=-1)
        o_aug, S_end_aug = run(sl, v_aug, S_aug)
        o_zero, q_t = o_aug[0, 0, :, :dv], o_aug[0, 0, :, dv:]
        B, A = S_end_aug[0, 0, :, :dv], S_end_aug[0, 0, :, dv:]
        outs.append(o_zero + q_t @ S_start)
        S_start = A @ S_start + B
    assert _rel(np.concatenate(outs), o_full[0, 0]) < 1e-12
    assert _rel(S_start, S_full[0, 0]) < 1e-12


def test_sequence_split_as_two_packed_calls():
    """The long-prefill plan in the packed-sequence calling convention
    (q, k, v, beta [H, T, d]; cu_seqlens at the segment cuts; one initial
    state per segment [N, H, dk, dv]): one call with [v, S0 = 0] and one with
    [0, S0 = I] (dv = dk there), then per head the scan over segments and
    the correction, against one unsplit run per head."""
    r = np.random.default_rng(8)
    H, T, d = 3, 150, 6
    q = _unit(r.standard_normal((H, T, d)))
    k = _unit(r.standard_normal((H, T, d)))
    v = r.standard_normal((H, T, d))
    beta = r.uniform(0.05, 1.5, (H, T))
    S0 = 0.5 * r.standard_normal((H, d, d))
    cu = [0, 40, 64, 129, 150]
    N = len(cu) - 1
    o_zero, B = oracle.forward_varlen(q, k, v, beta, cu)
    eye = np.broadcast_to(np.eye(d), (N, H, d, d))
    q_t, A = oracle.forward_varlen(q, k, np.zeros_like(v), beta, cu, S0=eye)
    o_full, S_full = oracle.forward(q[None], k[None], v[None], beta[None], S0[None])
    for h in range(H):
        S_start = S0[h]
        for n in range(N):
            sl = slice(cu[n], cu[n + 1])
            o_seg = o_zero[h, sl] + q_t[h, sl] @ S_start
            assert _rel(o_seg, o_full[0, h, sl]) < 1e-12
            S_start = A[n, h] @ S_start + B[n, h]
        assert _rel(S_start, S_full[0, h]) < 1e-12
