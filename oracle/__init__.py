"""fp64 CPU oracle for the DeltaNet delta-rule recurrence -- TEST INFRASTRUCTURE.

This package is not part of the product.  Only the tests, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The product library never calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``deltanet_oracle.c`` (plain C, fp64, OpenMP over the
independent (batch, head) pairs).  This module only compiles it with gcc and
passes numpy arrays to it.  The recurrence, per (b, h), token by token:

    p_t = S_{t-1} k_t;  u_t = beta_t (v_t - p_t);  S_t = S_{t-1} + u_t k_t^T;
    o_t = S_t q_t

is the error-correcting delta rule of "DeltaNet 引入 Delta Rule"
(garden.houmin.site/infra/delta-net) and of "DeltaNet : écrire l'erreur de
prédiction plutôt que la valeur" (fr.news.hada.io/topic?id=31925), reading
after writing as "Calcul de toutes les sorties internes au chunk" on the same
page states.

Layouts follow the library's: q, k ``[B, H, T, dk]``; v, o ``[B, H, T, dv]``;
beta ``[B, H, T]``; state ``[B, H, dk, dv]`` (the pages' dv x dk state stored
transposed, value channel contiguous).

Every function here is pinned by ``tests/test_oracle_pins.py`` to closed
forms, invariants and brute force that do not reuse this code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "deltanet_oracle.c"
_BUILD_DIR = _HERE / "_build"
_LIB_PATH = _BUILD_DIR / "libdn_oracle.so"

_lib = None


def build(force: bool = False) -> Path:
    """Compiles the C oracle with gcc (fp64, no FMA contraction, OpenMP)."""
    if (not force and _LIB_PATH.exists()
            and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime):
        return _LIB_PATH
    _BUILD_DIR.mkdir(exist_ok=True)
    tmp = _BUILD_DIR / f"libdn_oracle.{os.getpid()}.so"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", str(_SRC), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB_PATH))
        dp = ctypes.POINTER(ctypes.c_double)
        lib.dn_oracle_forward.argtypes = [dp, dp, dp, dp, dp, dp,
                                          ctypes.c_long, ctypes.c_long,
                                          ctypes.c_long, ctypes.c_long,
                                          ctypes.c_int]
        lib.dn_oracle_forward.restype = ctypes.c_int
        lib.dn_oracle_backward.argtypes = [dp] * 12 + [ctypes.c_long] * 4 + [ctypes.c_int]
        lib.dn_oracle_backward.restype = ctypes.c_int
        lib.dn_oracle_forward_gated.argtypes = [dp] * 7 + [ctypes.c_long] * 4 + [ctypes.c_int]
        lib.dn_oracle_backward_gated.argtypes = [dp] * 14 + [ctypes.c_long] * 4 + [ctypes.c_int]
        lib.dn_oracle_backward_gated.restype = ctypes.c_int
        lib.dn_oracle_forward_gated.restype = ctypes.c_int
        lib.dn_oracle_forward_kda.argtypes = [dp] * 7 + [ctypes.c_long] * 4 + [ctypes.c_int]
        lib.dn_oracle_forward_kda.restype = ctypes.c_int
        lib.dn_oracle_backward_kda.argtypes = [dp] * 14 + [ctypes.c_long] * 4 + [ctypes.c_int]
        lib.dn_oracle_backward_kda.restype = ctypes.c_int
        lib.dn_oracle_prepare_rows.argtypes = [dp, dp, ctypes.c_long, ctypes.c_long,
                                               ctypes.c_int, ctypes.c_double,
                                               ctypes.c_double]
        lib.dn_oracle_prepare_rows.restype = None
        lib.dn_oracle_prepare_rows_backward.argtypes = [dp, dp, dp, ctypes.c_long,
                                                        ctypes.c_long, ctypes.c_int,
                                                        ctypes.c_double, ctypes.c_double]
        lib.dn_oracle_prepare_rows_backward.restype = None
        _lib = lib
    return _lib


def host_cores() -> int:
    """Cores this process may run on (the count the oracle uses by default)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def forward(q, k, v, beta, S0=None, nthreads: int | None = None):
    """Runs the recurrence over a whole sequence.

    Args:
      q, k: ``[B, H, T, dk]``; v: ``[B, H, T, dv]``; beta: ``[B, H, T]``.
      S0: ``[B, H, dk, dv]`` initial state, or None for zeros.
      nthreads: OpenMP threads (default: every core this process may use).

    Returns ``(o, S_T)`` as fp64 numpy arrays, ``o`` ``[B, H, T, dv]`` and
    ``S_T`` ``[B, H, dk, dv]``.  Inputs of any float dtype are widened to fp64
    exactly, so bf16 inputs reach the oracle with the values the GPU sees.
    """
    q, k, v, beta = _f64(q), _f64(k), _f64(v), _f64(beta)
    if q.ndim != 4 or k.shape != q.shape or v.ndim != 4:
        raise ValueError("q, k must be [B,H,T,dk] and v [B,H,T,dv]")
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if v.shape[:3] != (B, H, T) or beta.shape != (B, H, T):
        raise ValueError("v must be [B,H,T,dv] and beta [B,H,T]")
    if S0 is None:
        S = np.zeros((B, H, dk, dv), dtype=np.float64)
    else:
        S = _f64(S0).copy()
        if S.shape != (B, H, dk, dv):
            raise ValueError("S0 must be [B,H,dk,dv]")
    o = np.zeros((B, H, T, dv), dtype=np.float64)
    if B * H == 0 or T == 0:
        return o, S
    n = host_cores() if nthreads is None else int(nthreads)
    rc = _load().dn_oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                   _ptr(S), _ptr(o), B * H, T, dk, dv, n)
    if rc != 0:
        raise MemoryError("oracle could not allocate its scratch vector")
    return o, S


def recurrent_step(q, k, v, beta, S, nthreads: int | None = None):
    """One decoding step: the recurrence applied to a single token.

    Args:
      q, k: ``[B, H, dk]``; v: ``[B, H, dv]``; beta: ``[B, H]``;
      S: ``[B, H, dk, dv]`` state before the step.

    Returns ``(o, S_new)``: ``o`` ``[B, H, dv]`` and the state after the step.
    """
    q, k, v, beta = _f64(q), _f64(k), _f64(v), _f64(beta)
    o, S_new = forward(q[:, :, None, :], k[:, :, None, :], v[:, :, None, :],
                       beta[:, :, None], S, nthreads=nthreads)
    return o[:, :, 0, :], S_new


def backward(q, k, v, beta, dO, S0=None, dS_T=None, nthreads: int | None = None,
             max_bytes: int = 4 << 30):
    """Gradients of L = <dO, o> + <dS_T, S_T> for the recurrence run by
    ``forward`` (its exact vector-Jacobian product, fp64).

    Args:
      q, k, v, beta, S0: as for ``forward``.
      dO: ``[B, H, T, dv]`` gradient of the outputs.
      dS_T: ``[B, H, dk, dv]`` gradient of the final state, or None (zeros).
      nthreads: OpenMP threads; lowered so that the per-thread copies of the
        T + 1 states of one head stay within ``max_bytes`` in total.

    Returns ``(dq, dk, dv, dbeta, dS0)`` as fp64 numpy arrays shaped like
    ``q, k, v, beta`` and the state.
    """
    q, k, v, beta, dO = _f64(q), _f64(k), _f64(v), _f64(beta), _f64(dO)
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or beta.shape != (B, H, T):
        raise ValueError("q, k must be [B,H,T,dk], v [B,H,T,dv] and beta [B,H,T]")
    if dO.shape != v.shape:
        raise ValueError("dO must be shaped like v")
    S0a = None if S0 is None else _f64(S0)
    dSa = None if dS_T is None else _f64(dS_T)
    for name, a in (("S0", S0a), ("dS_T", dSa)):
        if a is not None and a.shape != (B, H, dk, dv):
            raise ValueError(f"{name} must be [B,H,dk,dv]")
    dq = np.zeros_like(q)
    dkk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    db = np.zeros_like(beta)
    dS0 = np.zeros((B, H, dk, dv), dtype=np.float64)
    if B * H == 0:
        return dq, dkk, dvv, db, dS0
    if T == 0:
        if dSa is not None:
            dS0[...] = dSa
        return dq, dkk, dvv, db, dS0
    n = host_cores() if nthreads is None else int(nthreads)
    per_thread = 8 * dk * dv * (T + 2)
    n = max(1, min(n, max_bytes // max(per_thread, 1)))
    null = ctypes.POINTER(ctypes.c_double)()
    rc = _load().dn_oracle_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(S0a) if S0a is not None else null,
        _ptr(dO), _ptr(dSa) if dSa is not None else null, _ptr(dq), _ptr(dkk), _ptr(dvv),
        _ptr(db), _ptr(dS0), B * H, T, dk, dv, n)
    if rc != 0:
        raise MemoryError("oracle could not allocate its state history")
    return dq, dkk, dvv, db, dS0


def forward_gated(q, k, v, beta, g, S0=None, nthreads: int | None = None):
    """Gated DeltaNet over a whole sequence: the keep rate exp(g_t) decays the
    state before each delta-rule update (forget, predict, correct, write,
    read).  ``g``: ``[B, H, T]`` log keep rates.  Other arguments and the
    result ``(o, S_T)`` as for ``forward``."""
    q, k, v, beta, g = _f64(q), _f64(k), _f64(v), _f64(beta), _f64(g)
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if (k.shape != q.shape or v.shape[:3] != (B, H, T) or beta.shape != (B, H, T)
            or g.shape != (B, H, T)):
        raise ValueError("q, k [B,H,T,dk]; v [B,H,T,dv]; beta and g [B,H,T]")
    S = np.zeros((B, H, dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((B, H, T, dv))
    if B * H == 0 or T == 0:
        return o, S
    n = host_cores() if nthreads is None else int(nthreads)
    rc = _load().dn_oracle_forward_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                         _ptr(S), _ptr(o), B * H, T, dk, dv, n)
    if rc != 0:
        raise MemoryError("oracle could not allocate its scratch vector")
    return o, S


def backward_gated(q, k, v, beta, g, dO, S0=None, dS_T=None, nthreads: int | None = None,
                   max_bytes: int = 4 << 30):
    """Gradients of L = <dO, o> + <dS_T, S_T> for the recurrence run by
    ``forward_gated`` (its exact vector-Jacobian product, fp64).  Arguments as
    for ``backward`` plus ``g`` ``[B, H, T]`` (log keep rates).  Returns
    ``(dq, dk, dv, dbeta, dg, dS0)``."""
    q, k, v, beta, g, dO = _f64(q), _f64(k), _f64(v), _f64(beta), _f64(g), _f64(dO)
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if (k.shape != q.shape or v.shape[:3] != (B, H, T) or beta.shape != (B, H, T)
            or g.shape != (B, H, T) or dO.shape != v.shape):
        raise ValueError("q, k [B,H,T,dk]; v, dO [B,H,T,dv]; beta and g [B,H,T]")
    S0a = None if S0 is None else _f64(S0)
    dSa = None if dS_T is None else _f64(dS_T)
    for name, a in (("S0", S0a), ("dS_T", dSa)):
        if a is not None and a.shape != (B, H, dk, dv):
            raise ValueError(f"{name} must be [B,H,dk,dv]")
    dq, dkk, dvv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    db, dg = np.zeros_like(beta), np.zeros_like(g)
    dS0 = np.zeros((B, H, dk, dv), dtype=np.float64)
    if B * H == 0:
        return dq, dkk, dvv, db, dg, dS0
    if T == 0:
        if dSa is not None:
            dS0[...] = dSa
        return dq, dkk, dvv, db, dg, dS0
    n = host_cores() if nthreads is None else int(nthreads)
    n = max(1, min(n, max_bytes // max(8 * dk * dv * (T + 2), 1)))
    null = ctypes.POINTER(ctypes.c_double)()
    rc = _load().dn_oracle_backward_gated(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
        _ptr(S0a) if S0a is not None else null, _ptr(dO),
        _ptr(dSa) if dSa is not None else null, _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(db),
        _ptr(dg), _ptr(dS0), B * H, T, dk, dv, n)
    if rc != 0:
        raise MemoryError("oracle could not allocate its state history")
    return dq, dkk, dvv, db, dg, dS0


def recurrent_step_gated(q, k, v, beta, g, S, nthreads: int | None = None):
    """One gated decoding step (``g``: ``[B, H]``); returns ``(o, S_new)``."""
    q, k, v, beta, g = _f64(q), _f64(k), _f64(v), _f64(beta), _f64(g)
    o, S_new = forward_gated(q[:, :, None, :], k[:, :, None, :], v[:, :, None, :],
                             beta[:, :, None], g[:, :, None], S, nthreads=nthreads)
    return o[:, :, 0, :], S_new


def forward_varlen(q, k, v, beta, cu_seqlens, S0=None, nthreads: int | None = None):
    """Packed variable-length sequences: q, k ``[H, T, dk]``, v ``[H, T, dv]``,
    beta ``[H, T]`` hold N sequences back to back along T, sequence n being
    tokens ``cu_seqlens[n] .. cu_seqlens[n+1]-1``.  Each sequence runs the
    recurrence from its own initial state (``S0``: ``[N, H, dk, dv]`` or
    None).  Returns ``(o [H, T, dv], S_T [N, H, dk, dv])``."""
    q, k, v, beta = _f64(q), _f64(k), _f64(v), _f64(beta)
    cu = [int(x) for x in cu_seqlens]
    H, T, dk = q.shape
    dv = v.shape[2]
    N = len(cu) - 1
    if cu[0] != 0 or cu[-1] != T or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must rise from 0 to T")
    o = np.zeros((H, T, dv))
    S_T = np.zeros((N, H, dk, dv))
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        s0 = None if S0 is None else _f64(S0)[n][None]
        o_n, S_n = forward(q[None, :, a:b], k[None, :, a:b], v[None, :, a:b], beta[None, :, a:b],
                           s0, nthreads=nthreads)
        o[:, a:b] = o_n[0]
        S_T[n] = S_n[0]
    return o, S_T


def forward_kda(q, k, v, beta, g, S0=None, nthreads: int | None = None):
    """Kimi Delta Attention over a whole sequence: per-key-channel keep rates
    exp(g_t) (``g``: ``[B, H, T, dk]``) decay the state's key channels before
    each delta-rule update.  Other arguments and the result as ``forward``."""
    q, k, v, beta, g = _f64(q), _f64(k), _f64(v), _f64(beta), _f64(g)
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if (k.shape != q.shape or v.shape[:3] != (B, H, T) or beta.shape != (B, H, T)
            or g.shape != q.shape):
        raise ValueError("q, k, g [B,H,T,dk]; v [B,H,T,dv]; beta [B,H,T]")
    S = np.zeros((B, H, dk, dv)) if S0 is None else _f64(S0).copy()
    o = np.zeros((B, H, T, dv))
    if B * H == 0 or T == 0:
        return o, S
    n = host_cores() if nthreads is None else int(nthreads)
    rc = _load().dn_oracle_forward_kda(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                       _ptr(S), _ptr(o), B * H, T, dk, dv, n)
    if rc != 0:
        raise MemoryError("oracle could not allocate its scratch vector")
    return o, S


def backward_kda(q, k, v, beta, g, dO, S0=None, dS_T=None, nthreads: int | None = None,
                 max_bytes: int = 4 << 30):
    """Gradients of L = <dO, o> + <dS_T, S_T> for the recurrence run by
    ``forward_kda`` (its exact vector-Jacobian product, fp64).  Arguments as
    for ``backward`` plus ``g`` ``[B, H, T, dk]`` (per-channel log keep
    rates).  Returns ``(dq, dk, dv, dbeta, dg, dS0)``, ``dg`` shaped like g."""
    q, k, v, beta, g, dO = _f64(q), _f64(k), _f64(v), _f64(beta), _f64(g), _f64(dO)
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if (k.shape != q.shape or v.shape[:3] != (B, H, T) or beta.shape != (B, H, T)
            or g.shape != q.shape or dO.shape != v.shape):
        raise ValueError("q, k, g [B,H,T,dk]; v, dO [B,H,T,dv]; beta [B,H,T]")
    S0a = None if S0 is None else _f64(S0)
    dSa = None if dS_T is None else _f64(dS_T)
    for name, a in (("S0", S0a), ("dS_T", dSa)):
        if a is not None and a.shape != (B, H, dk, dv):
            raise ValueError(f"{name} must be [B,H,dk,dv]")
    dq, dkk, dvv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    db, dg = np.zeros_like(beta), np.zeros_like(g)
    dS0 = np.zeros((B, H, dk, dv), dtype=np.float64)
    if B * H == 0:
        return dq, dkk, dvv, db, dg, dS0
    if T == 0:
        if dSa is not None:
            dS0[...] = dSa
        return dq, dkk, dvv, db, dg, dS0
    n = host_cores() if nthreads is None else int(nthreads)
    n = max(1, min(n, max_bytes // max(8 * dk * dv * (T + 2), 1)))
    null = ctypes.POINTER(ctypes.c_double)()
    rc = _load().dn_oracle_backward_kda(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
        _ptr(S0a) if S0a is not None else null, _ptr(dO),
        _ptr(dSa) if dSa is not None else null, _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(db),
        _ptr(dg), _ptr(dS0), B * H, T, dk, dv, n)
    if rc != 0:
        raise MemoryError("oracle could not allocate its state history")
    return dq, dkk, dvv, db, dg, dS0


def recurrent_step_kda(q, k, v, beta, g, S, nthreads: int | None = None):
    """One KDA decoding step (``g``: ``[B, H, dk]``); returns ``(o, S_new)``."""
    q, k, v, beta, g = _f64(q), _f64(k), _f64(v), _f64(beta), _f64(g)
    o, S_new = forward_kda(q[:, :, None, :], k[:, :, None, :], v[:, :, None, :],
                           beta[:, :, None], g[:, :, None, :], S, nthreads=nthreads)
    return o[:, :, 0, :], S_new


def prepare_qk(q, k, scale: float = 1.0, l2norm: bool = False, eps: float = 1e-6):
    """The optional input preparation, in fp64: with ``l2norm`` every row of
    q and k (the last axis, the head dimension) becomes x / sqrt(sum x^2 + eps);
    then q is multiplied by ``scale``; k is never scaled.  Any leading shape.
    Returns ``(q', k')`` as fp64 numpy arrays; feed them to any form above."""
    q, k = _f64(q), _f64(k)
    if q.shape != k.shape or q.ndim < 1:
        raise ValueError("q and k must have the same shape")
    d = q.shape[-1]
    rows = q.size // d if d else 0
    qo, ko = np.empty_like(q), np.empty_like(k)
    lib = _load()
    lib.dn_oracle_prepare_rows(_ptr(q), _ptr(qo), rows, d, int(l2norm), float(scale),
                               float(eps))
    lib.dn_oracle_prepare_rows(_ptr(k), _ptr(ko), rows, d, int(l2norm), 1.0, float(eps))
    return qo, ko


def prepare_qk_backward(q, k, d_q, d_k, scale: float = 1.0, l2norm: bool = False,
                        eps: float = 1e-6):
    """Gradients of ``prepare_qk`` with respect to its raw inputs, in fp64:
    given the raw q, k and the gradients d_q, d_k of the prepared q', k',
    returns ``(dq_raw, dk_raw)`` (the keys carry no scale)."""
    q, k, d_q, d_k = _f64(q), _f64(k), _f64(d_q), _f64(d_k)
    if not (q.shape == k.shape == d_q.shape == d_k.shape) or q.ndim < 1:
        raise ValueError("q, k, d_q and d_k must share one shape")
    d = q.shape[-1]
    rows = q.size // d if d else 0
    gq, gk = np.empty_like(q), np.empty_like(k)
    lib = _load()
    lib.dn_oracle_prepare_rows_backward(_ptr(q), _ptr(d_q), _ptr(gq), rows, d, int(l2norm),
                                        float(scale), float(eps))
    lib.dn_oracle_prepare_rows_backward(_ptr(k), _ptr(d_k), _ptr(gk), rows, d, int(l2norm),
                                        1.0, float(eps))
    return gq, gk
