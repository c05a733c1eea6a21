"""GB300-native DeltaNet delta-rule operator.

Thin Python binding over the C ABI in ``include/deltanet.h``: these functions
only check tensors, allocate outputs with PyTorch and pass raw device
pointers plus the current CUDA stream to ``libdeltanet.so``.  Every step of
the computation runs in the library's sm_103a kernels.

    chunk_fwd(q, k, v, beta, initial_state=None, output_final_state=True)
        -> (o, final_state)          # training / prefill, chunkwise form
    recurrent_step(q, k, v, beta, state) -> o   # decoding, state in place
    chunk_bwd(q, k, v, beta, d_o, initial_state=None, d_final_state=None)
        -> (d_q, d_k, d_v, d_beta, d_initial_state)   # training backward
    DeltaRule.apply(q, k, v, beta, initial_state, scale)  # autograd: (o, final_state)
    chunk_fwd_varlen(q, k, v, beta, cu_seqlens, ...)  # packed sequences, [H, T, d]
    chunk_fwd_gated(q, k, v, beta, g, ...), recurrent_step_gated(q, k, v, beta, g, state)
        # Gated DeltaNet: log keep rate g per token (per head for a step)
    chunk_bwd_gated(q, k, v, beta, g, d_o, ...) -> (d_q, d_k, d_v, d_beta, d_g, d_initial_state)
    GatedDeltaRule.apply(q, k, v, beta, g, initial_state, scale, qk_l2norm)  # autograd
    chunk_bwd_kda(q, k, v, beta, g, d_o, ...), KdaDeltaRule.apply(...)  # KDA's gradients
    chunk_fwd_kda(q, k, v, beta, g, ...), recurrent_step_kda(q, k, v, beta, g, state)
        # KDA: one log keep rate per key channel
    qk_prepare(q, k, scale=1.0, l2norm=True)  # the q/k L2-norm and query scale as a pass
    qk_prepare_bwd(q, k, d_q_out, d_k_out, scale, l2norm)  # its gradient

Shapes: q, k ``[B, H, T, dk]``; v ``[B, H, T, dv]``; beta ``[B, H, T]``;
state ``[B, H, dk, dv]`` fp32 (the pages' dv x dk state, transposed).  For a
decoding step the T axis is absent.  q and k are used as given unless a
forward or step is called with ``qk_l2norm=True`` and/or ``scale=...``: the
kernels then L2-normalise q and k (and scale q) as they load them (the
``*_qk`` entry points); the backward takes prepared q and k, and
``DeltaRule`` chains the preparation's gradient after it.
"""
from __future__ import annotations

import torch

import ctypes

from ._lib import (DN_ALGO_AUTO, DN_ALGO_SIMT, DN_ALGO_TCGEN05, DN_BF16, DN_F32,
                   DeltaNetError, QkNorm, check, header_symbols, lib_path, load)

__all__ = ["chunk_fwd", "chunk_fwd_split", "chunk_bwd", "chunk_bwd_varlen", "chunk_bwd_gated", "chunk_bwd_kda", "recurrent_step", "chunk_fwd_varlen", "chunk_fwd_gated",
           "recurrent_step_gated", "chunk_fwd_kda", "recurrent_step_kda", "qk_prepare",
           "qk_prepare_bwd", "DeltaRule", "GatedDeltaRule", "KdaDeltaRule", "DeltaNetError", "load", "lib_path",
           "header_symbols", "ALGOS"]

ALGOS = {"auto": DN_ALGO_AUTO, "simt": DN_ALGO_SIMT, "tcgen05": DN_ALGO_TCGEN05}
_DT = {torch.float32: DN_F32, torch.bfloat16: DN_BF16}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")
    return _DT[t.dtype]


def _check_cuda(name: str, t: torch.Tensor, device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda" or (device is not None and t.device != device):
        raise ValueError(f"{name} must live on {device or 'a CUDA device'}, not {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def qk_prepare(q: torch.Tensor, k: torch.Tensor, scale: float = 1.0, l2norm: bool = True,
               eps: float = 1e-6, inplace: bool = False):
    """Optional input preparation (``dn_qk_prepare``): with ``l2norm`` every
    row of q and k (the last axis) becomes x / sqrt(sum x^2 + eps); q is then
    multiplied by ``scale``.  Returns ``(q', k')``, new tensors unless
    ``inplace``; without ``l2norm`` k is returned as it is."""
    dev = q.device
    _check_cuda("q", q, dev)
    _check_cuda("k", k, dev)
    dt = _dtype_code(q)
    if k.dtype != q.dtype or k.shape != q.shape or q.dim() < 1:
        raise ValueError("q and k must share one shape and dtype")
    d = q.shape[-1]
    rows = q.numel() // d if d else 0
    q_out = q if inplace else torch.empty_like(q)
    k_out = k if (inplace or not l2norm) else torch.empty_like(k)
    lib = load()
    with torch.cuda.device(dev):
        check(lib.dn_qk_prepare(q.data_ptr(), k.data_ptr(), q_out.data_ptr(), k_out.data_ptr(),
                                rows, d, int(bool(l2norm)), float(scale), float(eps), dt,
                                _stream_handle(dev)))
    return q_out, k_out


def qk_prepare_bwd(q: torch.Tensor, k: torch.Tensor, d_q_out: torch.Tensor,
                   d_k_out: torch.Tensor | None, scale: float = 1.0, l2norm: bool = True,
                   eps: float = 1e-6):
    """Gradient of ``qk_prepare`` (``dn_qk_prepare_bwd``): given the raw q, k
    and the gradients of the prepared q', k', returns ``(d_q, d_k)`` with
    respect to the raw inputs (``d_k`` is ``d_k_out`` itself without
    ``l2norm``, since k is then used as given)."""
    dev = q.device
    for name, t in (("q", q), ("k", k), ("d_q_out", d_q_out)):
        _check_cuda(name, t, dev)
    dt = _dtype_code(q)
    if k.shape != q.shape or d_q_out.shape != q.shape or k.dtype != q.dtype or \
            d_q_out.dtype != q.dtype:
        raise ValueError("q, k and d_q_out must share one shape and dtype")
    if l2norm:
        _check_cuda("d_k_out", d_k_out, dev)
        if d_k_out.shape != q.shape or d_k_out.dtype != q.dtype:
            raise ValueError("d_k_out must match q")
    d = q.shape[-1]
    rows = q.numel() // d if d else 0
    d_q = torch.empty_like(q)
    d_k = torch.empty_like(k) if l2norm else d_k_out
    lib = load()
    with torch.cuda.device(dev):
        check(lib.dn_qk_prepare_bwd(
            q.data_ptr(), k.data_ptr(), d_q_out.data_ptr(),
            d_k_out.data_ptr() if l2norm else None, d_q.data_ptr(),
            d_k.data_ptr() if l2norm else None, rows, d, int(bool(l2norm)), float(scale),
            float(eps), dt, _stream_handle(dev)))
    return d_q, d_k


def _norm(scale, qk_l2norm, eps=1e-6):
    """The dn_qk_norm a forward or step was asked for (None: none)."""
    if scale is None and not qk_l2norm:
        return None
    return ctypes.byref(QkNorm(int(bool(qk_l2norm)), 1.0 if scale is None else float(scale),
                               float(eps)))


def _forward_tensors(q, k, v, beta, initial_state, output_final_state, out, final_state):
    """Checks a [B,H,T,d] forward's tensors; allocates o and S_T when not given.
    Returns (device, dtype code, (B, H, T, dk, dv), o, S_T or None)."""
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta)):
        _check_cuda(name, t, dev)
    dt = _dtype_code(q)
    if not (k.dtype == v.dtype == beta.dtype == q.dtype):
        raise TypeError("q, k, v and beta must share one dtype")
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4:
        raise ValueError("q, k must be [B,H,T,dk] and v [B,H,T,dv]")
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if tuple(v.shape[:3]) != (B, H, T) or tuple(beta.shape) != (B, H, T):
        raise ValueError("v must be [B,H,T,dv] and beta [B,H,T]")
    if initial_state is not None:
        _check_cuda("initial_state", initial_state, dev)
        if initial_state.dtype != torch.float32 or tuple(initial_state.shape) != (B, H, dk, dv):
            raise ValueError("initial_state must be float32 [B,H,dk,dv]")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=dev)
    else:
        _check_cuda("out", out, dev)
        if out.dtype != q.dtype or tuple(out.shape) != (B, H, T, dv):
            raise ValueError("out must match v's shape and dtype")
    S_T = None
    if output_final_state:
        S_T = final_state if final_state is not None else torch.empty(
            (B, H, dk, dv), dtype=torch.float32, device=dev)
        _check_cuda("final_state", S_T, dev)
        if S_T.dtype != torch.float32 or tuple(S_T.shape) != (B, H, dk, dv):
            raise ValueError("final_state must be float32 [B,H,dk,dv]")
    return dev, dt, (B, H, T, dk, dv), out, S_T


def chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
              initial_state: torch.Tensor | None = None, output_final_state: bool = True,
              chunk_size: int = 64, algo: str = "auto", out: torch.Tensor | None = None,
              final_state: torch.Tensor | None = None, workspace="auto",
              scale: float | None = None, qk_l2norm: bool = False):
    """Chunkwise delta-rule forward (``dn_chunk_fwd``).

    Returns ``(o, S_T)``; ``S_T`` is None when ``output_final_state`` is
    False.  ``final_state`` may be ``initial_state`` itself to update it in
    place; ``out`` may supply the output buffer.  ``workspace``: "auto"
    allocates the scratch ``dn_chunk_fwd_workspace_bytes`` asks for (the
    two-pass tensor-core path), None runs without scratch (one fused kernel),
    and a uint8 CUDA tensor of at least that many bytes is used as given.
    ``qk_l2norm`` / ``scale``: the kernels L2-normalise q and k and scale q
    as they load them (``dn_chunk_fwd_qk``).
    """
    dev, dt, (B, H, T, dk, dv), out, S_T = _forward_tensors(
        q, k, v, beta, initial_state, output_final_state, out, final_state)
    lib = load()
    ws_bytes = lib.dn_chunk_fwd_workspace_bytes(B, H, T, dk, dv, chunk_size, dt)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', None or a uint8 CUDA tensor")
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    elif workspace is None:
        ws, ws_bytes = None, 0
    else:
        _check_cuda("workspace", workspace, dev)
        ws, ws_bytes = workspace, workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        check(lib.dn_chunk_fwd_qk(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(),
            initial_state.data_ptr() if initial_state is not None else None,
            out.data_ptr(), S_T.data_ptr() if S_T is not None else None,
            B, H, T, dk, dv, chunk_size, dt,
            ws.data_ptr() if ws is not None else None, ws_bytes,
            _stream_handle(dev), ALGOS[algo], _norm(scale, qk_l2norm)))
    return out, S_T


def chunk_fwd_split(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                    initial_state: torch.Tensor | None = None, output_final_state: bool = True,
                    segments: int = 0, chunk_size: int = 64, out: torch.Tensor | None = None,
                    final_state: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None):
    """The chunkwise forward for a few long sequences (``dn_chunk_fwd_split``):
    each sequence cut into ``segments`` runs scanned in parallel (0: enough
    to fill the GPU once).  bf16, dk = dv = 128.  Arguments and results as
    for ``chunk_fwd``; ``workspace`` is a uint8 CUDA tensor of at least
    ``dn_chunk_fwd_split_workspace_bytes`` bytes, or None to allocate one."""
    dev, dt, (B, H, T, dk, dv), out, S_T = _forward_tensors(
        q, k, v, beta, initial_state, output_final_state, out, final_state)
    lib = load()
    with torch.cuda.device(dev):
        ws_bytes = lib.dn_chunk_fwd_split_workspace_bytes(B, H, T, dk, dv, chunk_size, dt,
                                                          segments)
        if workspace is None:
            workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        _check_cuda("workspace", workspace, dev)
        check(lib.dn_chunk_fwd_split(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(),
            initial_state.data_ptr() if initial_state is not None else None,
            out.data_ptr(), S_T.data_ptr() if S_T is not None else None,
            B, H, T, dk, dv, chunk_size, dt, segments, workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(dev)))
    return out, S_T


def recurrent_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                   state: torch.Tensor, out: torch.Tensor | None = None,
                   scale: float | None = None, qk_l2norm: bool = False) -> torch.Tensor:
    """One fused decoding step (``dn_recurrent_step``); ``state`` is updated
    in place and the step's output ``o`` ``[B, H, dv]`` is returned.
    ``qk_l2norm`` / ``scale``: the step L2-normalises q and k and scales q
    as it loads them."""
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("state", state)):
        _check_cuda(name, t, dev)
    dt = _dtype_code(q)
    if not (k.dtype == v.dtype == beta.dtype == q.dtype):
        raise TypeError("q, k, v and beta must share one dtype")
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3:
        raise ValueError("q, k must be [B,H,dk] and v [B,H,dv]")
    B, H, dk = q.shape
    dv = v.shape[2]
    if tuple(v.shape[:2]) != (B, H) or tuple(beta.shape) != (B, H):
        raise ValueError("v must be [B,H,dv] and beta [B,H]")
    if state.dtype != torch.float32 or tuple(state.shape) != (B, H, dk, dv):
        raise ValueError("state must be float32 [B,H,dk,dv]")
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=dev)
    else:
        _check_cuda("out", out, dev)
        if out.dtype != q.dtype or tuple(out.shape) != (B, H, dv):
            raise ValueError("out must be [B,H,dv] in q's dtype")
    lib = load()
    with torch.cuda.device(dev):
        check(lib.dn_recurrent_step_qk(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                       beta.data_ptr(), state.data_ptr(), out.data_ptr(), B, H,
                                       dk, dv, dt, _stream_handle(dev), _norm(scale, qk_l2norm)))
    return out


def chunk_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
              d_o: torch.Tensor, initial_state: torch.Tensor | None = None,
              d_final_state: torch.Tensor | None = None, chunk_size: int = 64,
              workspace: torch.Tensor | None = None):
    """Gradients of the chunkwise forward (``dn_chunk_bwd``).

    Returns ``(d_q, d_k, d_v, d_beta, d_initial_state)`` for
    L = <d_o, o> + <d_final_state, final_state>; ``d_initial_state`` is fp32
    ``[B, H, dk, dv]`` (zeros-based even when ``initial_state`` is None).
    ``workspace``: a uint8 CUDA tensor of at least
    ``dn_chunk_bwd_workspace_bytes`` bytes, or None to allocate one.
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("d_o", d_o)):
        _check_cuda(name, t, dev)
    dt = _dtype_code(q)
    if not (k.dtype == v.dtype == beta.dtype == d_o.dtype == q.dtype):
        raise TypeError("q, k, v, beta and d_o must share one dtype")
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or d_o.shape != v.shape:
        raise ValueError("q, k must be [B,H,T,dk]; v and d_o [B,H,T,dv]")
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if tuple(v.shape[:3]) != (B, H, T) or tuple(beta.shape) != (B, H, T):
        raise ValueError("v must be [B,H,T,dv] and beta [B,H,T]")
    for name, t in (("initial_state", initial_state), ("d_final_state", d_final_state)):
        if t is not None:
            _check_cuda(name, t, dev)
            if t.dtype != torch.float32 or tuple(t.shape) != (B, H, dk, dv):
                raise ValueError(f"{name} must be float32 [B,H,dk,dv]")
    lib = load()
    need = lib.dn_chunk_bwd_workspace_bytes(B, H, T, dk, dv, chunk_size, dt)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    else:
        _check_cuda("workspace", workspace, dev)
    d_q, d_k = torch.empty_like(q), torch.empty_like(k)
    d_v, d_beta = torch.empty_like(v), torch.empty_like(beta)
    d_S0 = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        check(lib.dn_chunk_bwd(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(),
            initial_state.data_ptr() if initial_state is not None else None, d_o.data_ptr(),
            d_final_state.data_ptr() if d_final_state is not None else None,
            d_q.data_ptr(), d_k.data_ptr(), d_v.data_ptr(), d_beta.data_ptr(), d_S0.data_ptr(),
            B, H, T, dk, dv, chunk_size, dt, workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(dev)))
    return d_q, d_k, d_v, d_beta, d_S0


class DeltaRule(torch.autograd.Function):
    """Autograd wrapper: ``DeltaRule.apply(q, k, v, beta, initial_state,
    scale, qk_l2norm)`` returns ``(o, final_state)`` from ``chunk_fwd``; the
    backward pass calls ``chunk_bwd`` (the chunk states are recomputed there,
    not stored).  ``qk_l2norm`` L2-normalises q and k and ``scale`` (None for
    none) multiplies q, inside the forward's kernels; the backward forms the
    prepared q and k again (``qk_prepare``), takes the recurrence's gradient
    with respect to them and chains the preparation's gradient
    (``qk_prepare_bwd``) to reach the raw q and k."""

    @staticmethod
    def forward(ctx, q, k, v, beta, initial_state=None, scale=None, qk_l2norm=False):
        q, k, v, beta = (t.contiguous() for t in (q, k, v, beta))
        if initial_state is not None:
            initial_state = initial_state.contiguous()
        o, S_T = chunk_fwd(q, k, v, beta, initial_state=initial_state, output_final_state=True,
                           scale=scale, qk_l2norm=qk_l2norm)
        ctx.save_for_backward(q, k, v, beta, initial_state)
        ctx.scale, ctx.l2norm = scale, bool(qk_l2norm)
        return o, S_T

    @staticmethod
    def backward(ctx, d_o, d_S_T):
        q, k, v, beta, S0 = ctx.saved_tensors
        d_o = torch.zeros_like(v) if d_o is None else d_o.contiguous()
        d_S_T = None if d_S_T is None else d_S_T.contiguous().float()
        prepared = ctx.scale is not None or ctx.l2norm
        scale = 1.0 if ctx.scale is None else ctx.scale
        qp, kp = qk_prepare(q, k, scale=scale, l2norm=ctx.l2norm) if prepared else (q, k)
        d_q, d_k, d_v, d_beta, d_S0 = chunk_bwd(qp, kp, v, beta, d_o.to(v.dtype), S0, d_S_T)
        if prepared:
            d_q, d_k = qk_prepare_bwd(q, k, d_q, d_k, scale=scale, l2norm=ctx.l2norm)
        return d_q, d_k, d_v, d_beta, (d_S0 if S0 is not None else None), None, None


def _decayed_forward(ctx, per_channel, q, k, v, beta, g, initial_state, scale, qk_l2norm):
    q, k, v, beta, g = (t.contiguous() for t in (q, k, v, beta, g))
    if initial_state is not None:
        initial_state = initial_state.contiguous()
    fwd = chunk_fwd_kda if per_channel else chunk_fwd_gated
    o, S_T = fwd(q, k, v, beta, g, initial_state=initial_state, output_final_state=True,
                 scale=scale, qk_l2norm=qk_l2norm)
    ctx.save_for_backward(q, k, v, beta, g, initial_state)
    ctx.scale, ctx.l2norm = scale, bool(qk_l2norm)
    return o, S_T


def _decayed_backward(ctx, per_channel, d_o, d_S_T):
    q, k, v, beta, g, S0 = ctx.saved_tensors
    d_o = torch.zeros_like(v) if d_o is None else d_o.contiguous()
    d_S_T = None if d_S_T is None else d_S_T.contiguous().float()
    prepared = ctx.scale is not None or ctx.l2norm
    scale = 1.0 if ctx.scale is None else ctx.scale
    qp, kp = qk_prepare(q, k, scale=scale, l2norm=ctx.l2norm) if prepared else (q, k)
    bwd = chunk_bwd_kda if per_channel else chunk_bwd_gated
    d_q, d_k, d_v, d_beta, d_g, d_S0 = bwd(qp, kp, v, beta, g, d_o.to(v.dtype), S0, d_S_T)
    if prepared:
        d_q, d_k = qk_prepare_bwd(q, k, d_q, d_k, scale=scale, l2norm=ctx.l2norm)
    return (d_q, d_k, d_v, d_beta, d_g, (d_S0 if S0 is not None else None), None, None)


class GatedDeltaRule(torch.autograd.Function):
    """Autograd wrapper for Gated DeltaNet: ``GatedDeltaRule.apply(q, k, v,
    beta, g, initial_state, scale, qk_l2norm)`` returns ``(o, final_state)``
    from ``chunk_fwd_gated``; the backward calls ``chunk_bwd_gated`` (states
    recomputed there) and chains the q/k preparation's gradient as
    ``DeltaRule`` does.  ``g`` is the fp32 ``[B, H, T]`` log keep rate and
    receives a gradient."""

    @staticmethod
    def forward(ctx, q, k, v, beta, g, initial_state=None, scale=None, qk_l2norm=False):
        return _decayed_forward(ctx, False, q, k, v, beta, g, initial_state, scale, qk_l2norm)

    @staticmethod
    def backward(ctx, d_o, d_S_T):
        return _decayed_backward(ctx, False, d_o, d_S_T)


class KdaDeltaRule(torch.autograd.Function):
    """Autograd wrapper for KDA: as ``GatedDeltaRule`` with ``chunk_fwd_kda``
    and ``chunk_bwd_kda``; ``g`` is the fp32 ``[B, H, T, dk]`` per-key-channel
    log keep rate."""

    @staticmethod
    def forward(ctx, q, k, v, beta, g, initial_state=None, scale=None, qk_l2norm=False):
        return _decayed_forward(ctx, True, q, k, v, beta, g, initial_state, scale, qk_l2norm)

    @staticmethod
    def backward(ctx, d_o, d_S_T):
        return _decayed_backward(ctx, True, d_o, d_S_T)


def _check_gate(g: torch.Tensor, shape, dev) -> None:
    _check_cuda("g", g, dev)
    if g.dtype != torch.float32 or tuple(g.shape) != tuple(shape):
        raise ValueError(f"g must be float32 {list(shape)}")


def chunk_fwd_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                    g: torch.Tensor, initial_state: torch.Tensor | None = None,
                    output_final_state: bool = True, chunk_size: int = 64,
                    out: torch.Tensor | None = None, final_state: torch.Tensor | None = None,
                    workspace="auto", scale: float | None = None, qk_l2norm: bool = False):
    """Gated DeltaNet, chunkwise (``dn_chunk_fwd_gated``): ``g`` is the fp32
    ``[B, H, T]`` log keep rate.  Returns ``(o, S_T)`` as ``chunk_fwd``.
    ``workspace``: "auto" allocates the scratch of the two-pass tensor-core
    form where it applies (``dn_chunk_fwd_gated_workspace_bytes``), None runs
    the fp32 CUDA-core kernel, a uint8 CUDA tensor supplies the scratch.
    ``qk_l2norm`` / ``scale``: prepared inside the kernels, as ``chunk_fwd``."""
    return _chunk_decayed(q, k, v, beta, g, False, initial_state, output_final_state,
                          chunk_size, out, final_state, workspace, scale, qk_l2norm)


def chunk_fwd_kda(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                  g: torch.Tensor, initial_state: torch.Tensor | None = None,
                  output_final_state: bool = True, chunk_size: int = 64,
                  out: torch.Tensor | None = None, final_state: torch.Tensor | None = None,
                  workspace="auto", scale: float | None = None, qk_l2norm: bool = False):
    """Kimi Delta Attention, chunkwise (``dn_chunk_fwd_kda``): ``g`` is the
    fp32 ``[B, H, T, dk]`` per-key-channel log keep rate.  The page's read
    scales q by d_k^{-1/2}: ``scale=dk ** -0.5`` applies it.
    ``qk_l2norm`` / ``scale``: prepared inside the kernels, as ``chunk_fwd``.
    ``workspace``: "auto" allocates the scratch of the tensor-core form where
    it applies (``dn_chunk_fwd_kda_workspace_bytes``), None runs the fp32
    CUDA-core kernel, a uint8 CUDA tensor supplies the scratch."""
    return _chunk_decayed(q, k, v, beta, g, True, initial_state, output_final_state,
                          chunk_size, out, final_state, workspace, scale, qk_l2norm)


def _chunk_decayed(q, k, v, beta, g, per_channel, initial_state, output_final_state,
                   chunk_size, out, final_state, workspace, scale=None, qk_l2norm=False):
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta)):
        _check_cuda(name, t, dev)
    dt = _dtype_code(q)
    if not (k.dtype == v.dtype == beta.dtype == q.dtype):
        raise TypeError("q, k, v and beta must share one dtype")
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4:
        raise ValueError("q, k must be [B,H,T,dk] and v [B,H,T,dv]")
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if tuple(v.shape[:3]) != (B, H, T) or tuple(beta.shape) != (B, H, T):
        raise ValueError("v must be [B,H,T,dv] and beta [B,H,T]")
    _check_gate(g, (B, H, T, dk) if per_channel else (B, H, T), dev)
    if initial_state is not None:
        _check_cuda("initial_state", initial_state, dev)
        if initial_state.dtype != torch.float32 or tuple(initial_state.shape) != (B, H, dk, dv):
            raise ValueError("initial_state must be float32 [B,H,dk,dv]")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=dev)
    else:
        _check_cuda("out", out, dev)
        if out.dtype != q.dtype or tuple(out.shape) != (B, H, T, dv):
            raise ValueError("out must match v's shape and dtype")
    S_T = None
    if output_final_state:
        S_T = final_state if final_state is not None else torch.empty(
            (B, H, dk, dv), dtype=torch.float32, device=dev)
        _check_cuda("final_state", S_T, dev)
        if S_T.dtype != torch.float32 or tuple(S_T.shape) != (B, H, dk, dv):
            raise ValueError("final_state must be float32 [B,H,dk,dv]")
    lib = load()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(), g.data_ptr(),
            initial_state.data_ptr() if initial_state is not None else None, out.data_ptr(),
            S_T.data_ptr() if S_T is not None else None, B, H, T, dk, dv, chunk_size, dt)
    sizer = (lib.dn_chunk_fwd_kda_workspace_bytes if per_channel
             else lib.dn_chunk_fwd_gated_workspace_bytes)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', None or a uint8 CUDA tensor")
        need = sizer(B, H, T, dk, dv, chunk_size, dt)
        ws = torch.empty(need, dtype=torch.uint8, device=dev) if need else None
    else:
        ws = workspace
        if ws is not None:
            _check_cuda("workspace", ws, dev)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    entry = lib.dn_chunk_fwd_kda_qk if per_channel else lib.dn_chunk_fwd_gated_qk
    with torch.cuda.device(dev):
        check(entry(*args, ws.data_ptr() if ws is not None else None, ws_bytes,
                    _stream_handle(dev), _norm(scale, qk_l2norm)))
    return out, S_T


def recurrent_step_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                         g: torch.Tensor, state: torch.Tensor,
                         out: torch.Tensor | None = None, scale: float | None = None,
                         qk_l2norm: bool = False) -> torch.Tensor:
    """One Gated DeltaNet decoding step (``dn_recurrent_step_gated``); ``g``
    is the fp32 ``[B, H]`` log keep rate; ``state`` is updated in place.
    ``qk_l2norm`` / ``scale``: prepared inside the kernel."""
    return _step_decayed(q, k, v, beta, g, False, state, out, scale, qk_l2norm)


def recurrent_step_kda(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                       g: torch.Tensor, state: torch.Tensor,
                       out: torch.Tensor | None = None, scale: float | None = None,
                       qk_l2norm: bool = False) -> torch.Tensor:
    """One KDA decoding step (``dn_recurrent_step_kda``); ``g`` is the fp32
    ``[B, H, dk]`` per-key-channel log keep rate; ``state`` updated in place.
    ``qk_l2norm`` / ``scale``: prepared inside the kernel."""
    return _step_decayed(q, k, v, beta, g, True, state, out, scale, qk_l2norm)


def _step_decayed(q, k, v, beta, g, per_channel, state, out, scale=None, qk_l2norm=False):
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("state", state)):
        _check_cuda(name, t, dev)
    dt = _dtype_code(q)
    if not (k.dtype == v.dtype == beta.dtype == q.dtype):
        raise TypeError("q, k, v and beta must share one dtype")
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3:
        raise ValueError("q, k must be [B,H,dk] and v [B,H,dv]")
    B, H, dk = q.shape
    dv = v.shape[2]
    if tuple(v.shape[:2]) != (B, H) or tuple(beta.shape) != (B, H):
        raise ValueError("v must be [B,H,dv] and beta [B,H]")
    _check_gate(g, (B, H, dk) if per_channel else (B, H), dev)
    if state.dtype != torch.float32 or tuple(state.shape) != (B, H, dk, dv):
        raise ValueError("state must be float32 [B,H,dk,dv]")
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=dev)
    else:
        _check_cuda("out", out, dev)
        if out.dtype != q.dtype or tuple(out.shape) != (B, H, dv):
            raise ValueError("out must be [B,H,dv] in q's dtype")
    lib = load()
    with torch.cuda.device(dev):
        entry = lib.dn_recurrent_step_kda_qk if per_channel else lib.dn_recurrent_step_gated_qk
        check(entry(q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(), g.data_ptr(),
                    state.data_ptr(), out.data_ptr(), B, H, dk, dv, dt, _stream_handle(dev),
                    _norm(scale, qk_l2norm)))
    return out


def chunk_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                     cu_seqlens, initial_state: torch.Tensor | None = None,
                     output_final_state: bool = True, chunk_size: int = 64,
                     workspace="auto", scale: float | None = None, qk_l2norm: bool = False):
    """Packed variable-length sequences (``dn_chunk_fwd_varlen``).

    q, k ``[H, T, dk]``, v ``[H, T, dv]``, beta ``[H, T]`` hold N sequences
    back to back; ``cu_seqlens`` (a host sequence of N + 1 ints) gives their
    offsets.  Returns ``(o [H, T, dv], S_T [N, H, dk, dv] or None)``.
    ``workspace``: "auto" (the two-pass tensor-core path where it applies),
    None (the CUDA-core path) or a uint8 CUDA tensor.
    ``qk_l2norm`` / ``scale``: prepared inside the kernels, as ``chunk_fwd``.
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta)):
        _check_cuda(name, t, dev)
    dt = _dtype_code(q)
    if not (k.dtype == v.dtype == beta.dtype == q.dtype):
        raise TypeError("q, k, v and beta must share one dtype")
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3:
        raise ValueError("q, k must be [H,T,dk] and v [H,T,dv]")
    H, T, dk = q.shape
    dv = v.shape[2]
    if tuple(v.shape[:2]) != (H, T) or tuple(beta.shape) != (H, T):
        raise ValueError("v must be [H,T,dv] and beta [H,T]")
    cu = [int(x) for x in cu_seqlens]
    N = len(cu) - 1
    cu_arr = (ctypes.c_int * len(cu))(*cu)
    if initial_state is not None:
        _check_cuda("initial_state", initial_state, dev)
        if initial_state.dtype != torch.float32 or tuple(initial_state.shape) != (N, H, dk, dv):
            raise ValueError("initial_state must be float32 [N,H,dk,dv]")
    out = torch.empty((H, T, dv), dtype=q.dtype, device=dev)
    S_T = (torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
           if output_final_state else None)
    lib = load()
    need = lib.dn_chunk_fwd_varlen_workspace_bytes(cu_arr, N, H, dk, dv, chunk_size, dt)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', None or a uint8 CUDA tensor")
        ws = torch.empty(need, dtype=torch.uint8, device=dev) if need else None
    else:
        ws = workspace
        if ws is not None:
            _check_cuda("workspace", ws, dev)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    with torch.cuda.device(dev):
        check(lib.dn_chunk_fwd_varlen_qk(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(),
            initial_state.data_ptr() if initial_state is not None else None, out.data_ptr(),
            S_T.data_ptr() if S_T is not None else None, cu_arr, N, H, T, dk, dv, chunk_size, dt,
            ws.data_ptr() if ws is not None else None, ws_bytes, _stream_handle(dev),
            _norm(scale, qk_l2norm)))
    return out, S_T


def chunk_bwd_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                    g: torch.Tensor, d_o: torch.Tensor, initial_state: torch.Tensor | None = None,
                    d_final_state: torch.Tensor | None = None, chunk_size: int = 64,
                    workspace: torch.Tensor | None = None):
    """Gradients of ``chunk_fwd_gated`` (``dn_chunk_bwd_gated``).

    ``g``: fp32 ``[B, H, T]`` log keep rates.  Returns ``(d_q, d_k, d_v,
    d_beta, d_g, d_initial_state)`` for L = <d_o, o> + <d_final_state,
    final_state>; ``d_g`` fp32 like ``g``.
    """
    return _bwd_decayed(q, k, v, beta, g, d_o, initial_state, d_final_state, chunk_size,
                        workspace, per_channel=False)


def chunk_bwd_kda(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                  g: torch.Tensor, d_o: torch.Tensor, initial_state: torch.Tensor | None = None,
                  d_final_state: torch.Tensor | None = None, chunk_size: int = 64,
                  workspace: torch.Tensor | None = None):
    """Gradients of ``chunk_fwd_kda`` (``dn_chunk_bwd_kda``).

    ``g``: fp32 ``[B, H, T, dk]`` per-key-channel log keep rates.  Returns
    ``(d_q, d_k, d_v, d_beta, d_g, d_initial_state)`` for L = <d_o, o> +
    <d_final_state, final_state>; ``d_g`` fp32 like ``g``.
    """
    return _bwd_decayed(q, k, v, beta, g, d_o, initial_state, d_final_state, chunk_size,
                        workspace, per_channel=True)


def _bwd_decayed(q, k, v, beta, g, d_o, initial_state, d_final_state, chunk_size, workspace,
                 per_channel):
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g), ("d_o", d_o)):
        _check_cuda(name, t, dev)
    dt = _dtype_code(q)
    if not (k.dtype == v.dtype == beta.dtype == d_o.dtype == q.dtype):
        raise TypeError("q, k, v, beta and d_o must share one dtype")
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or d_o.shape != v.shape:
        raise ValueError("q, k must be [B,H,T,dk]; v and d_o [B,H,T,dv]")
    B, H, T, dk = q.shape
    dv = v.shape[3]
    if tuple(v.shape[:3]) != (B, H, T) or tuple(beta.shape) != (B, H, T):
        raise ValueError("v must be [B,H,T,dv] and beta [B,H,T]")
    gshape = (B, H, T, dk) if per_channel else (B, H, T)
    if g.dtype != torch.float32 or tuple(g.shape) != gshape:
        raise ValueError(f"g must be float32 {list(gshape)}")
    for name, t in (("initial_state", initial_state), ("d_final_state", d_final_state)):
        if t is not None:
            _check_cuda(name, t, dev)
            if t.dtype != torch.float32 or tuple(t.shape) != (B, H, dk, dv):
                raise ValueError(f"{name} must be float32 [B,H,dk,dv]")
    lib = load()
    fn, ws_fn = ((lib.dn_chunk_bwd_kda, lib.dn_chunk_bwd_kda_workspace_bytes) if per_channel else
                 (lib.dn_chunk_bwd_gated, lib.dn_chunk_bwd_gated_workspace_bytes))
    need = ws_fn(B, H, T, dk, dv, chunk_size, dt)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace, dev)
    grads = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
             torch.empty_like(beta), torch.empty_like(g),
             torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)]
    with torch.cuda.device(dev):
        check(fn(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(), g.data_ptr(),
            initial_state.data_ptr() if initial_state is not None else None, d_o.data_ptr(),
            d_final_state.data_ptr() if d_final_state is not None else None,
            *(x.data_ptr() for x in grads), B, H, T, dk, dv, chunk_size, dt,
            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _stream_handle(dev)))
    return tuple(grads)


def chunk_bwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                     d_o: torch.Tensor, cu_seqlens, initial_state: torch.Tensor | None = None,
                     d_final_state: torch.Tensor | None = None, chunk_size: int = 64,
                     workspace: torch.Tensor | None = None):
    """Gradients of ``chunk_fwd_varlen`` (``dn_chunk_bwd_varlen``).

    q, k ``[H, T, dk]``, v and d_o ``[H, T, dv]``, beta ``[H, T]`` packed as
    for the forward; ``cu_seqlens`` a host sequence of N + 1 ints; the states
    ``[N, H, dk, dv]`` fp32.  Returns ``(d_q, d_k, d_v, d_beta,
    d_initial_state)`` for L = <d_o, o> + <d_final_state, final_state>.
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("d_o", d_o)):
        _check_cuda(name, t, dev)
    dt = _dtype_code(q)
    if not (k.dtype == v.dtype == beta.dtype == d_o.dtype == q.dtype):
        raise TypeError("q, k, v, beta and d_o must share one dtype")
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or d_o.shape != v.shape:
        raise ValueError("q, k must be [H,T,dk] and v, d_o [H,T,dv]")
    H, T, dk = q.shape
    dv = v.shape[2]
    if tuple(v.shape[:2]) != (H, T) or tuple(beta.shape) != (H, T):
        raise ValueError("v must be [H,T,dv] and beta [H,T]")
    cu = [int(x) for x in cu_seqlens]
    N = len(cu) - 1
    cu_arr = (ctypes.c_int * len(cu))(*cu)
    for name, t in (("initial_state", initial_state), ("d_final_state", d_final_state)):
        if t is not None:
            _check_cuda(name, t, dev)
            if t.dtype != torch.float32 or tuple(t.shape) != (N, H, dk, dv):
                raise ValueError(f"{name} must be float32 [N,H,dk,dv]")
    grads = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
             torch.empty_like(beta),
             torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)]
    lib = load()
    need = lib.dn_chunk_bwd_varlen_workspace_bytes(cu_arr, N, H, dk, dv, chunk_size, dt)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace, dev)
    with torch.cuda.device(dev):
        check(lib.dn_chunk_bwd_varlen(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), beta.data_ptr(),
            initial_state.data_ptr() if initial_state is not None else None, d_o.data_ptr(),
            d_final_state.data_ptr() if d_final_state is not None else None,
            *(g.data_ptr() for g in grads), cu_arr, N, H, T, dk, dv, chunk_size, dt,
            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _stream_handle(dev)))
    return tuple(grads)
