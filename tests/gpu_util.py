"""Helpers for the GPU parity tests (imported only by tests marked gpu)."""
from __future__ import annotations

import numpy as np
import torch

import delta_rule_recurrent_gb300 as dn

# Relative L2 bounds: fp32 I/O with fp32 arithmetic, and bf16 I/O with fp32
# accumulation.
TOL = {torch.float32: 1e-4, torch.bfloat16: 1e-2}


def dev(t):
    return None if t is None else t.to("cuda:0", non_blocking=False).contiguous()


def run_chunk(inp, algo="auto", want_state=True, segments=0):
    """Runs the library on ChunkInputs; returns (o, S_T) as fp64 numpy.
    algo "tcgen05-fused" is the tensor-core path without a workspace (one
    fused kernel); "tcgen05" and "auto" get the workspace (two passes);
    "split" is dn_chunk_fwd_split with `segments` runs per sequence."""
    if algo == "split":
        o, S = dn.chunk_fwd_split(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta),
                                  initial_state=dev(inp.S0), output_final_state=want_state,
                                  segments=segments)
        torch.cuda.synchronize()
        return o.double().cpu().numpy(), (S.double().cpu().numpy() if S is not None else None)
    ws = "auto"
    if algo.endswith("-fused"):
        algo, ws = algo[: -len("-fused")], None
    o, S = dn.chunk_fwd(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta),
                        initial_state=dev(inp.S0), output_final_state=want_state, algo=algo,
                        workspace=ws)
    torch.cuda.synchronize()
    o = o.double().cpu().numpy()
    return o, (S.double().cpu().numpy() if S is not None else None)


def sample_heads(B, H, n, seed):
    """n distinct (b, h) pairs, always including the first and the last."""
    r = np.random.default_rng(seed)
    flat = r.choice(B * H, size=min(n, B * H), replace=False)
    flat = np.unique(np.concatenate([flat[: max(0, n - 2)], [0, B * H - 1]]))
    return flat // H, flat % H


def take_heads(x, bi, hi):
    """x[b, h, ...] for the sampled pairs, as a [1, n, ...] array."""
    if x is None:
        return None
    return x[torch.as_tensor(bi), torch.as_tensor(hi)].unsqueeze(0)


def per_head_rel_l2(x, ref):
    """Relative L2 error of every (batch, head) slice of [B, H, ...] arrays."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    B, H = ref.shape[:2]
    num = np.linalg.norm((x - ref).reshape(B, H, -1), axis=2)
    den = np.linalg.norm(ref.reshape(B, H, -1), axis=2)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), num)


def per_chunk_rel_l2(o, o_ref, C=64):
    """Relative L2 error of every (batch, head, C-token chunk) of [B, H, T, d]
    outputs; the last chunk may be short."""
    o = np.asarray(o, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    B, H, T, d = o_ref.shape
    n = (T + C - 1) // C
    pad = n * C - T
    diff = np.pad(o - o_ref, ((0, 0), (0, 0), (0, pad), (0, 0))).reshape(B, H, n, C * d)
    ref = np.pad(o_ref, ((0, 0), (0, 0), (0, pad), (0, 0))).reshape(B, H, n, C * d)
    num, den = np.linalg.norm(diff, axis=3), np.linalg.norm(ref, axis=3)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), num)


def check_every_head(o, S, o_ref, S_ref, tol, what=""):
    """The parity bar on every (batch, head) separately, for o and the final
    state, and on every 64-token chunk of o: one wrong head, or one wrong
    chunk inside a head, fails even when the whole-tensor error would hide
    it.  Returns the worst errors seen."""
    eo = per_head_rel_l2(o, o_ref)
    ec = per_chunk_rel_l2(o, o_ref)
    worst = {"o_head": float(eo.max()), "o_chunk": float(ec.max())}
    bo = np.unravel_index(int(np.argmax(eo)), eo.shape)
    assert eo.max() <= tol, f"{what} o rel L2 {eo.max():.3e} at (b, h) = {bo}"
    bc = np.unravel_index(int(np.argmax(ec)), ec.shape)
    assert ec.max() <= tol, f"{what} o rel L2 {ec.max():.3e} at (b, h, chunk) = {bc}"
    if S is not None or S_ref is not None:
        eS = per_head_rel_l2(S, S_ref)
        worst["S_head"] = float(eS.max())
        bS = np.unravel_index(int(np.argmax(eS)), eS.shape)
        assert eS.max() <= tol, f"{what} S_T rel L2 {eS.max():.3e} at (b, h) = {bS}"
    return worst
