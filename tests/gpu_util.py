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


def run_chunk(inp, algo="auto", want_state=True):
    """Runs the library on ChunkInputs; returns (o, S_T) as fp64 numpy.
    algo "tcgen05-fused" is the tensor-core path without a workspace (one
    fused kernel); "tcgen05" and "auto" get the workspace (two passes)."""
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
