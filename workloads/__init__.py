"""Seeded synthetic inputs for the DeltaNet delta-rule operator.

This module is shared by the tests, the smoke check and the benchmark; it is
the only code both the CUDA path's callers and the oracle's callers use.  It
draws random numbers and shapes them into the operator's inputs (feature map,
L2 normalisation, sigmoid write strength, casts).  It performs none of the
delta-rule arithmetic.

Input recipes (what the layer in front of the operator produces):
  - q, k: L2-normalised per head, optionally after a SiLU feature map, the
    pairing "DeltaNet transformer" (paperlayer.ai/abs/2406.06484v6, section 3)
    describes; normalisation is x * rsqrt(sum x^2 + 1e-6), the form
    "代码实现" (garden.houmin.site/infra/delta-net) prints.
  - beta = sigmoid(N(0,1)), times 2 for the negative-eigenvalue variant the
    DeltaNet layer's ``allow_neg_eigval`` flag selects
    (fla/layers/delta_net.py, class DeltaNet, constructor arguments).
  - v ~ N(0,1); initial state ~ N(0, s0_std^2) in fp32 when asked for.

All sampling is fp32 on the CPU with a ``torch.Generator`` seeded per
workload, in the fixed order q, k, v, beta, S0; normalisation and activation
run in fp32; the result is then cast to the I/O dtype.  The oracle receives
exactly the cast values widened to fp64.
"""
from __future__ import annotations

import dataclasses

import torch

__all__ = [
    "ChunkInputs", "DecodeInputs", "WORKLOADS", "l2norm", "chunk_inputs",
    "recall_inputs", "decode_state", "decode_step_inputs", "workload_inputs",
]


def l2norm(x: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    """x / sqrt(sum(x^2) + eps) over the last axis, in fp32."""
    x = x.float()
    return x * torch.rsqrt((x * x).sum(dim=-1, keepdim=True) + eps)


# The five workloads, by what they are.  Each names its shape, I/O dtype and
# input recipe; "seed" fixes the generator.
WORKLOADS = {
    "tiny_fp32": dict(B=1, H=2, T=256, dk=64, dv=64, C=64, dtype="f32",
                      recipe="plain", s0_std=None, seed=1000),
    "recall_bf16": dict(B=4, H=4, T=1024, dk=64, dv=64, C=64, dtype="bf16",
                        recipe="recall", s0_std=None, seed=1001,
                        n_write=64),
    "layer1p3b_bf16": dict(B=8, H=16, T=2048, dk=128, dv=128, C=64,
                           dtype="bf16", recipe="silu", s0_std=None,
                           seed=1002),
    "long_prefill_bf16": dict(B=1, H=16, T=32768, dk=128, dv=128, C=64,
                              dtype="bf16", recipe="silu", s0_std=0.1,
                              seed=1003),
    "decode_bf16": dict(B=256, H=16, dk=128, dv=128, dtype="bf16",
                        steps=1024, s0_std=0.1, beta_scale=2.0, seed=1004),
}

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


@dataclasses.dataclass
class ChunkInputs:
    """Inputs of one sequence-level call, CPU tensors in the I/O dtype."""
    q: torch.Tensor          # [B, H, T, dk]
    k: torch.Tensor          # [B, H, T, dk]
    v: torch.Tensor          # [B, H, T, dv]
    beta: torch.Tensor       # [B, H, T]
    S0: torch.Tensor | None  # [B, H, dk, dv] fp32, or None for zeros

    @property
    def shape(self):
        B, H, T, dk = self.q.shape
        return B, H, T, dk, self.v.shape[3]


@dataclasses.dataclass
class DecodeInputs:
    """Inputs of one decoding step, CPU tensors in the I/O dtype."""
    q: torch.Tensor     # [B, H, dk]
    k: torch.Tensor     # [B, H, dk]
    v: torch.Tensor     # [B, H, dv]
    beta: torch.Tensor  # [B, H]


def chunk_inputs(B: int, H: int, T: int, dk: int, dv: int, *, dtype="bf16",
                 seed: int = 0, feature_map: str = "none",
                 beta_scale: float = 1.0, s0_std: float | None = None,
                 normalize: bool = True) -> ChunkInputs:
    """Random sequence inputs.

    feature_map: "none" (q, k = l2norm(N(0,1))) or "silu"
    (q, k = l2norm(silu(N(0,1)))).  beta = beta_scale * sigmoid(N(0,1)).
    normalize=False leaves q and k as drawn (N(0,1), or silu of it), for
    calls that normalise them in the library.
    """
    g = torch.Generator().manual_seed(int(seed))
    q = torch.randn(B, H, T, dk, generator=g)
    k = torch.randn(B, H, T, dk, generator=g)
    v = torch.randn(B, H, T, dv, generator=g)
    b = torch.randn(B, H, T, generator=g)
    S0 = None
    if s0_std is not None:
        S0 = torch.randn(B, H, dk, dv, generator=g) * float(s0_std)
    if feature_map == "silu":
        q, k = torch.nn.functional.silu(q), torch.nn.functional.silu(k)
    elif feature_map != "none":
        raise ValueError(f"unknown feature map {feature_map!r}")
    if normalize:
        q, k = l2norm(q), l2norm(k)
    beta = torch.sigmoid(b) * float(beta_scale)
    dt = torch_dtype(dtype)
    return ChunkInputs(q.to(dt).contiguous(), k.to(dt).contiguous(),
                       v.to(dt).contiguous(), beta.to(dt).contiguous(),
                       None if S0 is None else S0.float().contiguous())


def _orthogonal(n: int, g: torch.Generator) -> torch.Tensor:
    """Haar-random n x n orthogonal matrix: QR of N(0,1), signs fixed."""
    a = torch.randn(n, n, generator=g, dtype=torch.float64)
    qm, r = torch.linalg.qr(a)
    return qm * torch.sign(torch.diagonal(r)).unsqueeze(0)


def recall_inputs(B: int, H: int, T: int, d: int, *, n_write: int | None = None,
                  dtype="bf16", seed: int = 0):
    """Associative-recall inputs with a closed-form answer.

    For each (b, h): the first ``n_write`` (= d) tokens write the rows of a
    seeded random orthogonal d x d matrix as keys, with beta = 1 and
    v ~ N(0,1), q = k.  Every later token re-queries one of those keys
    (index drawn uniformly) with q = k and beta = 0, v ~ N(0,1) (ignored).

    Returns (ChunkInputs, expected_o) where expected_o [B, H, T, d] fp64 is
    the stored value of the key each token reads; for exactly orthonormal
    keys the recurrence returns it exactly.
    """
    n_write = d if n_write is None else int(n_write)
    if n_write > d or n_write > T:
        raise ValueError("n_write must be <= d and <= T")
    g = torch.Generator().manual_seed(int(seed))
    dt = torch_dtype(dtype)
    k = torch.empty(B, H, T, d, dtype=torch.float64)
    beta = torch.empty(B, H, T, dtype=torch.float64)
    v = torch.randn(B, H, T, d, generator=g, dtype=torch.float64)
    idx = torch.empty(B, H, T, dtype=torch.long)
    for b in range(B):
        for h in range(H):
            basis = _orthogonal(d, g)
            which = torch.randint(0, n_write, (T - n_write,), generator=g)
            order = torch.cat([torch.arange(n_write), which])
            k[b, h] = basis[order]
            idx[b, h] = order
            beta[b, h, :n_write] = 1.0
            beta[b, h, n_write:] = 0.0
    kc, vc, bc = k.to(dt), v.to(dt), beta.to(dt)
    stored = torch.gather(vc.double(), 2,
                          idx.unsqueeze(-1).expand(B, H, T, d))
    inp = ChunkInputs(kc.contiguous(), kc.clone().contiguous(),
                      vc.contiguous(), bc.contiguous(), None)
    return inp, stored.numpy()


def decode_state(B: int, H: int, dk: int, dv: int, *, std: float = 0.1,
                 seed: int = 0) -> torch.Tensor:
    """fp32 state [B, H, dk, dv] ~ N(0, std^2)."""
    g = torch.Generator().manual_seed(int(seed))
    return (torch.randn(B, H, dk, dv, generator=g) * float(std)).contiguous()


def decode_step_inputs(B: int, H: int, dk: int, dv: int, *, step: int,
                       dtype="bf16", seed: int = 0,
                       beta_scale: float = 2.0, normalize: bool = True) -> DecodeInputs:
    """Inputs of decoding step ``step``: q, k = l2norm(N(0,1)), v ~ N(0,1),
    beta = beta_scale * sigmoid(N(0,1)); seeded by (seed, step).
    normalize=False leaves q and k as drawn."""
    g = torch.Generator().manual_seed(int(seed) * 100003 + 7919 * int(step) + 1)
    q = torch.randn(B, H, dk, generator=g)
    k = torch.randn(B, H, dk, generator=g)
    if normalize:
        q, k = l2norm(q), l2norm(k)
    v = torch.randn(B, H, dv, generator=g)
    beta = torch.sigmoid(torch.randn(B, H, generator=g)) * float(beta_scale)
    dt = torch_dtype(dtype)
    return DecodeInputs(q.to(dt).contiguous(), k.to(dt).contiguous(),
                        v.to(dt).contiguous(), beta.to(dt).contiguous())


def workload_inputs(name: str, **overrides):
    """Inputs of a named sequence workload (not the decode one).

    Keyword overrides replace shape entries (B, H, T) to draw a smaller case
    with the same recipe; normalize=False leaves q and k unnormalised.  Returns ChunkInputs, or (ChunkInputs, expected_o)
    for the recall workload.
    """
    w = dict(WORKLOADS[name])
    w.update(overrides)
    if w["recipe"] == "recall":
        return recall_inputs(w["B"], w["H"], w["T"], w["dk"],
                             n_write=w.get("n_write"), dtype=w["dtype"],
                             seed=w["seed"])
    return chunk_inputs(w["B"], w["H"], w["T"], w["dk"], w["dv"],
                        dtype=w["dtype"], seed=w["seed"],
                        feature_map="silu" if w["recipe"] == "silu" else "none",
                        s0_std=w["s0_std"], normalize=w.get("normalize", True))


def decode_inputs_on_device(B: int, H: int, dk: int, dv: int, steps: int, *,
                            dtype="bf16", seed: int = 0, beta_scale: float = 2.0,
                            device="cuda", block: int = 64):
    """All ``steps`` decoding steps' inputs drawn on the device (for timing
    runs, where CPU generation of gigabytes would dominate): same recipe as
    ``decode_step_inputs``, drawn from a seeded device generator ``block``
    steps at a time.  Returns q, k ``[steps, B, H, dk]``, v
    ``[steps, B, H, dv]``, beta ``[steps, B, H]`` in the I/O dtype."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    dt = torch_dtype(dtype)
    q = torch.empty(steps, B, H, dk, dtype=dt, device=device)
    k = torch.empty_like(q)
    v = torch.empty(steps, B, H, dv, dtype=dt, device=device)
    beta = torch.empty(steps, B, H, dtype=dt, device=device)
    for s0 in range(0, steps, block):
        n = min(block, steps - s0)
        sl = slice(s0, s0 + n)
        q[sl] = l2norm(torch.randn(n, B, H, dk, generator=g, device=device)).to(dt)
        k[sl] = l2norm(torch.randn(n, B, H, dk, generator=g, device=device)).to(dt)
        v[sl] = torch.randn(n, B, H, dv, generator=g, device=device).to(dt)
        beta[sl] = (torch.sigmoid(torch.randn(n, B, H, generator=g, device=device))
                    * float(beta_scale)).to(dt)
    return q, k, v, beta


def grad_inputs(B: int, H: int, T: int, dv: int, dk: int | None = None, *, dtype="bf16",
                seed: int = 0, ds_std: float | None = 0.1):
    """Upstream gradients for a backward pass: d_o ``[B, H, T, dv]`` ~ N(0, 1)
    in the I/O dtype, and d_S_T ``[B, H, dk, dv]`` ~ N(0, ds_std^2) fp32 (None
    when ds_std is None).  Seeded by (seed, "grad")."""
    g = torch.Generator().manual_seed(int(seed) * 7907 + 104729)
    d_o = torch.randn(B, H, T, dv, generator=g).to(torch_dtype(dtype)).contiguous()
    d_S = None
    if ds_std is not None:
        d_S = (torch.randn(B, H, dk if dk is not None else dv, dv, generator=g)
               * float(ds_std)).float().contiguous()
    return d_o, d_S


def gate_inputs(B: int, H: int, T: int | None = None, *, seed: int = 0, lo: float = 0.9,
                hi: float = 1.0, channels: int | None = None) -> torch.Tensor:
    """Log keep rates g = log(alpha), alpha ~ U(lo, hi) fp32, [B, H, T] (or
    [B, H] when T is None), with a trailing [channels] axis for per-channel
    rates; seeded by (seed, "gate")."""
    gen = torch.Generator().manual_seed(int(seed) * 6151 + 3571)
    shape = (B, H) if T is None else (B, H, T)
    if channels is not None:
        shape = shape + (channels,)
    alpha = lo + (hi - lo) * torch.rand(shape, generator=gen)
    return torch.log(alpha).float().contiguous()


def varlen_lengths(n: int, total: int, *, seed: int = 0) -> list[int]:
    """n sequence lengths summing to ``total``: seeded U(0, 1) weights, scaled
    and rounded (the remainder goes to the last sequence)."""
    gen = torch.Generator().manual_seed(int(seed) * 4409 + 2281)
    w = torch.rand(n, generator=gen) + 0.05
    lens = [int(x) for x in (w / w.sum() * total).floor().tolist()]
    lens[-1] += total - sum(lens)
    return lens
