"""Gated DeltaNet on the GPU (chunkwise forward and decoding step) against
the fp64 gated oracle, through the C ABI.  Bars as for the plain forms:
relative L2 <= 1e-4 (fp32 I/O) and <= 1e-2 (bf16 I/O) on o and the state.
The chunkwise form has two kernels: the fp32 CUDA-core one (workspace=None,
every shape) and the two-pass tcgen05 one (a workspace, dk = dv = 128 bf16).
"""
import functools
import numpy as np
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import oracle
import workloads
from tests.conftest import rel_l2
from tests.gpu_util import TOL, check_every_head, dev, sample_heads, take_heads

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def no_device_error():
    lib = dn.load()
    assert lib.dn_device_error() == 0
    yield
    assert lib.dn_device_error() == 0


def _check(o, S, o_ref, S_ref, dtype, what):
    eo, eS = rel_l2(o, o_ref), rel_l2(S, S_ref)
    assert eo <= TOL[dtype], f"{what} o rel L2 {eo:.3e}"
    assert eS <= TOL[dtype], f"{what} S_T rel L2 {eS:.3e}"


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gated_chunk_ragged(dk, dv, dtype):
    B, H, T = 2, 2, 200
    inp = workloads.chunk_inputs(B, H, T, dk, dv, dtype=dtype, seed=dk + 3 * dv,
                                 feature_map="silu", s0_std=0.1)
    g = workloads.gate_inputs(B, H, T, seed=dk + dv)
    o, S = dn.chunk_fwd_gated(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g),
                              initial_state=dev(inp.S0), workspace=None)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_gated(inp.q, inp.k, inp.v, inp.beta, g, inp.S0)
    _check(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
           workloads.torch_dtype(dtype), f"{dtype} {dk}x{dv}")


def test_gated_zero_decay_matches_the_plain_kernel_exactly():
    """g = 0 runs the CUDA-core kernel with every decay factor exactly 1."""
    inp = workloads.chunk_inputs(1, 2, 130, 64, 64, dtype="f32", seed=2, s0_std=0.1)
    q, k, v, b, S0 = (dev(x) for x in (inp.q, inp.k, inp.v, inp.beta, inp.S0))
    o1, S1 = dn.chunk_fwd(q, k, v, b, initial_state=S0, algo="simt")
    o2, S2 = dn.chunk_fwd_gated(q, k, v, b, torch.zeros(1, 2, 130, device="cuda"),
                                initial_state=S0)
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


def test_gated_strong_decay_and_edge_lengths():
    for T in (1, 64, 65):
        inp = workloads.chunk_inputs(1, 3, T, 128, 128, dtype="f32", seed=T, s0_std=0.5)
        g = workloads.gate_inputs(1, 3, T, seed=T, lo=0.05, hi=0.5)  # alpha far below 1
        o, S = dn.chunk_fwd_gated(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g),
                                  initial_state=dev(inp.S0))
        torch.cuda.synchronize()
        o_ref, S_ref = oracle.forward_gated(inp.q, inp.k, inp.v, inp.beta, g, inp.S0)
        _check(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
               torch.float32, f"T={T}")


def _tc_workspace(B, H, T):
    n = dn.load().dn_chunk_fwd_gated_workspace_bytes(B, H, T, 128, 128, 64, 1)
    assert n == B * H * ((T + 63) // 64) * 33792
    return torch.empty(n, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 1000])
@pytest.mark.parametrize("lo,hi", [(0.9, 1.0), (0.3, 1.0), (0.05, 0.3)],
                         ids=["mild", "strong", "extreme"])
def test_gated_tc_chunk_ragged(T, lo, hi):
    """The tcgen05 form over ragged lengths (one partial chunk to 16
    chunks), with an initial state, and three decay regimes: mild, strong
    (alpha down to 0.3) and extreme (alpha in (0.05, 0.3): a full chunk
    decays by more than exp(-80), so its ratios take one exponential per
    entry; a ragged tail chunk stays on the product form)."""
    B, H = 2, 3
    inp = workloads.chunk_inputs(B, H, T, 128, 128, dtype="bf16", seed=T + 7,
                                 feature_map="silu", s0_std=0.5)
    g = workloads.gate_inputs(B, H, T, seed=T, lo=lo, hi=hi)
    o, S = dn.chunk_fwd_gated(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g),
                              initial_state=dev(inp.S0), workspace=_tc_workspace(B, H, T))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_gated(inp.q, inp.k, inp.v, inp.beta, g, inp.S0)
    _check(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
           torch.bfloat16, f"tcgen05 T={T} alpha in ({lo}, {hi})")


def test_gated_tc_zero_decay_matches_the_plain_tc_kernel():
    """g = 0: every decay factor of the gated tcgen05 form is exactly 1, so it
    computes what the plain two-pass kernel computes."""
    B, H, T = 2, 4, 333
    inp = workloads.chunk_inputs(B, H, T, 128, 128, dtype="bf16", seed=12, s0_std=0.1)
    q, k, v, b, S0 = (dev(x) for x in (inp.q, inp.k, inp.v, inp.beta, inp.S0))
    o1, S1 = dn.chunk_fwd(q, k, v, b, initial_state=S0, algo="tcgen05")
    o2, S2 = dn.chunk_fwd_gated(q, k, v, b, torch.zeros(B, H, T, device="cuda"),
                                initial_state=S0, workspace=_tc_workspace(B, H, T))
    torch.cuda.synchronize()
    assert rel_l2(o2.double().cpu().numpy(), o1.double().cpu().numpy()) <= 1e-6
    assert rel_l2(S2.double().cpu().numpy(), S1.double().cpu().numpy()) <= 1e-6


def test_gated_tc_matches_the_cuda_core_kernel():
    """Both kernels of the gated form on one bf16 problem agree to the bf16 bar."""
    B, H, T = 2, 4, 777
    inp = workloads.chunk_inputs(B, H, T, 128, 128, dtype="bf16", seed=21, s0_std=0.2)
    g = workloads.gate_inputs(B, H, T, seed=21, lo=0.7)
    args = [dev(x) for x in (inp.q, inp.k, inp.v, inp.beta, g)]
    o1, S1 = dn.chunk_fwd_gated(*args, initial_state=dev(inp.S0), workspace=None)
    o2, S2 = dn.chunk_fwd_gated(*args, initial_state=dev(inp.S0), workspace="auto")
    torch.cuda.synchronize()
    _check(o2.double().cpu().numpy(), S2.double().cpu().numpy(), o1.double().cpu().numpy(),
           S1.double().cpu().numpy(), torch.bfloat16, "tcgen05 vs CUDA cores")


def test_gated_tc_workspace_too_small_is_rejected():
    B, H, T = 1, 2, 100
    inp = workloads.chunk_inputs(B, H, T, 128, 128, dtype="bf16", seed=1)
    g = workloads.gate_inputs(B, H, T, seed=1)
    ws = _tc_workspace(B, H, T)[:-16]
    with pytest.raises(RuntimeError, match="workspace"):
        dn.chunk_fwd_gated(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g),
                           workspace=ws)


@functools.lru_cache(maxsize=1)
def _oracle_gated_1p3b():
    """The gated oracle on the whole 1.3B-layer workload, once per session."""
    inp = workloads.workload_inputs("layer1p3b_bf16")
    B, H, T, d = inp.q.shape
    g = workloads.gate_inputs(B, H, T, seed=7)
    return inp, g, oracle.forward_gated(inp.q, inp.k, inp.v, inp.beta, g)


@pytest.mark.parametrize("workspace", ["auto", None], ids=["tcgen05", "cuda-cores"])
def test_gated_layer_1p3b_every_head(workspace):
    """The 1.3B-layer shape with keep rates in (0.9, 1): every head and every
    64-token chunk against the gated oracle."""
    inp, g, (o_ref, S_ref) = _oracle_gated_1p3b()
    o, S = dn.chunk_fwd_gated(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g),
                              workspace=workspace)
    torch.cuda.synchronize()
    check_every_head(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
                     TOL[torch.bfloat16], "gated 1.3B")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gated_decode_steps(dtype):
    B, H, d, steps, seed = 4, 4, 128, 24, 11
    S0 = workloads.decode_state(B, H, d, d, std=0.1, seed=seed)
    S = dev(S0)
    rec = {n: [] for n in ("q", "k", "v", "beta", "g", "o")}
    for step in range(steps):
        x = workloads.decode_step_inputs(B, H, d, d, step=step, dtype=dtype, seed=seed)
        g = workloads.gate_inputs(B, H, seed=seed * 100 + step, lo=0.8)
        o = dn.recurrent_step_gated(dev(x.q), dev(x.k), dev(x.v), dev(x.beta), dev(g), S)
        for n in ("q", "k", "v", "beta"):
            rec[n].append(getattr(x, n))
        rec["g"].append(g)
        rec["o"].append(o.cpu())
    torch.cuda.synchronize()
    st = {n: torch.stack(v_, dim=2) for n, v_ in rec.items()}  # [B, H, steps, ...]
    o_ref, S_ref = oracle.forward_gated(st["q"], st["k"], st["v"], st["beta"], st["g"], S0)
    _check(st["o"].double().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
           workloads.torch_dtype(dtype), f"decode {dtype}")


def test_gated_decode_zero_decay_matches_the_plain_step_exactly():
    B, H, d = 8, 2, 128
    S0 = dev(workloads.decode_state(B, H, d, d, std=0.1, seed=3))
    x = workloads.decode_step_inputs(B, H, d, d, step=0, dtype="bf16", seed=3)
    S1, S2 = S0.clone(), S0.clone()
    o1 = dn.recurrent_step(dev(x.q), dev(x.k), dev(x.v), dev(x.beta), S1)
    o2 = dn.recurrent_step_gated(dev(x.q), dev(x.k), dev(x.v), dev(x.beta),
                                 torch.zeros(B, H, device="cuda"), S2)
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


@pytest.mark.parametrize("form", ["gated", "kda"])
def test_zero_length_sequence_passes_the_state_through(form):
    """T = 0: no token, so S_T is S0 (or zeros without S0), and o is empty."""
    B, H, d = 2, 3, 128
    z = torch.zeros(B, H, 0, d, dtype=torch.bfloat16, device="cuda")
    beta = torch.zeros(B, H, 0, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((B, H, 0, d) if form == "kda" else (B, H, 0), device="cuda")
    S0 = workloads.decode_state(B, H, d, d, std=0.1, seed=3).cuda()
    fwd = dn.chunk_fwd_kda if form == "kda" else dn.chunk_fwd_gated
    o, S = fwd(z, z, z, beta, g, initial_state=S0)
    o0, S_zero = fwd(z, z, z, beta, g)
    torch.cuda.synchronize()
    assert o.shape == (B, H, 0, d) and torch.equal(S, S0)
    assert torch.count_nonzero(S_zero) == 0


@pytest.mark.parametrize("form", ["gated", "kda"])
def test_decode_at_the_bench_shape_sampled_heads(form):
    """B256 H16 d128 bf16 (the decode workload's shape and the bench's launch
    configuration), eight chained steps with one keep rate per head (gated)
    or per key channel (KDA); 12 heads replayed by the oracle."""
    w = workloads.WORKLOADS["decode_bf16"]
    B, H, d, seed = w["B"], w["H"], w["dk"], w["seed"]
    steps = 8
    bi, hi = sample_heads(B, H, 12, seed=13)
    S0 = workloads.decode_state(B, H, d, d, std=w["s0_std"], seed=seed)
    S = dev(S0)
    g = workloads.gate_inputs(B, H, seed=seed, channels=d if form == "kda" else None)
    step = dn.recurrent_step_kda if form == "kda" else dn.recurrent_step_gated
    rec = {n: [] for n in ("q", "k", "v", "beta", "o")}
    for t in range(steps):
        x = workloads.decode_step_inputs(B, H, d, d, step=t, dtype="bf16", seed=seed,
                                         beta_scale=w["beta_scale"])
        o = step(dev(x.q), dev(x.k), dev(x.v), dev(x.beta), dev(g), S)
        for n in ("q", "k", "v", "beta"):
            rec[n].append(take_heads(getattr(x, n), bi, hi))
        rec["o"].append(take_heads(o.cpu(), bi, hi))
    torch.cuda.synchronize()
    st = {n: torch.stack(v_, dim=2) for n, v_ in rec.items()}  # [1, n, steps, ...]
    g_s = take_heads(g, bi, hi)
    g_seq = (g_s[:, :, None, :] if form == "kda" else g_s[:, :, None]).expand(
        *st["beta"].shape, *([d] if form == "kda" else [])).contiguous()
    f = oracle.forward_kda if form == "kda" else oracle.forward_gated
    o_ref, S_ref = f(st["q"], st["k"], st["v"], st["beta"], g_seq, take_heads(S0, bi, hi))
    _check(st["o"].double().numpy(), take_heads(S.cpu(), bi, hi).double().numpy(), o_ref, S_ref,
           torch.bfloat16, f"{form} decode, bench shape")
