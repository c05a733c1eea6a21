"""Kimi Delta Attention on the GPU (chunkwise forward and decoding step)
against the fp64 KDA oracle, through the C ABI.  Bars: relative L2 <= 1e-4
(fp32 I/O) and <= 1e-2 (bf16 I/O) on o and the state.
"""
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import oracle
import workloads
from tests.conftest import rel_l2
from tests.gpu_util import TOL, check_every_head, dev

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
def test_kda_chunk_ragged(dk, dv, dtype):
    B, H, T = 2, 2, 200
    inp = workloads.chunk_inputs(B, H, T, dk, dv, dtype=dtype, seed=dk + 5 * dv,
                                 feature_map="silu", s0_std=0.1)
    g = workloads.gate_inputs(B, H, T, seed=dk * dv, channels=dk)
    o, S = dn.chunk_fwd_kda(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g),
                            initial_state=dev(inp.S0))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_kda(inp.q, inp.k, inp.v, inp.beta, g, inp.S0)
    _check(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
           workloads.torch_dtype(dtype), f"{dtype} {dk}x{dv}")


def test_kda_equal_channels_match_the_gated_kernel():
    B, H, T, d = 1, 2, 150, 64
    inp = workloads.chunk_inputs(B, H, T, d, d, dtype="f32", seed=4, s0_std=0.1)
    g = workloads.gate_inputs(B, H, T, seed=4)
    args = [dev(x) for x in (inp.q, inp.k, inp.v, inp.beta)]
    o1, S1 = dn.chunk_fwd_gated(*args, dev(g), initial_state=dev(inp.S0))
    o2, S2 = dn.chunk_fwd_kda(*args, dev(g)[..., None].expand(B, H, T, d).contiguous(),
                              initial_state=dev(inp.S0))
    assert rel_l2(o2.double().cpu().numpy(), o1.double().cpu().numpy()) <= 1e-5
    assert rel_l2(S2.double().cpu().numpy(), S1.double().cpu().numpy()) <= 1e-5


def test_kda_strong_decay_and_edge_lengths():
    for T in (1, 64, 65):
        inp = workloads.chunk_inputs(1, 2, T, 128, 128, dtype="f32", seed=T + 1, s0_std=0.5)
        g = workloads.gate_inputs(1, 2, T, seed=T, lo=0.05, hi=0.6, channels=128)
        o, S = dn.chunk_fwd_kda(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g),
                                initial_state=dev(inp.S0))
        torch.cuda.synchronize()
        o_ref, S_ref = oracle.forward_kda(inp.q, inp.k, inp.v, inp.beta, g, inp.S0)
        _check(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
               torch.float32, f"T={T}")


def test_kda_layer_1p3b_every_head():
    """The 1.3B-layer shape with per-channel keep rates in (0.9, 1): every head
    and every 64-token chunk against the KDA oracle."""
    inp = workloads.workload_inputs("layer1p3b_bf16")
    B, H, T, d = inp.q.shape
    g = workloads.gate_inputs(B, H, T, seed=9, channels=d)
    o, S = dn.chunk_fwd_kda(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_kda(inp.q, inp.k, inp.v, inp.beta, g)
    check_every_head(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
                     TOL[torch.bfloat16], "KDA 1.3B")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_kda_decode_steps(dtype):
    B, H, d, steps, seed = 4, 4, 128, 24, 13
    S0 = workloads.decode_state(B, H, d, d, std=0.1, seed=seed)
    S = dev(S0)
    rec = {n: [] for n in ("q", "k", "v", "beta", "g", "o")}
    for step in range(steps):
        x = workloads.decode_step_inputs(B, H, d, d, step=step, dtype=dtype, seed=seed)
        g = workloads.gate_inputs(B, H, seed=seed * 100 + step, lo=0.7, channels=d)
        o = dn.recurrent_step_kda(dev(x.q), dev(x.k), dev(x.v), dev(x.beta), dev(g), S)
        for n in ("q", "k", "v", "beta"):
            rec[n].append(getattr(x, n))
        rec["g"].append(g)
        rec["o"].append(o.cpu())
    torch.cuda.synchronize()
    st = {n: torch.stack(v_, dim=2) for n, v_ in rec.items()}
    o_ref, S_ref = oracle.forward_kda(st["q"], st["k"], st["v"], st["beta"], st["g"], S0)
    _check(st["o"].double().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
           workloads.torch_dtype(dtype), f"decode {dtype}")


def test_steps_reject_mismatched_inputs_before_any_launch():
    """The decayed steps check dtypes and shapes in the binding: a bf16 beta
    with fp32 q, or a beta of the wrong shape, would otherwise have the kernel
    read past the buffer it was given."""
    B, H, d = 2, 3, 64
    q = torch.zeros(B, H, d, device="cuda")
    S = torch.zeros(B, H, d, d, device="cuda")
    g = torch.zeros(B, H, d, device="cuda")
    with pytest.raises(TypeError, match="one dtype"):
        dn.recurrent_step_kda(q, q, q, torch.zeros(B, H, device="cuda",
                                                   dtype=torch.bfloat16), g, S)
    with pytest.raises(ValueError, match="beta"):
        dn.recurrent_step_kda(q, q, q, torch.zeros(B, device="cuda"), g, S)
    with pytest.raises(ValueError, match="beta"):
        dn.recurrent_step_gated(q, q, q, torch.zeros(B, H, 1, device="cuda"),
                                torch.zeros(B, H, device="cuda"), S)
    with pytest.raises(ValueError, match="out"):
        dn.recurrent_step_gated(q, q, q, torch.zeros(B, H, device="cuda"),
                                torch.zeros(B, H, device="cuda"), S,
                                out=torch.zeros(B, H, d + 1, device="cuda"))
    with pytest.raises(ValueError, match="final_state"):
        dn.chunk_fwd_kda(q[:, :, None], q[:, :, None], q[:, :, None],
                         torch.zeros(B, H, 1, device="cuda"), g[:, :, None],
                         final_state=torch.zeros(B, H, d, device="cuda"))


def _kda_tc_workspace(B, H, T):
    n = dn.load().dn_chunk_fwd_kda_workspace_bytes(B, H, T, 128, 128, 64, 1)
    assert n > 0
    return torch.empty(n, dtype=torch.uint8, device="cuda")


REGIMES = {"mild": (0.9, 1.0), "strong": (0.3, 1.0), "extreme": (0.05, 0.3)}


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 1000])
@pytest.mark.parametrize("regime", list(REGIMES))
def test_kda_tc_chunk_ragged(T, regime):
    """The tensor-core form (bf16, dk = dv = 128) over ragged lengths, with an
    initial state, in three decay regimes: mild and strong keep every chunk
    within the separable range (one tensor-core product forms A and P);
    extreme (per-token keep rates 0.05-0.3) takes whole chunks past exp(-80)
    on every channel, so their tiles come from the exact CUDA-core path."""
    B, H = 2, 3
    lo, hi = REGIMES[regime]
    inp = workloads.chunk_inputs(B, H, T, 128, 128, dtype="bf16", seed=T + 11,
                                 feature_map="silu", s0_std=0.5)
    g = workloads.gate_inputs(B, H, T, seed=T + 3, lo=lo, hi=hi, channels=128)
    o, S = dn.chunk_fwd_kda(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g),
                            initial_state=dev(inp.S0), workspace=_kda_tc_workspace(B, H, T))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_kda(inp.q, inp.k, inp.v, inp.beta, g, inp.S0)
    check_every_head(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
                     TOL[torch.bfloat16], f"KDA tcgen05 {regime} T{T}")


def test_kda_tc_mixed_channels_take_the_exact_path():
    """Half the key channels decay hard (keep 0.05-0.3) and half barely (0.95-1):
    every full chunk leaves the separable range on some channel, and the
    exact tiles must agree with the oracle with the slow channels intact."""
    B, H, T = 1, 4, 300
    inp = workloads.chunk_inputs(B, H, T, 128, 128, dtype="bf16", seed=71,
                                 feature_map="silu", s0_std=0.3)
    g_hard = workloads.gate_inputs(B, H, T, seed=72, lo=0.05, hi=0.3, channels=128)
    g_soft = workloads.gate_inputs(B, H, T, seed=73, lo=0.95, hi=1.0, channels=128)
    g = torch.where(torch.arange(128) % 2 == 0, g_hard, g_soft).contiguous()
    o, S = dn.chunk_fwd_kda(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g),
                            initial_state=dev(inp.S0))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_kda(inp.q, inp.k, inp.v, inp.beta, g, inp.S0)
    check_every_head(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
                     TOL[torch.bfloat16], "KDA tcgen05 mixed channels")


def test_kda_tc_agrees_with_the_cuda_core_kernel():
    B, H, T = 2, 2, 700
    inp = workloads.chunk_inputs(B, H, T, 128, 128, dtype="bf16", seed=74,
                                 feature_map="silu", s0_std=0.2)
    g = workloads.gate_inputs(B, H, T, seed=75, lo=0.8, channels=128)
    args = [dev(x) for x in (inp.q, inp.k, inp.v, inp.beta, g)]
    o1, S1 = dn.chunk_fwd_kda(*args, initial_state=dev(inp.S0), workspace="auto")
    o2, S2 = dn.chunk_fwd_kda(*args, initial_state=dev(inp.S0), workspace=None)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_kda(inp.q, inp.k, inp.v, inp.beta, g, inp.S0)
    for o, S, what in ((o1, S1, "tcgen05"), (o2, S2, "cuda cores")):
        check_every_head(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
                         TOL[torch.bfloat16], what)
    assert rel_l2(o1.double().cpu().numpy(), o2.double().cpu().numpy()) <= TOL[torch.bfloat16]


def test_kda_tc_workspace_too_small_is_rejected():
    B, H, T = 1, 2, 100
    inp = workloads.chunk_inputs(B, H, T, 128, 128, dtype="bf16", seed=1)
    g = workloads.gate_inputs(B, H, T, seed=1, channels=128)
    ws = _kda_tc_workspace(B, H, T)[:-16]
    with pytest.raises(RuntimeError, match="workspace"):
        dn.chunk_fwd_kda(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g), workspace=ws)
