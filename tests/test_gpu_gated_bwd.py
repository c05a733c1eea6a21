"""Gated DeltaNet backward (dn_chunk_bwd_gated) on the GPU against the fp64
oracle's gated gradient (``oracle.backward_gated``, pinned in
``tests/pins_gated_bwd.py``).

Bars on each of d_q, d_k, d_v, d_beta, d_g and d_S0 separately: relative
L2 <= 1e-4 for fp32 I/O and <= 1e-2 for bf16 I/O, and on every head at the
1.3B-layer shape.  Cases: the three decay regimes (mild U(0.9, 1), strong
U(0.3, 1), extreme U(0.05, 0.3), where a chunk's decay underflows fp32),
ragged lengths, both dtypes, 64- and 128-wide heads, with and without the
states; zero decay against the plain backward.
"""
import numpy as np
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import oracle
import workloads
from tests.conftest import rel_l2
from tests.gpu_util import TOL, dev, per_head_rel_l2

pytestmark = pytest.mark.gpu
NAMES = ("d_q", "d_k", "d_v", "d_beta", "d_g", "d_S0")
REGIMES = {"mild": (0.9, 1.0), "strong": (0.3, 1.0), "extreme": (0.05, 0.3)}


@pytest.fixture(autouse=True)
def no_device_error():
    lib = dn.load()
    assert lib.dn_device_error() == 0
    yield
    assert lib.dn_device_error() == 0


def _case(B, H, T, d, dtype, seed, regime="mild", states=True):
    inp = workloads.chunk_inputs(B, H, T, d, d, dtype=dtype, seed=seed, feature_map="silu",
                                 s0_std=0.2 if states else None)
    lo, hi = REGIMES[regime]
    g = workloads.gate_inputs(B, H, T, seed=seed, lo=lo, hi=hi)
    d_o, d_S = workloads.grad_inputs(B, H, T, d, d, dtype=dtype, seed=seed + 1, ds_std=0.1)
    return inp, g, d_o, (d_S if states else None)


def _run(inp, g, d_o, d_S):
    got = dn.chunk_bwd_gated(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g),
                             dev(d_o), initial_state=dev(inp.S0), d_final_state=dev(d_S))
    torch.cuda.synchronize()
    return [x.double().cpu().numpy() for x in got]


def _check(got, ref, tol, what):
    for name, a, b in zip(NAMES, got, ref):
        e = rel_l2(a, b)
        assert e <= tol, f"{what} {name} rel L2 {e:.3e}"


@pytest.mark.parametrize("regime", list(REGIMES))
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decay_regimes_and_ragged_lengths(regime, T, dtype):
    inp, g, d_o, d_S = _case(1, 2, T, 128, dtype, seed=17 * T + len(regime), regime=regime)
    ref = oracle.backward_gated(inp.q, inp.k, inp.v, inp.beta, g, d_o, inp.S0, d_S)
    _check(_run(inp, g, d_o, d_S), ref, TOL[workloads.torch_dtype(dtype)],
           f"{dtype} T={T} {regime}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("states", [False, True], ids=["no-states", "states"])
def test_head_widths_and_states(d, states):
    inp, g, d_o, d_S = _case(2, 2, 150, d, "f32", seed=d + 5, regime="strong", states=states)
    ref = oracle.backward_gated(inp.q, inp.k, inp.v, inp.beta, g, d_o, inp.S0, d_S)
    _check(_run(inp, g, d_o, d_S), ref, TOL[torch.float32], f"d={d} states={states}")


@pytest.mark.parametrize("regime", ["mild", "extreme"])
def test_bf16_64_wide_heads(regime):
    """bf16 with d = 64: the states from the CUDA-core recompute, the chain
    and gradients on the tf32 instances for 64-wide heads."""
    inp, g, d_o, d_S = _case(2, 2, 150, 64, "bf16", seed=21, regime=regime)
    ref = oracle.backward_gated(inp.q, inp.k, inp.v, inp.beta, g, d_o, inp.S0, d_S)
    _check(_run(inp, g, d_o, d_S), ref, TOL[torch.bfloat16], f"bf16 d=64 {regime}")


def test_zero_decay_matches_the_plain_backward():
    """g = 0: every gradient but d_g equals the plain backward's, both within
    fp32 rounding of each other."""
    inp, g, d_o, d_S = _case(1, 2, 130, 64, "f32", seed=3)
    g = torch.zeros_like(g)
    got = _run(inp, g, d_o, d_S)
    plain = [x.double().cpu().numpy() for x in dn.chunk_bwd(
        dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(d_o),
        initial_state=dev(inp.S0), d_final_state=dev(d_S))]
    for name, a, b in zip(NAMES[:4] + NAMES[5:], got[:4] + got[5:], plain):
        assert rel_l2(a, b) <= 1e-5, name


def test_layer_1p3b_workload_every_head():
    """B8 H16 T2048 d128 bf16 with keep rates U(0.9, 1): every gradient of
    every head held to the bar on its own."""
    inp = workloads.workload_inputs("layer1p3b_bf16")
    B, H, T, d = inp.q.shape
    g = workloads.gate_inputs(B, H, T, seed=7)
    d_o, d_S = workloads.grad_inputs(B, H, T, d, d, dtype="bf16", seed=2, ds_std=0.1)
    got = _run(inp, g, d_o, d_S)
    ref = oracle.backward_gated(inp.q, inp.k, inp.v, inp.beta, g, d_o, inp.S0, d_S)
    _check(got, ref, TOL[torch.bfloat16], "1.3B")
    for name, a, b in zip(NAMES, got, ref):
        e = per_head_rel_l2(a, b)
        assert e.max() <= TOL[torch.bfloat16], f"{name}: worst head {e.max():.3e}"


def test_workspace_is_checked():
    inp, g, d_o, d_S = _case(1, 1, 100, 64, "f32", seed=4)
    lib = dn.load()
    need = lib.dn_chunk_bwd_gated_workspace_bytes(1, 1, 100, 64, 64, 64, 0)
    assert need == 2 * 2 * 64 * 64 * 4
    with pytest.raises(dn.DeltaNetError, match="INVALID_ARG"):
        dn.chunk_bwd_gated(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(g), dev(d_o),
                           workspace=torch.empty(need - 16, dtype=torch.uint8, device="cuda"))


def test_autograd_function_matches_the_entry_point():
    """GatedDeltaRule.apply + torch.autograd gives chunk_bwd_gated's gradients
    exactly (the kernels' sums have a fixed order), and they match the
    oracle's."""
    inp, g, d_o, d_S = _case(2, 2, 150, 128, "bf16", seed=9, regime="strong")
    leaves = [dev(x).requires_grad_() for x in (inp.q, inp.k, inp.v, inp.beta, g, inp.S0)]
    o, S_T = dn.GatedDeltaRule.apply(*leaves)
    torch.autograd.backward([o, S_T], [dev(d_o), dev(d_S)])
    direct = dn.chunk_bwd_gated(*(dev(x) for x in (inp.q, inp.k, inp.v, inp.beta, g, d_o)),
                                initial_state=dev(inp.S0), d_final_state=dev(d_S))
    for leaf, want in zip(leaves, direct):
        assert torch.equal(leaf.grad, want)
    ref = oracle.backward_gated(inp.q, inp.k, inp.v, inp.beta, g, d_o, inp.S0, d_S)
    _check([x.grad.double().cpu().numpy() for x in leaves], ref, TOL[torch.bfloat16],
           "autograd")
