"""Chunkwise backward on the GPU against the fp64 oracle's gradient (through
the C ABI).

Bars, on each of d_q, d_k, d_v, d_beta and d_S0 separately: relative L2
<= 1e-4 for fp32 I/O and <= 1e-2 for bf16 I/O (fp32 arithmetic, bf16
gradients).  The full-size workload is checked on every (batch, head) pair
separately.
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
NAMES = ("d_q", "d_k", "d_v", "d_beta", "d_S0")


@pytest.fixture(autouse=True)
def no_device_error():
    lib = dn.load()
    assert lib.dn_device_error() == 0
    yield
    assert lib.dn_device_error() == 0


def _gpu_grads(inp, d_o, d_S):
    g = dn.chunk_bwd(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(d_o),
                     initial_state=dev(inp.S0), d_final_state=dev(d_S))
    torch.cuda.synchronize()
    return [x.double().cpu().numpy() for x in g]


def _check(got, ref, dtype, what=""):
    errs = {}
    for name, a, b in zip(NAMES, got, ref):
        errs[name] = rel_l2(a, b)
        assert errs[name] <= TOL[dtype], f"{what} {name} rel L2 {errs[name]:.3e}"
    return errs


def _case(B, H, T, dk, dv, dtype, seed, s0=0.1, ds=0.1):
    inp = workloads.chunk_inputs(B, H, T, dk, dv, dtype=dtype, seed=seed, feature_map="silu",
                                 s0_std=s0)
    d_o, d_S = workloads.grad_inputs(B, H, T, dv, dk, dtype=dtype, seed=seed, ds_std=ds)
    return inp, d_o, d_S


def test_tiny_fp32_workload_gradients():
    """The tiny fp32 workload (B1 H2 T256 d64), every gradient in full."""
    inp = workloads.workload_inputs("tiny_fp32")
    d_o, d_S = workloads.grad_inputs(1, 2, 256, 64, 64, dtype="f32", seed=0, ds_std=0.1)
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.beta, d_o, inp.S0, d_S)
    _check(_gpu_grads(inp, d_o, d_S), ref, torch.float32, "tiny")


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_shapes(dk, dv, dtype):
    """Several chunks and a ragged tail, initial state and final-state
    gradient present, every (dk, dv) the library covers."""
    inp, d_o, d_S = _case(2, 2, 200, dk, dv, dtype, seed=dk + dv)
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.beta, d_o, inp.S0, d_S)
    _check(_gpu_grads(inp, d_o, d_S), ref, workloads.torch_dtype(dtype), f"{dtype} {dk}x{dv}")


@pytest.mark.parametrize("T", [1, 63, 64, 65])
def test_edge_lengths_without_optional_states(T):
    """One token, one chunk short, exactly one chunk, one past it; no S0 and
    no final-state gradient (zeros)."""
    inp, d_o, _ = _case(1, 3, T, 128, 128, "f32", seed=T, s0=None, ds=None)
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.beta, d_o, None, None)
    _check(_gpu_grads(inp, d_o, None), ref, torch.float32, f"T={T}")


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
@pytest.mark.parametrize("states", [False, True], ids=["no-states", "states"])
def test_tensor_core_chain_edge_lengths(T, states):
    """bf16, dk = dv = 128: the tensor-core chain (chunks last to first, the
    ragged chunk first) from one token to a ragged third chunk, with and
    without the initial state and the final-state gradient."""
    inp, d_o, d_S = _case(1, 3, T, 128, 128, "bf16", seed=100 + T,
                          s0=0.3 if states else None, ds=0.3 if states else None)
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.beta, d_o, inp.S0, d_S)
    got = _gpu_grads(inp, d_o, d_S) if states else [
        x.double().cpu().numpy() for x in dn.chunk_bwd(
            dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(d_o))]
    _check(got, ref, torch.bfloat16, f"T={T} states={states}")


def test_beta_zero_gives_zero_key_and_value_gradients():
    inp, d_o, d_S = _case(1, 2, 130, 64, 64, "f32", seed=3)
    inp.beta.zero_()
    got = _gpu_grads(inp, d_o, d_S)
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.beta, d_o, inp.S0, d_S)
    _check(got, ref, torch.float32, "beta=0")


def test_empty_sequence_passes_the_state_gradient_through():
    q = torch.zeros(2, 2, 0, 64, device="cuda")
    v = torch.zeros(2, 2, 0, 64, device="cuda")
    d_S = torch.randn(2, 2, 64, 64, device="cuda")
    g = dn.chunk_bwd(q, q, v, torch.zeros(2, 2, 0, device="cuda"), v, d_final_state=d_S)
    assert torch.equal(g[4], d_S) and g[0].numel() == 0


def test_layer_1p3b_workload_every_head():
    """B8 H16 T2048 d128 bf16, full launch; every gradient of every head
    against the oracle's, each head held to the bar on its own."""
    inp = workloads.workload_inputs("layer1p3b_bf16")
    B, H, T, d = inp.q.shape
    d_o, d_S = workloads.grad_inputs(B, H, T, d, d, dtype="bf16", seed=2, ds_std=0.1)
    got = _gpu_grads(inp, d_o, d_S)
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.beta, d_o, inp.S0, d_S)
    _check(got, ref, torch.bfloat16, "1.3B")
    for name, a, b in zip(NAMES, got, ref):
        e = per_head_rel_l2(a, b)
        worst = np.unravel_index(int(np.argmax(e)), e.shape)
        assert e.max() <= TOL[torch.bfloat16], f"{name} rel L2 {e.max():.3e} at (b, h) = {worst}"


def test_workspace_is_checked():
    inp, d_o, d_S = _case(1, 1, 100, 64, 64, "f32", seed=4)
    need = dn.load().dn_chunk_bwd_workspace_bytes(1, 1, 100, 64, 64, 64, 0)
    assert need == 2 * 2 * 64 * 64 * 4
    short = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(dn.DeltaNetError, match="INVALID_ARG"):
        dn.chunk_bwd(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(d_o),
                     workspace=short)


def test_autograd_function_matches_the_entry_point():
    """DeltaRule.apply + torch.autograd gives chunk_bwd's gradients exactly,
    and they match the oracle."""
    inp, d_o, d_S = _case(2, 2, 150, 128, 128, "bf16", seed=6)
    leaves = [dev(x).requires_grad_() for x in (inp.q, inp.k, inp.v, inp.beta, inp.S0)]
    o, S_T = dn.DeltaRule.apply(*leaves)
    torch.autograd.backward([o, S_T], [dev(d_o), dev(d_S)])
    direct = dn.chunk_bwd(*(dev(x) for x in (inp.q, inp.k, inp.v, inp.beta, d_o)),
                          initial_state=dev(inp.S0), d_final_state=dev(d_S))
    for leaf, g in zip(leaves, direct):
        assert torch.equal(leaf.grad, g)
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.beta, d_o, inp.S0, d_S)
    _check([x.grad.double().cpu().numpy() for x in leaves], ref, torch.bfloat16, "autograd")


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_autograd_with_a_query_scale(dtype, d):
    """DeltaRule.apply(..., scale=s): the forward reads s q; the gradients are
    the oracle's for s q, with the q gradient multiplied by s (chain rule)."""
    inp, d_o, d_S = _case(1, 2, 130, d, d, dtype, seed=8)
    s = d ** -0.5
    leaves = [dev(x).requires_grad_() for x in (inp.q, inp.k, inp.v, inp.beta, inp.S0)]
    o, S_T = dn.DeltaRule.apply(*leaves, s)
    torch.autograd.backward([o, S_T], [dev(d_o), dev(d_S)])
    qs, _ = oracle.prepare_qk(inp.q, inp.k, scale=s)
    o_ref, _ = oracle.forward(qs, inp.k, inp.v, inp.beta, inp.S0)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    assert rel_l2(o.detach().double().cpu().numpy(), o_ref) <= TOL[dt]
    ref = list(oracle.backward(qs, inp.k, inp.v, inp.beta, d_o, inp.S0, d_S))
    ref[0] = ref[0] * s
    _check([x.grad.double().cpu().numpy() for x in leaves], ref, dt, "autograd, scaled q")
