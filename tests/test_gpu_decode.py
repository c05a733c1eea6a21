"""Fused decoding step on the GPU against the fp64 oracle (through the C ABI).

The full decode workload (B256 H16 d128, fp32 state, bf16 q/k/v/beta,
beta in (0, 2), 1024 chained steps with fresh inputs) runs in full on the
GPU; sampled heads are replayed by the oracle over all 1024 steps.
"""
import numpy as np
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import oracle
import workloads
from tests.conftest import rel_l2
from tests.gpu_util import TOL, dev, sample_heads

pytestmark = pytest.mark.gpu


def _run_steps(B, H, dk, dv, steps, dtype, seed, beta_scale=2.0, s0_std=0.1, sample=None):
    """Runs `steps` chained decoding steps; returns the sampled heads' inputs,
    outputs and initial/final states."""
    S0 = workloads.decode_state(B, H, dk, dv, std=s0_std, seed=seed)
    S = dev(S0)
    bi, hi = sample if sample is not None else (np.repeat(np.arange(B), H), np.tile(np.arange(H), B))
    ib, ih = torch.as_tensor(bi), torch.as_tensor(hi)
    rec = {name: [] for name in ("q", "k", "v", "beta", "o")}
    for step in range(steps):
        x = workloads.decode_step_inputs(B, H, dk, dv, step=step, dtype=dtype, seed=seed,
                                         beta_scale=beta_scale)
        o = dn.recurrent_step(dev(x.q), dev(x.k), dev(x.v), dev(x.beta), S)
        for name in ("q", "k", "v", "beta"):
            rec[name].append(getattr(x, name)[ib, ih])
        rec["o"].append(o[ib.cuda(), ih.cuda()].cpu())
    torch.cuda.synchronize()
    stack = {n: torch.stack(v, dim=1).unsqueeze(0) for n, v in rec.items()}  # [1, n, steps, ...]
    return stack, S0[ib, ih].unsqueeze(0), S[ib.cuda(), ih.cuda()].double().cpu().numpy()[None]


def test_decode_workload_1024_steps_sampled_heads():
    w = workloads.WORKLOADS["decode_bf16"]
    B, H, dk, dv, steps = w["B"], w["H"], w["dk"], w["dv"], w["steps"]
    sample = sample_heads(B, H, 24, seed=11)
    rec, S0, S_gpu = _run_steps(B, H, dk, dv, steps, "bf16", w["seed"], sample=sample,
                                beta_scale=w["beta_scale"], s0_std=w["s0_std"])
    o_ref, S_ref = oracle.forward(rec["q"], rec["k"], rec["v"], rec["beta"], S0)
    eo = rel_l2(rec["o"].double().numpy(), o_ref)
    eS = rel_l2(S_gpu, S_ref)
    assert eo <= TOL[torch.bfloat16], f"o rel L2 {eo:.3e}"
    assert eS <= TOL[torch.bfloat16], f"S rel L2 {eS:.3e}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_decode_shapes(dtype, dk, dv):
    rec, S0, S_gpu = _run_steps(3, 5, dk, dv, 12, dtype, seed=dk * 3 + dv)
    o_ref, S_ref = oracle.forward(rec["q"], rec["k"], rec["v"], rec["beta"], S0)
    tol = TOL[workloads.torch_dtype(dtype)]
    assert rel_l2(rec["o"].double().numpy(), o_ref) <= tol
    assert rel_l2(S_gpu, S_ref) <= tol


def test_decode_beta_zero_leaves_state_bitwise():
    B, H, d = 4, 3, 128
    S = dev(workloads.decode_state(B, H, d, d, seed=1))
    S_before = S.clone()
    x = workloads.decode_step_inputs(B, H, d, d, step=0, dtype="f32", seed=2)
    o = dn.recurrent_step(dev(x.q), dev(x.k), dev(x.v), torch.zeros(B, H, device="cuda:0"), S)
    torch.cuda.synchronize()
    assert torch.equal(S, S_before)
    o_ref = torch.einsum("bhij,bhi->bhj", S_before.double(), dev(x.q).double())
    assert rel_l2(o.double().cpu().numpy(), o_ref.cpu().numpy()) <= 1e-6


def test_decode_rejects_bad_pointers():
    from delta_rule_recurrent_gb300 import _lib
    lib = _lib.load()
    B, H, d = 2, 2, 64
    q = torch.zeros(B, H, d, device="cuda:0")
    beta = torch.zeros(B, H, device="cuda:0")
    S = torch.zeros(B, H, d, d, device="cuda:0")
    o = torch.zeros(B, H, d, device="cuda:0")
    call = lambda Sp, op: lib.dn_recurrent_step(q.data_ptr(), q.data_ptr(), q.data_ptr(),
                                                beta.data_ptr(), Sp, op, B, H, d, d, 0, None)
    assert call(S.cpu().data_ptr(), o.data_ptr()) == _lib.DN_ERR_INVALID_ARG
    assert call(S.data_ptr(), q.data_ptr()) == _lib.DN_ERR_INVALID_ARG
    assert call(S.data_ptr() + 4, o.data_ptr()) == _lib.DN_ERR_INVALID_ARG
    assert call(S.data_ptr(), o.data_ptr()) == _lib.DN_OK
    torch.cuda.synchronize()
