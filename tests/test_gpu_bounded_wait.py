"""The bounded-wait failure path, exercised once on purpose.

The tensor-core gradient kernel (dn_chunk_bwd, bf16, dk = dv = 128) is given
a zero limit on its first wait through dn_debug_first_wait_ns, so that wait
gives up before looking.  The kernel must then record the timeout code, wait
for the loads it had started, free its tensor memory and return; nothing
hangs and the context stays usable: with the default limit back, the next
call must match the oracle.  No fault, trap or endless wait is involved.
"""
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import oracle
import workloads
from tests.conftest import rel_l2
from tests.gpu_util import TOL, dev

pytestmark = pytest.mark.gpu
DEFAULT_LIMIT_NS = 2_000_000_000


def _call(inp, d_o, d_S):
    g = dn.chunk_bwd(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), dev(d_o),
                     initial_state=dev(inp.S0), d_final_state=dev(d_S))
    torch.cuda.synchronize()
    return [x.double().cpu().numpy() for x in g]


def test_first_wait_giving_up_is_recorded_and_the_next_call_is_right():
    lib = dn.load()
    inp = workloads.chunk_inputs(1, 2, 130, 128, 128, dtype="bf16", seed=11,
                                 feature_map="silu", s0_std=0.1)
    d_o, d_S = workloads.grad_inputs(1, 2, 130, 128, 128, dtype="bf16", seed=11, ds_std=0.1)
    assert lib.dn_device_error() == 0
    assert lib.dn_debug_first_wait_ns(0) == 0
    try:
        _call(inp, d_o, d_S)
        assert lib.dn_device_error() == 1, "the zero-limit wait did not record its code"
    finally:
        assert lib.dn_debug_first_wait_ns(DEFAULT_LIMIT_NS) == 0
    got = _call(inp, d_o, d_S)
    assert lib.dn_device_error() == 0
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.beta, d_o, inp.S0, d_S)
    for name, a, b in zip(("d_q", "d_k", "d_v", "d_beta", "d_S0"), got, ref):
        e = rel_l2(a, b)
        assert e <= TOL[torch.bfloat16], f"{name} rel L2 {e:.3e} after the failed call"
