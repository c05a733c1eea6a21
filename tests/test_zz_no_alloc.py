"""dn_chunk_fwd_noalloc, the entry point that allocates nothing, through the C ABI.

Its [PT; T] tiles live in a static device array instead of a caller
workspace; the kernels are the same as dn_chunk_fwd's two-pass tensor-core
path, so on the same inputs the outputs must be identical, call after call.
This file is collected last and also runs on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from delta_rule_recurrent_gb300 import _lib
import delta_rule_recurrent_gb300 as dn
from tests.conftest import rel_l2

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, b, S0, o, S_T):
    B, H, T, d = q.shape
    return lib.dn_chunk_fwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), b.data_ptr(),
        S0.data_ptr() if S0 is not None else None, o.data_ptr(), S_T.data_ptr(),
        B, H, T, d, d, 64, _lib.DN_BF16, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("B,H,T,s0", [(2, 4, 1000, 0.1), (1, 16, 2048, None)])
def test_noalloc_matches_the_workspace_entry_point_twice(B, H, T, s0):
    lib = _lib.load()
    assert lib.dn_device_error() == 0
    inp = workloads.chunk_inputs(B, H, T, 128, 128, dtype="bf16", seed=900 + T,
                                 feature_map="silu", s0_std=s0)
    q, k, v, b = (x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta))
    S0 = inp.S0.cuda() if inp.S0 is not None else None
    o_ref, S_ref = dn.chunk_fwd(q, k, v, b, initial_state=S0, algo="tcgen05", workspace="auto")
    for call in range(2):  # the shared static scratch is reused by the second call
        o = torch.full_like(o_ref, float("nan"))
        S_T = torch.full_like(S_ref, float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _noalloc(lib, q, k, v, b, S0, o, S_T) == _lib.DN_OK, lib.dn_last_error()
        torch.cuda.synchronize()
        if call == 1:  # after the first call has loaded everything: no device memory taken
            assert torch.cuda.mem_get_info()[0] == free_before
        assert torch.equal(o, o_ref)
        assert torch.equal(S_T, S_ref)
    assert lib.dn_device_error() == 0
    # and one head against the oracle, independently of the workspace path
    s0 = None if inp.S0 is None else inp.S0[:1, :1]
    o1, S1 = oracle.forward(inp.q[:1, :1], inp.k[:1, :1], inp.v[:1, :1], inp.beta[:1, :1], s0)
    assert rel_l2(o[:1, :1].double().cpu().numpy(), o1) <= 1e-2
    assert rel_l2(S_T[:1, :1].double().cpu().numpy(), S1) <= 1e-2


def test_noalloc_refuses_more_than_its_scratch():
    lib = _lib.load()
    B, H, T = 1, 8, 64 * 65  # 520 chunk tiles > 512
    q = torch.zeros(B, H, T, 128, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(B, H, T, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    S_T = torch.empty(B, H, 128, 128, device="cuda")
    assert _noalloc(lib, q, q, q, b, None, o, S_T) == _lib.DN_ERR_INVALID_ARG
    assert b"512" in lib.dn_last_error()
