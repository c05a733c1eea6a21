"""dn_chunk_fwd_split on the GPU against the fp64 oracle: each sequence cut
into runs of whole chunks scanned in parallel, the runs' start states joined
through their transitions.

Bar: relative L2 <= 1e-2 on o and S_T (bf16 I/O), per (batch, head) and per
64-token chunk of o.  Cases: one run (the plain scan), runs that do and do
not divide the chunk count, a ragged last chunk, more runs asked for than
there are chunks, with and without an initial state, and the automatic
count; argument errors.
"""
import numpy as np
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import oracle
import workloads
from tests.gpu_util import TOL, check_every_head, dev, run_chunk

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def no_device_error():
    lib = dn.load()
    assert lib.dn_device_error() == 0
    yield
    assert lib.dn_device_error() == 0


@pytest.mark.parametrize("T,segments", [(1, 1), (200, 2), (200, 3), (1000, 1), (1000, 3),
                                        (1000, 5), (4100, 7), (4100, 64), (130, 9), (4096, 0)])
@pytest.mark.parametrize("s0", [None, 0.3], ids=["zero-start", "S0"])
def test_runs_match_the_oracle(T, segments, s0):
    inp = workloads.chunk_inputs(1, 2, T, 128, 128, dtype="bf16", seed=T + segments,
                                 feature_map="silu", s0_std=s0)
    o, S = run_chunk(inp, "split", segments=segments)
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    check_every_head(o, S, o_ref, S_ref, TOL[torch.bfloat16], f"T={T} runs={segments}")


def test_several_sequences_automatic_runs():
    """B2 H3: six sequences, as many runs each as fill the GPU once."""
    inp = workloads.chunk_inputs(2, 3, 2500, 128, 128, dtype="bf16", seed=5,
                                 feature_map="silu", s0_std=0.1)
    o, S = run_chunk(inp, "split")
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    check_every_head(o, S, o_ref, S_ref, TOL[torch.bfloat16], "B2 H3 automatic runs")


def test_in_place_final_state():
    inp = workloads.chunk_inputs(1, 2, 1000, 128, 128, dtype="bf16", seed=9,
                                 feature_map="silu", s0_std=0.2)
    S = dev(inp.S0).clone()
    o, S_out = dn.chunk_fwd_split(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta),
                                  initial_state=S, final_state=S, segments=4)
    torch.cuda.synchronize()
    assert S_out.data_ptr() == S.data_ptr()
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    check_every_head(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref,
                     TOL[torch.bfloat16], "in place")


def test_arguments_are_checked():
    lib = dn.load()
    inp = workloads.chunk_inputs(1, 1, 300, 128, 128, dtype="bf16", seed=1)
    need = lib.dn_chunk_fwd_split_workspace_bytes(1, 1, 300, 128, 128, 64, 1, 2)
    assert need == 5 * 16384 + 3 * 2 * 128 * 128 * 4
    with pytest.raises(dn.DeltaNetError, match="INVALID_ARG"):
        dn.chunk_fwd_split(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), segments=2,
                           workspace=torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
    with pytest.raises(dn.DeltaNetError, match="INVALID_ARG"):
        dn.chunk_fwd_split(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta), segments=1025)
    f32 = workloads.chunk_inputs(1, 1, 300, 128, 128, dtype="f32", seed=1)
    with pytest.raises(dn.DeltaNetError, match="UNSUPPORTED"):
        dn.chunk_fwd_split(dev(f32.q), dev(f32.k), dev(f32.v), dev(f32.beta), segments=2)
