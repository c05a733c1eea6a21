"""CUDA-graph capture of both entry points.

The library enqueues kernels only (no allocation, no synchronisation), so a
sequence of calls can be captured into a CUDA graph and replayed.  A replay
must give exactly what the same calls give eagerly: the kernels and their
inputs are the same, only the launch route differs.
"""
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import workloads
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu


def _capture(fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        fn()
    return g


def test_decode_steps_replayed_from_a_graph_equal_eager():
    B, H, d, steps, seed = 8, 4, 128, 16, 77
    xs = [workloads.decode_step_inputs(B, H, d, d, step=i, dtype="bf16", seed=seed,
                                       beta_scale=2.0) for i in range(steps)]
    q, k, v, b = (torch.stack([dev(getattr(x, n)) for x in xs]) for n in ("q", "k", "v", "beta"))
    S0 = dev(workloads.decode_state(B, H, d, d, std=0.1, seed=seed))

    S_e = S0.clone()
    o_e = torch.empty(steps, B, H, d, dtype=torch.bfloat16, device="cuda")
    for i in range(steps):
        dn.recurrent_step(q[i], k[i], v[i], b[i], S_e, out=o_e[i])

    S_g = S0.clone()
    o_g = torch.zeros_like(o_e)
    g = _capture(lambda: [dn.recurrent_step(q[i], k[i], v[i], b[i], S_g, out=o_g[i])
                          for i in range(steps)])
    torch.cuda.synchronize()
    assert torch.equal(S_g, S0) and not o_g.any()  # capture ran nothing
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e)
    assert torch.equal(S_g, S_e)
    assert dn.load().dn_device_error() == 0


@pytest.mark.parametrize("workspace", ["auto", None], ids=["two-pass", "fused"])
def test_chunk_fwd_replayed_from_a_graph_equal_eager(workspace):
    inp = workloads.chunk_inputs(B=2, H=4, T=1000, dk=128, dv=128, dtype="bf16",
                                 seed=5, s0_std=0.1)
    q, k, v, b, S0 = (dev(x) for x in (inp.q, inp.k, inp.v, inp.beta, inp.S0))
    ws = workspace
    if workspace == "auto":
        ws = torch.empty(dn.load().dn_chunk_fwd_workspace_bytes(2, 4, 1000, 128, 128, 64, 1),
                         dtype=torch.uint8, device="cuda")
    o_e, S_e = dn.chunk_fwd(q, k, v, b, initial_state=S0, output_final_state=True,
                            algo="tcgen05", workspace=ws)
    o_g, S_g = torch.zeros_like(o_e), torch.zeros_like(S_e)
    g = _capture(lambda: dn.chunk_fwd(q, k, v, b, initial_state=S0, out=o_g, final_state=S_g,
                                      algo="tcgen05", workspace=ws))
    for _ in range(2):  # a replay depends on nothing a previous one left behind
        o_g.zero_()
        S_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_e)
        assert torch.equal(S_g, S_e)
    assert dn.load().dn_device_error() == 0


def test_gated_tensor_core_call_replayed_from_a_graph_equals_eager():
    """The gated two-pass call (decay-scaled tiles and decay vectors in the
    caller's workspace) captured and replayed: the same bits as eager."""
    B, H, T, d = 2, 4, 700, 128
    inp = workloads.chunk_inputs(B, H, T, d, d, dtype="bf16", seed=9, s0_std=0.1)
    q, k, v, b, S0 = (dev(x) for x in (inp.q, inp.k, inp.v, inp.beta, inp.S0))
    g = dev(workloads.gate_inputs(B, H, T, seed=9, lo=0.5))
    ws = torch.empty(dn.load().dn_chunk_fwd_gated_workspace_bytes(B, H, T, d, d, 64, 1),
                     dtype=torch.uint8, device="cuda")
    o_e, S_e = dn.chunk_fwd_gated(q, k, v, b, g, initial_state=S0, workspace=ws)
    o_g, S_g = torch.zeros_like(o_e), torch.zeros_like(S_e)
    gr = _capture(lambda: dn.chunk_fwd_gated(q, k, v, b, g, initial_state=S0, out=o_g,
                                             final_state=S_g, workspace=ws))
    for _ in range(2):
        o_g.zero_()
        S_g.zero_()
        gr.replay()
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_e)
        assert torch.equal(S_g, S_e)
    assert dn.load().dn_device_error() == 0
