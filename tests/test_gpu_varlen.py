"""Packed variable-length sequences on the GPU (dn_chunk_fwd_varlen) against
the oracle, and against separate calls per sequence.  Bars: relative L2
<= 1e-2 (bf16 I/O) and <= 1e-4 (fp32 I/O) on o and on every final state.
"""
import numpy as np
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import oracle
import workloads
from tests.conftest import rel_l2
from tests.gpu_util import TOL

pytestmark = pytest.mark.gpu
LENS = [0, 1, 63, 64, 65, 200, 130, 7]


@pytest.fixture(autouse=True)
def no_device_error():
    lib = dn.load()
    assert lib.dn_device_error() == 0
    yield
    assert lib.dn_device_error() == 0


def _packed(lens, H, d, dtype, seed):
    T = int(sum(lens))
    inp = workloads.chunk_inputs(1, H, T, d, d, dtype=dtype, seed=seed, feature_map="silu")
    S0 = workloads.decode_state(len(lens), H, d, d, std=0.1, seed=seed)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(int).tolist()
    return inp, S0, cu


@pytest.mark.parametrize("path", ["tcgen05", "simt"])
def test_varlen_bf16_d128(path):
    H, d = 3, 128
    inp, S0, cu = _packed(LENS, H, d, "bf16", seed=21)
    q, k, v, b = (x[0].cuda() for x in (inp.q, inp.k, inp.v, inp.beta))
    o, S = dn.chunk_fwd_varlen(q, k, v, b, cu, initial_state=S0.cuda(),
                               workspace="auto" if path == "tcgen05" else None)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_varlen(inp.q[0], inp.k[0], inp.v[0], inp.beta[0], cu, S0)
    assert rel_l2(o.double().cpu().numpy(), o_ref) <= TOL[torch.bfloat16]
    for n, ln in enumerate(LENS):  # every state, including the empty sequences'
        assert rel_l2(S[n].double().cpu().numpy(), S_ref[n]) <= TOL[torch.bfloat16], n


def test_varlen_tensor_core_equals_separate_calls_exactly():
    """Tokens of the neighbouring sequence that a chunk's tiles read past the
    end meet exact zeros (strength 0), so each sequence's result is the one a
    separate call gives, bit for bit."""
    H, d = 2, 128
    lens = [65, 130, 1, 64]
    inp, S0, cu = _packed(lens, H, d, "bf16", seed=22)
    q, k, v, b = (x[0].cuda() for x in (inp.q, inp.k, inp.v, inp.beta))
    o, S = dn.chunk_fwd_varlen(q, k, v, b, cu, initial_state=S0.cuda())
    for n, (a, e) in enumerate(zip(cu[:-1], cu[1:])):
        o_n, S_n = dn.chunk_fwd(q[None, :, a:e].contiguous(), k[None, :, a:e].contiguous(),
                                v[None, :, a:e].contiguous(), b[None, :, a:e].contiguous(),
                                initial_state=S0[n][None].cuda(), algo="tcgen05")
        assert torch.equal(o[:, a:e], o_n[0]), n
        assert torch.equal(S[n], S_n[0]), n


@pytest.mark.parametrize("d", [64, 128])
def test_varlen_fp32(d):
    H = 2
    inp, S0, cu = _packed([5, 64, 0, 100, 70], H, d, "f32", seed=23 + d)
    q, k, v, b = (x[0].cuda() for x in (inp.q, inp.k, inp.v, inp.beta))
    o, S = dn.chunk_fwd_varlen(q, k, v, b, cu, initial_state=S0.cuda())
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_varlen(inp.q[0], inp.k[0], inp.v[0], inp.beta[0], cu, S0)
    assert rel_l2(o.double().cpu().numpy(), o_ref) <= TOL[torch.float32]
    assert rel_l2(S.double().cpu().numpy(), S_ref) <= TOL[torch.float32]


def test_varlen_all_empty_passes_the_states_through():
    H, d = 2, 128
    S0 = torch.randn(3, H, d, d, device="cuda")
    z = torch.zeros(H, 0, d, dtype=torch.bfloat16, device="cuda")
    o, S = dn.chunk_fwd_varlen(z, z, z, torch.zeros(H, 0, dtype=torch.bfloat16, device="cuda"),
                               [0, 0, 0, 0], initial_state=S0)
    assert torch.equal(S, S0) and o.numel() == 0


def test_varlen_bench_packing_sampled_sequences():
    """The bench's packing: the 1.3B-layer tokens (B8 x T2048 per head, H16,
    d128, bf16) re-read head-major as 64 packed sequences of seeded lengths,
    on the tensor-core path; five sequences on two heads checked against
    the oracle (outputs and final states), first and last included."""
    w = workloads.WORKLOADS["layer1p3b_bf16"]
    inp = workloads.workload_inputs("layer1p3b_bf16")
    B, H, T, d = inp.q.shape
    lens = workloads.varlen_lengths(64, B * T, seed=w["seed"])
    cu = [0]
    for ln in lens:
        cu.append(cu[-1] + ln)
    vq, vk, vv = (x.transpose(0, 1).reshape(H, B * T, -1).contiguous() for x in (inp.q, inp.k, inp.v))
    vb = inp.beta.transpose(0, 1).reshape(H, B * T).contiguous()
    o, S = dn.chunk_fwd_varlen(vq.cuda(), vk.cuda(), vv.cuda(), vb.cuda(), cu)
    torch.cuda.synchronize()
    o, S = o.cpu(), S.cpu()
    for n in (0, 17, 40, 62, 63):
        a, b = cu[n], cu[n + 1]
        for h in (0, H - 1):
            o_ref, S_ref = oracle.forward(vq[None, h:h + 1, a:b], vk[None, h:h + 1, a:b],
                                          vv[None, h:h + 1, a:b], vb[None, h:h + 1, a:b])
            assert rel_l2(o[h, a:b].double().numpy(), o_ref[0, 0]) <= TOL[torch.bfloat16], (n, h)
            assert rel_l2(S[n, h].double().numpy(), S_ref[0, 0]) <= TOL[torch.bfloat16], (n, h)
