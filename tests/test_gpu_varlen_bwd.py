"""dn_chunk_bwd_varlen on the GPU: every packed sequence's gradients against
the fp64 oracle's gradient of that sequence alone.

Bars per gradient and per sequence: relative L2 <= 1e-4 (fp32 I/O) and
<= 1e-2 (bf16 I/O).  Cases: ragged lengths, an empty sequence, a one-token
sequence, both dtypes, 64- and 128-wide heads, with and without the states;
and equality with the batched backward when the sequences are equally long.
"""
import numpy as np
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import oracle
import workloads
from tests.conftest import rel_l2
from tests.gpu_util import TOL, dev

pytestmark = pytest.mark.gpu
NAMES = ("d_q", "d_k", "d_v", "d_beta", "d_S0")


@pytest.fixture(autouse=True)
def no_device_error():
    lib = dn.load()
    assert lib.dn_device_error() == 0
    yield
    assert lib.dn_device_error() == 0


def _packed_case(lens, H, d, dtype, seed, states):
    T = sum(lens)
    inp = workloads.chunk_inputs(1, H, T, d, d, dtype=dtype, seed=seed, feature_map="silu")
    d_o, _ = workloads.grad_inputs(1, H, T, d, d, dtype=dtype, seed=seed + 1, ds_std=0.1)
    g = torch.Generator().manual_seed(seed + 2)
    N = len(lens)
    S0 = (0.2 * torch.randn(N, H, d, d, generator=g)) if states else None
    dS = (0.1 * torch.randn(N, H, d, d, generator=g)) if states else None
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(int).tolist()
    return [x[0] for x in (inp.q, inp.k, inp.v, inp.beta, d_o)], S0, dS, cu


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 64), ("f32", 128)])
@pytest.mark.parametrize("states", [False, True], ids=["no-states", "states"])
def test_each_sequence_matches_the_oracle(dtype, d, states):
    lens = [130, 0, 1, 64, 257, 63]
    (q, k, v, b, do), S0, dS, cu = _packed_case(lens, 2, d, dtype, 7 * d + len(dtype), states)
    got = dn.chunk_bwd_varlen(dev(q), dev(k), dev(v), dev(b), dev(do), cu,
                              initial_state=dev(S0), d_final_state=dev(dS))
    torch.cuda.synchronize()
    got = [x.double().cpu().numpy() for x in got]
    tol = TOL[workloads.torch_dtype(dtype)]
    for n in range(len(lens)):
        a, e = cu[n], cu[n + 1]
        s0 = None if S0 is None else S0[n][None]
        ds = None if dS is None else dS[n][None]
        if e == a:  # empty: the state gradient passes through
            want = np.zeros((2, d, d)) if dS is None else dS[n].double().numpy()
            assert np.array_equal(got[4][n], want)
            continue
        ref = oracle.backward(q[None, :, a:e], k[None, :, a:e], v[None, :, a:e],
                              b[None, :, a:e], do[None, :, a:e], s0, ds)
        mine = [got[0][:, a:e], got[1][:, a:e], got[2][:, a:e], got[3][:, a:e], got[4][n]]
        for name, x, r in zip(NAMES, mine, ref):
            err = rel_l2(x, np.asarray(r)[0])
            assert err <= tol, f"sequence {n} (len {e - a}) {name} rel L2 {err:.3e}"


def test_equal_lengths_match_the_batched_backward():
    """Three sequences of 200 tokens packed, against the batched backward of
    the same data laid out [3, H, 200, d]: the same kernels per sequence, so
    the gradients are equal bit for bit."""
    lens, H, d = [200, 200, 200], 2, 128
    (q, k, v, b, do), S0, dS, cu = _packed_case(lens, H, d, "bf16", 11, True)
    got = dn.chunk_bwd_varlen(dev(q), dev(k), dev(v), dev(b), dev(do), cu,
                              initial_state=dev(S0), d_final_state=dev(dS))

    def batched(x):  # [H, 3*200, ...] -> [3, H, 200, ...]
        return dev(torch.stack([x[:, cu[n]:cu[n + 1]] for n in range(3)]))

    ref = dn.chunk_bwd(batched(q), batched(k), batched(v), batched(b), batched(do),
                       initial_state=dev(S0), d_final_state=dev(dS))
    torch.cuda.synchronize()
    for name, x, r in zip(NAMES[:4], got[:4], ref[:4]):
        packed = torch.stack([x[:, cu[n]:cu[n + 1]] for n in range(3)])
        assert torch.equal(packed, r), name
    assert torch.equal(got[4], ref[4])


def test_arguments_are_checked():
    lib = dn.load()
    (q, k, v, b, do), _, _, cu = _packed_case([100, 50], 2, 64, "f32", 3, False)
    need = lib.dn_chunk_bwd_varlen_workspace_bytes((__import__("ctypes").c_int * 3)(*cu), 2, 2,
                                                   64, 64, 64, 0)
    assert need > 0
    with pytest.raises(dn.DeltaNetError, match="INVALID_ARG"):
        dn.chunk_bwd_varlen(dev(q), dev(k), dev(v), dev(b), dev(do), cu,
                            workspace=torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
    with pytest.raises(dn.DeltaNetError, match="INVALID_ARG"):  # offsets not ending at T
        dn.chunk_bwd_varlen(dev(q), dev(k), dev(v), dev(b), dev(do), [0, 100, 140])
