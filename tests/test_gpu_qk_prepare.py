"""The q/k preparation (dn_qk_prepare: optional L2 normalisation and query
scale) on the GPU against the oracle's fp64 preparation, element by element,
and the forms that take ``qk_l2norm`` / ``scale`` against the oracle run on
the oracle's own prepared inputs.

Element bars, from the arithmetic: the fp32 sum of d squares carries at most
(d - 1) roundings of 2^-24, the reciprocal square root and the two products
a few more, so an fp32 result sits within (d + 4) 2^-24 of the exact value,
relative; a bf16 result adds one rounding to 8 significant bits (2^-8).
Whole-call bars as everywhere: relative L2 <= 1e-4 (fp32 I/O), <= 1e-2
(bf16 I/O).
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
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def no_device_error():
    lib = dn.load()
    assert lib.dn_device_error() == 0
    yield
    assert lib.dn_device_error() == 0


def _raw(B, H, T, d, dtype, seed, zero_rows=()):
    inp = workloads.chunk_inputs(B, H, T, d, d, dtype=dtype, seed=seed, normalize=False)
    q, k = inp.q.clone(), inp.k.clone()
    for idx in zero_rows:  # rows the normalisation must leave at zero
        q[idx] = 0
        k[idx] = 0
    return inp, q, k


def _check_elements(got, ref, dtype):
    got = got.double().cpu().numpy()
    f32 = (ref.shape[-1] + 4) * 2.0 ** -24
    rel = f32 if dtype == "f32" else 2.0 ** -8 * (1 + f32) + f32
    bound = rel * np.abs(ref) + 1e-30
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{bad.sum()} elements off, worst at {np.argwhere(bad)[0]}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_prepare_matches_the_oracle_elementwise(dtype, d):
    """Ragged row count (3 * 257 rows: not a multiple of the 16 rows a block
    takes), zero rows, and the 1/sqrt(d) query scale."""
    _, q, k = _raw(1, 3, 257, d, dtype, seed=31, zero_rows=[(0, 0, 0), (0, 2, 256)])
    s = d ** -0.5
    qo, ko = dn.qk_prepare(q.cuda(), k.cuda(), scale=s, l2norm=True)
    torch.cuda.synchronize()
    q_ref, k_ref = oracle.prepare_qk(q, k, scale=s, l2norm=True)
    _check_elements(qo, q_ref, dtype)
    _check_elements(ko, k_ref, dtype)
    assert torch.all(qo[0, 0, 0] == 0) and torch.all(ko[0, 2, 256] == 0)


@pytest.mark.parametrize("rows", [1, 31, 33])
def test_prepare_tiny_row_counts(rows):
    """Fewer rows than one block takes (8 warps x 2 rows), and one partial block."""
    _, q, k = _raw(1, 1, rows, 128, "bf16", seed=32)
    qo, ko = dn.qk_prepare(q.cuda(), k.cuda(), scale=0.5, l2norm=True)
    torch.cuda.synchronize()
    q_ref, k_ref = oracle.prepare_qk(q, k, scale=0.5, l2norm=True)
    _check_elements(qo, q_ref, "bf16")
    _check_elements(ko, k_ref, "bf16")


def test_in_place_equals_out_of_place_bit_for_bit():
    _, q, k = _raw(2, 2, 130, 128, "bf16", seed=33)
    qg, kg = q.cuda(), k.cuda()
    qo, ko = dn.qk_prepare(qg, kg, scale=0.125, l2norm=True)
    qi, ki = dn.qk_prepare(qg.clone(), kg.clone(), scale=0.125, l2norm=True, inplace=True)
    torch.cuda.synchronize()
    assert torch.equal(qo, qi) and torch.equal(ko, ki)


def test_scale_alone_scales_q_and_leaves_k():
    _, q, k = _raw(1, 2, 65, 64, "f32", seed=34)
    qg, kg = q.cuda(), k.cuda()
    k_before = kg.clone()
    qo, ko = dn.qk_prepare(qg, kg, scale=0.25, l2norm=False)
    torch.cuda.synchronize()
    assert ko is kg and torch.equal(kg, k_before)
    assert torch.equal(qo.cpu(), q * 0.25)  # a power of two: exact


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_chunk_forward_with_normalisation_and_scale(dtype, d):
    """chunk_fwd(..., qk_l2norm=True, scale=d^-1/2) on raw q, k against the
    oracle's recurrence on the oracle's prepared q, k (ragged T)."""
    inp, q, k = _raw(2, 2, 200, d, dtype, seed=35)
    S0 = workloads.decode_state(2, 2, d, d, std=0.1, seed=35)
    s = d ** -0.5
    o, S = dn.chunk_fwd(q.cuda(), k.cuda(), inp.v.cuda(), inp.beta.cuda(),
                        initial_state=S0.cuda(), qk_l2norm=True, scale=s)
    torch.cuda.synchronize()
    qp, kp = oracle.prepare_qk(q, k, scale=s, l2norm=True)
    o_ref, S_ref = oracle.forward(qp, kp, inp.v, inp.beta, S0)
    assert rel_l2(o.double().cpu().numpy(), o_ref) <= TOL[DT[dtype]]
    assert rel_l2(S.double().cpu().numpy(), S_ref) <= TOL[DT[dtype]]


def test_decode_step_with_normalisation_and_scale():
    B, H, d = 4, 3, 128
    inp, q, k = _raw(B, H, 1, d, "bf16", seed=36)
    S0 = workloads.decode_state(B, H, d, d, std=0.1, seed=36)
    Sg = S0.cuda()
    o = dn.recurrent_step(q[:, :, 0].contiguous().cuda(), k[:, :, 0].contiguous().cuda(),
                          inp.v[:, :, 0].contiguous().cuda(),
                          inp.beta[:, :, 0].contiguous().cuda(), Sg, qk_l2norm=True,
                          scale=d ** -0.5)
    torch.cuda.synchronize()
    qp, kp = oracle.prepare_qk(q[:, :, 0], k[:, :, 0], scale=d ** -0.5, l2norm=True)
    o_ref, S_ref = oracle.recurrent_step(qp, kp, inp.v[:, :, 0], inp.beta[:, :, 0], S0)
    assert rel_l2(o.double().cpu().numpy(), o_ref) <= TOL[torch.bfloat16]
    assert rel_l2(Sg.double().cpu().numpy(), S_ref) <= TOL[torch.bfloat16]


def test_gated_and_kda_forward_with_normalisation():
    B, H, T, d = 1, 2, 130, 128
    inp, q, k = _raw(B, H, T, d, "bf16", seed=37)
    g = workloads.gate_inputs(B, H, T, seed=37)
    qp, kp = oracle.prepare_qk(q, k, scale=d ** -0.5, l2norm=True)
    o, S = dn.chunk_fwd_gated(q.cuda(), k.cuda(), inp.v.cuda(), inp.beta.cuda(), g.cuda(),
                              qk_l2norm=True, scale=d ** -0.5)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_gated(qp, kp, inp.v, inp.beta, g)
    assert rel_l2(o.double().cpu().numpy(), o_ref) <= TOL[torch.bfloat16]
    assert rel_l2(S.double().cpu().numpy(), S_ref) <= TOL[torch.bfloat16]
    gk = g[..., None].expand(B, H, T, d).contiguous()
    o, S = dn.chunk_fwd_kda(q.cuda(), k.cuda(), inp.v.cuda(), inp.beta.cuda(), gk.cuda(),
                            qk_l2norm=True, scale=d ** -0.5)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_kda(qp, kp, inp.v, inp.beta, gk)
    assert rel_l2(o.double().cpu().numpy(), o_ref) <= TOL[torch.bfloat16]
    assert rel_l2(S.double().cpu().numpy(), S_ref) <= TOL[torch.bfloat16]


def test_full_size_rows_sampled():
    """The 1.3B-layer shape (B8 H16 T2048 d128, bf16; 2 x 262144 rows) in the
    launch configuration the bench times, checked on 4096 sampled rows of q
    and of k."""
    B, H, T, d = 8, 16, 2048, 128
    _, q, k = _raw(B, H, T, d, "bf16", seed=38)
    qo, ko = dn.qk_prepare(q.cuda(), k.cuda(), scale=d ** -0.5, l2norm=True)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.random.default_rng(38).choice(B * H * T, 4094, False),
                                     [0, B * H * T - 1]]))
    idx = torch.as_tensor(rows)
    q, k = q.view(-1, d), k.view(-1, d)
    q_ref, k_ref = oracle.prepare_qk(q[idx], k[idx], scale=d ** -0.5, l2norm=True)
    _check_elements(qo.view(-1, d).cpu()[idx], q_ref, "bf16")
    _check_elements(ko.view(-1, d).cpu()[idx], k_ref, "bf16")


def test_rejections():
    q = torch.zeros(4, 128, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(4, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(dn.DeltaNetError, match="UNSUPPORTED"):
        dn.qk_prepare(q[:, :96].contiguous(), k[:, :96].contiguous())
    with pytest.raises(dn.DeltaNetError, match="overlaps"):
        lib = dn.load()
        from delta_rule_recurrent_gb300._lib import check
        check(lib.dn_qk_prepare(q.data_ptr(), k.data_ptr(), k.data_ptr(), q.data_ptr(), 4, 128,
                                1, 1.0, 1e-6, 1, None))


def test_empty_tensors_are_a_no_op():
    z = torch.zeros(2, 3, 0, 128, dtype=torch.bfloat16, device="cuda")
    qo, ko = dn.qk_prepare(z, z, scale=0.5, l2norm=True)
    torch.cuda.synchronize()
    assert qo.shape == z.shape and ko.shape == z.shape
