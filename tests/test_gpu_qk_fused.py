"""q/k L2 normalisation and query scale inside the kernels (the ``*_qk``
entry points: ``qk_l2norm=`` / ``scale=`` on every forward and step), and the
preparation's gradient kernel (dn_qk_prepare_bwd), on the GPU against the
oracle.

The forms run on raw q and k; the oracle runs its recurrence on its own
fp64 preparation of them (``oracle.prepare_qk``), which the pages' layer
applies before its kernels (use_qk_l2norm_in_kernel).  Bars as everywhere:
relative L2 <= 1e-4 (fp32 I/O), <= 1e-2 (bf16 I/O), on every (batch, head).
"""
import numpy as np
import pytest
import torch

import delta_rule_recurrent_gb300 as dn
import oracle
import workloads
from tests.conftest import rel_l2
from tests.gpu_util import TOL, check_every_head

pytestmark = pytest.mark.gpu
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def no_device_error():
    lib = dn.load()
    assert lib.dn_device_error() == 0
    yield
    assert lib.dn_device_error() == 0


def _raw(B, H, T, d, dtype, seed, dv=None, s0=0.1):
    """Raw (unnormalised) silu features, as the 1.3B-layer recipe draws them
    before its L2 normalisation, with an initial state."""
    return workloads.chunk_inputs(B, H, T, d, dv or d, dtype=dtype, seed=seed,
                                  feature_map="silu", normalize=False, s0_std=s0)


def _np(t):
    return t.double().cpu().numpy()


FORMS = [  # (algo, workspace) of chunk_fwd
    ("tcgen05", "auto"),   # two passes: prepare kernel + scan
    ("tcgen05", None),     # one fused kernel
    ("simt", "auto"),      # CUDA cores
]


@pytest.mark.parametrize("algo,ws", FORMS, ids=["two-pass", "fused", "simt"])
@pytest.mark.parametrize("T", [1, 63, 65, 200, 700])
@pytest.mark.parametrize("l2norm,scale", [(True, 128 ** -0.5), (True, None), (False, 0.25)],
                         ids=["norm+scale", "norm", "scale"])
def test_plain_forward_prepares_in_kernel(algo, ws, T, l2norm, scale):
    """The scale alone is applied to normalised q, k (as the recipe draws
    them); unnormalised keys would make the recurrence itself unstable."""
    inp = _raw(2, 3, T, 128, "bf16", seed=500 + T) if l2norm else workloads.chunk_inputs(
        2, 3, T, 128, 128, dtype="bf16", seed=500 + T, feature_map="silu", s0_std=0.1)
    o, S = dn.chunk_fwd(*(x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta)),
                        initial_state=inp.S0.cuda(), algo=algo, workspace=ws,
                        qk_l2norm=l2norm, scale=scale)
    torch.cuda.synchronize()
    qp, kp = oracle.prepare_qk(inp.q, inp.k, 1.0 if scale is None else scale, l2norm)
    o_ref, S_ref = oracle.forward(qp, kp, inp.v, inp.beta, inp.S0)
    check_every_head(_np(o), _np(S), o_ref, S_ref, TOL[torch.bfloat16], f"{algo} {ws} T{T}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_cuda_core_forward_every_shape(dtype, dk, dv):
    inp = workloads.chunk_inputs(2, 2, 130, dk, dv, dtype=dtype, seed=dk + dv,
                                 feature_map="silu", normalize=False, s0_std=0.2)
    o, S = dn.chunk_fwd(*(x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta)),
                        initial_state=inp.S0.cuda(), algo="simt", qk_l2norm=True,
                        scale=dk ** -0.5)
    torch.cuda.synchronize()
    qp, kp = oracle.prepare_qk(inp.q, inp.k, dk ** -0.5, True)
    o_ref, S_ref = oracle.forward(qp, kp, inp.v, inp.beta, inp.S0)
    check_every_head(_np(o), _np(S), o_ref, S_ref, TOL[DT[dtype]], f"simt {dtype} {dk}x{dv}")


def test_in_kernel_preparation_against_the_separate_pass():
    """The separate pass rounds the prepared rows to bf16 before the
    recurrence; inside the kernels the products of the raw rows are scaled
    in fp32 instead (and only the scan's k rows are rounded after scaling).
    Both routes meet the bar against the oracle and agree with each other to
    it, and neither touches q or k in memory."""
    inp = _raw(2, 4, 500, 128, "bf16", seed=41)
    q, k, v, b, S0 = (x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta, inp.S0))
    o1, S1 = dn.chunk_fwd(q, k, v, b, initial_state=S0, qk_l2norm=True, scale=0.125)
    qp, kp = dn.qk_prepare(q, k, scale=0.125, l2norm=True)
    o2, S2 = dn.chunk_fwd(qp, kp, v, b, initial_state=S0)
    torch.cuda.synchronize()
    qo, ko = oracle.prepare_qk(inp.q, inp.k, 0.125, True)
    o_ref, S_ref = oracle.forward(qo, ko, inp.v, inp.beta, inp.S0)
    bar = TOL[torch.bfloat16]
    for o, S in ((o1, S1), (o2, S2)):
        check_every_head(_np(o), _np(S), o_ref, S_ref, bar, "route")
    assert rel_l2(_np(o1), _np(o2)) <= bar and rel_l2(_np(S1), _np(S2)) <= bar
    assert torch.equal(q, inp.q.cuda()) and torch.equal(k, inp.k.cuda())  # inputs untouched


def test_layer_1p3b_every_head_with_normalisation():
    """The 1.3B-layer call (B8 H16 T2048 d128, bf16) on raw silu features with
    the normalisation and 1/sqrt(d) scale inside the two-pass kernels (the
    bench's qk_l2norm leg): every head and chunk against the oracle."""
    inp = workloads.workload_inputs("layer1p3b_bf16", normalize=False)
    s = 128 ** -0.5
    o, S = dn.chunk_fwd(*(x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta)),
                        qk_l2norm=True, scale=s)
    torch.cuda.synchronize()
    qp, kp = oracle.prepare_qk(inp.q, inp.k, s, True)
    o_ref, S_ref = oracle.forward(qp, kp, inp.v, inp.beta, inp.S0)
    check_every_head(_np(o), _np(S), o_ref, S_ref, TOL[torch.bfloat16], "1.3B qk_l2norm")


@pytest.mark.parametrize("ws", ["auto", None], ids=["tcgen05", "cuda-cores"])
def test_gated_forward_prepares_in_kernel(ws):
    inp = _raw(2, 2, 300, 128, "bf16", seed=42)
    g = workloads.gate_inputs(2, 2, 300, seed=42, lo=0.5)
    o, S = dn.chunk_fwd_gated(*(x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta, g)),
                              initial_state=inp.S0.cuda(), workspace=ws, qk_l2norm=True,
                              scale=128 ** -0.5)
    torch.cuda.synchronize()
    qp, kp = oracle.prepare_qk(inp.q, inp.k, 128 ** -0.5, True)
    o_ref, S_ref = oracle.forward_gated(qp, kp, inp.v, inp.beta, g, inp.S0)
    check_every_head(_np(o), _np(S), o_ref, S_ref, TOL[torch.bfloat16], f"gated {ws}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_kda_forward_prepares_in_kernel(dtype):
    inp = _raw(1, 3, 200, 128, dtype, seed=43)
    g = workloads.gate_inputs(1, 3, 200, seed=43, lo=0.7, channels=128)
    o, S = dn.chunk_fwd_kda(*(x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta, g)),
                            initial_state=inp.S0.cuda(), qk_l2norm=True, scale=128 ** -0.5)
    torch.cuda.synchronize()
    qp, kp = oracle.prepare_qk(inp.q, inp.k, 128 ** -0.5, True)
    o_ref, S_ref = oracle.forward_kda(qp, kp, inp.v, inp.beta, g, inp.S0)
    check_every_head(_np(o), _np(S), o_ref, S_ref, TOL[DT[dtype]], f"kda {dtype}")


@pytest.mark.parametrize("ws", ["auto", None], ids=["tcgen05", "cuda-cores"])
def test_varlen_forward_prepares_in_kernel(ws):
    H, d = 2, 128
    lens = [5, 64, 130, 0, 77]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    inp = _raw(1, H, T, d, "bf16", seed=44)
    q, k, v, b = (x[0] for x in (inp.q, inp.k, inp.v, inp.beta))
    o, S = dn.chunk_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), b.cuda(), cu, workspace=ws,
                               qk_l2norm=True, scale=d ** -0.5)
    torch.cuda.synchronize()
    qp, kp = oracle.prepare_qk(q, k, d ** -0.5, True)
    o_ref, S_ref = oracle.forward_varlen(qp, kp, v, b, cu)
    assert rel_l2(_np(o), o_ref) <= TOL[torch.bfloat16]
    assert rel_l2(_np(S), S_ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("form", ["plain", "gated", "kda"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_steps_prepare_in_kernel(form, dtype):
    """Twelve chained steps on raw q, k with the normalisation and scale
    inside the step kernel."""
    B, H, d, steps, seed = 4, 3, 128, 12, 45
    S0 = workloads.decode_state(B, H, d, d, std=0.1, seed=seed)
    S = S0.cuda()
    rec = {n: [] for n in ("q", "k", "v", "beta", "g", "o")}
    for t in range(steps):
        x = workloads.decode_step_inputs(B, H, d, d, step=t, dtype=dtype, seed=seed,
                                         normalize=False)
        g = workloads.gate_inputs(B, H, seed=seed + t, lo=0.8,
                                  channels=d if form == "kda" else None)
        args = [x.q.cuda(), x.k.cuda(), x.v.cuda(), x.beta.cuda()]
        if form == "plain":
            o = dn.recurrent_step(*args, S, qk_l2norm=True, scale=d ** -0.5)
        elif form == "gated":
            o = dn.recurrent_step_gated(*args, g.cuda(), S, qk_l2norm=True, scale=d ** -0.5)
        else:
            o = dn.recurrent_step_kda(*args, g.cuda(), S, qk_l2norm=True, scale=d ** -0.5)
        for n in ("q", "k", "v", "beta"):
            rec[n].append(getattr(x, n))
        rec["g"].append(g)
        rec["o"].append(o.cpu())
    torch.cuda.synchronize()
    st = {n: torch.stack(v_, dim=2) for n, v_ in rec.items()}
    qp, kp = oracle.prepare_qk(st["q"], st["k"], d ** -0.5, True)
    if form == "plain":
        o_ref, S_ref = oracle.forward(qp, kp, st["v"], st["beta"], S0)
    elif form == "gated":
        o_ref, S_ref = oracle.forward_gated(qp, kp, st["v"], st["beta"], st["g"], S0)
    else:
        o_ref, S_ref = oracle.forward_kda(qp, kp, st["v"], st["beta"], st["g"], S0)
    check_every_head(_np(st["o"]), _np(S), o_ref, S_ref, TOL[DT[dtype]], f"{form} steps")


def _grad_bound(x, dy, ref, scale, d, dtype):
    """Elementwise bound on the preparation's gradient: fp32 error in the row
    reductions and the products, relative to the magnitudes that enter each
    element (a difference of two terms can cancel), plus one rounding of the
    result to bf16."""
    n2 = (x * x).sum(-1, keepdims=True) + 1e-6
    c = (x * dy).sum(-1, keepdims=True) / n2
    mag = np.abs(scale) / np.sqrt(n2) * (np.abs(dy) + np.abs(x) * np.abs(c))
    bound = (2 * d + 16) * 2.0 ** -24 * mag
    if dtype == "bf16":
        bound = bound + 2.0 ** -8 * np.abs(ref)
    return bound + 1e-30


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("l2norm", [True, False])
def test_prepare_gradient_matches_the_oracle_elementwise(dtype, d, l2norm):
    """dn_qk_prepare_bwd on 3 x 257 rows (ragged against the kernel's 8 rows
    per block) against the oracle's gradient of the preparation."""
    inp = _raw(1, 3, 257, d, dtype, seed=46)
    dq_out, dk_out = (torch.randn(inp.q.shape, generator=torch.Generator().manual_seed(s))
                      .to(inp.q.dtype) for s in (1, 2))
    s = d ** -0.5
    dq, dk = dn.qk_prepare_bwd(inp.q.cuda(), inp.k.cuda(), dq_out.cuda(), dk_out.cuda(),
                               scale=s, l2norm=l2norm)
    torch.cuda.synchronize()
    gq, gk = oracle.prepare_qk_backward(inp.q, inp.k, dq_out, dk_out, s, l2norm)
    for got, ref, x, dy, sc in ((dq, gq, inp.q, dq_out, s), (dk, gk, inp.k, dk_out, 1.0)):
        if not l2norm and got is not None and sc == 1.0:
            assert torch.equal(got.cpu(), dk_out)  # k passes through untouched
            continue
        x64, dy64 = x.double().numpy(), dy.double().numpy()
        # without the normalisation: the fp32 scale and the product, two roundings
        bound = _grad_bound(x64, dy64, ref, sc, d, dtype) if l2norm else (
            ((2.0 ** -8 if dtype == "bf16" else 0.0) + 4 * 2.0 ** -24) * np.abs(ref) + 1e-30)
        err = np.abs(_np(got) - ref)
        assert (err <= bound).all(), f"{(err > bound).sum()} elements off"


def test_prepare_gradient_in_place():
    inp = _raw(2, 2, 65, 128, "bf16", seed=47)
    dq_out = torch.randn(inp.q.shape).to(torch.bfloat16).cuda()
    dk_out = torch.randn(inp.q.shape).to(torch.bfloat16).cuda()
    q, k = inp.q.cuda(), inp.k.cuda()
    dq, dk = dn.qk_prepare_bwd(q, k, dq_out, dk_out, scale=0.5, l2norm=True)
    lib = dn.load()
    from delta_rule_recurrent_gb300._lib import check
    rows = q.numel() // 128
    check(lib.dn_qk_prepare_bwd(q.data_ptr(), k.data_ptr(), dq_out.data_ptr(), dk_out.data_ptr(),
                                dq_out.data_ptr(), dk_out.data_ptr(), rows, 128, 1, 0.5, 1e-6, 1,
                                torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert torch.equal(dq, dq_out) and torch.equal(dk, dk_out)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_autograd_through_the_normalisation(dtype, d):
    """DeltaRule.apply(..., scale, qk_l2norm=True) on raw q, k: the forward
    matches the oracle on the prepared inputs and every gradient matches the
    oracle's recurrence gradient chained through its preparation gradient."""
    inp = _raw(1, 2, 130, d, dtype, seed=48, s0=0.1)
    d_o, d_S = workloads.grad_inputs(1, 2, 130, d, d, dtype=dtype, seed=48, ds_std=0.1)
    s = d ** -0.5
    leaves = [x.cuda().requires_grad_() for x in (inp.q, inp.k, inp.v, inp.beta, inp.S0)]
    o, S_T = dn.DeltaRule.apply(*leaves, s, True)
    torch.autograd.backward([o, S_T], [d_o.cuda(), d_S.cuda()])
    qp, kp = oracle.prepare_qk(inp.q, inp.k, s, True)
    o_ref, _ = oracle.forward(qp, kp, inp.v, inp.beta, inp.S0)
    assert rel_l2(_np(o.detach()), o_ref) <= TOL[DT[dtype]]
    ref = list(oracle.backward(qp, kp, inp.v, inp.beta, d_o, inp.S0, d_S))
    ref[0], ref[1] = oracle.prepare_qk_backward(inp.q, inp.k, ref[0], ref[1], s, True)
    for name, leaf, want in zip(("d_q", "d_k", "d_v", "d_beta", "d_S0"), leaves, ref):
        e = rel_l2(_np(leaf.grad), want)
        assert e <= TOL[DT[dtype]], f"{name} rel L2 {e:.3e}"


def test_rejects_a_bad_norm_before_any_launch():
    import ctypes
    from delta_rule_recurrent_gb300._lib import QkNorm
    lib = dn.load()
    q = torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(1, 1, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    for bad in (QkNorm(1, float("nan"), 1e-6), QkNorm(1, 1.0, -1.0), QkNorm(0, float("inf"), 0)):
        st = lib.dn_chunk_fwd_qk(q.data_ptr(), q.data_ptr(), q.data_ptr(), b.data_ptr(), None,
                                 o.data_ptr(), None, 1, 1, 64, 128, 128, 64, 1, None, 0, None, 0,
                                 ctypes.byref(bad))
        assert st == dn._lib.DN_ERR_INVALID_ARG
