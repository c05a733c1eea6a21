"""Chunkwise forward on the GPU against the fp64 oracle (through the C ABI).

Bars: relative L2 <= 1e-4 for fp32 I/O and <= 1e-2 for bf16 I/O, separately
on o and on the final state.  Full-size workloads are checked on every
(batch, head) pair and every 64-token chunk of o separately, each against
the oracle's full recurrence.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.conftest import rel_l2
from tests.gpu_util import TOL, check_every_head, dev, run_chunk

pytestmark = pytest.mark.gpu

ALGOS_BF16 = ["simt", "tcgen05", "tcgen05-fused"]


@pytest.fixture(autouse=True)
def no_device_error():
    """Every test must leave no device-side error recorded by a kernel."""
    from delta_rule_recurrent_gb300 import _lib
    lib = _lib.load()
    assert lib.dn_device_error() == 0
    yield
    assert lib.dn_device_error() == 0


def _check(o, S, o_ref, S_ref, dtype, what=""):
    eo, eS = rel_l2(o, o_ref), rel_l2(S, S_ref)
    assert eo <= TOL[dtype], f"{what} o rel L2 {eo:.3e}"
    assert eS <= TOL[dtype], f"{what} S_T rel L2 {eS:.3e}"
    return eo, eS


def test_tiny_fp32_workload():
    """B1 H2 T256 d64, fp32 I/O: the whole output and state."""
    inp = workloads.workload_inputs("tiny_fp32")
    o, S = run_chunk(inp)
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    _check(o, S, o_ref, S_ref, torch.float32, "tiny")


@pytest.mark.parametrize("algo", ["simt", "tcgen05", "auto"])
def test_recall_workload(algo):
    """B4 H4 T1024 d64 bf16 associative recall: oracle parity and the closed
    form (each re-queried key returns its stored value)."""
    inp, expect = workloads.workload_inputs("recall_bf16")
    o, S = run_chunk(inp, algo)
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    _check(o, S, o_ref, S_ref, torch.bfloat16, "recall")
    assert rel_l2(o, expect) <= 1e-2


@functools.lru_cache(maxsize=2)
def _oracle_workload(name):
    """The oracle's outputs for a full-size workload (every head), computed
    once per test session and shared by the kernels compared with it."""
    inp = workloads.workload_inputs(name)
    return inp, oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)


@pytest.mark.parametrize("algo", ALGOS_BF16)
def test_layer_1p3b_workload_every_head(algo):
    """B8 H16 T2048 d128 bf16 (the 1.3B-layer shape), full launch; all 128
    heads and all 4096 chunks held to the bar against the oracle.  At this
    size the persistent prepare kernel walks several work items per CTA."""
    inp, (o_ref, S_ref) = _oracle_workload("layer1p3b_bf16")
    o, S = run_chunk(inp, algo)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    check_every_head(o, S, o_ref, S_ref, TOL[torch.bfloat16], f"1.3B layer {algo}")


@pytest.mark.parametrize("algo", ALGOS_BF16 + ["split"])
def test_long_prefill_workload_every_head(algo):
    """B1 H16 T32768 d128 bf16 with an fp32 initial state; all 16 heads and
    all 512 chunks of each ("split": the sequence cut into as many runs as
    fill the GPU once, as the long-prefill benchmark runs it)."""
    inp, (o_ref, S_ref) = _oracle_workload("long_prefill_bf16")
    o, S = run_chunk(inp, algo)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    check_every_head(o, S, o_ref, S_ref, TOL[torch.bfloat16], f"long prefill {algo}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_shapes_and_ragged_tails(dtype, dk, dv, T):
    """Every supported (dk, dv), both dtypes, sequences shorter than, equal
    to and not a multiple of the 64-token chunk, with a carried state."""
    inp = workloads.chunk_inputs(2, 3, T, dk, dv, dtype=dtype, seed=T * 7 + dk + dv,
                                 s0_std=0.3)
    o, S = run_chunk(inp)
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    _check(o, S, o_ref, S_ref, inp.q.dtype, f"{dtype} dk{dk} dv{dv} T{T}")


@pytest.mark.parametrize("T", [1, 37, 64, 65, 200, 1000])
@pytest.mark.parametrize("with_s0", [False, True])
@pytest.mark.parametrize("algo", ["tcgen05", "tcgen05-fused"])
def test_tensor_core_path_ragged(T, with_s0, algo):
    """The tcgen05 kernels (two-pass and fused) on sequences shorter than,
    equal to and not a multiple of the chunk, with and without a carried
    state."""
    inp = workloads.chunk_inputs(3, 2, T, 128, 128, dtype="bf16", seed=100 + T,
                                 feature_map="silu", s0_std=0.1 if with_s0 else None)
    o, S = run_chunk(inp, algo)
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    _check(o, S, o_ref, S_ref, torch.bfloat16, f"{algo} T{T}")


@pytest.mark.parametrize("T", [1, 37, 64, 65, 200, 1000])
@pytest.mark.parametrize("with_s0", [False, True])
def test_tensor_core_path_64_wide_heads(T, with_s0):
    """dk = dv = 64 on the two-pass tcgen05 path (128-wide tiles whose second
    halves stay zero): ragged lengths, with and without a carried state, and
    the inputs prepared inside the kernels."""
    inp = workloads.chunk_inputs(3, 2, T, 64, 64, dtype="bf16", seed=300 + T,
                                 feature_map="silu", s0_std=0.2 if with_s0 else None)
    o, S = run_chunk(inp, "tcgen05")
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    _check(o, S, o_ref, S_ref, torch.bfloat16, f"d64 T{T}")
    raw = workloads.chunk_inputs(3, 2, T, 64, 64, dtype="bf16", seed=300 + T,
                                 feature_map="silu", s0_std=0.2 if with_s0 else None,
                                 normalize=False)
    import delta_rule_recurrent_gb300 as dn
    o2, S2 = dn.chunk_fwd(dev(raw.q), dev(raw.k), dev(raw.v), dev(raw.beta),
                          initial_state=dev(raw.S0), algo="tcgen05", qk_l2norm=True,
                          scale=0.125)
    torch.cuda.synchronize()
    qp, kp = oracle.prepare_qk(raw.q, raw.k, scale=0.125, l2norm=True)
    o_ref2, S_ref2 = oracle.forward(qp, kp, raw.v, raw.beta, raw.S0)
    _check(o2.double().cpu().numpy(), S2.double().cpu().numpy(), o_ref2, S_ref2,
           torch.bfloat16, f"d64 prepared T{T}")


def test_64_wide_heads_need_a_workspace_on_tensor_cores():
    """The fused tensor-core kernel covers 128-wide heads only: tcgen05 without
    a workspace is refused at d = 64, and auto falls back to the CUDA cores."""
    import delta_rule_recurrent_gb300 as dn
    inp = workloads.chunk_inputs(1, 2, 100, 64, 64, dtype="bf16", seed=5, s0_std=0.1)
    args = [dev(x) for x in (inp.q, inp.k, inp.v, inp.beta)]
    with pytest.raises(dn.DeltaNetError, match="UNSUPPORTED"):
        dn.chunk_fwd(*args, algo="tcgen05", workspace=None)
    o, S = dn.chunk_fwd(*args, initial_state=dev(inp.S0), algo="auto", workspace=None)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    _check(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref, torch.bfloat16,
           "d64 auto without workspace")


def test_split_and_fused_agree():
    """The two tensor-core forms differ only in how the triangular inverse is
    rounded (tf32 block merges in the prepare kernel, fp32 in the fused one)
    before both round it to bf16, so they agree with each other to the bf16
    bar and each meets it against the oracle."""
    inp = workloads.chunk_inputs(2, 4, 700, 128, 128, dtype="bf16", seed=404,
                                 feature_map="silu", s0_std=0.1)
    o1, S1 = run_chunk(inp, "tcgen05")
    o2, S2 = run_chunk(inp, "tcgen05-fused")
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    _check(o1, S1, o_ref, S_ref, torch.bfloat16, "split")
    _check(o2, S2, o_ref, S_ref, torch.bfloat16, "fused")
    assert rel_l2(o1, o2) <= TOL[torch.bfloat16] and rel_l2(S1, S2) <= TOL[torch.bfloat16]


def test_workspace_checks():
    """A short, misaligned or overlapping workspace is refused before any
    launch; NULL selects the fused kernel."""
    from delta_rule_recurrent_gb300 import _lib
    import delta_rule_recurrent_gb300 as dn
    inp = workloads.chunk_inputs(1, 2, 130, 128, 128, dtype="bf16", seed=9, feature_map="silu")
    q, k, v, b = (dev(x) for x in (inp.q, inp.k, inp.v, inp.beta))
    lib = _lib.load()
    need = lib.dn_chunk_fwd_workspace_bytes(1, 2, 130, 128, 128, 64, 1)
    assert need == 2 * 3 * (16384 + 1024)
    short = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.DeltaNetError, match="INVALID_ARG"):
        dn.chunk_fwd(q, k, v, b, workspace=short)
    big = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.DeltaNetError, match="INVALID_ARG"):
        dn.chunk_fwd(q, k, v, b, workspace=big[8:])
    buf = torch.empty(need // 2 + 2 * 130 * 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.DeltaNetError, match="INVALID_ARG"):  # workspace covers o
        dn.chunk_fwd(q, k, v, b, out=buf[: 2 * 130 * 128].view(1, 2, 130, 128),
                     workspace=buf.view(torch.uint8))
    o, S = dn.chunk_fwd(q, k, v, b, workspace=None)
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    torch.cuda.synchronize()
    _check(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref, torch.bfloat16)


@pytest.mark.parametrize("dk,dv,dtype", [(128, 64, "bf16"), (64, 128, "bf16"), (128, 128, "f32")])
def test_tensor_core_rejects_other_shapes(dk, dv, dtype):
    """The tcgen05 path covers bf16 with dk = dv in {64, 128}; asking for it
    on anything else is refused rather than run elsewhere."""
    from delta_rule_recurrent_gb300 import _lib
    inp = workloads.chunk_inputs(1, 1, 64, dk, dv, dtype=dtype, seed=1)
    with pytest.raises(_lib.DeltaNetError, match="UNSUPPORTED"):
        run_chunk(inp, "tcgen05")


def test_negative_eigenvalue_beta():
    """beta in (0, 2) through the chunk path."""
    inp = workloads.chunk_inputs(2, 2, 300, 128, 128, dtype="bf16", seed=77, beta_scale=2.0,
                                 s0_std=0.1)
    o, S = run_chunk(inp)
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    _check(o, S, o_ref, S_ref, torch.bfloat16, "beta in (0,2)")


def test_beta_zero_keeps_state_fp32():
    inp = workloads.chunk_inputs(1, 2, 130, 64, 64, dtype="f32", seed=3, s0_std=0.5)
    inp.beta.zero_()
    o, S = run_chunk(inp)
    assert rel_l2(S, inp.S0.double().numpy()) <= 1e-6
    o_ref = np.einsum("bhij,bhti->bhtj", inp.S0.double().numpy(), inp.q.double().numpy())
    assert rel_l2(o, o_ref) <= 1e-5


def test_zero_length_sequence_copies_state():
    import delta_rule_recurrent_gb300 as dn
    S0 = torch.randn(2, 3, 64, 64, device="cuda:0")
    q = torch.zeros(2, 3, 0, 64, device="cuda:0")
    beta = torch.zeros(2, 3, 0, device="cuda:0")
    o, S = dn.chunk_fwd(q, q, q, beta, initial_state=S0)
    torch.cuda.synchronize()
    assert o.shape == (2, 3, 0, 64) and torch.equal(S, S0)
    _, Sz = dn.chunk_fwd(q, q, q, beta)
    torch.cuda.synchronize()
    assert torch.count_nonzero(Sz) == 0


def test_state_updated_in_place_and_optional():
    import delta_rule_recurrent_gb300 as dn
    inp = workloads.chunk_inputs(1, 2, 100, 128, 128, dtype="bf16", seed=9, s0_std=0.2)
    o_ref, S_ref = oracle.forward(inp.q, inp.k, inp.v, inp.beta, inp.S0)
    S = dev(inp.S0)
    o, S_out = dn.chunk_fwd(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta),
                            initial_state=S, final_state=S)
    torch.cuda.synchronize()
    assert S_out.data_ptr() == S.data_ptr()
    _check(o.double().cpu().numpy(), S.double().cpu().numpy(), o_ref, S_ref, torch.bfloat16)
    o2, none = dn.chunk_fwd(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.beta),
                            initial_state=dev(inp.S0), output_final_state=False)
    torch.cuda.synchronize()
    assert none is None
    assert rel_l2(o2.double().cpu().numpy(), o_ref) <= 1e-2


def test_prefill_then_decode_handoff():
    """Chunk forward over a prefix, then decoding steps from its final state,
    equals the oracle over the whole sequence."""
    import delta_rule_recurrent_gb300 as dn
    full = workloads.chunk_inputs(2, 4, 150, 128, 128, dtype="bf16", seed=12)
    o_ref, S_ref = oracle.forward(full.q, full.k, full.v, full.beta, None)
    P = 140
    o_pre, S = dn.chunk_fwd(dev(full.q[:, :, :P].contiguous()), dev(full.k[:, :, :P].contiguous()),
                            dev(full.v[:, :, :P].contiguous()),
                            dev(full.beta[:, :, :P].contiguous()))
    outs = [o_pre]
    for t in range(P, 150):
        outs.append(dn.recurrent_step(dev(full.q[:, :, t].contiguous()),
                                      dev(full.k[:, :, t].contiguous()),
                                      dev(full.v[:, :, t].contiguous()),
                                      dev(full.beta[:, :, t].contiguous()), S)[:, :, None])
    torch.cuda.synchronize()
    o = torch.cat(outs, dim=2).double().cpu().numpy()
    _check(o, S.double().cpu().numpy(), o_ref, S_ref, torch.bfloat16, "handoff")


def test_rejects_bad_pointers_without_launching():
    from delta_rule_recurrent_gb300 import _lib
    lib = _lib.load()
    B, H, T, d = 1, 2, 64, 64
    q = torch.zeros(B, H, T, d, dtype=torch.bfloat16, device="cuda:0")
    beta = torch.zeros(B, H, T, dtype=torch.bfloat16, device="cuda:0")
    o = torch.zeros_like(q)
    host = torch.zeros_like(q, device="cpu")
    call = lambda qp, op: lib.dn_chunk_fwd(qp, q.data_ptr(), q.data_ptr(), beta.data_ptr(),
                                           None, op, None, B, H, T, d, d, 64, 1, None, 0, None)
    assert call(host.data_ptr(), o.data_ptr()) == _lib.DN_ERR_INVALID_ARG      # host memory
    assert call(q.data_ptr() + 2, o.data_ptr()) == _lib.DN_ERR_INVALID_ARG     # misaligned
    assert call(q.data_ptr(), q.data_ptr()) == _lib.DN_ERR_INVALID_ARG         # o aliases q
    assert call(None, o.data_ptr()) == _lib.DN_ERR_INVALID_ARG                 # NULL
    assert call(q.data_ptr(), o.data_ptr()) == _lib.DN_OK
    torch.cuda.synchronize()


def test_tensor_core_path_from_a_fresh_thread():
    """A thread that has made no CUDA runtime call has no current context;
    the library makes the device's primary context current before it
    encodes its tensor maps (through the driver), so the call works there."""
    import threading
    inp = workloads.chunk_inputs(1, 2, 130, 128, 128, dtype="bf16", seed=12, feature_map="silu")
    q, k, v, b = (dev(x) for x in (inp.q, inp.k, inp.v, inp.beta))
    o_main, S_main = dn_chunk(q, k, v, b)
    out = {}

    def worker():
        try:
            out["res"] = dn_chunk(q, k, v, b)
        except Exception as exc:  # reported below
            out["err"] = exc

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert "err" not in out, out.get("err")
    torch.cuda.synchronize()
    assert torch.equal(out["res"][0], o_main) and torch.equal(out["res"][1], S_main)


def dn_chunk(q, k, v, b):
    import delta_rule_recurrent_gb300 as dn
    o, S = dn.chunk_fwd(q, k, v, b, algo="tcgen05")
    torch.cuda.current_stream().synchronize()
    return o, S
