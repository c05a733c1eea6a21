"""The C-ABI library loads and exports what include/deltanet.h declares.

CPU only: nothing here launches a kernel.  The argument checks exercised
return before the library makes any CUDA call.
"""
import ctypes
import re
import subprocess

import pytest

import delta_rule_recurrent_gb300 as dn
from delta_rule_recurrent_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_boundary():
    names = _lib.header_symbols()
    for required in ("dn_chunk_fwd", "dn_recurrent_step", "dn_status_string",
                     "dn_last_error"):
        assert required in names
    assert set(names) == set(_lib.SIGNATURES), "binding signatures drift from the header"


def test_binding_argument_counts_match_the_header():
    """Each ctypes signature has as many parameters as the header's
    declaration (a miscount would shift every later argument)."""
    text = _lib.HEADER.read_text()
    for name, (_res, args) in _lib.SIGNATURES.items():
        m = re.search(r"DN_API\s+[\w\s\*]*?\b" + name + r"\s*\(([^)]*)\)", text)
        assert m, name
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(params) == len(args), f"{name}: header {len(params)}, binding {len(args)}"


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", str(_lib.lib_path())],
                         check=True, capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in _lib.header_symbols():
        assert name in exported, f"{name} declared but not exported"
        assert getattr(lib, name) is not None


def test_abi_version_and_status_strings(lib):
    assert lib.dn_abi_version() == 9
    assert lib.dn_status_string(0) == b"DN_OK"
    assert lib.dn_status_string(1) == b"DN_ERR_INVALID_ARG"
    assert lib.dn_status_string(2) == b"DN_ERR_UNSUPPORTED"
    assert lib.dn_status_string(3) == b"DN_ERR_CUDA"
    assert lib.dn_status_string(99) == b"DN_UNKNOWN_STATUS"


def test_workspace_bytes(lib):
    """The tensor-core path (bf16, dk = dv = 128 or 64, C = 64) asks for one
    16 KB [PT; Tm] tile and 1 KB of side vectors per (batch, head, chunk);
    every other case needs none."""
    f = lib.dn_chunk_fwd_workspace_bytes
    # one 16 KB [PT; T] tile and 1 KB of row factors (prepared inputs) per chunk
    assert f(8, 16, 2048, 128, 128, 64, 1) == 8 * 16 * 32 * (16384 + 1024)
    assert f(1, 2, 130, 128, 128, 64, 1) == 2 * 3 * (16384 + 1024)
    assert f(1, 1, 1, 128, 128, 64, 1) == 16384 + 1024
    assert f(1, 1, 0, 128, 128, 64, 1) == 0
    assert f(0, 4, 64, 128, 128, 64, 1) == 0
    assert f(8, 16, 2048, 128, 128, 64, 0) == 0  # fp32 I/O
    assert f(8, 16, 2048, 64, 64, 64, 1) == 8 * 16 * 32 * (16384 + 1024)  # d = 64, same tiles
    assert f(8, 16, 2048, 128, 64, 64, 1) == 0
    assert f(8, 16, 2048, 128, 128, 32, 1) == 0  # other chunk length


def test_gated_workspace_bytes(lib):
    """The gated tensor-core form needs two 16 KB tiles and 1 KB of fp32
    decay factors per chunk; where that form does not apply it needs none."""
    f = lib.dn_chunk_fwd_gated_workspace_bytes
    assert f(8, 16, 2048, 128, 128, 64, 1) == 8 * 16 * 32 * (2 * 16384 + 1024)
    assert f(1, 2, 130, 128, 128, 64, 1) == 2 * 3 * 33792
    assert f(1, 1, 0, 128, 128, 64, 1) == 0
    assert f(8, 16, 2048, 128, 128, 64, 0) == 0
    assert f(8, 16, 2048, 64, 128, 64, 1) == 0
    assert f(8, 16, 2048, 128, 128, 32, 1) == 0


def test_kda_workspace_bytes(lib):
    """The KDA tensor-core form needs, per chunk, a 16 KB [PT; Tm] tile and
    1 KB of side vectors, four bf16 [B, H, T, 128] operands (K . exp G,
    Q . exp G, K . exp(G_C - G), K . exp(-G)), and a list of the chunks past
    the separable range (a count and one int per chunk, rounded up to 256
    bytes); elsewhere none."""
    f = lib.dn_chunk_fwd_kda_workspace_bytes

    def size(BH, T):
        chunks = BH * ((T + 63) // 64)
        return chunks * (16384 + 1024) + 4 * BH * T * 256 + -(-(chunks + 1) * 4 // 256) * 256

    assert f(8, 16, 2048, 128, 128, 64, 1) == size(128, 2048)
    assert f(1, 2, 130, 128, 128, 64, 1) == size(2, 130)
    assert size(2, 130) == 2 * (3 * (16384 + 1024) + 4 * 130 * 256) + 256
    assert f(1, 1, 0, 128, 128, 64, 1) == 0
    assert f(8, 16, 2048, 128, 128, 64, 0) == 0
    assert f(8, 16, 2048, 64, 64, 64, 1) == 0


def test_kda_backward_workspace_bytes(lib):
    """KDA's backward keeps the fp32 state and state gradient of every chunk,
    plus the tensor-core forward's scratch where it recomputes the states;
    invalid arguments need none."""
    f = lib.dn_chunk_bwd_kda_workspace_bytes
    tc = lib.dn_chunk_fwd_kda_workspace_bytes(8, 16, 2048, 128, 128, 64, 1)
    assert tc > 0
    assert f(8, 16, 2048, 128, 128, 64, 1) == 2 * 8 * 16 * 32 * 128 * 128 * 4 + tc
    assert f(8, 16, 2048, 128, 128, 64, 0) == 2 * 8 * 16 * 32 * 128 * 128 * 4
    assert f(1, 2, 130, 64, 128, 64, 0) == 2 * 2 * 3 * 64 * 128 * 4
    assert f(1, 1, 0, 128, 128, 64, 1) == 0
    assert f(1, 1, 64, 96, 128, 64, 1) == 0
    assert f(1, 1, 64, 128, 128, 32, 1) == 0


def test_gated_backward_workspace_bytes(lib):
    """The gated backward keeps the fp32 state and state gradient of every
    chunk; for bf16 with d = 128 also the tensor-core KDA forward's scratch
    (256-byte aligned) and the rates on every key channel."""
    f = lib.dn_chunk_bwd_gated_workspace_bytes
    states = 2 * 8 * 16 * 32 * 128 * 128 * 4
    kda = lib.dn_chunk_fwd_kda_workspace_bytes(8, 16, 2048, 128, 128, 64, 1)
    assert f(8, 16, 2048, 128, 128, 64, 1) == states + (kda + 255) // 256 * 256 + 8 * 16 * 2048 * 128 * 4
    assert f(8, 16, 2048, 128, 128, 64, 0) == states
    assert f(1, 2, 130, 64, 64, 64, 1) == 2 * 2 * 3 * 64 * 64 * 4
    assert f(1, 1, 0, 128, 128, 64, 1) == 0


def test_kda_backward_rejects_a_short_workspace_before_any_cuda_call(lib):
    need = lib.dn_chunk_bwd_kda_workspace_bytes(1, 2, 130, 64, 64, 64, 0)
    st = lib.dn_chunk_bwd_kda(*([None] * 14), 1, 2, 130, 64, 64, 64, 0,
                              ctypes.c_void_p(4096), need - 1, None)
    assert st == _lib.DN_ERR_INVALID_ARG
    assert b"workspace" in lib.dn_last_error()


def test_gated_rejects_a_short_workspace_before_any_cuda_call(lib):
    need = lib.dn_chunk_fwd_gated_workspace_bytes(1, 2, 130, 128, 128, 64, 1)
    st = lib.dn_chunk_fwd_gated(None, None, None, None, None, None, None, None, 1, 2, 130,
                                128, 128, 64, 1, ctypes.c_void_p(4096), need - 1, None)
    assert st == _lib.DN_ERR_INVALID_ARG
    assert b"workspace" in lib.dn_last_error()


def _chunk(lib, B=1, H=1, T=64, dk=64, dv=64, C=64, dt=1, algo=0):
    return lib.dn_chunk_fwd_algo(None, None, None, None, None, None, None, B, H, T, dk, dv,
                                 C, dt, None, 0, None, algo)


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), _lib.DN_ERR_INVALID_ARG),
    (dict(T=-5), _lib.DN_ERR_INVALID_ARG),
    (dict(dt=7), _lib.DN_ERR_INVALID_ARG),
    (dict(algo=9), _lib.DN_ERR_INVALID_ARG),
    (dict(dk=0), _lib.DN_ERR_INVALID_ARG),
    (dict(dk=96), _lib.DN_ERR_UNSUPPORTED),
    (dict(dv=256), _lib.DN_ERR_UNSUPPORTED),
    (dict(C=32), _lib.DN_ERR_UNSUPPORTED),
    (dict(B=0), _lib.DN_OK),
    (dict(H=0, T=100), _lib.DN_OK),
])
def test_chunk_argument_checks_before_cuda(lib, kw, status):
    assert _chunk(lib, **kw) == status
    if status != _lib.DN_OK:
        assert lib.dn_last_error()  # a detail message is set


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), _lib.DN_ERR_INVALID_ARG),
    (dict(dt=3), _lib.DN_ERR_INVALID_ARG),
    (dict(dk=32), _lib.DN_ERR_UNSUPPORTED),
    (dict(B=0), _lib.DN_OK),
])
def test_decode_argument_checks_before_cuda(lib, kw, status):
    a = dict(B=2, H=2, dk=128, dv=128, dt=1)
    a.update(kw)
    assert lib.dn_recurrent_step(None, None, None, None, None, None, a["B"], a["H"], a["dk"],
                                 a["dv"], a["dt"], None) == status


def test_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 4, 64)
    with pytest.raises(ValueError):
        dn.chunk_fwd(q, q, q, torch.zeros(1, 1, 4))


def test_check_raises_with_detail(lib):
    _chunk(lib, dk=96)
    with pytest.raises(dn.DeltaNetError, match="UNSUPPORTED"):
        _lib.check(_lib.DN_ERR_UNSUPPORTED)


def test_last_error_is_per_thread(lib):
    import threading
    _chunk(lib, dk=96)
    seen = {}

    def other():
        seen["msg"] = lib.dn_last_error()
    th = threading.Thread(target=other)
    th.start()
    th.join()
    assert seen["msg"] == b""
    assert lib.dn_last_error() != b""


def test_noalloc_entry_point_rejects_before_any_cuda_call(lib):
    """dn_chunk_fwd_noalloc refuses shapes it does not cover and problems
    larger than its static scratch (DN_NOALLOC_MAX_TILES chunk tiles) from
    the sizes alone, before touching a pointer or the device."""
    f = lib.dn_chunk_fwd_noalloc
    null = [None] * 7

    def call(B, H, T, dk=128, dv=128, C=64, dt=1):
        return f(*null, B, H, T, dk, dv, C, dt, None)

    assert call(1, 8, 64 * 65) == _lib.DN_ERR_INVALID_ARG  # 520 tiles > 512
    assert b"512" in lib.dn_last_error()
    assert call(1, 8, 64 * 64 + 1) == _lib.DN_ERR_INVALID_ARG  # a ragged tail counts as a tile
    assert call(1, 1, 64, dt=0) == _lib.DN_ERR_UNSUPPORTED
    assert call(1, 1, 64, dk=64, dv=64) == _lib.DN_ERR_UNSUPPORTED
    assert call(1, 1, 64, C=32) == _lib.DN_ERR_UNSUPPORTED
    assert call(-1, 1, 64) == _lib.DN_ERR_INVALID_ARG
    assert call(0, 4, 64) == _lib.DN_OK  # nothing to do, nothing touched


def test_varlen_rejects_bad_offsets_before_any_cuda_call(lib):
    """cu_seqlens is checked on the host first: it must run from 0 to T
    without decreasing, with 0 < N <= DN_MAX_VARLEN_SEQS."""
    f = lib.dn_chunk_fwd_varlen
    null = [None] * 7

    def call(cu, N, T, H=2):
        arr = (ctypes.c_int * len(cu))(*cu)
        return f(*null, arr, N, H, T, 128, 128, 64, 1, None, 0, None)

    assert call([0, 5, 3, 9], 3, 9) == _lib.DN_ERR_INVALID_ARG  # decreases
    assert call([1, 5, 9], 2, 9) == _lib.DN_ERR_INVALID_ARG     # does not start at 0
    assert call([0, 5, 8], 2, 9) == _lib.DN_ERR_INVALID_ARG     # does not end at T
    assert call([0] * 1026, 1025, 0) == _lib.DN_ERR_INVALID_ARG  # too many sequences
    assert b"1024" in lib.dn_last_error()
    size = lib.dn_chunk_fwd_varlen_workspace_bytes
    arr = (ctypes.c_int * 4)(0, 65, 65, 100)
    assert size(arr, 3, 2, 128, 128, 64, 1) == 2 * (2 + 0 + 1) * (16384 + 1024)
    assert size(arr, 3, 2, 64, 64, 64, 1) == 0


def test_qk_prepare_rejects_before_any_cuda_call(lib):
    """dn_qk_prepare checks its sizes, dtype, scale and eps on the host
    first; an empty problem is a no-op that touches nothing."""
    f = lib.dn_qk_prepare
    null = [None] * 4

    def call(rows=8, d=128, normalize=1, scale=1.0, eps=1e-6, dt=1):
        return f(*null, rows, d, normalize, scale, eps, dt, None)

    assert call(rows=-1) == _lib.DN_ERR_INVALID_ARG
    assert call(dt=7) == _lib.DN_ERR_INVALID_ARG
    assert call(d=0) == _lib.DN_ERR_INVALID_ARG
    assert call(d=96) == _lib.DN_ERR_UNSUPPORTED
    assert call(scale=float("inf")) == _lib.DN_ERR_INVALID_ARG
    assert call(scale=float("nan")) == _lib.DN_ERR_INVALID_ARG
    assert call(eps=-1e-6) == _lib.DN_ERR_INVALID_ARG
    assert b"eps" in lib.dn_last_error()
    assert call(rows=0) == _lib.DN_OK
    assert call(rows=0, normalize=0) == _lib.DN_OK
