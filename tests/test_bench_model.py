"""The bench's cost model against the workload figures it reports against.

CPU only.  The chunk forward's algorithmic FLOPs and bytes per call on the
1.3B-layer shape (B8 H16 T2048 d128, bf16 I/O) and the decoding step's bytes
are the roofline numerators; these tests hold them to independently
tabulated values (FLOPs counted per matrix product of the chunk algebra, bytes
per tensor) and check which roof binds.
"""
import json
from pathlib import Path

import pytest

import bench

B, H, T, D, C = 8, 16, 2048, 128, 64


def _chunk_flops_by_product(C, dk, dv):
    """FLOPs per token and head, one term per product of the chunk algebra
    (a C x C triangle counted as half its square, 2 FLOPs per multiply-add),
    divided over the chunk's C tokens."""
    per_chunk = (
        C * C * dk            # A = tril(K K^T, -1): half of a C x C x dk product
        + C * C * dk          # P = tril(Q K^T): half of it
        + C ** 3 / 3          # the triangular solve (C^3 / 3 multiply-adds, x 2 / 2)
        + 2 * C * C * dk / 2  # W = T K (T lower triangular: half)
        + 2 * C * C * dv / 2  # U = T V (half)
        + 2 * C * dk * dv     # W S
        + 2 * C * dk * dv     # Q S
        + 2 * C * C * dv / 2  # P U' (P lower triangular: half)
        + 2 * C * dk * dv     # K^T U'
    )
    return per_chunk / C


def test_chunk_flops_match_the_product_count():
    assert bench.chunk_flops_per_token_head(C, D, D) == pytest.approx(
        _chunk_flops_by_product(C, D, D), rel=1e-12)
    total = bench.chunk_flops_per_token_head(C, D, D) * B * H * T
    assert total == pytest.approx(36.87e9, rel=1e-3)


def test_dense_tile_flops_count_the_triangles_in_full():
    """Every triangular product counted as its full square: A and P as full
    C x C x dk products, T K, T V and P U' as full C x C products; the
    solve's C^3/3 and the three dk x dv products as before."""
    per_chunk = (2 * C * C * D + 2 * C * C * D + C ** 3 / 3 + 2 * C * C * D + 2 * C * C * D
                 + 2 * C * D * D * 3 + 2 * C * C * D)
    assert bench.chunk_dense_flops_per_token_head(C, D, D) == pytest.approx(per_chunk / C,
                                                                           rel=1e-12)
    assert bench.chunk_dense_flops_per_token_head(C, D, D) * B * H * T == pytest.approx(
        47.6e9, rel=1e-3)


def test_chunk_bytes_count_each_tensor_once():
    q = k = B * H * T * D * 2
    v = o = B * H * T * D * 2
    beta = B * H * T * 2
    s_t = B * H * D * D * 4
    assert bench.chunk_bytes(B, H, T, D, D, 2, False, True) == q + k + v + o + beta + s_t
    assert bench.chunk_bytes(B, H, T, D, D, 2, False, True) == pytest.approx(277.3e6, rel=1e-3)


def test_decode_bytes_read_and_write_the_state_once():
    Bd = 256
    state = Bd * H * D * D * 4
    io = Bd * H * (2 * D + 2 * D + 1) * 2
    assert bench.decode_bytes(Bd, H, D, D, 2) == 2 * state + io
    assert bench.decode_bytes(Bd, H, D, D, 2) == pytest.approx(541.1e6, rel=1e-3)


def test_the_chunk_forward_is_bound_by_hbm():
    """Arithmetic intensity below the ridge of the measured peaks."""
    peaks, _ = bench.load_peaks()
    flops = bench.chunk_flops_per_token_head(C, D, D) * B * H * T
    nbytes = bench.chunk_bytes(B, H, T, D, D, 2, False, True)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    assert flops / nbytes < ridge


def test_traffic_table_entries_name_their_capture():
    """Each entry names its capture; one scaled from a smaller case says how."""
    table = json.loads((Path(bench.ROOT) / "profiles" / "traffic.json").read_text())
    for name, entry in table.items():
        assert set(entry) - {"scaled"} == {"bytes_per_launch", "source_sha", "capture"}, name
        assert (Path(bench.ROOT) / entry["capture"]).exists(), entry["capture"]
        assert entry["bytes_per_launch"] > 0


def test_varlen_packing_covers_every_token_once():
    """The bench's packed-sequence leg: 64 seeded lengths that tile the
    headline's B * T tokens per head exactly, none negative, the same for the
    same seed (so the bench and its full-size parity test pack alike)."""
    import workloads
    lens = workloads.varlen_lengths(64, B * T, seed=1002)
    assert len(lens) == 64 and sum(lens) == B * T and min(lens) >= 0
    assert lens == workloads.varlen_lengths(64, B * T, seed=1002)
    assert max(lens) > min(lens)  # ragged, not an even split
