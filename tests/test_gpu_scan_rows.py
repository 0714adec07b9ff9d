"""Batched (per-row) scans against the CPU oracle: int32/uint32 bit-exact,
fp32 within the normalised bound, with the normaliser taken per row."""

from __future__ import annotations

import functools

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import FP32_TOL, Guarded, assert_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import stream_compaction_pass_gb300 as m
    return m


@functools.lru_cache(maxsize=None)
def rows_input(kind: str, rows: int, cols: int) -> np.ndarray:
    n = rows * cols
    if kind == "i32":
        return si.uniform_int32(n, -1000, 1000, seed=80).reshape(rows, cols)
    if kind == "u32":
        return si.uniform_u32(n, seed=81).reshape(rows, cols)
    return si.uniform_f32(n, seed=82).reshape(rows, cols)  # probabilities-like, in [0, 1)


def run_rows(ss, kind, inclusive, x, offset=0, inplace=False):
    rows, cols = x.shape
    src = Guarded(rows * cols, offset, fill=x.reshape(-1))
    dst = src if inplace else Guarded(rows * cols, offset)
    dt = {"i32": ss.SS_I32, "u32": ss.SS_U32, "f32": ss.SS_F32}[kind]
    ss.ss_scan_rows(dt, inclusive, src.view, dst.view, rows, cols)
    st, tile = ss.ss_stream_status()
    assert st == ss.SS_OK, f"device status {st} at tile {tile}"
    assert dst.guards_intact(), "a store landed outside the output"
    np_dt = {"i32": np.int32, "u32": np.uint32, "f32": np.float32}[kind]
    return dst.numpy(np_dt).reshape(rows, cols).copy()


def check(ss, kind, inclusive, x, **kw):
    got = run_rows(ss, kind, inclusive, x, **kw)
    ref = oracle.scan_rows(x, inclusive)
    if kind != "f32":
        assert_equal(got.reshape(-1), ref.reshape(-1), tile=x.shape[1])
        return
    norm = np.maximum(1.0, oracle.abs_prefix_rows_f32(x))
    err = float(np.max(np.abs(got.astype(np.float64) - ref) / norm))
    assert err <= FP32_TOL, f"normalised fp32 error {err:.3e}"


SHAPES = [(1, 1), (1, 5), (3, 7), (1000, 1), (17, 128), (5, 2047), (5, 2048), (5, 2049), (3, 4096),
          (3, 4097), (100, 4095), (64, 32000), (4, 128256), (2, 1_000_003), (1000, 100), (4096, 256),
          # persistent long-row kernel: one tile per row, a short last tile, many rows per CTA;
          # its tile is chosen from the row length: 10240 (20000), 14336 (40000, 27000),
          # 16384 (32000, 49152) or 18432 (16388, 32772, 128256, 2^20) elements
          (3, 16384), (5, 16388), (7, 32772), (1, 1 << 20), (300, 20000), (153, 16384 * 3),
          (5, 40000), (11, 27000),
          # rows of at most 64 elements, several to a warp (lanes per row 1, 2, 4, 8, 16),
          # lengths that are and are not multiples of 4, row counts that leave a warp's
          # last group short
          (5001, 4), (3001, 3), (2001, 8), (999, 17), (1000, 33), (777, 64), (4097, 61), (70001, 2),
          # rows of 65-224 elements take one step each with two vectors per lane; 225 and
          # longer go back to one warp per row
          (2001, 65), (999, 128), (1001, 129), (777, 200), (501, 224), (502, 225), (333, 250),
          (1000, 255)]


@pytest.mark.parametrize("kind", ["i32", "u32", "f32"])
@pytest.mark.parametrize("inclusive", [True, False])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"{r}x{c}" for r, c in SHAPES])
def test_shapes(ss, kind, inclusive, shape):
    check(ss, kind, inclusive, rows_input(kind, *shape))


@pytest.mark.parametrize("shape", [(512, 128256), (262144, 256), (3, (1 << 21) + 5)],
                         ids=["topp_512x128256", "short_262144x256", "long_rows_as_flat_scans"])
def test_bench_shapes(ss, shape):
    check(ss, "f32", True, rows_input("f32", *shape))
    check(ss, "i32", False, rows_input("i32", *shape))


# (333, 100), (257, 224), (300, 160), (301, 65), (129, 128): the one-step kernel with two
# 16-byte vectors per lane (rows of 65-224 elements), whose per-vector bounds and the
# scalar path of a misaligned base need their own cases.
@pytest.mark.parametrize("shape", [(9, 5000), (33, 300), (7, 2051), (5, 40000), (1001, 20), (513, 64),
                                   (333, 100), (257, 224), (301, 65), (129, 128)])
@pytest.mark.parametrize("offset", [1, 3])
def test_unaligned(ss, shape, offset):
    check(ss, "i32", True, rows_input("i32", *shape), offset=offset)


@pytest.mark.parametrize("shape", [(6, 9000), (300, 64), (9, 50000), (300, 160), (257, 224), (333, 100)])
def test_in_place(ss, shape):
    check(ss, "i32", False, rows_input("i32", *shape), inplace=True)


def test_structured_fp32_rows_are_exact(ss):
    # (i % 8) + 1 per row: every prefix is an integer below 2^24, exact in any add order
    rows, cols = 40, 70_001
    x = np.tile(si.structured_i_mod_8(cols), (rows, 1))
    got = run_rows(ss, "f32", True, x)
    assert_equal(got.reshape(-1), oracle.scan_rows(x, True).astype(np.float32).reshape(-1), tile=cols)


def test_empty(ss):
    import torch
    e = torch.empty(0, dtype=torch.float32, device="cuda")
    ss.ss_scan_rows(ss.SS_F32, True, e, e, 0, 10)
    ss.ss_scan_rows(ss.SS_F32, True, e, e, 10, 0)
    assert ss.ss_stream_status()[0] == ss.SS_OK


def test_row_tile_timeout_is_reported_and_recovered(ss):
    import torch
    # 4 tiles per row: tile 5 is row 1's second tile, and tiles 6 and 7 of the same row wait on it
    rows, cols = 3, 3 * 4096 + 100
    x = rows_input("i32", rows, cols)
    d = torch.from_numpy(x.reshape(-1)).cuda()
    o = torch.empty_like(d)
    ss.ss_debug_set_lookback_fault(5, 2_000_000)
    try:
        ss.ss_scan_rows(ss.SS_I32, True, d, o, rows, cols)
        st, tile = ss.ss_stream_status()
    finally:
        ss.ss_debug_set_lookback_fault(-1, 0)
    assert st == ss.SS_ERR_LOOKBACK_TIMEOUT and tile in (6, 7)
    ss.ss_scan_rows(ss.SS_I32, True, d, o, rows, cols)
    assert ss.ss_stream_status() == (ss.SS_OK, -1)
    assert_equal(o.cpu().numpy(), oracle.scan_rows(x, True).reshape(-1), tile=cols)


def test_long_row_pipe_timeout_is_reported_and_recovered(ss):
    # 3 tiles of 16384 per row: tile 4 is row 1's second tile, and tile 5 waits on it
    import torch
    rows, cols = 3, 40000
    x = rows_input("i32", rows, cols)
    d = torch.from_numpy(x.reshape(-1)).cuda()
    o = torch.empty_like(d)
    ss.ss_debug_set_lookback_fault(4, 2_000_000)
    try:
        ss.ss_scan_rows(ss.SS_I32, False, d, o, rows, cols)
        st, tile = ss.ss_stream_status()
    finally:
        ss.ss_debug_set_lookback_fault(-1, 0)
    assert st == ss.SS_ERR_LOOKBACK_TIMEOUT and tile == 5
    ss.ss_scan_rows(ss.SS_I32, False, d, o, rows, cols)
    assert ss.ss_stream_status() == (ss.SS_OK, -1)
    assert_equal(o.cpu().numpy(), oracle.scan_rows(x, False).reshape(-1), tile=cols)
