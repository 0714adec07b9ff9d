"""Segmented scans against the CPU oracle: int32/uint32 bit-exact, fp32
within the normalised bound, the normaliser taken per segment."""

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
def seg_input(kind: str, n: int) -> np.ndarray:
    if kind == "i32":
        return si.uniform_int32(n, -1000, 1000, seed=94)
    if kind == "u32":
        return si.uniform_u32(n, seed=95)
    return si.uniform_f32(n, seed=96)


def run_segments(ss, kind, inclusive, x, offsets, offset=0, inplace=False, num_segments=None):
    import torch
    n = x.size
    src = Guarded(n, offset, fill=x)
    dst = src if inplace else Guarded(n, offset)
    d_off = torch.from_numpy(offsets.astype(np.int64)).cuda()
    dt = {"i32": ss.SS_I32, "u32": ss.SS_U32, "f32": ss.SS_F32}[kind]
    ss.ss_scan_segments(dt, inclusive, src.view, dst.view, d_off, num_segments=num_segments)
    st, tile = ss.ss_stream_status()
    assert st == ss.SS_OK, f"device status {st} at tile {tile}"
    assert dst.guards_intact(), "a store landed outside the output"
    return dst.numpy({"i32": np.int32, "u32": np.uint32, "f32": np.float32}[kind]).copy()


def check(ss, kind, inclusive, x, offsets, **kw):
    got = run_segments(ss, kind, inclusive, x, offsets, **kw)
    ref = oracle.scan_segments(x, offsets, inclusive)
    if kind != "f32":
        assert_equal(got, ref, tile=16384)
        return
    norm = np.maximum(1.0, oracle.abs_prefix_segments_f32(x, offsets))
    err = float(np.max(np.abs(got.astype(np.float64) - ref) / norm))
    assert err <= FP32_TOL, f"normalised fp32 error {err:.3e}"


CASES = [(1, 1.0), (5, 2.0), (4096, 3.5), (12287, 50.0), (12288, 12288.0), (12289, 3.0), (16383, 100.0),
         (16384, 16384.0), (16385, 1.0), (100_003, 700.0),
         (100_003, 40_000.0), (1 << 20, 7.0), (1 << 20, 300_000.0), (3_000_017, 5000.0), (3_000_017, 1e9)]


@pytest.mark.parametrize("kind", ["i32", "u32", "f32"])
@pytest.mark.parametrize("inclusive", [True, False])
@pytest.mark.parametrize("n,mean", CASES, ids=[f"{n}_{int(m)}" for n, m in CASES])
def test_segments(ss, kind, inclusive, n, mean):
    offsets = si.segment_offsets(n, mean, seed=97, empty_frac=0.1 if mean < 50 else 0.0)
    check(ss, kind, inclusive, seg_input(kind, n), offsets)


FORMS = {1: "rows", 2: "blocked-256", 3: "blocked-128", 4: "blocked-512", 5: "blocked-64"}


@pytest.fixture(params=list(FORMS), ids=list(FORMS.values()))
def form(request, ss):
    ss.ss_set_segments_config(request.param)
    yield request.param
    ss.ss_set_segments_config(0)  # the library's default


# sizes about the tiles of every form (4096, 8192, 16384) and their ragged tails
FORM_CASES = [(1, 1.0), (4095, 3.0), (4096, 4096.0), (4097, 2.0), (8191, 20.0), (8192, 8192.0), (8193, 1.5),
              (16385, 5.0), (49_153, 30_000.0), (100_003, 700.0), (1 << 20, 7.0), (3_000_017, 5000.0),
              (3_000_017, 1e9)]


@pytest.mark.parametrize("kind,inclusive", [("i32", True), ("u32", False), ("f32", True), ("f32", False)])
@pytest.mark.parametrize("n,mean", FORM_CASES, ids=[f"{n}_{int(m)}" for n, m in FORM_CASES])
def test_each_form(ss, form, kind, inclusive, n, mean):
    offsets = si.segment_offsets(n, mean, seed=97, empty_frac=0.1 if mean < 50 else 0.0)
    check(ss, kind, inclusive, seg_input(kind, n), offsets)


@functools.lru_cache(maxsize=3)
def full_size_case(mean: float):
    n = 100_000_000
    x = seg_input("i32", n)
    offsets = si.segment_offsets(n, mean, seed=98)
    return x, offsets, oracle.scan_segments(x, offsets, True)


@pytest.mark.parametrize("mean", [4.0, 100.0, 128256.0])
def test_each_form_full_size(ss, form, mean):
    x, offsets, ref = full_size_case(mean)
    assert_equal(run_segments(ss, "i32", True, x, offsets), ref, tile=4096)


def test_forms_agree_bitwise_on_integers(ss):
    n = 2_000_003
    x = seg_input("u32", n)
    offsets = si.segment_offsets(n, 60.0, seed=102, empty_frac=0.05)
    outs = []
    try:
        for f in FORMS:
            ss.ss_set_segments_config(f)
            outs.append(run_segments(ss, "u32", False, x, offsets))
    finally:
        ss.ss_set_segments_config(0)
    for o in outs[1:]:
        assert_equal(o, outs[0], tile=4096)


def test_unknown_form_is_rejected(ss):
    with pytest.raises(ss.StreamScanError):
        ss.ss_set_segments_config(6)
    with pytest.raises(ss.StreamScanError):
        ss.ss_set_segments_config(-1)


@pytest.mark.parametrize("mean", [128256.0, 1000.0])
def test_full_size(ss, mean):
    n = 100_000_000
    offsets = si.segment_offsets(n, mean, seed=98)
    check(ss, "f32", True, seg_input("f32", n), offsets)
    check(ss, "i32", False, seg_input("i32", n), offsets)


def test_equal_lengths_match_batched_rows(ss):
    import torch
    rows, cols = 300, 20_000
    x = seg_input("i32", rows * cols)
    offsets = np.arange(0, rows * cols + 1, cols, dtype=np.uint64)
    got = run_segments(ss, "i32", True, x, offsets)
    d = torch.from_numpy(x).cuda()
    o = torch.empty_like(d)
    ss.ss_scan_rows(ss.SS_I32, True, d, o, rows, cols)
    assert_equal(got, o.cpu().numpy(), tile=16384)


@pytest.mark.parametrize("offset", [1, 3])
def test_unaligned(ss, offset):
    n = 500_001
    check(ss, "i32", True, seg_input("i32", n), si.segment_offsets(n, 900.0, seed=99), offset=offset)


@pytest.mark.parametrize("mean", [3.5, 40.0])
def test_offsets_not_16_byte_aligned(ss, mean):
    # the offsets array starts 8 bytes past a 16-byte boundary: the start
    # marking reads it element by element instead of in 16-byte pairs
    import torch
    n = 300_007
    x = seg_input("i32", n)
    offsets = si.segment_offsets(n, mean, seed=101, empty_frac=0.1)
    buf = torch.zeros(offsets.size + 1, dtype=torch.int64, device="cuda")
    buf[1:] = torch.from_numpy(offsets.astype(np.int64)).cuda()
    d_off = buf[1:]
    assert d_off.data_ptr() % 16 == 8
    src = torch.from_numpy(x).cuda()
    dst = torch.empty_like(src)
    ss.ss_scan_segments(ss.SS_I32, True, src, dst, d_off)
    assert ss.ss_stream_status()[0] == ss.SS_OK
    assert_equal(dst.cpu().numpy(), oracle.scan_segments(x, offsets, True), tile=16384)


def test_in_place(ss):
    n = 700_001
    check(ss, "u32", False, seg_input("u32", n), si.segment_offsets(n, 2000.0, seed=100), inplace=True)


def test_no_segments_is_one_segment(ss):
    n = 200_000
    x = seg_input("i32", n)
    got = run_segments(ss, "i32", True, x, np.array([0, n], dtype=np.uint64), num_segments=0)
    assert_equal(got, oracle.scan_i32(x, True), tile=16384)


@pytest.mark.parametrize("seg_form", [0, 1, 2, 3, 4, 5])
def test_segmented_timeout_short_segments(ss, seg_form):
    # Segments of mean length 40 (the blocked form unless one is forced).  A tile holding a start
    # publishes its inclusive prefix before its look-back, but still looks
    # back for the elements before its first start; the fault hook makes
    # tile 7 publish nothing, so tile 8's look-back runs out.
    import torch
    n = 30 * 16384 + 5
    x = seg_input("i32", n)
    offsets = si.segment_offsets(n, 40.0, seed=101)
    d = torch.from_numpy(x).cuda()
    o = torch.empty_like(d)
    d_off = torch.from_numpy(offsets.astype(np.int64)).cuda()
    ss.ss_set_segments_config(seg_form)
    ss.ss_debug_set_lookback_fault(7, 2_000_000)
    try:
        ss.ss_scan_segments(ss.SS_I32, True, d, o, d_off)
        st, tile = ss.ss_stream_status()
        ss.ss_debug_set_lookback_fault(-1, 0)
        assert st == ss.SS_ERR_LOOKBACK_TIMEOUT and tile > 7
        ss.ss_scan_segments(ss.SS_I32, True, d, o, d_off)
        assert ss.ss_stream_status() == (ss.SS_OK, -1)
    finally:
        ss.ss_debug_set_lookback_fault(-1, 0)
        ss.ss_set_segments_config(0)
    assert_equal(o.cpu().numpy(), oracle.scan_segments(x, offsets, True), tile=16384)


def test_segmented_timeout_is_reported_and_recovered(ss):
    # one long segment: tile 7 publishes nothing and tile 8 waits on it
    import torch
    n = 30 * 16384 + 5
    x = seg_input("i32", n)
    offsets = np.array([0, n], dtype=np.uint64)
    d = torch.from_numpy(x).cuda()
    o = torch.empty_like(d)
    d_off = torch.from_numpy(offsets.astype(np.int64)).cuda()
    ss.ss_debug_set_lookback_fault(7, 2_000_000)
    try:
        ss.ss_scan_segments(ss.SS_I32, True, d, o, d_off)
        st, tile = ss.ss_stream_status()
    finally:
        ss.ss_debug_set_lookback_fault(-1, 0)
    assert st == ss.SS_ERR_LOOKBACK_TIMEOUT and tile > 7
    ss.ss_scan_segments(ss.SS_I32, True, d, o, d_off)
    assert ss.ss_stream_status() == (ss.SS_OK, -1)
    assert_equal(o.cpu().numpy(), oracle.scan_i32(x, True), tile=16384)
