"""Scans with 64-bit sums against the CPU oracle.

uint32 -> uint64, int32 -> int64 and int64 (modulo 2^64) are bit-exact.  fp64
is compared with a bound derived from the kernel's add order; integer-valued
fp64 inputs with every prefix below 2^53 are bit-exact too."""

from __future__ import annotations

import functools
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import SENTINEL, Guarded, assert_equal

pytestmark = pytest.mark.gpu

TILE = 8192      # integer kinds: 8192-element tiles of a 64-bit input (one 512-thread CTA per SM)
TILE_W32 = 4096  # ... and 4096 of a 32-bit one (four 128-thread CTAs per SM)
TILE_F64 = 4096  # fp64: two 256-thread CTAs per SM, 16 elements per lane
U = 2.0 ** -53

KINDS = {
    # kind: (input dtype, output dtype, oracle, ss wide type name)
    "u32_u64": (np.uint32, np.uint64, oracle.scan_u32_u64, "SS_WIDE_U32_U64"),
    "i32_i64": (np.int32, np.int64, oracle.scan_i32_i64, "SS_WIDE_I32_I64"),
    "i64": (np.int64, np.int64, oracle.scan_i64, "SS_WIDE_I64"),
    "f64": (np.float64, np.float64, oracle.scan_f64, "SS_WIDE_F64"),
}


@pytest.fixture(scope="module")
def ss():
    import stream_compaction_pass_gb300 as m
    return m


@functools.lru_cache(maxsize=None)
def wide_input(kind: str, n: int) -> np.ndarray:
    if kind == "u32_u64":
        return si.uniform_u32(n, seed=60)
    if kind == "i32_i64":
        return si.uniform_int32(n, -(2**31), 2**31 - 1, seed=61)
    if kind == "i64":
        hi = si.uniform_u32(n, seed=62).astype(np.uint64)
        lo = si.uniform_u32(n, seed=63).astype(np.uint64)
        return ((hi << np.uint64(32)) | lo).view(np.int64)
    # fp64: 24-bit fractions in [-0.5, 0.5) scaled over 2^-10 .. 2^10
    u = si.uniform_f32(n, seed=64).astype(np.float64) - 0.5
    return u * np.exp2(si.uniform_int32(n, -10, 10, seed=65).astype(np.float64))


def run_wide(ss, kind: str, inclusive: bool, x: np.ndarray, offset: int = 0, inplace: bool = False):
    """offset is in elements of the input; buffers are int32 words underneath."""
    import torch
    in_dt, out_dt, _, tname = KINDS[kind]
    n = x.size
    iw = np.dtype(in_dt).itemsize // 4  # 32-bit words per input element
    src = Guarded(n * iw, offset * iw, fill=x.view(np.int32))
    dst = src if inplace else Guarded(n * 2, offset * 2)
    d_in = src.view.view(torch.int64 if iw == 2 else torch.int32)
    d_out = dst.view.view(torch.int64)
    ss.ss_scan_wide(getattr(ss, tname), inclusive, d_in, d_out, n)
    st, tile = ss.ss_stream_status()
    assert st == ss.SS_OK, f"device status {st} at tile {tile}"
    assert dst.guards_intact(), "a store landed outside the output"
    return dst.numpy(np.int32).view(out_dt).copy()


def f64_bound(n: int) -> float:
    # Every output is a sum whose add tree has depth at most 16 (a lane's 16
    # elements, in sequence) + 5 (warp scan) + 5 (scan of the 8 warp totals)
    # + 2 (the tile's prefix into the warp offset, then the lane offset) + 7
    # per tile of the look-back chain (one add to the predecessor's prefix, a
    # 5-level warp reduction of a window, one add of the window sums).  So
    # the normalised error is at most (7 * tiles + 28) * u (first order),
    # plus the oracle's own rounding of about u; 64 leaves room.
    tiles = max(1, math.ceil(n / TILE_F64))
    return (7 * tiles + 64) * U


def check(ss, kind, inclusive, x, **kw):
    got = run_wide(ss, kind, inclusive, x, **kw)
    ref = KINDS[kind][2](x, inclusive)
    if kind != "f64":
        assert_equal(got, ref, tile=TILE)
        return
    norm = np.maximum(1.0, oracle.abs_prefix_f64(x))
    err = float(np.max(np.abs(got - ref) / norm)) if x.size else 0.0
    assert err <= f64_bound(x.size), f"normalised fp64 error {err:.3e} > {f64_bound(x.size):.3e}"


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("inclusive", [True, False])
@pytest.mark.parametrize("n", [1, 2, 3, 7, 4095, 4096, 4097, 8191, 8192, 8193, 16383, 16384, 16385, 3 * 8192 + 5,
                               152 * 8192,
                               152 * 8192 + 1, 152 * 16384 + 3, 1_000_003,
                               # a whole round of 608 CTAs on 4096-element tiles, and ragged ones
                               608 * TILE_W32, 608 * TILE_W32 + 1, 3 * 608 * TILE_W32 + TILE_W32 - 1])
def test_sizes(ss, kind, inclusive, n):
    check(ss, kind, inclusive, wide_input(kind, n))


@pytest.mark.parametrize("kind", ["u32_u64", "f64"])
def test_full_size(ss, kind):
    n = 100_000_000
    check(ss, kind, True, wide_input(kind, n))


def test_widened_exceeds_32_bits(ss):
    # all-max uint32: the inclusive sum at i is (i + 1) * (2^32 - 1)
    n = 5 * 8192 + 3
    x = np.full(n, 0xFFFFFFFF, dtype=np.uint32)
    got = run_wide(ss, "u32_u64", True, x)
    assert_equal(got, (np.arange(1, n + 1, dtype=np.uint64) * np.uint64(0xFFFFFFFF)))


def test_f64_integer_valued_is_exact(ss):
    n = 3_000_017
    x = si.uniform_int32(n, -(2**20), 2**20, seed=66).astype(np.float64)
    for inclusive in (True, False):
        got = run_wide(ss, "f64", inclusive, x)
        assert_equal(got, oracle.scan_f64(x, inclusive), tile=TILE)


@pytest.mark.parametrize("kind", ["i64", "f64"])
def test_in_place(ss, kind):
    x = wide_input(kind, 40 * 8192 + 9)
    check(ss, kind, False, x, inplace=True)


@pytest.mark.parametrize("kind,offset", [("u32_u64", 1), ("u32_u64", 3), ("i64", 1), ("f64", 1)])
def test_unaligned(ss, kind, offset):
    # 4- or 8-byte aligned but not 16: every tile takes the checked element-wise path
    check(ss, kind, True, wide_input(kind, 20 * 8192 + 13), offset=offset)


def test_named_entry_points(ss):
    import torch
    n = 12345
    x = wide_input("u32_u64", n)
    d = torch.from_numpy(x.view(np.int32)).cuda()
    o = torch.empty(n, dtype=torch.int64, device="cuda")
    ss.scan_exclusive_u32_u64(d, o)
    assert_equal(o.cpu().numpy().view(np.uint64), oracle.scan_u32_u64(x, False))
    xf = wide_input("f64", n)
    df = torch.from_numpy(xf).cuda()
    of = torch.empty_like(df)
    ss.scan_inclusive_f64(df, of)
    ss.scan_exclusive_i64(df.view(torch.int64), of.view(torch.int64))
    assert ss.ss_stream_status()[0] == ss.SS_OK
    assert_equal(of.cpu().numpy().view(np.int64), oracle.scan_i64(xf.view(np.int64), False))


def test_empty(ss):
    import torch
    e = torch.empty(0, dtype=torch.int64, device="cuda")
    ss.scan_inclusive_i64(e, e, 0)
    assert ss.ss_stream_status()[0] == ss.SS_OK


def test_repeated_launches_alternate_with_32_bit_scans(ss):
    # the 16-byte and 8-byte descriptors share one workspace: epochs keep them apart
    import torch
    n = 77 * 8192 + 1
    x = wide_input("i64", n)
    d = torch.from_numpy(x).cuda()
    o = torch.empty_like(d)
    x32 = si.workload_int_pm1000(n, seed=2)
    d32 = torch.from_numpy(x32).cuda()
    o32 = torch.empty_like(d32)
    for _ in range(3):
        ss.scan_inclusive_i64(d, o)
        ss.scan_exclusive_i32(d32, o32)
    assert ss.ss_stream_status()[0] == ss.SS_OK
    assert_equal(o.cpu().numpy(), oracle.scan_i64(x, True), tile=TILE)
    assert_equal(o32.cpu().numpy(), oracle.scan_i32(x32, False))
