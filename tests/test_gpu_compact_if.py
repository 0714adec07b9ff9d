"""Predicate compaction (keep v > 0, no flag array) and the unordered
warp-aggregated-atomic compaction, against the CPU oracle.

The ordered calls are compared bit for bit, output and count.  The unordered
calls keep the same elements in another order.  For them, the count is
compared exactly and the output as a multiset: both sides are sorted by bit
pattern and compared bit for bit."""

from __future__ import annotations

import functools

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import SENTINEL, Guarded, assert_equal

pytestmark = pytest.mark.gpu

DT = {"f32": (np.float32, "SS_F32", oracle.compact_positive_f32),
      "i32": (np.int32, "SS_I32", oracle.compact_positive_i32),
      "u32": (np.uint32, "SS_U32", oracle.compact_positive_u32)}


@pytest.fixture(scope="module")
def ss():
    import stream_compaction_pass_gb300 as m
    return m


@functools.lru_cache(maxsize=None)
def positive_input(n: int, p: float, kind: str) -> np.ndarray:
    if kind == "f32":
        return si.workload_positive_f32(n, p, seed=5)
    if kind == "i32":
        return si.uniform_int32(n, -int(round((1 - p) * 1000)), int(round(p * 1000)), seed=5)
    x = si.uniform_u32(n, seed=5)
    return np.where(si.bernoulli_flags(n, p, seed=15) != 0, x | 1, 0).astype(np.uint32)


def run_positive(ss, kind: str, x: np.ndarray, unordered: bool = False, in_offset: int = 0, out_offset: int = 0):
    import torch
    n = x.size
    src = Guarded(n, in_offset, fill=x)
    dst = Guarded(n, out_offset)
    cnt = torch.full((1,), -1, dtype=torch.int64, device="cuda:0")
    dtype = getattr(ss, DT[kind][1])
    if unordered:
        ss.ss_compact_positive_unordered(dtype, src.view, dst.view, cnt, n)
    elif kind == "f32":
        ss.compact_positive_f32(src.view, dst.view, cnt, n)
    else:
        ss.ss_compact_positive(dtype, src.view, dst.view, cnt, n)
    st, tile = ss.ss_stream_status()
    assert st == ss.SS_OK, f"device status {st} at tile {tile}"
    assert dst.guards_intact(), "a store landed outside the output"
    c = int(cnt.item())
    full = dst.numpy(np.uint32)
    assert (full[c:].view(np.int32) == SENTINEL).all(), "an element past the count was written"
    return full[:c].copy(), c


def expected_bits(kind: str, x: np.ndarray) -> np.ndarray:
    return DT[kind][2](x).view(np.uint32)


@pytest.mark.parametrize("p", [0.01, 0.5, 0.99])
def test_positive_f32_full_size(ss, p):
    n = 1 << 28
    x = positive_input(n, p, "f32")
    got, c = run_positive(ss, "f32", x)
    ref = expected_bits("f32", x)
    assert c == ref.size
    assert_equal(got, ref)


@pytest.mark.parametrize("kind", ["f32", "i32", "u32"])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 31, 33, 513, 4095, 4096, 4097, 16383, 16384, 16385, 16389,
                               3 * 16384 + 7, 100_003, 1 << 20, (1 << 20) + 3])
def test_positive_edges(ss, kind, n):
    x = positive_input(n, 0.4, kind)
    got, c = run_positive(ss, kind, x)
    ref = expected_bits(kind, x)
    assert c == ref.size
    assert_equal(got, ref)


@pytest.mark.parametrize("kind", ["f32", "i32", "u32"])
@pytest.mark.parametrize("p", [0.001, 0.01, 0.0155, 0.06])
def test_positive_sparse_and_mixed_tiles(ss, kind, p):
    # Low keep rates: tiles keeping fewer than 256 keys, none of whose threads
    # keeps more than four, take the sparse form (at 0.001 and 0.01), the
    # others the staged one; ragged last tile.
    n = 150 * 16384 + 4093
    x = positive_input(n, p, kind)
    got, c = run_positive(ss, kind, x)
    ref = expected_bits(kind, x)
    assert c == ref.size
    assert_equal(got, ref)


@pytest.mark.parametrize("run", [3, 5, 17, 40])
def test_positive_clustered_runs(ss, run):
    # Runs of `run` consecutive positive values in a negative background, at
    # seeded positions, about 128 kept keys a tile: a thread holding five or
    # more kept keys sends its tile to the staged form while tiles without
    # one stay sparse.
    n = 64 * 16384 + 999
    x = -np.abs(si.uniform_f32(n, seed=42)) - np.float32(1.0)
    starts = si.uniform_int32(max(1, n // (128 * run)), 0, n - 1, seed=43).astype(np.int64)
    for st in starts:
        x[st: st + run] = np.abs(x[st: st + run])
    got, c = run_positive(ss, "f32", x)
    ref = expected_bits("f32", x)
    assert c == ref.size
    assert_equal(got, ref)


@pytest.mark.parametrize("p", [0.0, 1.0])
@pytest.mark.parametrize("n", [4096, 5 * 16384 + 1])
def test_positive_none_or_all(ss, p, n):
    x = positive_input(n, p, "f32").copy()
    if p == 0.0:  # all negative, with signed zeros mixed in: none is kept
        x[::3] = np.float32(0.0)
        x[1::3] = np.float32(-0.0)
    got, c = run_positive(ss, "f32", x)
    ref = expected_bits("f32", x)
    assert c == ref.size == (0 if p == 0.0 else n)
    assert_equal(got, ref)


def test_ieee_special_values_in_every_tile(ss):
    specials = np.array([0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000, 0x00000000, 0x80000000,
                         0x00000001, 0x80000001, 0x3F800000, 0x7F7FFFFF], dtype=np.uint32)
    n = 40 * 16384 + 11
    x = si.workload_positive_f32(n, 0.5, seed=21).view(np.uint32).copy()
    idx = (np.arange(0, n, 997)).astype(np.int64)
    x[idx] = specials[np.arange(idx.size) % specials.size]
    xf = x.view(np.float32)
    got, c = run_positive(ss, "f32", xf)
    assert_equal(got, expected_bits("f32", xf))


@pytest.mark.parametrize("ioff,ooff", [(1, 0), (0, 1), (3, 2)])
def test_positive_misaligned(ss, ioff, ooff):
    n = 7 * 16384 + 100
    x = positive_input(n, 0.5, "f32")
    got, c = run_positive(ss, "f32", x, in_offset=ioff, out_offset=ooff)
    assert_equal(got, expected_bits("f32", x))


@pytest.mark.parametrize("p", [0.02, 0.5, 0.99])
@pytest.mark.parametrize("ooff", [1, 2, 3])
def test_positive_output_phase(ss, p, ooff):
    # aligned keys take the persistent kernel; the output starts 4, 8 or 12
    # bytes past a 16-byte boundary, so every staged run has a ragged head
    n = 9 * 16384 + 77
    x = positive_input(n, p, "f32")
    got, c = run_positive(ss, "f32", x, out_offset=ooff)
    assert_equal(got, expected_bits("f32", x))


def test_positive_zero_length(ss):
    import torch
    cnt = torch.full((1,), 77, dtype=torch.int64, device="cuda:0")
    e = torch.empty(0, dtype=torch.float32, device="cuda:0")
    ss.compact_positive_f32(e, e, cnt, 0)
    assert int(cnt.item()) == 0
    ss.ss_compact_positive_unordered(ss.SS_F32, e, e, cnt, 0)
    assert int(cnt.item()) == 0


def test_positive_repeated_and_non_default_stream(ss):
    import torch
    n = 9 * 16384 + 5
    x = positive_input(n, 0.5, "f32")
    ref = expected_bits("f32", x)
    s = torch.cuda.Stream()
    src = torch.from_numpy(x).cuda()
    dst = torch.empty_like(src)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda:0")
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(5):
            ss.compact_positive_f32(src, dst, cnt, n, stream=s.cuda_stream)
    s.synchronize()
    assert ss.ss_stream_status(stream=s.cuda_stream)[0] == ss.SS_OK
    c = int(cnt.item())
    assert_equal(dst[:c].cpu().numpy().view(np.uint32), ref)


def test_flag_form_equals_predicate_form(ss):
    # compact_u32 with flags (x > 0) gives the same bits as the predicate call.
    import torch
    n = 11 * 16384 + 3
    x = positive_input(n, 0.3, "f32")
    got_pred, c_pred = run_positive(ss, "f32", x)
    keys = torch.from_numpy(x.view(np.int32)).cuda()
    flags = torch.from_numpy((x > 0).astype(np.uint8)).cuda()
    out = torch.empty_like(keys)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda:0")
    ss.compact_u32(keys, flags, out, cnt)
    c = int(cnt.item())
    assert c == c_pred
    assert_equal(out[:c].cpu().numpy().view(np.uint32), got_pred)


# ---- unordered (warp-aggregated atomics) ----

def assert_same_multiset(got_bits: np.ndarray, ref_bits: np.ndarray):
    assert got_bits.size == ref_bits.size
    assert_equal(np.sort(got_bits), np.sort(ref_bits))


@pytest.mark.parametrize("kind", ["f32", "i32", "u32"])
@pytest.mark.parametrize("n", [1, 31, 32, 33, 511, 512, 513, 4097, 100_003, 1 << 20])
def test_unordered_positive_multiset(ss, kind, n):
    x = positive_input(n, 0.5, kind)
    got, c = run_positive(ss, kind, x, unordered=True)
    assert_same_multiset(got, expected_bits(kind, x))


@pytest.mark.parametrize("p", [0.01, 0.5, 0.99])
def test_unordered_full_size(ss, p):
    n = 1 << 28
    x = positive_input(n, p, "f32")
    got, c = run_positive(ss, "f32", x, unordered=True)
    assert_same_multiset(got, expected_bits("f32", x))


def test_unordered_keeps_order_inside_each_batch(ss):
    # With one warp's 512-element batch as the whole input, the unordered
    # kernel makes a single claim, so its output is the ordered one.
    n = 512
    x = positive_input(n, 0.5, "f32")
    got, c = run_positive(ss, "f32", x, unordered=True)
    assert_equal(got, expected_bits("f32", x))


@pytest.mark.parametrize("ioff", [0, 1, 2])
def test_unordered_flags_multiset(ss, ioff):
    import torch
    n = 3 * 16384 + 77
    keys, flags = si.workload_compaction(n, 0.5, seed=3)
    k = Guarded(n, ioff, fill=keys)
    fbuf = torch.zeros(n + 64 + ioff, dtype=torch.uint8, device="cuda:0")
    fview = fbuf[ioff: ioff + n]
    fview.copy_(torch.from_numpy(flags))
    out = Guarded(n)
    cnt = torch.full((1,), -1, dtype=torch.int64, device="cuda:0")
    ss.ss_compact_u32_unordered(k.view, fview, out.view, cnt, n)
    assert ss.ss_stream_status()[0] == ss.SS_OK
    assert out.guards_intact()
    c = int(cnt.item())
    assert_same_multiset(out.numpy(np.uint32)[:c], oracle.compact_u32(keys, flags))
