"""Pins for the CPU oracle: it is checked against what the pages and plain
mathematics fix, never against itself or the GPU.

Which pin covers which oracle function:

* scan_i32 / scan_u32 / scan_f32 (inclusive and exclusive):
  worked examples (tests/golden/scan_worked_examples.txt), closed forms
  (iota, constants, the (i % 8) + 1 and period-4 patterns), invariants
  (inclusive - exclusive = x, last inclusive = total, exclusive[0] = 0),
  O(n^2) brute force with Python big integers / exact fractions, and
  wraparound through an independent uint32 running sum.
* abs_prefix_f32: brute force with exact fractions.
* compact_u32 / compact_positive_*: brute-force list filter, the count
  identity pos[n-1] + flags[n-1], subsequence check, all-zero / all-one
  flags, IEEE special values written out by hand, agreement of the
  predicate form with the flag form.
* scan_u32_u64 / scan_i32_i64 / scan_i64: the worked examples, brute force
  with Python integers (mod 2^64 for int64), the low 32 bits against the
  pinned 32-bit scans.
* scan_f64 / abs_prefix_f64: exact rational brute force within the
  compensated-sum bound, Neumaier's classic cancellation case,
  integer-valued inputs exactly.
* scan_rows / abs_prefix_rows_f32: a worked example by hand, all-ones rows
  restart at every row, brute force with Python integers, each row equal to
  the pinned one-dimensional scan.
* scan_segments / abs_prefix_segments_f32: a worked example by hand with an
  empty segment, one segment = the flat scan, unit segments, equal lengths =
  the batched rows, brute force with Python integers.
* moe_counts_offsets: a worked example by hand, the histogram against
  numpy's bincount, tile size 1 against the (pinned) exclusive scan, the
  rounding invariants, one-expert and out-of-range cases.
* the tile model: the pages' printed tables (tests/golden/).
"""

from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import seeded_inputs as si

M32 = 1 << 32


def _parse_ints(field: str):
    field = field.strip()
    return [int(t) for t in field.split()] if field else None


def _worked_examples(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "scan_worked_examples.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, x, inc, exc, src = [p.strip() for p in line.split("|")]
            rows.append((name, _parse_ints(x), _parse_ints(inc), _parse_ints(exc), src))
    return rows


def test_worked_examples_int(golden_dir):
    rows = _worked_examples(golden_dir)
    assert len(rows) == 4
    for name, x, inc, exc, _src in rows:
        xa = np.array(x, dtype=np.int32)
        if inc is not None:
            assert oracle.scan_i32(xa, True).tolist() == inc, name
            assert oracle.scan_u32(xa.astype(np.uint32), True).tolist() == inc, name
        if exc is not None:
            assert oracle.scan_i32(xa, False).tolist() == exc, name
            assert oracle.scan_u32(xa.astype(np.uint32), False).tolist() == exc, name


def test_worked_examples_f32(golden_dir):
    for name, x, inc, exc, _src in _worked_examples(golden_dir):
        xa = np.array(x, dtype=np.float32)
        if inc is not None:
            assert oracle.scan_f32(xa, True).tolist() == [float(v) for v in inc], name
        if exc is not None:
            assert oracle.scan_f32(xa, False).tolist() == [float(v) for v in exc], name


@pytest.mark.parametrize("n", [1, 2, 7, 64, 4096, 100_003])
def test_closed_form_all_ones_is_iota(n):
    ones = np.ones(n, dtype=np.int32)
    assert np.array_equal(oracle.scan_i32(ones, False), np.arange(n, dtype=np.int32))
    assert np.array_equal(oracle.scan_i32(ones, True), np.arange(1, n + 1, dtype=np.int32))
    f = np.ones(n, dtype=np.float32)
    assert np.array_equal(oracle.scan_f32(f, True), np.arange(1, n + 1, dtype=np.float64))


@pytest.mark.parametrize("c", [-7, 3, 1000])
def test_closed_form_constant(c):
    n = 5000
    x = np.full(n, c, dtype=np.int32)
    i = np.arange(n, dtype=np.int64)
    assert np.array_equal(oracle.scan_i32(x, False).astype(np.int64), c * i)
    assert np.array_equal(oracle.scan_i32(x, True).astype(np.int64), c * (i + 1))


def test_closed_form_i_mod_8(golden_dir):
    n = 1_049_187  # the page's element count, a partial tile at every block size
    x = si.structured_i_mod_8(n)
    i1 = np.arange(1, n + 1, dtype=np.int64)
    r = i1 % 8
    expect = 36 * (i1 // 8) + r * (r + 1) // 2
    assert np.array_equal(oracle.scan_f32(x, True), expect.astype(np.float64))
    # the page's tile bound: a 1024-element tile never exceeds 4608
    assert oracle.scan_f32(x[:1024], True)[-1] == 4608.0


def test_closed_form_period4_total():
    n = 10_000_000
    x = si.structured_period4(n)
    inc = oracle.scan_f32(x, True)
    i1 = np.arange(1, n + 1, dtype=np.int64)
    assert np.array_equal(inc, (i1 + i1 // 4).astype(np.float64))
    assert inc[-1] == 12_500_000.0  # total printed on the page
    assert np.array_equal(oracle.scan_f32(x, False)[1:], inc[:-1])


def test_structured_fixture_values(golden_dir):
    with open(os.path.join(golden_dir, "structured_inputs.txt")) as f:
        rows = [l.split("|") for l in f if l.strip() and not l.startswith("#")]
    vals = {r[0].strip(): (int(r[1]), float(r[2])) for r in rows}
    n, total = vals["period4_total"]
    assert oracle.scan_f32(si.structured_period4(n), True)[-1] == total
    n, peak = vals["i_mod_8_tile1024_max_prefix"]
    assert oracle.scan_f32(si.structured_i_mod_8(n), True).max() == peak


def _brute_force_mod32(x, inclusive):
    out = []
    for i in range(len(x)):
        s = sum(int(v) for v in (x[: i + 1] if inclusive else x[:i]))
        out.append(s % M32)
    return out


@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 31, 32, 33, 63, 64])
@pytest.mark.parametrize("inclusive", [True, False])
def test_brute_force_int_full_range(n, inclusive):
    rng = np.random.default_rng(1000 + n)
    x = rng.integers(-(1 << 31), 1 << 31, size=n, dtype=np.int64).astype(np.int32)
    got_i = oracle.scan_i32(x, inclusive).astype(np.int64) % M32
    assert got_i.tolist() == _brute_force_mod32(x, inclusive)
    xu = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    got_u = oracle.scan_u32(xu, inclusive).astype(np.int64)
    assert got_u.tolist() == _brute_force_mod32(xu, inclusive)


@pytest.mark.parametrize("n", [1, 2, 17, 64])
@pytest.mark.parametrize("inclusive", [True, False])
def test_brute_force_f32_exact_fractions(n, inclusive):
    # Inputs of the workload's form k * 2**-24 (and signed): every partial sum
    # of <= 64 of them is exact in float64, so the oracle must equal the exact
    # rational prefix sum.
    x = si.uniform_f32(n, seed=77)
    x = np.where(np.arange(n) % 3 == 1, -x, x).astype(np.float32)
    got = oracle.scan_f32(x, inclusive)
    for i in range(n):
        part = x[: i + 1] if inclusive else x[:i]
        exact = sum((Fraction(float(v)) for v in part), Fraction(0))
        assert Fraction(float(got[i])) == exact
    a = oracle.abs_prefix_f32(x)
    for i in range(n):
        assert Fraction(float(a[i])) == sum((abs(Fraction(float(v))) for v in x[: i + 1]), Fraction(0))


def test_wraparound_two_routes():
    # Route 1: the oracle (64-bit exact sum, low 32 bits kept).
    # Route 2: a uint32 running sum that wraps at every step, in numpy.
    x = si.workload_int_pm1000(1 << 20, seed=2)
    big = np.full(1 << 16, 2_000_000_000, dtype=np.int32)  # forces many wraps
    for arr in (x, big, np.concatenate([big, x])):
        acc = np.uint32(0)
        route2 = np.empty(arr.size, dtype=np.uint32)
        u = arr.view(np.uint32)
        with np.errstate(over="ignore"):
            for s in range(0, arr.size, 1 << 16):
                blk = np.cumsum(u[s:s + (1 << 16)], dtype=np.uint32) + acc
                route2[s:s + blk.size] = blk
                acc = blk[-1]
        assert np.array_equal(oracle.scan_i32(arr, True).view(np.uint32), route2)


def test_invariants_random():
    for seed, n in [(2, 1 << 16), (3, 100_003)]:
        x = si.workload_int_pm1000(n, seed=seed)
        inc = oracle.scan_i32(x, True)
        exc = oracle.scan_i32(x, False)
        assert exc[0] == 0
        with np.errstate(over="ignore"):
            assert np.array_equal((inc.view(np.uint32) - exc.view(np.uint32)), x.view(np.uint32))
        assert int(inc[-1]) == int(np.sum(x.astype(np.int64)))  # no wrap at this size
        assert np.array_equal(exc[1:], inc[:-1])
    # Nonnegative counts give a monotone exclusive scan.
    c = si.workload_poisson_counts(1 << 16, seed=4)
    e = oracle.scan_u32(c, False)
    assert np.all(np.diff(e.astype(np.int64)) >= 0)


def test_fp32_integer_valued_is_exact():
    # Integer-valued fp32 inputs with every prefix below 2**24 have a unique
    # exact answer whatever the add order.
    x = si.uniform_int32(200_000, 0, 9, seed=11).astype(np.float32)
    inc = oracle.scan_f32(x, True)
    assert inc[-1] < 2 ** 24
    assert np.array_equal(inc, np.cumsum(x.astype(np.int64)).astype(np.float64))


def _brute_compact(keys, flags):
    return [int(k) for k, f in zip(keys, flags) if int(f) != 0]


@pytest.mark.parametrize("n", [0, 1, 5, 64, 1000])
def test_compact_brute_force(n):
    keys = si.uniform_u32(n, seed=5)
    flags = si.bernoulli_flags(n, 0.5, seed=6)
    flags = np.where(np.arange(n) % 7 == 3, 200, flags).astype(np.uint8)  # any nonzero keeps
    got = oracle.compact_u32(keys, flags)
    assert got.tolist() == _brute_compact(keys, flags)


def test_compact_count_identity_and_subsequence():
    n = 1 << 16
    for p in (0.01, 0.5, 0.99):
        keys, flags = si.workload_compaction(n, p, seed=3)
        got = oracle.compact_u32(keys, flags)
        f01 = (flags != 0).astype(np.uint32)
        pos = oracle.scan_u32(f01, False)
        assert got.size == int(pos[-1]) + int(f01[-1])
        # out[pos[i]] = keys[i] for kept i  (the scatter reading of the page)
        kept = np.nonzero(f01)[0]
        assert np.array_equal(got[pos[kept]], keys[kept])
        # subsequence: the kept keys appear in index order
        assert np.array_equal(got, keys[kept])


def test_compact_degenerate():
    n = 4099
    keys = si.uniform_u32(n, seed=9)
    assert oracle.compact_u32(keys, np.zeros(n, np.uint8)).size == 0
    assert np.array_equal(oracle.compact_u32(keys, np.ones(n, np.uint8)), keys)


def test_compact_positive_predicate():
    x = np.array([0.5, -1.0, 0.0, 2.0, -0.0, 3.5, float("nan")], dtype=np.float32)
    assert oracle.compact_positive_f32(x).tolist() == [0.5, 2.0, 3.5]


def test_compact_positive_ieee_special_values():
    # IEEE 754 ordering: NaN compares false, -0 == +0 is not > 0, infinities
    # and the smallest subnormal order as numbers.  Expected output written
    # out by hand, as bit patterns.
    bits = np.array([0x7F800000,   # +inf   kept
                     0xFF800000,   # -inf
                     0x7FC00000,   # NaN
                     0xFFC00000,   # -NaN
                     0x00000000,   # +0
                     0x80000000,   # -0
                     0x00000001,   # smallest subnormal  kept
                     0x80000001,   # its negative
                     0x3F800000,   # 1.0    kept
                     0x7F7FFFFF],  # FLT_MAX  kept
                    dtype=np.uint32)
    got = oracle.compact_positive_f32(bits.view(np.float32)).view(np.uint32)
    assert got.tolist() == [0x7F800000, 0x00000001, 0x3F800000, 0x7F7FFFFF]


def test_compact_positive_int_special_values():
    xi = np.array([-2147483648, -1, 0, 1, 2147483647, 0, 42], dtype=np.int32)
    assert oracle.compact_positive_i32(xi).tolist() == [1, 2147483647, 42]
    xu = np.array([0, 1, 0x80000000, 0xFFFFFFFF, 0], dtype=np.uint32)
    assert oracle.compact_positive_u32(xu).tolist() == [1, 0x80000000, 0xFFFFFFFF]


@pytest.mark.parametrize("n", [0, 1, 7, 64])
def test_compact_positive_brute_force(n):
    x = si.workload_positive_f32(n, 0.5, seed=11)
    got = oracle.compact_positive_f32(x)
    assert [float(v) for v in got] == [float(v) for v in x if float(v) > 0.0]


def test_compact_positive_agrees_with_flag_form():
    # The predicate form equals the flag form with flags = (x > 0), through
    # the separately pinned compact_u32 and the exclusive flag scan.
    n = 1 << 15
    for p in (0.01, 0.5, 0.99):
        x = si.workload_positive_f32(n, p, seed=12)
        f01 = (x > 0).astype(np.uint8)
        got = oracle.compact_positive_f32(x)
        assert np.array_equal(got.view(np.uint32), oracle.compact_u32(x.view(np.uint32), f01))
        pos = oracle.scan_u32(f01.astype(np.uint32), False)
        assert got.size == int(pos[-1]) + int(f01[-1])
    xi = si.uniform_int32(n, -50, 50, seed=13)
    assert np.array_equal(oracle.compact_positive_i32(xi).view(np.uint32),
                          oracle.compact_u32(xi.view(np.uint32), (xi > 0).astype(np.uint8)))


def test_moe_worked_example():
    # E = 4 experts, GEMM tile 4: counts [2, 0, 4, 1] round up to segments
    # [4, 0, 4, 4], so the starts are [0, 4, 4, 8] and the padded total 12.
    counts, offsets = oracle.moe_counts_offsets(np.array([0, 2, 2, 3, 0, 2, 2]), 4, 4)
    assert counts.tolist() == [2, 0, 4, 1]
    assert offsets.tolist() == [0, 4, 4, 8, 12]


def test_moe_histogram_is_bincount_and_align1_is_the_scan():
    ids = si.topk_ids(4096, 8, 256, seed=6)
    counts, offsets = oracle.moe_counts_offsets(ids, 256, 1)
    assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=256).astype(np.uint32))
    assert counts.sum() == ids.size
    # with a tile of one element the starts are the exclusive scan of the counts
    assert np.array_equal(offsets[:-1].astype(np.uint32), oracle.scan_u32(counts, False))
    assert int(offsets[-1]) == ids.size


@pytest.mark.parametrize("align", [1, 16, 64, 128])
def test_moe_alignment_invariants(align):
    ids = si.topk_ids(1000, 6, 160, seed=7)
    counts, offsets = oracle.moe_counts_offsets(ids, 160, align)
    seg = np.diff(offsets.astype(np.int64))
    assert (seg % align == 0).all()
    assert (seg >= counts).all() and (seg < counts.astype(np.int64) + align).all()
    assert ((counts == 0) == (seg == 0)).all()
    assert offsets[0] == 0


def test_moe_degenerate():
    m = 1000
    # every token on one expert: a single segment of ceil(m / 64) tiles
    counts, offsets = oracle.moe_counts_offsets(np.full(m, 3), 5, 64)
    assert counts.tolist() == [0, 0, 0, m, 0]
    assert offsets.tolist() == [0, 0, 0, 0, 1024, 1024]
    # ids outside [0, E) belong to no expert
    counts, offsets = oracle.moe_counts_offsets(np.array([-1, 5, 7, 0, 4]), 5, 8)
    assert counts.tolist() == [1, 0, 0, 0, 1]
    assert offsets.tolist() == [0, 8, 8, 8, 8, 16]
    counts, offsets = oracle.moe_counts_offsets(np.zeros(0, np.int32), 3, 64)
    assert counts.tolist() == [0, 0, 0] and offsets.tolist() == [0, 0, 0, 0]


def test_tile_model_against_page_tables(golden_dir):
    levels, totals = [], {}
    with open(os.path.join(golden_dir, "blelloch_tile_model.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            if parts[0] == "total":
                totals[parts[1]] = int(parts[2])
            else:
                levels.append([int(p) for p in parts])
    assert len(levels) == 12
    tile = 4096
    for stride, lanes, warps, plain, pad1, pad2 in levels:
        assert tile // (2 * stride) == lanes
        assert oracle.blelloch_level_warps(tile, stride) == warps
        assert oracle.blelloch_level_degree(tile, stride, oracle.LAYOUT_PLAIN) == plain
        assert oracle.blelloch_level_degree(tile, stride, oracle.LAYOUT_PAD32) == pad1
        assert oracle.blelloch_level_degree(tile, stride, oracle.LAYOUT_PAD32_1024) == pad2
    assert oracle.hillis_steele_adds(tile) == totals["hillis_steele_adds"]
    assert oracle.hillis_steele_requests(tile) == totals["hillis_steele_requests"]
    assert oracle.blelloch_adds(tile) == totals["blelloch_adds"]
    assert oracle.blelloch_requests(tile, oracle.LAYOUT_PLAIN) == totals["blelloch_plain_requests"]
    assert oracle.blelloch_requests(tile, oracle.LAYOUT_PAD32) == totals["blelloch_pad32_requests"]
    assert oracle.blelloch_requests(tile, oracle.LAYOUT_PAD32_1024) == totals["blelloch_pad32_1024_requests"]


def test_work_closed_forms(golden_dir):
    with open(os.path.join(golden_dir, "hillis_steele_work.txt")) as f:
        rows = [[int(v) for v in l.split()] for l in f if l.strip() and not l.startswith("#")]
    for threads, steps, adds, seq in rows:
        assert int(math.log2(threads)) == steps
        assert oracle.hillis_steele_adds(threads) == adds
        assert threads - 1 == seq
    for k in range(1, 13):
        n = 1 << k
        assert oracle.hillis_steele_adds(n) == n * k - (n - 1)  # n log2 n - (n - 1)
        assert oracle.blelloch_adds(n) == 2 * (n - 1)


# ---- widened and 64-bit scans ----

M64 = 1 << 64


def _py_scan(vals, inclusive, mod=None):
    out, acc = [], 0
    for v in vals:
        if inclusive:
            acc += v
            out.append(acc if mod is None else acc % mod)
        else:
            out.append(acc if mod is None else acc % mod)
            acc += v
    return out


def test_worked_examples_wide(golden_dir):
    for name, x, inc, exc, src in _worked_examples(golden_dir):
        if x is None or any(v < 0 for v in x):
            continue
        a = np.array(x)
        for inclusive, want in ((True, inc), (False, exc)):
            if want is None:
                continue
            assert oracle.scan_u32_u64(a, inclusive).tolist() == want, name
            assert oracle.scan_i32_i64(a, inclusive).tolist() == want, name
            assert oracle.scan_i64(a, inclusive).tolist() == want, name
            assert oracle.scan_f64(a.astype(np.float64), inclusive).tolist() == want, name


@pytest.mark.parametrize("n", [1, 2, 17, 64])
@pytest.mark.parametrize("inclusive", [True, False])
def test_brute_force_widened(n, inclusive):
    xu = si.uniform_u32(n, seed=40)
    xu[::3] = 0xFFFFFFFF  # sums pass 2^32 quickly
    assert oracle.scan_u32_u64(xu, inclusive).tolist() == _py_scan([int(v) for v in xu], inclusive)
    xi = si.uniform_int32(n, -(2**31), 2**31 - 1, seed=41)
    assert oracle.scan_i32_i64(xi, inclusive).tolist() == _py_scan([int(v) for v in xi], inclusive)


@pytest.mark.parametrize("inclusive", [True, False])
def test_brute_force_i64_wraps_mod_2_64(inclusive):
    n = 64
    hi = si.uniform_u32(n, seed=42).astype(np.uint64)
    lo = si.uniform_u32(n, seed=43).astype(np.uint64)
    x = ((hi << np.uint64(32)) | lo).view(np.int64)
    want = [(v - M64 if v >= 1 << 63 else v) for v in _py_scan([int(v) for v in x], inclusive, mod=M64)]
    assert oracle.scan_i64(x, inclusive).tolist() == want


def test_widened_low_bits_are_the_32_bit_scan():
    n = 1 << 16
    x = si.uniform_u32(n, seed=44)
    for inclusive in (True, False):
        wide = oracle.scan_u32_u64(x, inclusive)
        assert np.array_equal((wide & np.uint64(0xFFFFFFFF)).astype(np.uint32), oracle.scan_u32(x, inclusive))
        xi = x.view(np.int32)
        wi = oracle.scan_i32_i64(xi, inclusive)
        assert np.array_equal(wi.astype(np.uint64).astype(np.uint32).view(np.int32), oracle.scan_i32(xi, inclusive))


def test_f64_compensation_classic_case():
    # 1 + 1e100 + 1 - 1e100 = 2 exactly; an uncompensated float64 running
    # sum returns 0 for the last prefix.
    x = np.array([1.0, 1e100, 1.0, -1e100], dtype=np.float64)
    assert oracle.scan_f64(x, True).tolist() == [1.0, 1e100, 1e100, 2.0]
    assert oracle.scan_f64(x, False).tolist() == [0.0, 1.0, 1e100, 1e100]


@pytest.mark.parametrize("n", [1, 5, 64])
def test_f64_within_one_rounding_of_exact(n):
    # random doubles over 40 binades, both signs: exact rational prefixes
    u = si.uniform_f32(n, seed=45).astype(np.float64)
    e = si.uniform_int32(n, -20, 20, seed=46).astype(np.float64)
    sgn = np.where(si.bernoulli_flags(n, 0.5, seed=47) != 0, 1.0, -1.0)
    x = sgn * (u + 0.5) * np.exp2(e)
    u64 = 2.0 ** -53
    for inclusive in (True, False):
        got = oracle.scan_f64(x, inclusive)
        acc = Fraction(0)
        abs_acc = Fraction(0)
        for i in range(n):
            if inclusive:
                acc += Fraction(float(x[i]))
                abs_acc += abs(Fraction(float(x[i])))
            err = abs(Fraction(float(got[i])) - acc)
            bound = 2 * u64 * abs(acc) + 8 * n * u64 * u64 * abs_acc
            assert err <= bound, (i, float(err), float(bound))
            if not inclusive:
                acc += Fraction(float(x[i]))
                abs_acc += abs(Fraction(float(x[i])))


def test_f64_integer_valued_is_exact():
    n = 100_000
    x = si.uniform_int32(n, -(2**20), 2**20, seed=48).astype(np.float64)
    want = np.cumsum(x.astype(np.int64))  # |prefix| < 2^37, exact in float64
    assert np.array_equal(oracle.scan_f64(x, True), want.astype(np.float64))


def test_abs_prefix_f64_exact():
    n = 64
    x = (si.uniform_f32(n, seed=49).astype(np.float64) - 0.5) * np.exp2(si.uniform_int32(n, -30, 30, seed=50))
    got = oracle.abs_prefix_f64(x)
    acc = Fraction(0)
    for i in range(n):
        acc += abs(Fraction(float(x[i])))
        assert abs(Fraction(float(got[i])) - acc) <= 2 * (2.0 ** -53) * acc


# ---- batched (per-row) scans ----

def test_rows_worked_example():
    x = np.array([[3, 1, 7, 0], [4, 1, 6, 3]], dtype=np.int32)
    assert oracle.scan_rows(x, True).tolist() == [[3, 4, 11, 11], [4, 5, 11, 14]]
    assert oracle.scan_rows(x, False).tolist() == [[0, 3, 4, 11], [0, 4, 5, 11]]


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 1), (1, 7), (5, 64), (64, 3)])
def test_rows_all_ones_restart_at_every_row(rows, cols):
    x = np.ones((rows, cols), dtype=np.uint32)
    inc = np.tile(np.arange(1, cols + 1, dtype=np.uint32), (rows, 1))
    assert np.array_equal(oracle.scan_rows(x, True), inc)
    assert np.array_equal(oracle.scan_rows(x, False), inc - 1)


def test_rows_brute_force_and_one_row_is_the_flat_scan():
    x = si.uniform_int32(7 * 33, -(2**31), 2**31 - 1, seed=70).reshape(7, 33)
    got = oracle.scan_rows(x, True)
    for r in range(7):
        acc = 0
        for c in range(33):
            acc += int(x[r, c])
            assert int(got[r, c]) == (acc + 2**31) % 2**32 - 2**31
    flat = si.workload_int_pm1000(1000, seed=2)
    assert np.array_equal(oracle.scan_rows(flat.reshape(1, -1), False)[0], oracle.scan_i32(flat, False))
    xf = si.uniform_f32(4 * 50, seed=71).reshape(4, 50)
    for r in range(4):
        assert np.array_equal(oracle.scan_rows(xf, True)[r], oracle.scan_f32(xf[r], True))
        assert np.array_equal(oracle.abs_prefix_rows_f32(xf)[r], oracle.abs_prefix_f32(xf[r]))


# ---- segmented scans ----

def test_segments_worked_example():
    x = np.array([3, 1, 7, 0, 4, 1, 6, 3], dtype=np.int32)
    # segments [0,3), [3,3) (empty), [3,8)
    assert oracle.scan_segments(x, [0, 3, 3, 8], True).tolist() == [3, 4, 11, 0, 4, 5, 11, 14]
    assert oracle.scan_segments(x, [0, 3, 3, 8], False).tolist() == [0, 3, 4, 0, 0, 4, 5, 11]


def test_segments_special_cases():
    x = si.workload_int_pm1000(1000, seed=2)
    assert np.array_equal(oracle.scan_segments(x, [0, 1000], True), oracle.scan_i32(x, True))
    unit = np.arange(1001, dtype=np.uint64)  # every element its own segment
    assert np.array_equal(oracle.scan_segments(x, unit, True), x)
    assert (oracle.scan_segments(x, unit, False) == 0).all()
    rows = np.arange(0, 1001, 100, dtype=np.uint64)  # equal lengths: the batched rows
    assert np.array_equal(oracle.scan_segments(x, rows, False), oracle.scan_rows(x.reshape(10, 100), False).ravel())


@pytest.mark.parametrize("inclusive", [True, False])
def test_segments_brute_force(inclusive):
    n = 300
    x = si.uniform_int32(n, -(2**31), 2**31 - 1, seed=91)
    offsets = si.segment_offsets(n, 7.0, seed=92, empty_frac=0.2)
    got = oracle.scan_segments(x, offsets, inclusive)
    want = np.empty(n, dtype=np.int64)
    for s in range(offsets.size - 1):
        acc = 0
        for i in range(int(offsets[s]), int(offsets[s + 1])):
            if inclusive:
                acc += int(x[i])
                want[i] = acc
            else:
                want[i] = acc
                acc += int(x[i])
    assert got.tolist() == [((v + 2**31) % 2**32) - 2**31 for v in want.tolist()]
    xf = si.uniform_f32(n, seed=93)
    assert np.array_equal(oracle.abs_prefix_segments_f32(xf, offsets), oracle.scan_segments(xf, offsets, True))
