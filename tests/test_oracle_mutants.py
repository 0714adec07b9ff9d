"""The oracle's pins must catch plausible mistakes.  Each case below plants
one mistake in a copy of the oracle's C source (in a temporary directory,
on the CPU), builds it, and checks that at least one pin fails against it.
The oracle itself is never modified."""

from __future__ import annotations

import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
import seeded_inputs as si

HERE = os.path.dirname(os.path.abspath(__file__))
M64 = 1 << 64
ORACLE_DIR = os.path.join(os.path.dirname(HERE), "oracle")

# (file, text to find, replacement, what the mistake is)
MUTANTS = [
    ("scan_ref.c", "            y[i] = (int32_t)(uint32_t)acc;\n            acc += xi;",
     "            acc += xi;\n            y[i] = (int32_t)(uint32_t)acc;", "int32 exclusive becomes inclusive"),
    ("scan_ref.c", "for (size_t i = 0; i < n; ++i) {\n        uint64_t xi",
     "for (size_t i = 1; i < n; ++i) {\n        uint64_t xi", "int32 scan skips element 0"),
    ("scan_ref.c", "uint64_t xi = (uint64_t)(int64_t)x[i];",
     "uint64_t xi = (uint64_t)(int64_t)(int16_t)x[i];", "int32 inputs truncated to 16 bits"),
    ("scan_ref.c", "    double acc = 0.0;\n    for (size_t i = 0; i < n; ++i) {\n        if (inclusive) {\n            acc += (double)x[i];",
     "    float acc = 0.0f;\n    for (size_t i = 0; i < n; ++i) {\n        if (inclusive) {\n            acc += x[i];",
     "fp32 inclusive summed in fp32"),
    ("scan_ref.c", "            acc += x[i];\n            y[i] = (uint32_t)acc;",
     "            acc += x[i] - 1u;\n            y[i] = (uint32_t)acc;", "uint32 inclusive drops a term"),
    ("scan_ref.c", "acc += v < 0.0 ? -v : v;", "acc += v;", "normaliser without the absolute value"),
    ("scan_ref.c", "if (flags[i] != 0) {", "if (flags[i] == 1) {", "compaction only keeps flag value 1"),
    ("scan_ref.c", "            out[count] = keys[i];\n            count += 1;",
     "            count += 1;\n            out[count - 1] = keys[i - (i > 0)];", "compaction copies the wrong index"),
    ("scan_ref.c", "if (x[i] > 0.0f) {", "if (x[i] >= 0.0f) {", "predicate keeps zeros"),
    ("scan_ref.c", "if (x[i] > 0) {", "if (x[i] >= 0) {", "int32 predicate keeps zeros"),
    ("scan_ref.c", "if (x[i] > 0u) {", "if ((int32_t)x[i] > 0) {", "uint32 predicate compares signed"),
    ("scan_ref.c", "uint64_t blocks = ((uint64_t)counts[e] + align - 1) / align;",
     "uint64_t blocks = (uint64_t)counts[e] / align;", "MoE segments rounded down"),
    ("scan_ref.c", "offsets[e + 1] = offsets[e] + blocks * align;",
     "offsets[e + 1] = blocks * align;", "MoE offsets not accumulated"),
    ("scan_ref.c", "counts[ids[i]] += 1;", "counts[ids[i]] += (i + 1 < m);", "MoE histogram drops the last id"),
    ("scan_ref.c", "uint64_t *y, size_t n, int inclusive)\n{\n    uint64_t acc = 0;",
     "uint64_t *y, size_t n, int inclusive)\n{\n    uint32_t acc = 0;", "widened scan keeps a 32-bit sum"),
    ("scan_ref.c", "int64_t *y, size_t n, int inclusive)\n{\n    int64_t acc = 0;",
     "int64_t *y, size_t n, int inclusive)\n{\n    uint32_t acc = 0;", "int32 -> int64 loses the sign"),
    ("scan_ref.c", "            acc += (uint64_t)x[i];\n            y[i] = (int64_t)acc;",
     "            y[i] = (int64_t)acc;\n            acc += (uint64_t)x[i];", "int64 inclusive becomes exclusive"),
    ("scan_ref.c", "if (inclusive)\n            y[i] = sum + comp;", "if (inclusive)\n            y[i] = sum;",
     "fp64 inclusive drops the compensation"),
    ("scan_ref.c", "if (as >= av)", "if (as <= av)", "fp64 compensation takes the wrong branch"),
    ("scan_ref.c", "        oracle_scan_u32(x + r * cols, y + r * cols, cols, inclusive);",
     "        oracle_scan_u32(x + r * cols, y + r * cols, cols - (r > 0), inclusive);", "batched scan skips a column"),
    ("scan_ref.c", "        oracle_scan_i32(x + r * cols, y + r * cols, cols, inclusive);",
     "        oracle_scan_i32(x + r * cols, y + r * cols, cols, !inclusive);",
     "batched int32 scan flips inclusive"),
    ("scan_ref.c", "oracle_scan_i32(x + offsets[s], y + offsets[s], (size_t)(offsets[s + 1] - offsets[s]), inclusive);",
     "oracle_scan_i32(x + offsets[s], y + offsets[s], (size_t)(offsets[s + 1] - offsets[s]) - (s + 1 == S), inclusive);",
     "segmented scan drops the last element"),
    ("tile_model.c", "return i + i / 32 + i / 1024;", "return i + i / 32 + i / 512;", "two-term padding uses /512"),
    ("tile_model.c", "return i + i / 32;\n", "return i + i / 16;\n", "one-term padding uses /16"),
    ("tile_model.c", "total += 2 * level;", "total += level;", "model counts one sweep"),
    ("tile_model.c", "for (uint64_t i = offset; i < n; ++i)",
     "for (uint64_t i = offset - 1; i < n; ++i)", "Hillis-Steele counts one add too many"),
]


def _checks(lib):
    """A compact run of the pins, parameterised on the library under test.
    Returns the names of the pins that failed."""
    failed = []

    def pin(name, fn):
        try:
            ok = fn()
        except Exception:
            ok = False
        if not ok:
            failed.append(name)

    x8 = np.array([3, 1, 7, 0, 4, 1, 6, 3], dtype=np.int32)
    inc8 = [3, 4, 11, 11, 15, 16, 22, 25]
    exc8 = [0, 3, 4, 11, 11, 15, 16, 22]
    pin("worked_i32_incl", lambda: oracle.scan_i32(x8, True, lib=lib).tolist() == inc8)
    pin("worked_i32_excl", lambda: oracle.scan_i32(x8, False, lib=lib).tolist() == exc8)
    pin("worked_u32_incl", lambda: oracle.scan_u32(x8.astype(np.uint32), True, lib=lib).tolist() == inc8)
    pin("worked_u32_excl", lambda: oracle.scan_u32(x8.astype(np.uint32), False, lib=lib).tolist() == exc8)
    pin("worked_f32_incl", lambda: oracle.scan_f32(x8.astype(np.float32), True, lib=lib).tolist() == inc8)
    pin("worked_f32_excl", lambda: oracle.scan_f32(x8.astype(np.float32), False, lib=lib).tolist() == exc8)

    big = np.full(4096, 2_000_000_000, dtype=np.int32)
    pin("wrap_two_routes", lambda: np.array_equal(
        oracle.scan_i32(big, True, lib=lib).view(np.uint32),
        (np.arange(1, 4097, dtype=np.uint64) * 2_000_000_000 % (1 << 32)).astype(np.uint32)))

    xf = si.uniform_f32(64, seed=77)
    xf = np.where(np.arange(64) % 3 == 1, -xf, xf).astype(np.float32)

    def exact_f32():
        got = oracle.scan_f32(xf, True, lib=lib)
        acc = Fraction(0)
        for i in range(64):
            acc += Fraction(float(xf[i]))
            if Fraction(float(got[i])) != acc:
                return False
        return True

    pin("brute_force_f32", exact_f32)

    def abs_pin():
        a = oracle.abs_prefix_f32(xf, lib=lib)
        return Fraction(float(a[-1])) == sum((abs(Fraction(float(v))) for v in xf), Fraction(0))

    pin("abs_prefix", abs_pin)

    keys = si.uniform_u32(1000, seed=5)
    flags = si.bernoulli_flags(1000, 0.5, seed=6)
    flags = np.where(np.arange(1000) % 7 == 3, 200, flags).astype(np.uint8)
    pin("compact_brute", lambda: oracle.compact_u32(keys, flags, lib=lib).tolist()
        == [int(k) for k, f in zip(keys, flags) if f != 0])
    xp = np.array([0.5, -1.0, 0.0, 2.0, -0.0, 3.5], dtype=np.float32)
    pin("compact_positive", lambda: oracle.compact_positive_f32(xp, lib=lib).tolist() == [0.5, 2.0, 3.5])
    xi = np.array([5, 0, -3, 2147483647, -2147483648, 1], dtype=np.int32)
    pin("compact_positive_i32", lambda: oracle.compact_positive_i32(xi, lib=lib).tolist() == [5, 2147483647, 1])
    xu = np.array([0, 7, 0x80000000, 0, 0xFFFFFFFF], dtype=np.uint32)
    pin("compact_positive_u32",
        lambda: oracle.compact_positive_u32(xu, lib=lib).tolist() == [7, 0x80000000, 0xFFFFFFFF])

    def moe_pin():
        c, o = oracle.moe_counts_offsets(np.array([0, 2, 2, 3, 0, 2, 2]), 4, 4, lib=lib)
        return c.tolist() == [2, 0, 4, 1] and o.tolist() == [0, 4, 4, 8, 12]

    pin("moe_worked", moe_pin)

    xw = np.array([0xFFFFFFFF, 0xFFFFFFFF, 5, 0xFFFFFFFF], dtype=np.uint32)
    pin("widened_u64", lambda: oracle.scan_u32_u64(xw, True, lib=lib).tolist()
        == [4294967295, 8589934590, 8589934595, 12884901890])
    xs = np.array([-5, 3, -(2**31), 7], dtype=np.int32)
    pin("widened_i64", lambda: oracle.scan_i32_i64(xs, False, lib=lib).tolist() == [0, -5, -2, -2147483650])
    x64 = np.array([2**62, 2**62, 2**62, 5], dtype=np.int64)
    pin("i64_wrap", lambda: oracle.scan_i64(x64, True, lib=lib).tolist()
        == [2**62, 2**63 - M64, 3 * 2**62 - M64, 3 * 2**62 + 5 - M64])
    xn = np.array([1.0, 1e100, 1.0, -1e100], dtype=np.float64)
    pin("f64_neumaier", lambda: oracle.scan_f64(xn, True, lib=lib).tolist() == [1.0, 1e100, 1e100, 2.0]
        and oracle.scan_f64(xn[::-1].copy(), True, lib=lib).tolist() == [-1e100, -1e100, 1.0, 2.0])

    xr = np.array([[3, 1, 7, 0], [4, 1, 6, 3]], dtype=np.int32)
    pin("rows_i32", lambda: oracle.scan_rows(xr, True, lib=lib).tolist() == [[3, 4, 11, 11], [4, 5, 11, 14]])
    pin("rows_u32", lambda: oracle.scan_rows(xr.astype(np.uint32), False, lib=lib).tolist()
        == [[0, 3, 4, 11], [0, 4, 5, 11]])

    xs = np.array([3, 1, 7, 0, 4, 1, 6, 3], dtype=np.int32)
    pin("segments_i32", lambda: oracle.scan_segments(xs, [0, 3, 3, 8], True, lib=lib).tolist()
        == [3, 4, 11, 0, 4, 5, 11, 14])

    pin("model_plain", lambda: oracle.blelloch_requests(4096, oracle.LAYOUT_PLAIN, lib=lib) == 1534)
    pin("model_pad32", lambda: oracle.blelloch_requests(4096, oracle.LAYOUT_PAD32, lib=lib) == 294)
    pin("model_pad2", lambda: oracle.blelloch_requests(4096, oracle.LAYOUT_PAD32_1024, lib=lib) == 264)
    pin("model_hs_adds", lambda: oracle.hillis_steele_adds(4096, lib=lib) == 45057)
    return failed


def test_unmutated_oracle_passes_every_pin():
    assert _checks(oracle.load()) == []


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[3] for m in MUTANTS])
def test_mutant_is_caught(mutant, tmp_path):
    fname, find, repl, _what = mutant
    for src in ("scan_ref.c", "tile_model.c"):
        shutil.copy(os.path.join(ORACLE_DIR, src), tmp_path / src)
    text = (tmp_path / fname).read_text()
    assert text.count(find) == 1, "mutation anchor no longer matches the oracle source"
    (tmp_path / fname).write_text(text.replace(find, repl))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-w", "-o", str(so),
                    str(tmp_path / "scan_ref.c"), str(tmp_path / "tile_model.c")], check=True)
    lib = oracle.load(str(so))
    assert _checks(lib), "no pin caught the planted mistake"
