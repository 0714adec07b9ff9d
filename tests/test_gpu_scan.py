"""Single-pass look-back scans against the CPU oracle, through the C ABI.

Integer results must match bit for bit (int32 wraps modulo 2^32); fp32
results must satisfy max_i |y_i - ref_i| / max(1, sum_{j<=i} |x_j|) <= 1e-4
against the float64 oracle, and be bit-exact on integer-valued inputs whose
prefixes stay below 2^24.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import (FP32_TOL, Guarded, assert_equal, assert_fp32_close, f32_input,
                         f32_reference, oracle_scan, poisson_input, run_named_scan, sweep_input,
                         sweep_reference)

pytestmark = pytest.mark.gpu

TILE = 4096
SWEEP_MAX = (1 << 30) + 1


DEFAULT_CONFIG = 8  # the library's row for large n (18432-element tiles claimed from the counter)


@pytest.fixture(scope="module")
def ss():
    # Most of this module runs on the large-n row; the library's
    # own initial setting (-1, chosen per call by size) is restored after it,
    # so later modules run what a caller gets.
    import stream_compaction_pass_gb300 as m
    m.ss_set_scan_config(DEFAULT_CONFIG)
    yield m
    m.ss_set_scan_config(-1)


# --- the single-tile case: int32 in [0, 100), seed 0 ----------------------

@pytest.mark.parametrize("inclusive", [True, False])
def test_single_tile_int32(ss, inclusive):
    x = si.workload_int_0_100(4096, seed=0)
    got = run_named_scan("i32", inclusive, x)
    assert_equal(got, oracle.scan_i32(x, inclusive))


# --- the pages' worked examples through the GPU ---------------------------

@pytest.mark.parametrize("kind", ["i32", "u32", "f32"])
def test_worked_example(ss, kind):
    x = np.array([3, 1, 7, 0, 4, 1, 6, 3]).astype(np.dtype({"i32": np.int32, "u32": np.uint32, "f32": np.float32}[kind]))
    assert run_named_scan(kind, True, x).tolist() == [3, 4, 11, 11, 15, 16, 22, 25]
    assert run_named_scan(kind, False, x).tolist() == [0, 3, 4, 11, 11, 15, 16, 22]


# --- int32 exclusive size sweep, seed 2, wraparound -----------------------

def _sweep_sizes():
    sizes = {1 << k for k in range(10, 31)}
    for k in (10, 12, 13, 16, 20, 24, 27, 30):
        sizes |= {(1 << k) - 1, (1 << k) + 1}
    sizes |= {10 ** k for k in range(3, 10)}
    return sorted(sizes)


@pytest.mark.parametrize("n", _sweep_sizes())
def test_int32_exclusive_size_sweep(ss, n):
    x = sweep_input(SWEEP_MAX)[:n]
    ref = sweep_reference(SWEEP_MAX)[:n]
    got = run_named_scan("i32", False, x)
    assert_equal(got, ref)


def test_int32_wraparound_happens_and_matches(ss):
    # 2^30 values of +-1000 drift far enough that partial sums leave the int32
    # range only with large inputs; force wrapping with big constants too.
    x = np.full(3 * TILE + 5, 1_900_000_000, dtype=np.int32)
    got = run_named_scan("i32", True, x)
    ref = oracle.scan_i32(x, True)
    assert_equal(got, ref)
    assert (ref < 0).any()  # it did wrap


# --- fp32 at the pages' sizes, seed 1 --------------------------------------

@pytest.mark.parametrize("n", [1_000_000, 10_000_000, 100_000_000])
@pytest.mark.parametrize("inclusive", [True, False])
def test_fp32_unit_uniform(ss, n, inclusive):
    x = f32_input(n)
    got = run_named_scan("f32", inclusive, x)
    assert_fp32_close(got, f32_reference(n, inclusive), x)


@pytest.mark.parametrize("config", [2, DEFAULT_CONFIG, -1], ids=["row2", "row8", "automatic"])
def test_fp32_runs_agree_within_the_bound(ss, config):
    # The grouping of fp32 adds depends on timing (a look-back stops at the
    # nearest published prefix), so repeated runs may differ in the last bits.
    # What every run guarantees: the bound against the float64 oracle, and so
    # at most twice the bound between two runs.
    import torch
    n = 10_000_000
    x = f32_input(n)
    ref = f32_reference(n, True)
    norm = np.maximum(1.0, oracle.abs_prefix_f32(x))
    d_in = torch.from_numpy(x).to("cuda:0")
    d_out = torch.empty_like(d_in)
    ss.ss_set_scan_config(config)
    try:
        runs = []
        for _ in range(8):
            ss.scan_inclusive_f32(d_in, d_out)
            runs.append(d_out.cpu().numpy().astype(np.float64))
    finally:
        ss.ss_set_scan_config(DEFAULT_CONFIG)
    for r in runs:
        assert float((np.abs(r - ref) / norm).max()) <= FP32_TOL
    for r in runs[1:]:
        assert float((np.abs(r - runs[0]) / norm).max()) <= 2 * FP32_TOL


def test_fp32_structured_exact(ss):
    # Every prefix is an exact integer < 2^24, so any add order is exact.
    x = si.structured_period4(10_000_000)
    got = run_named_scan("f32", True, x)
    assert_equal(got, oracle.scan_f32(x, True).astype(np.float32))
    assert got[-1] == 12_500_000.0
    y = si.structured_i_mod_8(1_049_187)
    for inclusive in (True, False):
        got = run_named_scan("f32", inclusive, y)
        assert_equal(got, oracle.scan_f32(y, inclusive).astype(np.float32))


# --- uint32 Poisson(8) digit histograms, seed 4, in-place and not ----------

@pytest.mark.parametrize("inplace", [False, True])
def test_uint32_poisson_counts(ss, inplace):
    n = 1 << 27
    x = poisson_input(n)
    got = run_named_scan("u32", False, x, inplace=inplace)
    assert_equal(got, oracle.scan_u32(x, False))


# --- edge cases --------------------------------------------------------------

# (whole tiles of the configured size, extra elements): sizes around tile
# boundaries of whatever tile the library runs with, plus small absolutes.
EDGE = [(0, 1), (0, 2), (0, 3), (0, 4), (0, 5), (0, 31), (0, 32), (0, 33), (0, 127), (0, 128),
        (0, 129), (0, 511), (0, 512), (0, 513), (0, 4095), (0, 4096), (0, 4097), (1, -1), (1, 0),
        (1, 1), (2, -1), (2, 0), (2, 1), (33, 7)]


@pytest.mark.parametrize("edge", EDGE, ids=[f"{t}T{d:+d}" for t, d in EDGE])
@pytest.mark.parametrize("kind", ["i32", "u32", "f32"])
def test_edge_sizes(ss, edge, kind):
    n = edge[0] * ss.ss_scan_tile_elems() + edge[1]
    if kind == "f32":
        x = si.structured_i_mod_8(n)  # exact in any order
    elif kind == "u32":
        x = si.uniform_u32(n, seed=21)
    else:
        x = si.uniform_int32(n, -(1 << 31), (1 << 31) - 1, seed=22)
    for inclusive in (True, False):
        got = run_named_scan(kind, inclusive, x)
        ref = oracle_scan(kind, inclusive, x)
        assert_equal(got, ref.astype(got.dtype) if kind == "f32" else ref)


def test_zero_length(ss):
    import torch
    t = torch.empty(0, dtype=torch.int32, device="cuda:0")
    ss.scan_inclusive_i32(t, t)
    st, _ = ss.ss_stream_status()
    assert st == ss.SS_OK


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_pointers(ss, offset):
    n = 5 * TILE + 77
    x = sweep_input(SWEEP_MAX)[:n]
    got = run_named_scan("i32", False, x, offset=offset)
    assert_equal(got, sweep_reference(SWEEP_MAX)[:n])


@pytest.mark.parametrize("kind", ["i32", "u32", "f32"])
def test_in_place(ss, kind):
    n = 40 * TILE + 3
    x = {"i32": sweep_input(SWEEP_MAX)[:n], "u32": poisson_input(1 << 27)[:n],
         "f32": si.structured_i_mod_8(n)}[kind]
    for inclusive in (True, False):
        got = run_named_scan(kind, inclusive, x, inplace=True)
        ref = oracle_scan(kind, inclusive, x)
        assert_equal(got, ref.astype(got.dtype) if kind == "f32" else ref)


NUM_CONFIGS = 13


@pytest.mark.parametrize("config", range(NUM_CONFIGS))
def test_every_tile_configuration(ss, config):
    assert ss.ss_scan_config_count() == NUM_CONFIGS
    default = ss.ss_scan_tile_elems()
    ss.ss_set_scan_config(config)
    try:
        tile = ss.ss_scan_tile_elems()
        for n in (tile - 1, tile, tile + 1, 17 * tile + 5, 1_000_003):
            x = sweep_input(SWEEP_MAX)[:n]
            for inclusive in (True, False):
                assert_equal(run_named_scan("i32", inclusive, x), oracle.scan_i32(x, inclusive), tile)
            f = f32_input(n)
            assert_fp32_close(run_named_scan("f32", True, f), oracle.scan_f32(f, True), f)
    finally:
        ss.ss_set_scan_config(DEFAULT_CONFIG)
    assert ss.ss_scan_tile_elems() == default


def test_repeated_launches_are_deterministic_and_epochs_advance(ss):
    # Many launches of varying size on one workspace: descriptors from a
    # previous launch must never be taken for this launch's.
    import torch
    rng = np.random.default_rng(5)
    big = sweep_input(SWEEP_MAX)[: 300 * TILE]
    d_in = torch.from_numpy(big.view(np.int32)).to("cuda:0")
    d_out = torch.empty_like(d_in)
    ref = oracle.scan_i32(big, True)
    for it in range(60):
        n = int(rng.integers(1, 300 * TILE))
        ss.scan_inclusive_i32(d_in[:n], d_out[:n])
        if it % 10 == 9 or n < 2 * TILE:
            got = d_out[:n].cpu().numpy()
            assert_equal(got, oracle.scan_i32(big[:n], True))
    ss.scan_inclusive_i32(d_in, d_out)
    first = d_out.cpu().numpy()
    ss.scan_inclusive_i32(d_in, d_out)
    assert np.array_equal(first, d_out.cpu().numpy())
    assert_equal(first, ref)
    assert ss.ss_stream_status()[0] == ss.SS_OK


def test_seeded_chunks_compose(ss):
    import torch
    n = 10 * TILE + 999
    x = sweep_input(SWEEP_MAX)[:n]
    d_in = torch.from_numpy(x.view(np.int32)).to("cuda:0")
    d_out = torch.empty_like(d_in)
    carry = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    cuts = [0, 1, TILE + 3, 3 * TILE, 7 * TILE + 1, n]
    for a, b in zip(cuts[:-1], cuts[1:]):
        ss.ss_scan_seeded(ss.SS_I32, False, d_in[a:b], d_out[a:b], carry, carry)
    assert_equal(d_out.cpu().numpy(), oracle.scan_i32(x, False))
    assert int(carry.item()) == int(oracle.scan_i32(x, True)[-1])


def test_nondefault_stream(ss):
    import torch
    s = torch.cuda.Stream()
    n = 100 * TILE + 1
    x = sweep_input(SWEEP_MAX)[:n]
    with torch.cuda.stream(s):
        d_in = torch.from_numpy(x.view(np.int32)).to("cuda:0")
        d_out = torch.empty_like(d_in)
        ss.scan_exclusive_i32(d_in, d_out)
        st, _ = ss.ss_stream_status(s)
        assert st == ss.SS_OK
        got = d_out.cpu().numpy()
    assert_equal(got, sweep_reference(SWEEP_MAX)[:n])


@pytest.mark.parametrize("config", range(NUM_CONFIGS))
def test_trace_build_scans_and_records(ss, config):
    import torch
    n = 10_000_000 + 123
    x = sweep_input(SWEEP_MAX)[:n]
    ss.ss_set_scan_config(config)
    try:
        tile = ss.ss_scan_tile_elems()
    finally:
        ss.ss_set_scan_config(DEFAULT_CONFIG)
    tiles = (n + tile - 1) // tile
    d_in = torch.from_numpy(x).to("cuda:0")
    d_out = torch.empty_like(d_in)
    tr = torch.zeros(tiles * 8, dtype=torch.int64, device="cuda:0")
    ss.ss_scan_trace(config, d_in, d_out, tr)
    assert ss.ss_stream_status()[0] == ss.SS_OK
    assert_equal(d_out.cpu().numpy(), sweep_reference(SWEEP_MAX)[:n], tile)
    rec = tr.cpu().numpy().reshape(tiles, 8)
    t = rec[:, :5]
    assert (t > 0).all()
    assert (np.diff(t, axis=1) >= 0).all()        # begin <= aggregate <= published <= resolved <= end
    assert (rec[1:, 5] >= 1).all()                # every tile after the first read a window
    assert (rec[0, 5] == 0)


@pytest.mark.parametrize("n", [1_000_003, 1_999_999, 2_000_000, 3_000_017, 49_999_999, 50_000_000, 60_000_001])
def test_automatic_configuration(ss, n):
    # the initial setting (-1) picks the 16384-element-tile row from 2e6 to
    # 5e7 elements and the 18432 row (tiles claimed from the counter) below
    # and above; both sides of each switch, int32 exclusive and fp32
    # inclusive and exclusive
    import torch
    ss.ss_set_scan_config(-1)
    try:
        x = sweep_input(SWEEP_MAX)[:n]
        d_in = torch.from_numpy(x).to("cuda:0")
        d_out = torch.empty_like(d_in)
        ss.scan_exclusive_i32(d_in, d_out)
        assert ss.ss_stream_status()[0] == ss.SS_OK
        assert_equal(d_out.cpu().numpy(), sweep_reference(SWEEP_MAX)[:n], 16384)
        f = si.workload_f32_unit(n, seed=1)
        d_f = torch.from_numpy(f).to("cuda:0")
        d_g = torch.empty_like(d_f)
        for inclusive in (True, False):
            (ss.scan_inclusive_f32 if inclusive else ss.scan_exclusive_f32)(d_f, d_g)
            assert ss.ss_stream_status()[0] == ss.SS_OK
            err = oracle.fp32_normalised_error(d_g.cpu().numpy(), oracle.scan_f32(f, inclusive), f)
            assert err <= 1e-4, f"fp32 error {err:.3e} (inclusive={inclusive})"
    finally:
        ss.ss_set_scan_config(DEFAULT_CONFIG)


def test_automatic_configuration_carries_between_chunks(ss):
    # under the automatic choice the first chunk (1e6) takes the 18432 row
    # and the others the 16384-element-tile row: a carried prefix must chain
    # through both
    import torch
    ss.ss_set_scan_config(-1)
    try:
        n = 7_000_003
        x = sweep_input(SWEEP_MAX)[:n]
        d_in = torch.from_numpy(x).to("cuda:0")
        d_out = torch.empty_like(d_in)
        carry = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        bounds = [0, 1_000_001, 4_500_000, n]
        for a, b in zip(bounds[:-1], bounds[1:]):
            ss.ss_scan_seeded(ss.SS_I32, False, d_in[a:b], d_out[a:b], carry, carry)
        assert ss.ss_stream_status()[0] == ss.SS_OK
        assert_equal(d_out.cpu().numpy(), sweep_reference(SWEEP_MAX)[:n], 16384)
        assert int(carry.item()) == int(oracle.scan_i32(x, True)[-1])
    finally:
        ss.ss_set_scan_config(DEFAULT_CONFIG)
