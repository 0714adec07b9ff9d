"""The measured ablations (reduce-then-scan with the shuffle tile scan, and
with the Blelloch tree unpadded / padded) give the oracle's results too."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import Guarded, assert_equal, assert_fp32_close, f32_input, f32_reference

pytestmark = pytest.mark.gpu

ALGOS = ["REDUCE_THEN_SCAN", "RTS_BLELLOCH", "RTS_BLELLOCH_PAD32", "RTS_BLELLOCH_PAD2"]


@pytest.fixture(scope="module")
def ss():
    import stream_compaction_pass_gb300 as m
    return m


def run_algo(ss, algo: str, dtype: int, inclusive: bool, x: np.ndarray, inplace=False):
    n = x.size
    src = Guarded(n, fill=x)
    dst = src if inplace else Guarded(n)
    ss.ss_scan(dtype, inclusive, getattr(ss, "SS_ALGO_" + algo), src.view, dst.view)
    st, _ = ss.ss_stream_status()
    assert st == ss.SS_OK
    assert dst.guards_intact()
    return dst.numpy(x.dtype)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("n", [1, 4095, 4096, 4097, 1_000_003, 10_000_000])
def test_int32(ss, algo, n):
    x = si.workload_int_pm1000(n, seed=2)
    for inclusive in (True, False):
        assert_equal(run_algo(ss, algo, ss.SS_I32, inclusive, x), oracle.scan_i32(x, inclusive))


@pytest.mark.parametrize("algo", ALGOS)
def test_uint32_inplace_and_wrap(ss, algo):
    n = 3 * 4096 + 11
    x = si.uniform_u32(n, seed=41)
    for inclusive in (True, False):
        assert_equal(run_algo(ss, algo, ss.SS_U32, inclusive, x, inplace=True), oracle.scan_u32(x, inclusive))


@pytest.mark.parametrize("algo", ALGOS)
def test_fp32(ss, algo):
    n = 100_000_000
    x = f32_input(n)
    for inclusive in (True, False):
        assert_fp32_close(run_algo(ss, algo, ss.SS_F32, inclusive, x), f32_reference(n, inclusive), x)
    y = si.structured_period4(10_000_000)
    assert_equal(run_algo(ss, algo, ss.SS_F32, True, y), oracle.scan_f32(y, True).astype(np.float32))


def test_lookback_through_generic_entry(ss):
    n = 123_457
    x = si.workload_int_pm1000(n, seed=2)
    assert_equal(run_algo(ss, "LOOKBACK", ss.SS_I32, False, x), oracle.scan_i32(x, False))
