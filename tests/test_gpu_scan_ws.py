"""The explicit-workspace scan (CUB's two-call shape) against the CPU oracle:
int32/uint32 bit-exact, fp32 within the normalised bound, with the caller's
scratch left full of garbage before every call."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import assert_equal

pytestmark = pytest.mark.gpu

KINDS = {"i32": (np.int32, "SS_I32"), "u32": (np.uint32, "SS_U32"), "f32": (np.float32, "SS_F32")}


@pytest.fixture(scope="module")
def ss():
    import stream_compaction_pass_gb300 as m
    return m


def _temp(ss, n, fill=0xA5):
    import torch
    bytes_ = ss.ss_scan_temp_bytes(n)
    t = torch.full((max(bytes_, 256) + 256,), fill, dtype=torch.uint8, device="cuda:0")
    off = (-t.data_ptr()) % 256  # 256-byte aligned view
    return t[off: off + max(bytes_, 256)]


def _input(kind, n):
    if kind == "i32":
        return si.workload_int_pm1000(n, seed=2)
    if kind == "u32":
        return si.uniform_u32(n, seed=95)
    return si.workload_f32_unit(n, seed=1)


def _reference(kind, x, inclusive):
    if kind == "i32":
        return oracle.scan_i32(x, inclusive)
    if kind == "u32":
        return oracle.scan_u32(x, inclusive)
    return oracle.scan_f32(x, inclusive)


@pytest.mark.parametrize("kind", ["i32", "u32", "f32"])
@pytest.mark.parametrize("n", [1, 4095, 4097, 1_000_003, 2_000_000, 50_000_001])
def test_workspace_scan_matches_oracle(ss, kind, n):
    # the sizes straddle the automatic choice (row 8 below 2e6 and from 5e7, row 7 between)
    import torch
    x = _input(kind, n)
    d_in = torch.from_numpy(x).to("cuda:0")
    d_out = torch.empty_like(d_in)
    temp = _temp(ss, n)
    for inclusive in (True, False):
        temp.fill_(0xFF)  # the call must not depend on what the scratch held
        ss.ss_scan_ws(getattr(ss, KINDS[kind][1]), inclusive, d_in, d_out, temp)
        assert ss.ss_temp_status(temp) == (ss.SS_OK, -1)
        got = d_out.cpu().numpy()
        ref = _reference(kind, x, inclusive)
        if kind == "f32":
            err = oracle.fp32_normalised_error(got, ref, x)
            assert err <= 1e-4, f"fp32 error {err:.3e}"
        else:
            assert_equal(got, ref)


def test_one_scratch_for_many_sizes_and_in_place(ss):
    import torch
    big = si.workload_int_pm1000(3_000_017, seed=2)
    temp = _temp(ss, big.size)
    d = torch.from_numpy(big).to("cuda:0")
    o = torch.empty_like(d)
    for n in (3_000_017, 17, 1_000_000, 65_537, 3_000_017):
        ss.ss_scan_ws(ss.SS_I32, True, d[:n], o[:n], temp)
        assert_equal(o[:n].cpu().numpy(), oracle.scan_i32(big[:n], True))
    d2 = d.clone()
    ss.ss_scan_ws(ss.SS_I32, False, d2, d2, temp)  # in place
    assert_equal(d2.cpu().numpy(), oracle.scan_i32(big, False))
    assert ss.ss_temp_status(temp) == (ss.SS_OK, -1)
    assert ss.ss_stream_status()[0] == ss.SS_OK  # the per-stream workspace is not involved


def test_workspace_timeout_is_reported_through_temp(ss):
    import torch
    n = 64 * 18432 + 9
    x = si.workload_int_pm1000(n, seed=2)
    d = torch.from_numpy(x).to("cuda:0")
    o = torch.empty_like(d)
    temp = _temp(ss, n)
    ss.ss_debug_set_lookback_fault(5, 2_000_000)
    try:
        ss.ss_scan_ws(ss.SS_I32, True, d, o, temp)
        st, tile = ss.ss_temp_status(temp)
    finally:
        ss.ss_debug_set_lookback_fault(-1, 0)
    assert st == ss.SS_ERR_LOOKBACK_TIMEOUT and tile > 5
    ss.ss_scan_ws(ss.SS_I32, True, d, o, temp)
    assert ss.ss_temp_status(temp) == (ss.SS_OK, -1)
    assert_equal(o.cpu().numpy(), oracle.scan_i32(x, True))


def test_too_small_scratch_is_rejected(ss):
    import torch
    n = 100_000
    d = torch.zeros(n, dtype=torch.int32, device="cuda:0")
    temp = _temp(ss, n)
    with pytest.raises(ss.StreamScanError):
        ss.ss_scan_ws(ss.SS_I32, True, d, d, temp, temp_bytes=ss.ss_scan_temp_bytes(n) - 8)
