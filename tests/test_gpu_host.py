"""The host-memory scan (chunked copies overlapped with seeded scans)
against the oracle."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import assert_equal, assert_fp32_close, f32_input, f32_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import stream_compaction_pass_gb300 as m
    return m


@pytest.mark.parametrize("n", [1, 4097, 16 << 20, (16 << 20) + 1, 50_000_017])
def test_host_scan_int32_pinned(ss, n):
    import torch
    x = si.workload_int_pm1000(n, seed=2)
    h_in = torch.from_numpy(x).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    for inclusive in (True, False):
        ss.ss_scan_host(ss.SS_I32, inclusive, h_in, h_out)
        assert_equal(h_out.numpy(), oracle.scan_i32(x, inclusive))


def test_host_scan_in_place_pageable(ss):
    n = 40_000_001
    x = si.uniform_u32(n, seed=51)
    y = x.copy()
    ss.ss_scan_host(ss.SS_U32, False, y, y)
    assert_equal(y, oracle.scan_u32(x, False))


def test_host_scan_fp32(ss):
    n = 100_000_000
    x = f32_input(n)
    out = np.empty_like(x)
    ss.ss_scan_host(ss.SS_F32, True, x, out)
    assert_fp32_close(out, f32_reference(n, True), x)
