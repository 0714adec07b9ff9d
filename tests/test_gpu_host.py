"""The host-memory scan against the oracle, on both of its paths: direct
device access to mapped pinned buffers, and chunked copies overlapped with
seeded scans (pageable buffers, or the staged mode forced)."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import assert_equal, assert_fp32_close, f32_input, f32_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[0, 1], ids=["direct", "staged"])
def ss(request):
    import stream_compaction_pass_gb300 as m
    m.ss_set_host_mode(request.param)
    yield m
    m.ss_set_host_mode(0)


@pytest.mark.parametrize("n", [1, 4097, 16 << 20, (16 << 20) + 1, 50_000_017])
def test_host_scan_int32_pinned(ss, n):
    import torch
    x = si.workload_int_pm1000(n, seed=2)
    h_in = torch.from_numpy(x).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    for inclusive in (True, False):
        ss.ss_scan_host(ss.SS_I32, inclusive, h_in, h_out)
        assert_equal(h_out.numpy(), oracle.scan_i32(x, inclusive))


def test_host_scan_pinned_in_place_and_offset(ss):
    # an interior pointer of a pinned allocation, and in == out
    import torch
    n = 3_000_001
    x = si.uniform_u32(n + 3, seed=52)
    h = torch.from_numpy(x.view(np.int32)).pin_memory()
    view = h[3:]
    ss.ss_scan_host(ss.SS_U32, True, view, view)
    assert_equal(view.numpy().view(np.uint32), oracle.scan_u32(x[3:], True))
    assert_equal(h[:3].numpy().view(np.uint32), x[:3])


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


def test_host_scan_fp32_pinned(ss):
    import torch
    n = 100_000_000
    x = f32_input(n)
    h_in = torch.from_numpy(x).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    ss.ss_scan_host(ss.SS_F32, False, h_in, h_out)
    assert_fp32_close(h_out.numpy(), f32_reference(n, False), x)
