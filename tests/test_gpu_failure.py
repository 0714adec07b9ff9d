"""The look-back's failure path, exercised without faulting the GPU: a test
hook makes one tile skip publishing, so its successor's bounded wait runs
out (a 2 ms limit); the kernel records the error in the stream's status word
and returns, the host reads it, and the context stays usable."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import assert_equal

pytestmark = pytest.mark.gpu

TILE = 4096


@pytest.fixture(scope="module", params=[0, 2, 5, 6, 8, 10],
                ids=["one-cta-per-tile", "persistent", "warp-specialised", "lean", "claimed-tiles", "two-level"])
def ss(request):
    import stream_compaction_pass_gb300 as m
    m.ss_set_scan_config(request.param)
    yield m
    m.ss_debug_set_lookback_fault(-1, 0)
    m.ss_set_scan_config(-1)  # the library's initial, automatic setting


def _scan(ss, x):
    import torch
    d_in = torch.from_numpy(x.view(np.int32)).to("cuda:0")
    d_out = torch.zeros_like(d_in)
    ss.scan_inclusive_i32(d_in, d_out)
    return d_out


@pytest.mark.parametrize("dead_tile", [0, 5, 63])
def test_scan_timeout_is_reported_and_recovered(ss, dead_tile):
    x = si.workload_int_pm1000(64 * ss.ss_scan_tile_elems() + 9, seed=2)
    ss.ss_debug_set_lookback_fault(dead_tile, 2_000_000)
    try:
        _scan(ss, x)
        st, tile = ss.ss_stream_status()
    finally:
        ss.ss_debug_set_lookback_fault(-1, 0)
    assert st == ss.SS_ERR_LOOKBACK_TIMEOUT
    assert tile > dead_tile
    # The status was cleared by reading it, and the next call is correct.
    d_out = _scan(ss, x)
    assert ss.ss_stream_status() == (ss.SS_OK, -1)
    assert_equal(d_out.cpu().numpy(), oracle.scan_i32(x, True))


@pytest.mark.parametrize("p", [0.5, 0.01])
def test_compaction_timeout_is_reported_and_recovered(ss, p):
    import torch
    n = 50 * 65536 + 17  # tile 7 exists for every compaction tile size (4096 to 65536)
    keys, flags = si.workload_compaction(n, p, seed=3)
    d_k = torch.from_numpy(keys.view(np.int32)).to("cuda:0")
    d_f = torch.from_numpy(flags).to("cuda:0")
    d_o = torch.empty_like(d_k)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda:0")
    ss.ss_debug_set_lookback_fault(7, 2_000_000)
    try:
        ss.compact_u32(d_k, d_f, d_o, cnt)
        st, tile = ss.ss_stream_status()
    finally:
        ss.ss_debug_set_lookback_fault(-1, 0)
    assert st == ss.SS_ERR_LOOKBACK_TIMEOUT and tile > 7
    ss.compact_u32(d_k, d_f, d_o, cnt)
    assert ss.ss_stream_status()[0] == ss.SS_OK
    c = int(cnt.item())
    assert_equal(d_o[:c].cpu().numpy().view(np.uint32), oracle.compact_u32(keys, flags))


def test_predicate_compaction_timeout_is_reported_and_recovered(ss):
    import torch
    n = 50 * 16384 + 5
    x = si.workload_positive_f32(n, 0.5, seed=5)
    d_x = torch.from_numpy(x).to("cuda:0")
    d_o = torch.empty_like(d_x)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda:0")
    ss.ss_debug_set_lookback_fault(7, 2_000_000)
    try:
        ss.compact_positive_f32(d_x, d_o, cnt)
        st, tile = ss.ss_stream_status()
    finally:
        ss.ss_debug_set_lookback_fault(-1, 0)
    assert st == ss.SS_ERR_LOOKBACK_TIMEOUT and tile > 7
    ss.compact_positive_f32(d_x, d_o, cnt)
    assert ss.ss_stream_status()[0] == ss.SS_OK
    c = int(cnt.item())
    assert_equal(d_o[:c].cpu().numpy().view(np.uint32), oracle.compact_positive_f32(x).view(np.uint32))


def test_wide_scan_timeout_is_reported_and_recovered(ss):
    import torch
    n = 40 * 8192 + 3
    x = si.uniform_int32(n, -1000, 1000, seed=2).astype(np.int64)
    d = torch.from_numpy(x).to("cuda:0")
    o = torch.empty_like(d)
    ss.ss_debug_set_lookback_fault(9, 2_000_000)
    try:
        ss.scan_inclusive_i64(d, o)
        st, tile = ss.ss_stream_status()
    finally:
        ss.ss_debug_set_lookback_fault(-1, 0)
    assert st == ss.SS_ERR_LOOKBACK_TIMEOUT and tile > 9
    ss.scan_inclusive_i64(d, o)
    assert ss.ss_stream_status() == (ss.SS_OK, -1)
    assert_equal(o.cpu().numpy(), oracle.scan_i64(x, True))


def test_f64_scan_timeout_is_reported_and_recovered(ss):
    # the fp64 kernel has its own tiles (4096 elements) and look-back loop
    import torch
    n = 80 * 4096 + 3
    x = si.uniform_int32(n, -1000, 1000, seed=2).astype(np.float64)
    d = torch.from_numpy(x).to("cuda:0")
    o = torch.empty_like(d)
    ss.ss_debug_set_lookback_fault(9, 2_000_000)
    try:
        ss.scan_exclusive_f64(d, o)
        st, tile = ss.ss_stream_status()
    finally:
        ss.ss_debug_set_lookback_fault(-1, 0)
    assert st == ss.SS_ERR_LOOKBACK_TIMEOUT and tile > 9
    ss.scan_exclusive_f64(d, o)
    assert ss.ss_stream_status() == (ss.SS_OK, -1)
    assert_equal(o.cpu().numpy(), oracle.scan_f64(x, False))
