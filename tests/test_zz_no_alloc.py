"""ss_scan_noalloc, the scan entry point that allocates nothing, must give
what the regular entry points give.

Some callers cannot call cudaMalloc: an application that serves every byte
of device memory from its own pool and forbids other allocations, or a loop
that may never pay for an allocation.  For them ss_scan_noalloc keeps its
scratch in a fixed device array instead of a per-stream workspace.  Each
case calls it through the C ABI twice in a row (the second call reuses the
scratch the first one left) and compares both outputs with the regular
entry point's: bit for bit for integers, within the fp32 bound the other
tests use.  This file is collected last; it also passes on its own in a
fresh process.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import FP32_TOL, SENTINEL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import stream_compaction_pass_gb300 as m
    return m


def _regular(ss, dtype, inclusive, d_in, d_out):
    name = {(ss.SS_I32, True): "scan_inclusive_i32", (ss.SS_I32, False): "scan_exclusive_i32",
            (ss.SS_U32, True): "scan_inclusive_u32", (ss.SS_U32, False): "scan_exclusive_u32",
            (ss.SS_F32, True): "scan_inclusive_f32", (ss.SS_F32, False): "scan_exclusive_f32"}[(dtype, inclusive)]
    getattr(ss, name)(d_in, d_out)


def _noalloc(ss, dtype, inclusive, d_in, d_out, n):
    import torch
    st = ss.lib().ss_scan_noalloc(dtype, int(inclusive), d_in.data_ptr(), d_out.data_ptr(), n,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == ss.SS_OK, ss.ss_status_string(st)


def _same(ss, dtype, got, want, x):
    if dtype == ss.SS_F32:
        g, w = got.view(np.float32).astype(np.float64), want.view(np.float32).astype(np.float64)
        err = float((np.abs(g - w) / np.maximum(1.0, oracle.abs_prefix_f32(x.view(np.float32)))).max())
        assert err <= FP32_TOL, f"normalised difference {err:.3e}"
    else:
        assert np.array_equal(got, want), f"first difference at {int(np.argmax(got != want))}"


CASES = [
    ("int32 exclusive, ragged", "SS_I32", False, lambda: si.workload_int_pm1000(10_000_007, seed=2)),
    ("int32 inclusive, one tile", "SS_I32", True, lambda: si.workload_int_0_100(4096, seed=0)),
    ("uint32 exclusive, digit counts", "SS_U32", False, lambda: si.workload_poisson_counts(1 << 24, seed=4)),
    ("fp32 inclusive", "SS_F32", True, lambda: si.workload_f32_unit(10_000_000, seed=1)),
    ("fp32 exclusive", "SS_F32", False, lambda: si.workload_f32_unit(1_000_003, seed=1)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_matches_regular_entry_twice(ss, case):
    import torch
    _name, dt_name, inclusive, make = case
    dtype = getattr(ss, dt_name)
    x = make()
    n = x.size
    d_in = torch.from_numpy(np.ascontiguousarray(x).view(np.int32)).to("cuda:0")
    want = torch.empty_like(d_in)
    _regular(ss, dtype, inclusive, d_in, want)
    want_np = want.cpu().numpy()
    out = torch.empty_like(d_in)
    for _ in range(2):
        out.fill_(SENTINEL)
        _noalloc(ss, dtype, inclusive, d_in, out, n)
        torch.cuda.synchronize()
        _same(ss, dtype, out.cpu().numpy(), want_np, x)


def test_in_place_at_the_maximum_size(ss):
    import torch
    n = 1 << 30
    x = si.workload_int_pm1000(n, seed=2)
    d = torch.from_numpy(x).to("cuda:0")
    want = torch.empty_like(d)
    ss.scan_inclusive_i32(d, want)
    want_np = want.cpu().numpy()
    del want
    for _ in range(2):
        d.copy_(torch.from_numpy(x))
        _noalloc(ss, ss.SS_I32, True, d, d, n)
        torch.cuda.synchronize()
        assert np.array_equal(d.cpu().numpy(), want_np)


def test_rejects_sizes_beyond_the_maximum(ss):
    import torch
    d = torch.zeros(16, dtype=torch.int32, device="cuda:0")
    st = ss.lib().ss_scan_noalloc(ss.SS_I32, 0, d.data_ptr(), d.data_ptr(), (1 << 30) + 1,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == ss.SS_ERR_INVALID_ARG
    with pytest.raises(ss.StreamScanError):
        ss.ss_scan_noalloc(ss.SS_F32, True, d, d, n=(1 << 31))
