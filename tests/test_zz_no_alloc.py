"""ss_scan_noalloc, the scan entry point that allocates nothing, checked
against the CPU oracle.

Some callers cannot call cudaMalloc: an application that serves every byte
of device memory from its own pool and forbids other allocations, or a loop
that may never pay for an allocation.  For them ss_scan_noalloc keeps its
scratch in a fixed device array instead of a per-stream workspace.  Each
case calls it through the C ABI twice in a row (the second call reuses the
scratch the first one left) and compares both outputs with the oracle: bit
for bit for integers, within the fp32 bound the other tests use (max |y -
ref| / max(1, sum_{j<=i} |x_j|) <= 1e-4); the regular entry point's output
must agree too.  This file is collected last; it also passes on its own in
a fresh process.
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


def _reference(ss, dtype, inclusive, x):
    if dtype == ss.SS_F32:
        return oracle.scan_f32(x, inclusive)  # float64
    if dtype == ss.SS_U32:
        return oracle.scan_u32(x, inclusive)
    return oracle.scan_i32(x, inclusive)


def _matches_oracle(ss, dtype, got, ref, x):
    if dtype == ss.SS_F32:
        err = oracle.fp32_normalised_error(got.view(np.float32), ref, x.view(np.float32))
        assert err <= FP32_TOL, f"normalised error {err:.3e} against the oracle"
    else:
        got = got.view(ref.dtype)
        assert np.array_equal(got, ref), f"first difference from the oracle at {int(np.argmax(got != ref))}"


CASES = [
    ("int32 exclusive, ragged", "SS_I32", False, lambda: si.workload_int_pm1000(10_000_007, seed=2)),
    ("int32 inclusive, one tile", "SS_I32", True, lambda: si.workload_int_0_100(4096, seed=0)),
    ("uint32 exclusive, digit counts", "SS_U32", False, lambda: si.workload_poisson_counts(1 << 24, seed=4)),
    ("fp32 inclusive", "SS_F32", True, lambda: si.workload_f32_unit(10_000_000, seed=1)),
    ("fp32 exclusive", "SS_F32", False, lambda: si.workload_f32_unit(1_000_003, seed=1)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_matches_oracle_twice(ss, case):
    import torch
    _name, dt_name, inclusive, make = case
    dtype = getattr(ss, dt_name)
    x = make()
    n = x.size
    ref = _reference(ss, dtype, inclusive, x)
    d_in = torch.from_numpy(np.ascontiguousarray(x).view(np.int32)).to("cuda:0")
    out = torch.empty_like(d_in)
    for _ in range(2):
        out.fill_(SENTINEL)
        _noalloc(ss, dtype, inclusive, d_in, out, n)
        torch.cuda.synchronize()
        _matches_oracle(ss, dtype, out.cpu().numpy(), ref, x)
    # the regular entry point gives the same answer
    want = torch.empty_like(d_in)
    _regular(ss, dtype, inclusive, d_in, want)
    _matches_oracle(ss, dtype, want.cpu().numpy(), ref, x)


def test_in_place_at_the_maximum_size(ss):
    import torch
    n = 1 << 30
    x = si.workload_int_pm1000(n, seed=2)
    ref = oracle.scan_i32(x, True)
    d = torch.from_numpy(x).to("cuda:0")
    for _ in range(2):
        d.copy_(torch.from_numpy(x))
        _noalloc(ss, ss.SS_I32, True, d, d, n)
        torch.cuda.synchronize()
        got = d.cpu().numpy()
        assert np.array_equal(got, ref), f"first difference from the oracle at {int(np.argmax(got != ref))}"


def test_across_the_periodic_descriptor_clear(ss):
    # The descriptors are cleared before the call that makes the call count a
    # multiple of the clear period (so that 30-bit epoch tags never meet an
    # old descriptor of the same tag); step the count to just below it and
    # check the calls before, at and after the clear against the oracle.
    import torch
    x = si.workload_int_pm1000(3_000_001, seed=2)
    ref = oracle.scan_i32(x, False)
    d_in = torch.from_numpy(x).to("cuda:0")
    out = torch.empty_like(d_in)
    period = ss.ss_debug_noalloc_clear_period()
    assert period == 1 << 29
    ss.ss_debug_set_noalloc_calls(period - 2)
    try:
        for _ in range(4):
            out.fill_(SENTINEL)
            _noalloc(ss, ss.SS_I32, False, d_in, out, x.size)
            torch.cuda.synchronize()
            assert np.array_equal(out.cpu().numpy(), ref)
    finally:
        ss.ss_debug_set_noalloc_calls(0)


def test_rejects_sizes_beyond_the_maximum(ss):
    import torch
    d = torch.zeros(16, dtype=torch.int32, device="cuda:0")
    st = ss.lib().ss_scan_noalloc(ss.SS_I32, 0, d.data_ptr(), d.data_ptr(), (1 << 30) + 1,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == ss.SS_ERR_INVALID_ARG
    with pytest.raises(ss.StreamScanError):
        ss.ss_scan_noalloc(ss.SS_F32, True, d, d, n=(1 << 31))
