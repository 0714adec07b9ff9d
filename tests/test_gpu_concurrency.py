"""Several streams, and several host threads, calling the library at the
same time.  Every (device, stream) pair has its own workspace (counter,
descriptors, status word), so concurrent scans, compactions and MoE counts
must not disturb one another."""

from __future__ import annotations

import threading

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import assert_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import stream_compaction_pass_gb300 as m
    return m


def test_streams_run_concurrently(ss):
    import torch
    sizes = [3_000_017, 1_000_003, 5_000_011, 777_777]
    xs = [si.workload_int_pm1000(n, seed=2) for n in sizes]
    streams = [torch.cuda.Stream() for _ in sizes]
    ins = [torch.from_numpy(x).cuda() for x in xs]
    outs = [torch.empty_like(d) for d in ins]
    keys, flags = si.workload_compaction(2_000_003, 0.3, seed=3)
    d_k = torch.from_numpy(keys.view(np.int32)).cuda()
    d_f = torch.from_numpy(flags).cuda()
    torch.cuda.synchronize()
    compacted = []
    for rep in range(3):
        for i, s in enumerate(streams):
            with torch.cuda.stream(s):
                ss.scan_exclusive_i32(ins[i], outs[i], stream=s.cuda_stream)
                ss.scan_inclusive_i32(outs[i], outs[i], stream=s.cuda_stream)  # in place, on the exclusive result
        o = torch.empty_like(d_k)
        c = torch.zeros(1, dtype=torch.int64, device="cuda")
        with torch.cuda.stream(streams[rep % len(streams)]):
            ss.compact_u32(d_k, d_f, o, c, stream=streams[rep % len(streams)].cuda_stream)
        compacted.append((o, c))
    torch.cuda.synchronize()
    for i, s in enumerate(streams):
        assert ss.ss_stream_status(stream=s.cuda_stream)[0] == ss.SS_OK
        want = oracle.scan_i32(oracle.scan_i32(xs[i], False), True)
        assert_equal(outs[i].cpu().numpy(), want)
    ref = oracle.compact_u32(keys, flags)
    for o, c in compacted:
        assert int(c.item()) == ref.size
        assert_equal(o[: ref.size].cpu().numpy().view(np.uint32), ref)


def test_host_threads_with_their_own_streams(ss):
    import torch
    errors = []

    def worker(idx: int):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            n = 1_500_000 + 1_000 * idx
            x = si.workload_f32_unit(n, seed=1)
            ids = si.topk_ids(2048 + idx, 4, 64, seed=idx)
            with torch.cuda.stream(s):
                d = torch.from_numpy(x).cuda()
                o = torch.empty_like(d)
                d_ids = torch.from_numpy(ids).cuda()
                cnt = torch.empty(64, dtype=torch.int32, device="cuda")
                off = torch.empty(65, dtype=torch.int32, device="cuda")
                for _ in range(5):
                    ss.scan_inclusive_f32(d, o, stream=s.cuda_stream)
                    ss.ss_moe_counts_offsets(d_ids, 64, 16, cnt, off, stream=s.cuda_stream)
            s.synchronize()
            st, _ = ss.ss_stream_status(stream=s.cuda_stream)
            assert st == ss.SS_OK
            err = oracle.fp32_normalised_error(o.cpu().numpy(), oracle.scan_f32(x, True), x)
            assert err <= 1e-4, err
            c_ref, o_ref = oracle.moe_counts_offsets(ids, 64, 16)
            assert np.array_equal(cnt.cpu().numpy().view(np.uint32), c_ref)
            assert np.array_equal(off.cpu().numpy().view(np.uint32).astype(np.uint64), o_ref)
        except Exception as e:  # reported by the main thread
            errors.append((idx, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker did not finish"
    assert not errors, errors
