"""The library's calls inside a captured CUDA graph.

Every call only enqueues work on its stream and, after a first call of the same size
on that stream, allocates nothing. So a sequence of calls can be captured once and
replayed; each replay reruns the whole sequence with no host work per kernel. The
replays must match the oracle, and the descriptors' epochs must keep successive replays
apart."""

from __future__ import annotations

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


def test_scan_compaction_and_moe_replay_in_a_graph(ss):
    import torch
    n = 3_000_017
    x = si.workload_int_pm1000(n, seed=2)
    keys, flags = si.workload_compaction(n, 0.3, seed=3)
    ids = si.topk_ids(4096, 8, 256, seed=6)
    d_x = torch.from_numpy(x).cuda()
    d_y = torch.empty_like(d_x)
    d_k = torch.from_numpy(keys.view(np.int32)).cuda()
    d_f = torch.from_numpy(flags).cuda()
    d_o = torch.empty_like(d_k)
    d_c = torch.zeros(1, dtype=torch.int64, device="cuda")
    d_ids = torch.from_numpy(ids).cuda()
    d_cnt = torch.empty(256, dtype=torch.int32, device="cuda")
    d_off = torch.empty(257, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()

    def work():
        ss.scan_exclusive_i32(d_x, d_y, stream=s.cuda_stream)
        ss.compact_u32(d_k, d_f, d_o, d_c, stream=s.cuda_stream)
        ss.ss_moe_counts_offsets(d_ids, 256, 64, d_cnt, d_off, stream=s.cuda_stream)

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        work()  # sizes the stream's workspace before capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        work()
    for _ in range(3):
        d_y.zero_()
        d_o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert ss.ss_stream_status(stream=s.cuda_stream)[0] == ss.SS_OK
        assert_equal(d_y.cpu().numpy(), oracle.scan_i32(x, False))
        ref = oracle.compact_u32(keys, flags)
        c = int(d_c.item())
        assert c == ref.size
        assert_equal(d_o[:c].cpu().numpy().view(np.uint32), ref)
        cnt, off = oracle.moe_counts_offsets(ids, 256, 64)
        assert_equal(d_cnt.cpu().numpy().view(np.uint32), cnt)
        assert_equal(d_off.cpu().numpy().view(np.uint32).astype(np.uint64), off)
