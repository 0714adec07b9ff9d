"""MoE token counts and tile-aligned offsets against the CPU oracle, bit
for bit (integer work)."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import SENTINEL, Guarded, assert_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ss():
    import stream_compaction_pass_gb300 as m
    return m


def run_moe(ss, ids: np.ndarray, num_experts: int, align: int, offset: int = 0, stream=None):
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    src = Guarded(ids.size, offset, fill=ids)
    counts = Guarded(num_experts)
    offsets = Guarded(num_experts + 1)
    ss.ss_moe_counts_offsets(src.view, num_experts, align, counts.view, offsets.view, m=ids.size, stream=stream)
    st, _ = ss.ss_stream_status(stream=stream)
    assert st == ss.SS_OK
    assert counts.guards_intact() and offsets.guards_intact(), "a store landed outside counts/offsets"
    return counts.numpy(np.uint32), offsets.numpy(np.uint32)


def check(ss, ids, num_experts, align, **kw):
    got_c, got_o = run_moe(ss, ids, num_experts, align, **kw)
    ref_c, ref_o = oracle.moe_counts_offsets(ids, num_experts, align)
    assert_equal(got_c, ref_c)
    assert_equal(got_o.astype(np.uint64), ref_o)


@pytest.mark.parametrize("tokens,top_k,experts,align", [
    (4096, 8, 256, 64),      # decode-size batch, 256 experts, top-8
    (65536, 8, 256, 64),     # prefill-size batch
    (16384, 2, 8, 16),       # few experts, top-2
    (1000, 6, 160, 128),
    (8192, 8, 16384, 1),     # the largest expert count, no padding
    (100_003, 4, 64, 1),
    (333, 3, 1000, 7),
    (1, 1, 1, 1),
    (3, 2, 5, 64),
])
def test_counts_offsets(ss, tokens, top_k, experts, align):
    check(ss, si.topk_ids(tokens, top_k, experts, seed=6), experts, align)


def test_large_batch_many_ctas(ss):
    # 2^20 tokens x top-8: every SM takes a stretch
    check(ss, si.topk_ids(1 << 20, 8, 256, seed=8), 256, 64)


def test_out_of_range_ids_are_not_counted(ss):
    ids = si.topk_ids(5000, 4, 100, seed=9).reshape(-1).copy()
    ids[::7] = -1
    ids[3::11] = 100
    ids[5::13] = 2**31 - 1
    ids[6::17] = -(2**31)
    check(ss, ids, 100, 32)


def test_all_tokens_on_one_expert(ss):
    # every shared-memory atomic hits one bin
    check(ss, np.full(300_001, 17, dtype=np.int32), 64, 64)


def test_empty(ss):
    got_c, got_o = run_moe(ss, np.zeros(0, np.int32), 12, 64)
    assert (got_c == 0).all() and (got_o == 0).all()


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unaligned_ids(ss, offset):
    check(ss, si.topk_ids(20000, 8, 256, seed=10), 256, 64, offset=offset)


def test_repeated_calls_reuse_the_ticket(ss):
    # The last CTA returns the ticket to zero; calls of different shapes in a
    # row on one stream must each see a clean ticket.
    import torch
    s = torch.cuda.Stream()
    for i, (tok, k, e, a) in enumerate([(4096, 8, 256, 64), (100, 2, 8, 1), (65536, 8, 256, 64),
                                        (4096, 8, 256, 64), (7, 1, 3, 2)]):
        check(ss, si.topk_ids(tok, k, e, seed=20 + i), e, a, stream=s.cuda_stream)


def test_offsets_feed_a_scan_consistently(ss):
    # align = 1: the offsets are the exclusive scan of the counts; checked
    # against the library's own scan of the returned counts.
    import torch
    ids = si.topk_ids(65536, 8, 256, seed=11)
    c, o = run_moe(ss, ids, 256, 1)
    d = torch.from_numpy(c.view(np.int32)).cuda()
    out = torch.empty_like(d)
    ss.scan_exclusive_u32(d, out)
    assert_equal(out.cpu().numpy().view(np.uint32), o[:-1])
    assert int(o[-1]) == ids.size
