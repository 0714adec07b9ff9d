"""Fused single-pass compaction against the CPU oracle: output and count
bit-exact."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_helpers import SENTINEL, Guarded, assert_equal, compaction_input

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[2, 3, 4, 5, 6, 7, 1, 0],
                ids=["chunked", "chunked-dense", "chunked-sparse", "chunked-512", "chunked-512-dense",
                     "chunked-512-sparse", "selective-keys", "bulk-keys"])
def ss(request):
    import stream_compaction_pass_gb300 as m
    m.ss_set_compact_config(request.param)
    yield m
    m.ss_set_compact_config(2)  # the library's default


def run_compact(ss, keys: np.ndarray, flags: np.ndarray, key_offset: int = 0, flag_offset: int = 0):
    import torch
    n = keys.size
    k = Guarded(n, key_offset, fill=keys)
    fbuf = torch.zeros(n + 64 + flag_offset, dtype=torch.uint8, device="cuda:0")
    fview = fbuf[flag_offset: flag_offset + n]
    fview.copy_(torch.from_numpy(flags))
    out = Guarded(n)
    cnt = torch.full((1,), -1, dtype=torch.int64, device="cuda:0")
    ss.compact_u32(k.view, fview, out.view, cnt, n)
    st, tile = ss.ss_stream_status()
    assert st == ss.SS_OK, f"device status {st} at tile {tile}"
    assert out.guards_intact(), "a store landed outside the output"
    c = int(cnt.item())
    full = out.numpy(np.uint32)
    # nothing past the count was written
    assert (full[c:].view(np.int32) == SENTINEL).all()
    return full[:c], c


@pytest.mark.parametrize("p", [0.01, 0.5, 0.99])
def test_compaction_full_size(ss, p):
    n = 1 << 28
    keys, flags = compaction_input(n, p)
    got, c = run_compact(ss, keys, flags)
    ref = oracle.compact_u32(keys, flags)
    assert c == ref.size
    assert_equal(got, ref)


@pytest.mark.parametrize("p", [0.0625, 0.001])
def test_compaction_sparse_and_moderate(ss, p):
    # Keep rates between the bench's: a few kept keys per 16-byte key vector
    # (0.0625) and almost none (0.001), over 300 tiles of 65,536 and a ragged
    # last one.
    n = 300 * 65536 + 12_345
    keys = si.uniform_u32(n, seed=33)
    flags = si.bernoulli_flags(n, p, seed=34)
    got, c = run_compact(ss, keys, flags)
    ref = oracle.compact_u32(keys, flags)
    assert c == ref.size
    assert_equal(got, ref)


def test_compaction_sparse_and_dense_tiles_in_one_call(ss):
    # A keep rate of 3456 / 65536 puts about half of the chunked kernel's
    # tiles on each side of its sparse/dense switch (fewer than 1728 kept keys
    # in a 32768-element tile, 3456 in a 65536-element one), interleaved
    # across CTAs.
    n = 200 * 65536 + 77
    keys = si.uniform_u32(n, seed=38)
    flags = si.bernoulli_flags(n, 3456 / 65536, seed=39)
    got, c = run_compact(ss, keys, flags)
    ref = oracle.compact_u32(keys, flags)
    assert c == ref.size
    assert_equal(got, ref)


@pytest.mark.parametrize("run", [1, 5, 32, 33, 64, 500])
def test_compaction_clustered_runs(ss, run):
    # Runs of `run` consecutive kept flags at seeded positions, about 1024 kept
    # keys per 65,536 elements: sparse tiles in which one thread's 32 elements
    # can all be kept, so the sparse form's loads past its four slots per
    # chunk run too.  Runs straddle threads, warps, chunks and tiles; with
    # runs of 500 some tiles take the dense form.
    n = 97 * 65536 + 1234
    keys = si.uniform_u32(n, seed=40)
    starts = si.uniform_int32(max(1, n * 1024 // (65536 * run)), 0, n - 1, seed=41)
    flags = np.zeros(n, dtype=np.uint8)
    for st in starts.astype(np.int64):
        flags[st: st + run] = 1
    got, c = run_compact(ss, keys, flags)
    ref = oracle.compact_u32(keys, flags)
    assert c == ref.size
    assert_equal(got, ref)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 31, 33, 511, 512, 513, 4095, 4096, 4097, 8191, 8193,
                               65535, 65536, 65537, 65536 * 3 + 1000, 100_003, 1 << 20, 152 * 65536 + 17])
@pytest.mark.parametrize("p", [0.0, 0.3, 1.0])
def test_compaction_edges(ss, n, p):
    keys = si.uniform_u32(n, seed=31)
    flags = si.bernoulli_flags(n, p, seed=32)
    got, c = run_compact(ss, keys, flags)
    ref = oracle.compact_u32(keys, flags)
    assert c == ref.size
    assert_equal(got, ref)


def test_any_nonzero_flag_keeps(ss):
    n = 3 * 4096 + 17
    keys = si.uniform_u32(n, seed=33)
    flags = (si.uniform_int32(n, 0, 255, seed=34) * (si.bernoulli_flags(n, 0.5, seed=35))).astype(np.uint8)
    got, c = run_compact(ss, keys, flags)
    assert_equal(got, oracle.compact_u32(keys, flags))


@pytest.mark.parametrize("koff,foff", [(1, 0), (0, 1), (3, 2), (2, 3)])
def test_misaligned(ss, koff, foff):
    n = 9 * 4096 + 100
    keys = si.uniform_u32(n, seed=36)
    flags = si.bernoulli_flags(n, 0.5, seed=37)
    got, c = run_compact(ss, keys, flags, key_offset=koff, flag_offset=foff)
    assert_equal(got, oracle.compact_u32(keys, flags))


def test_zero_length_writes_zero_count(ss):
    import torch
    cnt = torch.full((1,), 77, dtype=torch.int64, device="cuda:0")
    e = torch.empty(0, dtype=torch.int32, device="cuda:0")
    f = torch.empty(0, dtype=torch.uint8, device="cuda:0")
    ss.compact_u32(e, f, e, cnt, 0)
    assert int(cnt.item()) == 0


def test_count_identity_with_scan(ss):
    # count = excl_scan(flags)[n-1] + flags[n-1], the scan computed on the GPU.
    import torch
    n = 1_000_003
    keys, flags = si.workload_compaction(n, 0.5, seed=3)
    _, c = run_compact(ss, keys, flags)
    f32 = torch.from_numpy(flags.astype(np.int32)).to("cuda:0")
    pos = torch.empty_like(f32)
    ss.scan_exclusive_i32(f32, pos)
    assert c == int(pos[-1].item()) + int(flags[-1])
