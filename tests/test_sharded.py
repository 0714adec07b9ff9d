"""The scan split over the ranks of a process group (one contiguous part per
rank, one exchange of the part totals), and the device reduction it starts
with.

CPU tests (two and three gloo ranks) cover the partition, the exchange and
the composition of the parts with the oracle standing in for each rank's
kernels.  GPU tests call the reduction through the C ABI against the oracle,
and run the whole split scan as two gloo ranks that share cuda:0 (their
kernels never wait on each other: the exchange is a host-side collective
between the reduction and the seeded scan), bit-exact against the oracle's
scan of the concatenated array for integers and within the fp32 bound.
"""

from __future__ import annotations

import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
import seeded_inputs as si
from stream_compaction_pass_gb300.sharded import ALIGN, shard_bounds

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("n", [0, 1, 5, 1023, 1024, 1025, 4096 * 3 + 7, 10_000_019])
def test_shard_bounds_cover_in_order(n, world):
    parts = [shard_bounds(n, world, r) for r in range(world)]
    assert parts[0][0] == 0 and parts[-1][1] == n
    for (a, b), (c, d) in zip(parts, parts[1:]):
        assert b == c                       # contiguous, in rank order
    for a, b in parts:
        assert a <= b and a % ALIGN == 0 or a == n
    sizes = [b - a for a, b in parts]
    assert max(sizes) - min(sizes) <= -(-n // world) + ALIGN


def _cpu_worker(rank, world, port, n, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import oracle as orc
    import seeded_inputs as sin
    from stream_compaction_pass_gb300.sharded import gather_totals, shard_bounds as sb
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = sin.uniform_int32(n, -(1 << 31), (1 << 31) - 1, seed=23)
    a, b = sb(n, world, rank)
    part = x[a:b]
    total = int(orc.scan_i32(part, True)[-1]) if b > a else 0
    totals = gather_totals(torch.tensor([total], dtype=torch.int32))
    offsets = orc.scan_i32(totals.numpy(), False)
    # this rank's part of the whole scan: its own exclusive scan plus its offset, modulo 2^32
    got = (orc.scan_i32(part, False).astype(np.int64) + int(offsets[rank])).astype(np.uint32).view(np.int32)
    q.put((rank, a, got.tobytes()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_parts_compose_to_the_whole_scan_cpu(world):
    n = 1_000_003
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_cpu_worker, args=(r, world, port, n, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got = np.concatenate([np.frombuffer(buf, dtype=np.int32) for _r, _a, buf in out])
    x = si.uniform_int32(n, -(1 << 31), (1 << 31) - 1, seed=23)
    assert np.array_equal(got, oracle.scan_i32(x, False))


# ----------------------------------------------------------------- GPU ---

def _reduce_ref(kind, x):
    return oracle.scan_f32(x, True)[-1] if kind == "f32" else (
        oracle.scan_u32(x, True)[-1] if kind == "u32" else oracle.scan_i32(x, True)[-1])


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["i32", "u32", "f32"])
@pytest.mark.parametrize("n", [0, 1, 3, 4, 5, 1023, 1_000_003, 100_000_000])
@pytest.mark.parametrize("offset", [0, 1])
def test_reduce_sum_matches_oracle(kind, n, offset):
    import torch
    import stream_compaction_pass_gb300 as ss
    if kind == "f32":
        x = si.workload_f32_unit(n + offset, seed=1)
    elif kind == "u32":
        x = si.uniform_u32(n + offset, seed=21)
    else:
        x = si.uniform_int32(n + offset, -(1 << 31), (1 << 31) - 1, seed=22)
    d = torch.from_numpy(x.view(np.int32)).to("cuda:0")[offset:]
    x = x[offset:]
    tot = torch.full((2,), -559038737, dtype=torch.int32, device="cuda:0")
    dtype = {"i32": ss.SS_I32, "u32": ss.SS_U32, "f32": ss.SS_F32}[kind]
    got = []
    for _ in range(2):
        ss.ss_reduce_sum(dtype, d, tot[:1], n=n)
        got.append(tot.cpu().numpy())
    assert got[1][1] == -559038737                      # nothing past the total written
    assert np.array_equal(got[0], got[1])               # same bits on every run
    if n == 0:
        assert got[0][0] == 0
        return
    ref = _reduce_ref(kind, x)
    if kind == "f32":
        err = abs(float(got[0][:1].view(np.float32)[0]) - float(ref)) / max(1.0, float(np.abs(x.astype(np.float64)).sum()))
        assert err <= 1e-4
    else:
        assert got[0][:1].view(np.uint32 if kind == "u32" else np.int32)[0] == ref


def _gpu_worker(rank, world, port, n, kind, inclusive, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import seeded_inputs as sin
    import stream_compaction_pass_gb300 as ss
    from stream_compaction_pass_gb300.sharded import scan_sharded, shard_bounds as sb
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = sin.workload_f32_unit(n, seed=1).view(np.int32) if kind == "f32" else \
        sin.uniform_int32(n, -(1 << 31), (1 << 31) - 1, seed=23)
    a, b = sb(n, world, rank)
    d_in = torch.from_numpy(x[a:b].copy()).to("cuda:0")
    d_out = torch.empty_like(d_in)
    dtype = {"i32": ss.SS_I32, "u32": ss.SS_U32, "f32": ss.SS_F32}[kind]
    scan_sharded(dtype, inclusive, d_in, d_out)
    torch.cuda.synchronize()
    st, _ = ss.ss_stream_status()
    q.put((rank, st, d_out.cpu().numpy().tobytes()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.gpu
@pytest.mark.parametrize("kind,inclusive,n", [("i32", False, 10_000_019), ("i32", True, 3_000_001),
                                              ("u32", False, 1_000_003), ("f32", True, 10_000_019),
                                              ("i32", False, 1_000)])
def test_two_ranks_on_one_gpu_match_the_whole_scan(kind, inclusive, n):
    import stream_compaction_pass_gb300 as ss
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gpu_worker, args=(r, world, port, n, kind, inclusive, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(st == ss.SS_OK for _r, st, _b in out)
    if kind == "f32":
        x = si.workload_f32_unit(n, seed=1)
        got = np.concatenate([np.frombuffer(buf, dtype=np.float32) for _r, _s, buf in out])
        err = oracle.fp32_normalised_error(got, oracle.scan_f32(x, inclusive), x)
        assert err <= 1e-4
    else:
        x = si.uniform_int32(n, -(1 << 31), (1 << 31) - 1, seed=23)
        got = np.concatenate([np.frombuffer(buf, dtype=np.int32) for _r, _s, buf in out])
        ref = oracle.scan_u32(x.view(np.uint32), inclusive).view(np.int32) if kind == "u32" else \
            oracle.scan_i32(x, inclusive)
        assert np.array_equal(got, ref)
