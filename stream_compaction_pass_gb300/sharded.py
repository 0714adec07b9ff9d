"""A scan of one array split into contiguous parts over the ranks of a
torch.distributed process group, one part per rank.

This is the device-level scan of "Prefix sum and other parallel patterns"
(A device-level scan: scan then propagate) one level up: the parts play the
role of the blocks.  Each rank

  1. sums its part on its GPU (`ss_reduce_sum`, n reads);
  2. all-gathers the P part totals (the one exchange step: one scalar per
     rank, NCCL when the group has it, else through host memory);
  3. exclusive-scans the P totals with the library's scan kernel, which gives
     the sum of every part before its own;
  4. scans its part seeded with that offset (`ss_scan_seeded`, 2n).

So 3n bytes move per rank and nothing waits on another rank's kernels.  All
arithmetic runs in the library's kernels; this module only moves the P
scalars and orders the calls.  int32 and uint32 results are bit-exact with a
scan of the whole array; fp32 results are within the scans' bound.
"""

from __future__ import annotations

from . import SS_F32, SS_I32, SS_U32, ss_reduce_sum, ss_scan_seeded, _check, lib, _addr

ALIGN = 1024  # parts start on multiples of 1024 elements (16-byte aligned vectors, whole rows)


def shard_bounds(n: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of rank's part of n elements split over `world` ranks:
    contiguous, in rank order, each a multiple of ALIGN elements long except
    the last; a rank past the end gets an empty part."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError("bad partition arguments")
    per = -(-n // world)            # ceil(n / world)
    per = -(-per // ALIGN) * ALIGN  # rounded up to ALIGN
    start = min(n, rank * per)
    stop = min(n, start + per)
    return start, stop


def gather_totals(total, group=None):
    """All ranks' one-element `total` tensors, in rank order, as one tensor
    on total's device (the exchange step)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    if total.is_cuda and dist.get_backend(group) == "nccl":
        out = torch.empty(world, dtype=total.dtype, device=total.device)
        dist.all_gather_into_tensor(out, total.reshape(1), group=group)
        return out
    host = total.reshape(1).cpu()
    parts = [torch.empty_like(host) for _ in range(world)]
    dist.all_gather(parts, host, group=group)
    return torch.cat(parts).to(total.device)


def _torch_dtype(dtype: int):
    import torch
    return {SS_I32: torch.int32, SS_U32: torch.int32, SS_F32: torch.float32}[dtype]


def scan_sharded(dtype: int, inclusive: bool, part_in, part_out, group=None, stream=None) -> None:
    """Scans this rank's part of an array split with shard_bounds(), so that
    the parts of all ranks together hold the scan of the whole array.  Every
    rank of `group` must call it (with empty parts where it has none).
    part_in/part_out: this rank's device tensors (out may be in)."""
    import torch
    import torch.distributed as dist
    dev = part_in.device
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    total = torch.empty(1, dtype=_torch_dtype(dtype), device=dev)
    ss_reduce_sum(dtype, part_in, total, stream=s)
    s.synchronize()  # the exchange below reads `total` outside the stream
    totals = gather_totals(total, group)
    offsets = torch.empty_like(totals)
    name = {SS_I32: "scan_exclusive_i32", SS_U32: "scan_exclusive_u32", SS_F32: "scan_exclusive_f32"}[dtype]
    _check(getattr(lib(), name)(_addr(totals), _addr(offsets), totals.numel(), int(s.cuda_stream)), name)
    rank = dist.get_rank(group)
    ss_scan_seeded(dtype, inclusive, part_in, part_out, carry_in=offsets[rank:rank + 1], stream=s)
