"""Helpers for the GPU parity tests: guarded device buffers, cached seeded
inputs, and comparisons that name the first bad element.

Outputs are written into buffers pre-filled with a sentinel and surrounded by
guard words, so an element nobody wrote keeps the sentinel and a store past
either end changes a guard word (the stand-in for a sanitizer's initcheck
and out-of-bounds reports)."""

from __future__ import annotations

import functools

import numpy as np

import oracle
import seeded_inputs as si

GUARD = 64                 # elements on each side; a multiple of 4 keeps 16-byte alignment
SENTINEL = -559038737      # 0xDEADBEEF as int32
FP32_TOL = 1e-4            # max |y - ref| / max(1, sum_{j<=i} |x_j|)


def torch_dev():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


class Guarded:
    """A device int32 buffer of n elements at `offset` elements past an
    aligned start, with GUARD sentinel elements on both sides."""

    def __init__(self, n: int, offset: int = 0, fill: np.ndarray | None = None):
        import torch
        self.n, self.offset = n, offset
        self.buf = torch.full((n + 2 * GUARD + offset,), SENTINEL, dtype=torch.int32, device=torch_dev())
        self.view = self.buf[GUARD + offset: GUARD + offset + n]
        if fill is not None:
            self.view.copy_(torch.from_numpy(np.ascontiguousarray(fill).view(np.int32)))

    def guards_intact(self) -> bool:
        b = self.buf
        head = b[: GUARD + self.offset]
        tail = b[GUARD + self.offset + self.n:]
        return bool((head == SENTINEL).all().item()) and bool((tail == SENTINEL).all().item())

    def numpy(self, dtype) -> np.ndarray:
        return self.view.cpu().numpy().view(dtype)


def first_bad(got: np.ndarray, ref: np.ndarray, tile: int) -> str:
    bad = np.nonzero(got != ref)[0]
    if bad.size == 0:
        return "no mismatch"
    i = int(bad[0])
    return (f"{bad.size} mismatches; first at element {i} (tile {i // tile}, position {i % tile}): "
            f"got {got[i]!r}, want {ref[i]!r}")


def assert_equal(got: np.ndarray, ref: np.ndarray, tile: int = 4096) -> None:
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if not np.array_equal(got, ref):
        raise AssertionError(first_bad(got, ref, tile))


def assert_fp32_close(got: np.ndarray, ref64: np.ndarray, x: np.ndarray) -> float:
    err = oracle.fp32_normalised_error(got, ref64, x)
    assert err <= FP32_TOL, f"normalised fp32 error {err:.3e} > {FP32_TOL}"
    return err


@functools.lru_cache(maxsize=None)
def sweep_input(n_max: int) -> np.ndarray:
    """int32 uniform [-1000, 1000], seed 2; prefixes of it are the smaller sizes."""
    return si.workload_int_pm1000(n_max, seed=2)


@functools.lru_cache(maxsize=None)
def sweep_reference(n_max: int) -> np.ndarray:
    return oracle.scan_i32(sweep_input(n_max), False)


@functools.lru_cache(maxsize=None)
def f32_input(n: int) -> np.ndarray:
    return si.workload_f32_unit(n, seed=1)


@functools.lru_cache(maxsize=None)
def f32_reference(n: int, inclusive: bool) -> np.ndarray:
    return oracle.scan_f32(f32_input(n), inclusive)


@functools.lru_cache(maxsize=None)
def compaction_input(n: int, p: float):
    return si.workload_compaction(n, p, seed=3)


@functools.lru_cache(maxsize=None)
def poisson_input(n: int) -> np.ndarray:
    return si.workload_poisson_counts(n, seed=4)


SCAN_FNS = {
    ("i32", True): "scan_inclusive_i32", ("i32", False): "scan_exclusive_i32",
    ("u32", True): "scan_inclusive_u32", ("u32", False): "scan_exclusive_u32",
    ("f32", True): "scan_inclusive_f32", ("f32", False): "scan_exclusive_f32",
}
NP_DTYPE = {"i32": np.int32, "u32": np.uint32, "f32": np.float32}


def run_named_scan(kind: str, inclusive: bool, x: np.ndarray, offset: int = 0,
                   inplace: bool = False) -> np.ndarray:
    """Runs one named scan through the C ABI on guarded buffers; checks the
    guards and the device status; returns the output as numpy."""
    import stream_compaction_pass_gb300 as ss
    n = x.size
    src = Guarded(n, offset, fill=x)
    dst = src if inplace else Guarded(n, offset)
    getattr(ss, SCAN_FNS[(kind, inclusive)])(src.view, dst.view)
    st, tile = ss.ss_stream_status()
    assert st == ss.SS_OK, f"device status {ss.ss_status_string(st)} at tile {tile}"
    assert dst.guards_intact(), "a store landed outside the output"
    if not inplace:
        assert src.guards_intact()
        assert np.array_equal(src.numpy(x.dtype), x), "the input was modified"
    return dst.numpy(NP_DTYPE[kind])


def oracle_scan(kind: str, inclusive: bool, x: np.ndarray) -> np.ndarray:
    if kind == "i32":
        return oracle.scan_i32(x, inclusive)
    if kind == "u32":
        return oracle.scan_u32(x, inclusive)
    return oracle.scan_f32(x, inclusive)
