"""Python access to the sequential CPU oracle (oracle/scan_ref.c, tile_model.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg call this; the library under test
never does.  The functions take and return numpy arrays and call the C code
through ctypes; no arithmetic of the method happens in Python here.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

LAYOUT_PLAIN = 0
LAYOUT_PAD32 = 1
LAYOUT_PAD32_1024 = 2


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  `path` selects another
    build of the same sources, e.g. a deliberately broken one in a test."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(_build.build()))
    return _lib


def _declare(lib):
    p, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    u64 = ctypes.c_uint64
    for name in ("oracle_scan_i32", "oracle_scan_u32", "oracle_scan_f32"):
        f = getattr(lib, name)
        f.argtypes = [p, p, sz, i]
        f.restype = None
    lib.oracle_abs_prefix_f32.argtypes = [p, p, sz]
    lib.oracle_abs_prefix_f32.restype = None
    for name in ("oracle_scan_u32_u64", "oracle_scan_i32_i64", "oracle_scan_i64", "oracle_scan_f64"):
        f = getattr(lib, name)
        f.argtypes = [p, p, sz, i]
        f.restype = None
    lib.oracle_abs_prefix_f64.argtypes = [p, p, sz]
    lib.oracle_abs_prefix_f64.restype = None
    for name in ("oracle_scan_rows_i32", "oracle_scan_rows_u32", "oracle_scan_rows_f32"):
        f = getattr(lib, name)
        f.argtypes = [p, p, sz, sz, i]
        f.restype = None
    lib.oracle_abs_prefix_rows_f32.argtypes = [p, p, sz, sz]
    lib.oracle_abs_prefix_rows_f32.restype = None
    for name in ("oracle_scan_segments_i32", "oracle_scan_segments_u32", "oracle_scan_segments_f32"):
        f = getattr(lib, name)
        f.argtypes = [p, p, sz, p, sz, i]
        f.restype = None
    lib.oracle_abs_prefix_segments_f32.argtypes = [p, p, sz, p, sz]
    lib.oracle_abs_prefix_segments_f32.restype = None
    lib.oracle_compact_u32.argtypes = [p, p, p, sz]
    lib.oracle_compact_u32.restype = u64
    for name in ("oracle_compact_positive_f32", "oracle_compact_positive_i32", "oracle_compact_positive_u32"):
        f = getattr(lib, name)
        f.argtypes = [p, p, sz]
        f.restype = u64
    lib.oracle_moe_counts_offsets.argtypes = [p, sz, ctypes.c_int32, ctypes.c_uint32, p, p]
    lib.oracle_moe_counts_offsets.restype = None
    lib.oracle_blelloch_adds.argtypes = [u64]
    lib.oracle_blelloch_adds.restype = u64
    lib.oracle_hillis_steele_adds.argtypes = [u64]
    lib.oracle_hillis_steele_adds.restype = u64
    lib.oracle_blelloch_level_warps.argtypes = [u64, u64]
    lib.oracle_blelloch_level_warps.restype = i
    lib.oracle_blelloch_level_degree.argtypes = [u64, u64, i]
    lib.oracle_blelloch_level_degree.restype = i
    lib.oracle_blelloch_requests.argtypes = [u64, i]
    lib.oracle_blelloch_requests.restype = u64
    lib.oracle_hillis_steele_requests.argtypes = [u64]
    lib.oracle_hillis_steele_requests.restype = u64
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def scan_i32(x: np.ndarray, inclusive: bool, lib=None) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.int32)
    y = np.empty_like(x)
    (lib or load()).oracle_scan_i32(_ptr(x), _ptr(y), x.size, int(bool(inclusive)))
    return y


def scan_u32(x: np.ndarray, inclusive: bool, lib=None) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint32)
    y = np.empty_like(x)
    (lib or load()).oracle_scan_u32(_ptr(x), _ptr(y), x.size, int(bool(inclusive)))
    return y


def scan_f32(x: np.ndarray, inclusive: bool, lib=None) -> np.ndarray:
    """fp32 input, float64 result (float64 running sum)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.size, dtype=np.float64)
    (lib or load()).oracle_scan_f32(_ptr(x), _ptr(y), x.size, int(bool(inclusive)))
    return y


def abs_prefix_f32(x: np.ndarray, lib=None) -> np.ndarray:
    """Normaliser sum_{j<=i} |x_j| in float64."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.size, dtype=np.float64)
    (lib or load()).oracle_abs_prefix_f32(_ptr(x), _ptr(y), x.size)
    return y


def _scan_typed(x, in_dtype, out_dtype, fn, inclusive, lib):
    x = np.ascontiguousarray(x, dtype=in_dtype)
    y = np.empty(x.size, dtype=out_dtype)
    getattr(lib or load(), fn)(_ptr(x), _ptr(y), x.size, int(bool(inclusive)))
    return y


def scan_u32_u64(x: np.ndarray, inclusive: bool, lib=None) -> np.ndarray:
    """uint32 in, exact uint64 prefix sums out."""
    return _scan_typed(x, np.uint32, np.uint64, "oracle_scan_u32_u64", inclusive, lib)


def scan_i32_i64(x: np.ndarray, inclusive: bool, lib=None) -> np.ndarray:
    """int32 in, exact int64 prefix sums out."""
    return _scan_typed(x, np.int32, np.int64, "oracle_scan_i32_i64", inclusive, lib)


def scan_i64(x: np.ndarray, inclusive: bool, lib=None) -> np.ndarray:
    """int64 prefix sums modulo 2^64."""
    return _scan_typed(x, np.int64, np.int64, "oracle_scan_i64", inclusive, lib)


def scan_f64(x: np.ndarray, inclusive: bool, lib=None) -> np.ndarray:
    """fp64 prefix sums, compensated, within about one rounding of exact."""
    return _scan_typed(x, np.float64, np.float64, "oracle_scan_f64", inclusive, lib)


def abs_prefix_f64(x: np.ndarray, lib=None) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(x.size, dtype=np.float64)
    (lib or load()).oracle_abs_prefix_f64(_ptr(x), _ptr(y), x.size)
    return y


def scan_rows(x: np.ndarray, inclusive: bool, lib=None) -> np.ndarray:
    """Every row of a 2-D int32 / uint32 / fp32 array scanned on its own
    (fp32 rows in float64)."""
    x = np.ascontiguousarray(x)
    assert x.ndim == 2
    rows, cols = x.shape
    kinds = {np.dtype(np.int32): ("oracle_scan_rows_i32", np.int32),
             np.dtype(np.uint32): ("oracle_scan_rows_u32", np.uint32),
             np.dtype(np.float32): ("oracle_scan_rows_f32", np.float64)}
    fn, out_dt = kinds[x.dtype]
    y = np.empty((rows, cols), dtype=out_dt)
    getattr(lib or load(), fn)(_ptr(x), _ptr(y), rows, cols, int(bool(inclusive)))
    return y


def abs_prefix_rows_f32(x: np.ndarray, lib=None) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    y = np.empty((rows, cols), dtype=np.float64)
    (lib or load()).oracle_abs_prefix_rows_f32(_ptr(x), _ptr(y), rows, cols)
    return y


def _check_offsets(offsets, n):
    offsets = np.ascontiguousarray(offsets, dtype=np.uint64)
    assert offsets.size >= 2 and offsets[0] == 0 and offsets[-1] == n, "offsets must run from 0 to n"
    assert (np.diff(offsets.astype(np.int64)) >= 0).all(), "offsets must not decrease"
    return offsets


def scan_segments(x: np.ndarray, offsets: np.ndarray, inclusive: bool, lib=None) -> np.ndarray:
    """Every segment [offsets[s], offsets[s+1]) of a 1-D int32 / uint32 / fp32
    array scanned on its own (fp32 in float64)."""
    x = np.ascontiguousarray(x)
    offsets = _check_offsets(offsets, x.size)
    kinds = {np.dtype(np.int32): ("oracle_scan_segments_i32", np.int32),
             np.dtype(np.uint32): ("oracle_scan_segments_u32", np.uint32),
             np.dtype(np.float32): ("oracle_scan_segments_f32", np.float64)}
    fn, out_dt = kinds[x.dtype]
    y = np.empty(x.size, dtype=out_dt)
    getattr(lib or load(), fn)(_ptr(x), _ptr(y), x.size, _ptr(offsets), offsets.size - 1, int(bool(inclusive)))
    return y


def abs_prefix_segments_f32(x: np.ndarray, offsets: np.ndarray, lib=None) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    offsets = _check_offsets(offsets, x.size)
    y = np.empty(x.size, dtype=np.float64)
    (lib or load()).oracle_abs_prefix_segments_f32(_ptr(x), _ptr(y), x.size, _ptr(offsets), offsets.size - 1)
    return y


def compact_u32(keys: np.ndarray, flags: np.ndarray, lib=None) -> np.ndarray:
    """Keys whose flag is nonzero, in index order."""
    keys = np.ascontiguousarray(keys, dtype=np.uint32)
    flags = np.ascontiguousarray(flags, dtype=np.uint8)
    assert keys.size == flags.size
    out = np.empty(keys.size, dtype=np.uint32)
    cnt = (lib or load()).oracle_compact_u32(_ptr(keys), _ptr(flags), _ptr(out), keys.size)
    return out[:cnt].copy()


def compact_positive_f32(x: np.ndarray, lib=None) -> np.ndarray:
    """Elements with x > 0 (fp32 compare), in index order."""
    return _compact_positive(x, np.float32, "oracle_compact_positive_f32", lib)


def compact_positive_i32(x: np.ndarray, lib=None) -> np.ndarray:
    """Elements with x > 0 (signed), in index order."""
    return _compact_positive(x, np.int32, "oracle_compact_positive_i32", lib)


def compact_positive_u32(x: np.ndarray, lib=None) -> np.ndarray:
    """Nonzero elements, in index order."""
    return _compact_positive(x, np.uint32, "oracle_compact_positive_u32", lib)


def _compact_positive(x, dtype, fn, lib):
    x = np.ascontiguousarray(x, dtype=dtype)
    out = np.empty(x.size, dtype=dtype)
    cnt = getattr(lib or load(), fn)(_ptr(x), _ptr(out), x.size)
    return out[:cnt].copy()


def moe_counts_offsets(ids: np.ndarray, num_experts: int, align: int, lib=None):
    """(counts[E] uint32, offsets[E+1] uint64): the histogram of expert ids
    and each expert's start, segments rounded up to a multiple of `align`."""
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    assert num_experts >= 1 and align >= 1
    counts = np.empty(num_experts, dtype=np.uint32)
    offsets = np.empty(num_experts + 1, dtype=np.uint64)
    (lib or load()).oracle_moe_counts_offsets(_ptr(ids), ids.size, num_experts, align, _ptr(counts),
                                              _ptr(offsets))
    return counts, offsets


def blelloch_adds(tile: int, lib=None) -> int:
    return int((lib or load()).oracle_blelloch_adds(tile))


def hillis_steele_adds(n: int, lib=None) -> int:
    return int((lib or load()).oracle_hillis_steele_adds(n))


def blelloch_level_warps(tile: int, stride: int, lib=None) -> int:
    return int((lib or load()).oracle_blelloch_level_warps(tile, stride))


def blelloch_level_degree(tile: int, stride: int, layout: int, lib=None) -> int:
    return int((lib or load()).oracle_blelloch_level_degree(tile, stride, layout))


def blelloch_requests(tile: int, layout: int, lib=None) -> int:
    return int((lib or load()).oracle_blelloch_requests(tile, layout))


def hillis_steele_requests(tile: int, lib=None) -> int:
    return int((lib or load()).oracle_hillis_steele_requests(tile))


def fp32_normalised_error(got: np.ndarray, ref: np.ndarray, x: np.ndarray, lib=None) -> float:
    """max_i |got_i - ref_i| / max(1, sum_{j<=i} |x_j|), the fp32 parity
    measure.  The same normaliser (sum up to and including i) is used for
    inclusive and exclusive scans."""
    a = abs_prefix_f32(x, lib=lib)
    if got.size == 0:
        return 0.0
    err = np.abs(got.astype(np.float64) - ref) / np.maximum(1.0, a)
    return float(err.max())


_here = os.path.dirname(os.path.abspath(__file__))
