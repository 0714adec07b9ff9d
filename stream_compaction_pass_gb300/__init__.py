"""Device-wide prefix sums and order-preserving stream compaction on one
NVIDIA GB300 (sm_103a): a thin ctypes binding of libstreamscan.so.

The functions carry the C ABI's names (include/streamscan.h) and only
marshal arguments: device pointers, element counts and the CUDA stream.
Every step of the computation runs in the library's CUDA kernels; there is
no CPU fallback.  If libstreamscan.so has not been built, every call raises
LibraryMissing (build it with ``python -m stream_compaction_pass_gb300.build``).

Arguments that are arrays may be torch tensors (CUDA tensors for device
pointers, CPU tensors or numpy arrays for host pointers) or raw integer
addresses.  For tensors, `n` defaults to the element count and `stream` to
torch's current stream on the tensor's device.
"""

from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libstreamscan.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "streamscan.h")

SS_OK = 0
SS_ERR_INVALID_ARG = 1
SS_ERR_CUDA = 2
SS_ERR_LOOKBACK_TIMEOUT = 3
SS_ERR_NO_MEMORY = 4
SS_ERR_UNSUPPORTED = 5

SS_I32, SS_U32, SS_F32 = 0, 1, 2

SS_ALGO_LOOKBACK = 0
SS_ALGO_REDUCE_THEN_SCAN = 1
SS_ALGO_RTS_BLELLOCH = 2
SS_ALGO_RTS_BLELLOCH_PAD32 = 3
SS_ALGO_RTS_BLELLOCH_PAD2 = 4

SS_WIDE_U32_U64, SS_WIDE_I32_I64, SS_WIDE_I64, SS_WIDE_F64 = 0, 1, 2, 3


class LibraryMissing(ImportError):
    pass


class StreamScanError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: status {status} ({detail})")
        self.status = status
        self.detail = detail


_lib = None


def _declare(lib):
    P, SZ, I, U64, I64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64, ctypes.c_int64
    sigs = {
        "scan_inclusive_i32": [P, P, SZ, P],
        "scan_exclusive_i32": [P, P, SZ, P],
        "scan_inclusive_u32": [P, P, SZ, P],
        "scan_exclusive_u32": [P, P, SZ, P],
        "scan_inclusive_f32": [P, P, SZ, P],
        "scan_exclusive_f32": [P, P, SZ, P],
        "compact_u32": [P, P, P, P, SZ, P],
        "compact_positive_f32": [P, P, P, SZ, P],
        "ss_compact_positive": [I, P, P, P, SZ, P],
        "ss_compact_u32_unordered": [P, P, P, P, SZ, P],
        "ss_compact_positive_unordered": [I, P, P, P, SZ, P],
        "ss_moe_counts_offsets": [P, SZ, ctypes.c_int32, ctypes.c_uint32, P, P, P],
        "scan_inclusive_u32_u64": [P, P, SZ, P],
        "scan_exclusive_u32_u64": [P, P, SZ, P],
        "scan_inclusive_i64": [P, P, SZ, P],
        "scan_exclusive_i64": [P, P, SZ, P],
        "scan_inclusive_f64": [P, P, SZ, P],
        "scan_exclusive_f64": [P, P, SZ, P],
        "ss_scan_wide": [I, I, P, P, SZ, P],
        "ss_scan_rows": [I, I, P, P, SZ, SZ, P],
        "ss_scan_segments": [I, I, P, P, SZ, P, SZ, P],
        "ss_set_host_mode": [I],
        "ss_scan": [I, I, I, P, P, SZ, P],
        "ss_scan_seeded": [I, I, P, P, SZ, P, P, P],
        "ss_reduce_sum": [I, P, P, SZ, P],
        "ss_scan_host": [I, I, P, P, SZ, P],
        "ss_copy_u32": [P, P, SZ, P],
        "ss_scan_trace": [I, P, P, SZ, P, P],
        "ss_stream_status": [P, ctypes.POINTER(I64)],
        "ss_set_scan_config": [I],
        "ss_set_compact_config": [I],
        "ss_set_segments_config": [I],
        "ss_debug_set_lookback_fault": [I64, U64],
        "ss_scan_noalloc": [I, I, P, P, SZ, P],
        "ss_debug_set_noalloc_calls": [U64],
        "ss_scan_temp_bytes": [SZ, ctypes.POINTER(SZ)],
        "ss_scan_ws": [I, I, P, P, SZ, P, SZ, P],
        "ss_temp_status": [P, P, ctypes.POINTER(I64)],
    }
    for name, args in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = I
    lib.ss_status_string.argtypes = [I]
    lib.ss_status_string.restype = ctypes.c_char_p
    lib.ss_last_error_detail.argtypes = []
    lib.ss_last_error_detail.restype = ctypes.c_char_p
    lib.ss_scan_tile_elems.argtypes = []
    lib.ss_scan_tile_elems.restype = SZ
    lib.ss_scan_config_count.argtypes = []
    lib.ss_scan_config_count.restype = I
    lib.ss_shutdown.argtypes = []
    lib.ss_shutdown.restype = None
    lib.ss_debug_noalloc_clear_period.argtypes = []
    lib.ss_debug_noalloc_clear_period.restype = U64
    return lib


def lib():
    """The loaded libstreamscan.so (raises LibraryMissing if not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise LibraryMissing(
                f"{LIB_PATH} is not built; run `python -m stream_compaction_pass_gb300.build` "
                "(needs nvcc); there is no CPU fallback")
        _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/streamscan.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                                 text, flags=re.M)))


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)!r}")


def _numel(x) -> int:
    if hasattr(x, "numel"):
        return int(x.numel())
    return int(x.size)


def _stream(stream, *tensors) -> int:
    if stream is not None:
        if isinstance(stream, int):
            return stream
        return int(stream.cuda_stream)
    for t in tensors:
        if hasattr(t, "is_cuda") and t.is_cuda:
            import torch
            return int(torch.cuda.current_stream(t.device).cuda_stream)
    return 0


def _check(st: int, where: str) -> None:
    if st != SS_OK:
        detail = lib().ss_last_error_detail().decode() or lib().ss_status_string(st).decode()
        raise StreamScanError(st, where, detail)


def _scan_named(name: str, inp, out, n, stream) -> None:
    if n is None:
        n = _numel(inp)
    _check(getattr(lib(), name)(_addr(inp), _addr(out), n, _stream(stream, inp, out)), name)


def scan_inclusive_i32(inp, out, n=None, stream=None):
    _scan_named("scan_inclusive_i32", inp, out, n, stream)


def scan_exclusive_i32(inp, out, n=None, stream=None):
    _scan_named("scan_exclusive_i32", inp, out, n, stream)


def scan_inclusive_u32(inp, out, n=None, stream=None):
    _scan_named("scan_inclusive_u32", inp, out, n, stream)


def scan_exclusive_u32(inp, out, n=None, stream=None):
    _scan_named("scan_exclusive_u32", inp, out, n, stream)


def scan_inclusive_f32(inp, out, n=None, stream=None):
    _scan_named("scan_inclusive_f32", inp, out, n, stream)


def scan_exclusive_f32(inp, out, n=None, stream=None):
    _scan_named("scan_exclusive_f32", inp, out, n, stream)


def compact_u32(keys, flags, out, d_count, n=None, stream=None):
    if n is None:
        n = _numel(keys)
    _check(lib().compact_u32(_addr(keys), _addr(flags), _addr(out), _addr(d_count), n,
                             _stream(stream, keys, flags, out)), "compact_u32")


def compact_positive_f32(inp, out, d_count, n=None, stream=None):
    if n is None:
        n = _numel(inp)
    _check(lib().compact_positive_f32(_addr(inp), _addr(out), _addr(d_count), n, _stream(stream, inp, out)),
           "compact_positive_f32")


def ss_compact_positive(dtype: int, inp, out, d_count, n=None, stream=None):
    if n is None:
        n = _numel(inp)
    _check(lib().ss_compact_positive(dtype, _addr(inp), _addr(out), _addr(d_count), n, _stream(stream, inp, out)),
           "ss_compact_positive")


def ss_compact_u32_unordered(keys, flags, out, d_count, n=None, stream=None):
    if n is None:
        n = _numel(keys)
    _check(lib().ss_compact_u32_unordered(_addr(keys), _addr(flags), _addr(out), _addr(d_count), n,
                                          _stream(stream, keys, flags, out)), "ss_compact_u32_unordered")


def ss_compact_positive_unordered(dtype: int, inp, out, d_count, n=None, stream=None):
    if n is None:
        n = _numel(inp)
    _check(lib().ss_compact_positive_unordered(dtype, _addr(inp), _addr(out), _addr(d_count), n,
                                               _stream(stream, inp, out)), "ss_compact_positive_unordered")


def scan_inclusive_u32_u64(inp, out, n=None, stream=None):
    _scan_named("scan_inclusive_u32_u64", inp, out, n, stream)


def scan_exclusive_u32_u64(inp, out, n=None, stream=None):
    _scan_named("scan_exclusive_u32_u64", inp, out, n, stream)


def scan_inclusive_i64(inp, out, n=None, stream=None):
    _scan_named("scan_inclusive_i64", inp, out, n, stream)


def scan_exclusive_i64(inp, out, n=None, stream=None):
    _scan_named("scan_exclusive_i64", inp, out, n, stream)


def scan_inclusive_f64(inp, out, n=None, stream=None):
    _scan_named("scan_inclusive_f64", inp, out, n, stream)


def scan_exclusive_f64(inp, out, n=None, stream=None):
    _scan_named("scan_exclusive_f64", inp, out, n, stream)


def ss_scan_wide(wide_type: int, inclusive: bool, inp, out, n=None, stream=None):
    if n is None:
        n = _numel(inp)
    _check(lib().ss_scan_wide(wide_type, int(bool(inclusive)), _addr(inp), _addr(out), n,
                              _stream(stream, inp, out)), "ss_scan_wide")


def ss_scan_rows(dtype: int, inclusive: bool, inp, out, rows: int, cols: int, stream=None):
    _check(lib().ss_scan_rows(dtype, int(bool(inclusive)), _addr(inp), _addr(out), rows, cols,
                              _stream(stream, inp, out)), "ss_scan_rows")


def ss_scan_segments(dtype: int, inclusive: bool, inp, out, offsets, num_segments=None, n=None, stream=None):
    """offsets: device uint64/int64 tensor of num_segments + 1 entries."""
    if n is None:
        n = _numel(inp)
    if num_segments is None:
        num_segments = _numel(offsets) - 1
    _check(lib().ss_scan_segments(dtype, int(bool(inclusive)), _addr(inp), _addr(out), n, _addr(offsets),
                                  num_segments, _stream(stream, inp, out)), "ss_scan_segments")


def ss_moe_counts_offsets(topk_ids, num_experts: int, align: int, counts, offsets, m=None, stream=None):
    if m is None:
        m = _numel(topk_ids)
    _check(lib().ss_moe_counts_offsets(_addr(topk_ids), m, num_experts, align, _addr(counts), _addr(offsets),
                                       _stream(stream, topk_ids, counts, offsets)), "ss_moe_counts_offsets")


def ss_scan(dtype: int, inclusive: bool, algo: int, inp, out, n=None, stream=None):
    if n is None:
        n = _numel(inp)
    _check(lib().ss_scan(dtype, int(bool(inclusive)), algo, _addr(inp), _addr(out), n,
                         _stream(stream, inp, out)), "ss_scan")


def ss_scan_seeded(dtype: int, inclusive: bool, inp, out, carry_in=None, carry_out=None, n=None,
                   stream=None):
    if n is None:
        n = _numel(inp)
    _check(lib().ss_scan_seeded(dtype, int(bool(inclusive)), _addr(inp), _addr(out), n,
                                _addr(carry_in), _addr(carry_out), _stream(stream, inp, out)),
           "ss_scan_seeded")


def ss_reduce_sum(dtype: int, inp, d_total, n=None, stream=None):
    """Sum of `inp` (device) into d_total (device, one element)."""
    if n is None:
        n = _numel(inp)
    _check(lib().ss_reduce_sum(dtype, _addr(inp), _addr(d_total), n, _stream(stream, inp, d_total)),
           "ss_reduce_sum")


def ss_scan_host(dtype: int, inclusive: bool, h_in, h_out, n=None, stream=None):
    if n is None:
        n = _numel(h_in)
    _check(lib().ss_scan_host(dtype, int(bool(inclusive)), _addr(h_in), _addr(h_out), n,
                              _stream(stream)), "ss_scan_host")


def ss_copy_u32(inp, out, n=None, stream=None):
    if n is None:
        n = _numel(inp)
    _check(lib().ss_copy_u32(_addr(inp), _addr(out), n, _stream(stream, inp, out)), "ss_copy_u32")


def ss_scan_trace(config: int, inp, out, trace, n=None, stream=None):
    """Exclusive uint32 scan recording 8 uint64 per tile of look-back timing."""
    if n is None:
        n = _numel(inp)
    _check(lib().ss_scan_trace(config, _addr(inp), _addr(out), n, _addr(trace),
                               _stream(stream, inp, out)), "ss_scan_trace")


def ss_stream_status(stream=None):
    """Waits for the stream; returns (status, failing_tile) and clears it."""
    tile = ctypes.c_int64(-1)
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    st = lib().ss_stream_status(_stream(stream), ctypes.byref(tile))
    return st, tile.value


def ss_status_string(status: int) -> str:
    return lib().ss_status_string(status).decode()


def ss_last_error_detail() -> str:
    return lib().ss_last_error_detail().decode()


def ss_scan_tile_elems() -> int:
    return int(lib().ss_scan_tile_elems())


def ss_scan_config_count() -> int:
    return int(lib().ss_scan_config_count())


def ss_set_scan_config(config: int) -> None:
    _check(lib().ss_set_scan_config(config), "ss_set_scan_config")


def ss_set_host_mode(mode: int) -> None:
    _check(lib().ss_set_host_mode(mode), "ss_set_host_mode")


def ss_set_compact_config(config: int) -> None:
    _check(lib().ss_set_compact_config(config), "ss_set_compact_config")


def ss_set_segments_config(config: int) -> None:
    _check(lib().ss_set_segments_config(config), "ss_set_segments_config")


def ss_shutdown() -> None:
    lib().ss_shutdown()


def ss_debug_set_lookback_fault(tile: int, timeout_ns: int = 0) -> None:
    _check(lib().ss_debug_set_lookback_fault(tile, timeout_ns), "ss_debug_set_lookback_fault")


def ss_debug_set_noalloc_calls(calls: int) -> None:
    _check(lib().ss_debug_set_noalloc_calls(calls), "ss_debug_set_noalloc_calls")


def ss_debug_noalloc_clear_period() -> int:
    return int(lib().ss_debug_noalloc_clear_period())


def ss_scan_noalloc(dtype: int, inclusive: bool, inp, out, n=None, stream=None):
    """Single-pass scan whose scratch is a fixed device array: allocates
    nothing (n <= 2^30; the first call on a device sets that device up)."""
    if n is None:
        n = _numel(inp)
    st = lib().ss_scan_noalloc(dtype, int(bool(inclusive)), _addr(inp), _addr(out), n,
                               _stream(stream, inp, out))
    if st != SS_OK:
        raise StreamScanError(st, "ss_scan_noalloc", ss_status_string(st))


def ss_scan_temp_bytes(n: int) -> int:
    """Device scratch bytes that ss_scan_ws needs for n elements."""
    b = ctypes.c_size_t(0)
    _check(lib().ss_scan_temp_bytes(n, ctypes.byref(b)), "ss_scan_temp_bytes")
    return int(b.value)


def ss_scan_ws(dtype: int, inclusive: bool, inp, out, temp, n=None, temp_bytes=None, stream=None):
    """The library's scan with caller-provided scratch `temp` (device,
    256-byte aligned, at least ss_scan_temp_bytes(n) bytes)."""
    if n is None:
        n = _numel(inp)
    if temp_bytes is None:
        temp_bytes = temp.numel() * temp.element_size()
    st = lib().ss_scan_ws(dtype, int(bool(inclusive)), _addr(inp), _addr(out), n, _addr(temp), temp_bytes,
                          _stream(stream, inp, out))
    if st != SS_OK:
        raise StreamScanError(st, "ss_scan_ws", ss_status_string(st))


def ss_temp_status(temp, stream=None):
    """Waits for the stream; returns (status, failing_tile) held in `temp`
    and clears it."""
    tile = ctypes.c_int64(-1)
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    st = lib().ss_temp_status(_addr(temp), _stream(stream), ctypes.byref(tile))
    return st, tile.value
