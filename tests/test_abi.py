"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments before touching CUDA."""

import ctypes

import pytest

import stream_compaction_pass_gb300 as ss


@pytest.fixture(scope="module")
def lib():
    from stream_compaction_pass_gb300 import build
    build.build()
    return ss.lib()


def test_every_declared_function_is_exported(lib):
    names = ss.header_functions()
    assert len(names) >= 19
    raw = ctypes.CDLL(ss.LIB_PATH)
    for name in names:
        assert hasattr(raw, name), f"{name} declared in streamscan.h but not exported"
    for name in ("scan_inclusive_i32", "scan_exclusive_i32", "scan_inclusive_u32",
                 "scan_exclusive_u32", "scan_inclusive_f32", "scan_exclusive_f32", "compact_u32"):
        assert name in names


def test_status_strings(lib):
    for code in range(6):
        assert ss.ss_status_string(code)
    assert ss.ss_status_string(99) == "unknown status"


def test_null_pointers_rejected_before_cuda(lib):
    for name in ("scan_inclusive_i32", "scan_exclusive_f32", "scan_exclusive_u32"):
        assert getattr(lib, name)(None, None, 5, None) == ss.SS_ERR_INVALID_ARG
    assert lib.compact_u32(None, None, None, None, 5, None) == ss.SS_ERR_INVALID_ARG
    assert "null" in ss.ss_last_error_detail()


def test_zero_length_is_a_noop(lib):
    assert lib.scan_inclusive_i32(None, None, 0, None) == ss.SS_OK
    assert lib.ss_scan(ss.SS_F32, 1, ss.SS_ALGO_REDUCE_THEN_SCAN, None, None, 0, None) == ss.SS_OK
    assert lib.ss_scan_host(ss.SS_I32, 0, None, None, 0, None) == ss.SS_OK


def test_misaligned_and_overlapping_rejected(lib):
    assert lib.scan_inclusive_i32(0x1002, 0x2000, 4, None) == ss.SS_ERR_INVALID_ARG
    assert "aligned" in ss.ss_last_error_detail()
    # out starts inside in's range: partial overlap
    assert lib.scan_inclusive_u32(0x10000, 0x10010, 64, None) == ss.SS_ERR_INVALID_ARG
    assert "overlap" in ss.ss_last_error_detail()
    # compaction output overlapping the keys
    assert lib.compact_u32(0x10000, 0x90000, 0x10040, 0xA0000, 64, None) == ss.SS_ERR_INVALID_ARG
    assert lib.compact_u32(0x10000, 0x90000, 0x20000, 0xA0004, 64, None) == ss.SS_ERR_INVALID_ARG


def test_predicate_and_unordered_compaction_arguments(lib):
    inv = ss.SS_ERR_INVALID_ARG
    assert lib.compact_positive_f32(None, None, None, 5, None) == inv
    assert lib.compact_positive_f32(0x10000, 0x20000, None, 5, None) == inv          # no count
    assert lib.compact_positive_f32(0x10000, 0x20000, 0xA0004, 5, None) == inv       # count misaligned
    assert lib.compact_positive_f32(0x10000, 0x10040, 0xA0000, 64, None) == inv      # out overlaps in
    assert lib.compact_positive_f32(0x10002, 0x20000, 0xA0000, 64, None) == inv      # in misaligned
    assert lib.ss_compact_positive(9, 0x10000, 0x20000, 0xA0000, 4, None) == ss.SS_ERR_UNSUPPORTED
    assert lib.ss_compact_positive(ss.SS_I32, 0x10000, 0x20000, 0xA0000, 1 << 33, None) == inv
    assert lib.ss_compact_positive(ss.SS_U32, 0x10000, 0x20000, 0x10008, 64, None) == inv  # count in input
    assert lib.ss_compact_u32_unordered(0x10000, None, 0x20000, 0xA0000, 5, None) == inv  # flags required
    assert lib.ss_compact_u32_unordered(0x10000, 0x90000, 0x90010, 0xA0000, 64, None) == inv
    assert lib.ss_compact_positive_unordered(7, 0x10000, 0x20000, 0xA0000, 4, None) == ss.SS_ERR_UNSUPPORTED
    assert lib.ss_compact_positive_unordered(ss.SS_F32, 0x10000, 0x10000, 0xA0000, 4, None) == inv


def test_wide_scan_arguments(lib):
    inv = ss.SS_ERR_INVALID_ARG
    assert lib.scan_inclusive_f64(None, None, 5, None) == inv
    assert lib.scan_inclusive_f64(0x10004, 0x20000, 5, None) == inv          # fp64 input 4-byte aligned
    assert lib.scan_exclusive_u32_u64(0x10004, 0x20004, 5, None) == inv      # output not 8-byte aligned
    assert lib.scan_exclusive_u32_u64(0x10000, 0x10000, 5, None) == inv      # widened in place
    assert "widened" in ss.ss_last_error_detail()
    assert lib.scan_inclusive_i64(0x10000, 0x10008, 64, None) == inv         # partial overlap
    assert lib.ss_scan_wide(9, 1, 0x10000, 0x20000, 4, None) == ss.SS_ERR_UNSUPPORTED
    assert lib.scan_inclusive_i64(None, None, 0, None) == ss.SS_OK           # empty


def test_rows_scan_arguments(lib):
    inv = ss.SS_ERR_INVALID_ARG
    assert lib.ss_scan_rows(ss.SS_F32, 1, None, None, 0, 100, None) == ss.SS_OK     # no rows
    assert lib.ss_scan_rows(ss.SS_F32, 1, None, None, 4, 0, None) == ss.SS_OK       # empty rows
    assert lib.ss_scan_rows(ss.SS_F32, 1, None, None, 4, 5, None) == inv
    assert lib.ss_scan_rows(ss.SS_I32, 0, 0x10000, 0x10004, 4, 100, None) == inv    # partial overlap
    assert lib.ss_scan_rows(ss.SS_U32, 0, 0x10000, 0x20000, 1 << 40, 1 << 30, None) == inv  # too large
    assert lib.ss_scan_rows(7, 0, 0x10000, 0x20000, 4, 4, None) == ss.SS_ERR_UNSUPPORTED


def test_segments_arguments(lib):
    inv = ss.SS_ERR_INVALID_ARG
    f = lib.ss_scan_segments
    assert f(ss.SS_I32, 1, None, None, 0, None, 0, None) == ss.SS_OK                 # empty
    assert f(ss.SS_I32, 1, 0x10000, 0x20000, 64, None, 3, None) == inv               # no offsets
    assert f(ss.SS_I32, 1, 0x10000, 0x20000, 64, 0x30004, 3, None) == inv            # offsets misaligned
    assert f(ss.SS_I32, 1, 0x10000, 0x20000, 64, 0x20010, 3, None) == inv            # offsets overlap out
    assert f(ss.SS_I32, 1, 0x10000, 0x10004, 64, 0x30000, 3, None) == inv            # in/out partial overlap
    assert f(9, 1, 0x10000, 0x20000, 64, 0x30000, 3, None) == ss.SS_ERR_UNSUPPORTED


def test_moe_arguments(lib):
    inv = ss.SS_ERR_INVALID_ARG
    f = lib.ss_moe_counts_offsets
    assert f(0x10000, 64, 0, 64, 0x20000, 0x30000, None) == inv           # no experts
    assert f(0x10000, 64, 16385, 64, 0x20000, 0x30000, None) == inv       # too many experts
    assert f(0x10000, 64, 8, 0, 0x20000, 0x30000, None) == inv            # align 0
    assert f(0x10000, 1 << 31, 8, 1, 0x20000, 0x30000, None) == inv       # m too large
    assert f(0x10000, (1 << 31) - 1, 16384, 1 << 20, 0x20000, 0x30000, None) == inv  # total overflows
    assert f(None, 64, 8, 64, 0x20000, 0x30000, None) == inv              # null ids
    assert f(0x10000, 64, 8, 64, None, 0x30000, None) == inv              # null counts
    assert f(0x10002, 64, 8, 64, 0x20000, 0x30000, None) == inv           # misaligned ids
    assert f(0x10000, 64, 8, 64, 0x20000, 0x20010, None) == inv           # counts overlap offsets
    assert f(0x10000, 64, 8, 64, 0x10010, 0x30000, None) == inv           # counts overlap ids
    assert "overlap" in ss.ss_last_error_detail()


def test_bad_enums_and_sizes(lib):
    assert lib.ss_scan(7, 1, 0, 0x1000, 0x2000, 4, None) == ss.SS_ERR_UNSUPPORTED
    assert lib.ss_scan(0, 1, 9, 0x1000, 0x2000, 4, None) == ss.SS_ERR_UNSUPPORTED
    assert lib.compact_u32(0x10000, 0x90000, 0x20000, 0xA0000, 1 << 33, None) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_set_scan_config(99) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_debug_set_lookback_fault(-5, 0) == ss.SS_ERR_INVALID_ARG


def test_form_switches(lib):
    # host-only: each switch takes exactly its documented values
    for c in range(8):
        assert lib.ss_set_compact_config(c) == ss.SS_OK
    assert lib.ss_set_compact_config(8) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_set_compact_config(-1) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_set_compact_config(2) == ss.SS_OK  # the default
    for c in range(6):
        assert lib.ss_set_segments_config(c) == ss.SS_OK
    assert lib.ss_set_segments_config(6) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_set_segments_config(-1) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_set_segments_config(0) == ss.SS_OK  # the default


def test_explicit_workspace_arguments(lib):
    # the CUB-shape calls: the size query is host-only; argument errors come
    # back before anything is enqueued
    b = ctypes.c_size_t(7)
    assert lib.ss_scan_temp_bytes(0, ctypes.byref(b)) == ss.SS_OK and b.value == 0
    assert lib.ss_scan_temp_bytes(5, None) == ss.SS_ERR_INVALID_ARG
    for n in (1, 4096, 4097, 1_000_003, 100_000_000):
        tiles = (n + 4095) // 4096
        assert ss.ss_scan_temp_bytes(n) == 256 + 8 * (tiles + (tiles + 31) // 32)
    need = ss.ss_scan_temp_bytes(10_000)
    IN, OUT, TEMP = 0x100000, 0x200000, 0x300000
    assert lib.ss_scan_ws(ss.SS_I32, 1, IN, OUT, 10_000, None, need, None) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_scan_ws(ss.SS_I32, 1, IN, OUT, 10_000, TEMP + 16, need, None) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_scan_ws(ss.SS_I32, 1, IN, OUT, 10_000, TEMP, need - 1, None) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_scan_ws(ss.SS_I32, 1, IN, OUT, 10_000, IN + 256, need, None) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_scan_ws(7, 1, IN, OUT, 10_000, TEMP, need, None) == ss.SS_ERR_UNSUPPORTED
    assert lib.ss_scan_ws(ss.SS_F32, 0, None, None, 0, None, 0, None) == ss.SS_OK  # n = 0: nothing to do
    t = ctypes.c_int64(0)
    assert lib.ss_temp_status(TEMP + 8, None, ctypes.byref(t)) == ss.SS_ERR_INVALID_ARG and t.value == -1


def test_config_table(lib):
    n = ss.ss_scan_config_count()
    tiles = []
    for c in range(n):
        ss.ss_set_scan_config(c)
        tiles.append(ss.ss_scan_tile_elems())
    assert tiles[0] == 4096 and all(t % 128 == 0 for t in tiles)
    # -1: chosen per call by size; the tile reported is the large-n row's (8)
    assert lib.ss_set_scan_config(-2) == ss.SS_ERR_INVALID_ARG
    ss.ss_set_scan_config(-1)
    assert ss.ss_scan_tile_elems() == tiles[8]


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(ss, "_lib", None)
    monkeypatch.setattr(ss, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(ss.LibraryMissing):
        ss.scan_inclusive_i32(0, 0, 0)
