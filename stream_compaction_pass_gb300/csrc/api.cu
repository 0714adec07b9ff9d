// api.cu -- the C ABI declared in include/streamscan.h: argument checks,
// per-(device, stream) workspaces, device status read-back and the
// host-memory pipeline.  All arithmetic runs in the kernels of scan.cu,
// compact.cu and ablations.cu.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "../../include/streamscan.h"
#include "internal.h"

namespace {

using ss::Dtype;

thread_local std::string g_detail;

// The scan's configuration row; -1 = chosen per call by size.
std::atomic<int> g_config{-1};

// Between these sizes the 16384-element-tile row (7) beats the default row
// (8): its shorter tiles fill and drain the persistent pipeline sooner
// (measured with L2 flushed at 3e6 .. 3e7 elements).  Below, there are fewer
// tiles than SMs and row 8's claims win (1e6: 11.9 against 12.6 us); from
// 1e8 on row 8 is ahead.
constexpr size_t kAutoMidLow = 2'000'000;
constexpr size_t kAutoMidHigh = 50'000'000;

int effective_config(size_t n) {
    const int c = g_config.load();
    if (c >= 0) return c;
    return (n >= kAutoMidLow && n < kAutoMidHigh) ? 7 : ss::scan_default_config();
}

std::atomic<int64_t> g_fault_tile{-1};
std::atomic<uint64_t> g_timeout_ns{0};
std::atomic<int> g_host_mode{0};  // 0: direct access to mapped host buffers when possible; 1: always stage
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

// Descriptor epochs are 30 bits; clear the descriptors well before a tag can
// come round again.
constexpr uint64_t kClearEvery = 1ull << 29;

constexpr size_t kHostChunk = (size_t)16 << 20;  // elements per host-pipeline chunk
constexpr size_t kRowsFlat = (size_t)1 << 21;    // batched rows at least this long run as flat scans
constexpr int kHostBuffers = 3;

ss_status fail(ss_status st, const std::string& why) {
    g_detail = why;
    return st;
}

ss_status cuda_fail(cudaError_t e, const char* where) {
    g_detail = std::string(where) + ": " + cudaGetErrorString(e);
    return SS_ERR_CUDA;
}

struct HostPipe {
    void* buf[kHostBuffers] = {nullptr, nullptr, nullptr};
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev_in[kHostBuffers] = {}, ev_scan[kHostBuffers] = {}, ev_out[kHostBuffers] = {};
    bool ready = false;
};

struct Workspace {
    int device = 0;
    cudaStream_t stream = nullptr;
    // Header: [0] tile counter (u64), [8] status words (2 x u32), [16] carry (8 B),
    // [24] MoE ticket (u32), [28] reduction ticket (u32).
    unsigned char* header = nullptr;
    unsigned long long* desc = nullptr;
    size_t desc_cap = 0;  // descriptors
    void* totals = nullptr;
    size_t totals_cap = 0;  // bytes
    uint32_t* moe_acc = nullptr;  // MoE bin accumulator, kept all-zero between launches
    size_t moe_acc_cap = 0;       // words
    uint64_t launches_since_clear = 0;
    HostPipe pipe;
    std::mutex pipe_mu;  // one host pipeline at a time per workspace
};

std::mutex g_mu;
std::map<std::pair<int, uintptr_t>, Workspace*> g_ws;

unsigned long long* ws_counter(Workspace* w) { return reinterpret_cast<unsigned long long*>(w->header); }
uint32_t* ws_status(Workspace* w) { return reinterpret_cast<uint32_t*>(w->header + 8); }
void* ws_carry(Workspace* w) { return w->header + 16; }
uint32_t* ws_ticket(Workspace* w) { return reinterpret_cast<uint32_t*>(w->header + 24); }
uint32_t* ws_reduce_ticket(Workspace* w) { return reinterpret_cast<uint32_t*>(w->header + 28); }

ss_status get_workspace(cudaStream_t s, Workspace** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_pair(dev, reinterpret_cast<uintptr_t>(s));
    auto it = g_ws.find(key);
    if (it != g_ws.end()) {
        *out = it->second;
        return SS_OK;
    }
    Workspace* w = new Workspace();
    w->device = dev;
    w->stream = s;
    e = cudaMallocAsync(reinterpret_cast<void**>(&w->header), 256, s);
    if (e != cudaSuccess) {
        delete w;
        return e == cudaErrorMemoryAllocation ? fail(SS_ERR_NO_MEMORY, "workspace header")
                                              : cuda_fail(e, "cudaMallocAsync");
    }
    e = cudaMemsetAsync(w->header, 0, 256, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    g_ws[key] = w;
    *out = w;
    return SS_OK;
}

ss_status ensure_desc(Workspace* w, size_t tiles) {
    if (tiles > w->desc_cap) {
        size_t cap = w->desc_cap ? w->desc_cap : (size_t)1 << 16;
        while (cap < tiles) cap *= 2;
        if (w->desc) {
            cudaError_t e = cudaFreeAsync(w->desc, w->stream);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
            w->desc = nullptr;
            w->desc_cap = 0;
        }
        cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&w->desc), cap * 8, w->stream);
        if (e != cudaSuccess)
            return e == cudaErrorMemoryAllocation ? fail(SS_ERR_NO_MEMORY, "descriptor array")
                                                  : cuda_fail(e, "cudaMallocAsync");
        e = cudaMemsetAsync(w->desc, 0, cap * 8, w->stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
        w->desc_cap = cap;
        w->launches_since_clear = 0;
    } else if (w->launches_since_clear >= kClearEvery) {
        cudaError_t e = cudaMemsetAsync(w->desc, 0, w->desc_cap * 8, w->stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
        w->launches_since_clear = 0;
    }
    w->launches_since_clear += 1;
    return SS_OK;
}

ss_status ensure_totals(Workspace* w, size_t bytes) {
    if (bytes <= w->totals_cap) return SS_OK;
    size_t cap = w->totals_cap ? w->totals_cap : (size_t)1 << 18;
    while (cap < bytes) cap *= 2;
    if (w->totals) {
        cudaError_t e = cudaFreeAsync(w->totals, w->stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
        w->totals = nullptr;
        w->totals_cap = 0;
    }
    cudaError_t e = cudaMallocAsync(&w->totals, cap, w->stream);
    if (e != cudaSuccess)
        return e == cudaErrorMemoryAllocation ? fail(SS_ERR_NO_MEMORY, "totals array")
                                              : cuda_fail(e, "cudaMallocAsync");
    w->totals_cap = cap;
    return SS_OK;
}

ss_status ensure_moe_acc(Workspace* w, size_t words) {
    if (words <= w->moe_acc_cap) return SS_OK;
    if (w->moe_acc) {
        cudaError_t e = cudaFreeAsync(w->moe_acc, w->stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
        w->moe_acc = nullptr;
        w->moe_acc_cap = 0;
    }
    const size_t cap = (size_t)ss::kMoeMaxExperts;
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&w->moe_acc), cap * 4, w->stream);
    if (e != cudaSuccess)
        return e == cudaErrorMemoryAllocation ? fail(SS_ERR_NO_MEMORY, "MoE accumulator")
                                              : cuda_fail(e, "cudaMallocAsync");
    e = cudaMemsetAsync(w->moe_acc, 0, cap * 4, w->stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    w->moe_acc_cap = cap;
    return SS_OK;
}

int device_sms(int dev) {
    static std::atomic<int> cached[64];
    if (dev < 0 || dev >= 64) return 1;
    int v = cached[dev].load();
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
        cached[dev].store(v);
    }
    return v;
}

ss::LookbackWs make_ws(Workspace* w) {
    ss::LookbackWs ws;
    if (w) {
        ws.desc = w->desc;
        ws.counter = ws_counter(w);
        ws.status = ws_status(w);
    }
    const uint64_t t = g_timeout_ns.load();
    ws.timeout_ns = t ? t : kDefaultTimeoutNs;
    ws.fault_tile = g_fault_tile.load();
    return ws;
}

bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bbytes && y < x + abytes;
}

ss_status check_scan_args(const void* in, const void* out, size_t n, size_t tile) {
    if (n == 0) return SS_OK;
    if (in == nullptr || out == nullptr) return fail(SS_ERR_INVALID_ARG, "null pointer with n > 0");
    if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 3u)
        return fail(SS_ERR_INVALID_ARG, "in/out must be 4-byte aligned");
    if (n / tile >= ((size_t)1 << 31) - 1) return fail(SS_ERR_INVALID_ARG, "n too large");
    if (n > (SIZE_MAX / 8)) return fail(SS_ERR_INVALID_ARG, "n too large");
    if (in != out && overlaps(in, n * 4, out, n * 4))
        return fail(SS_ERR_INVALID_ARG, "in and out partially overlap");
    return SS_OK;
}

// Descriptors a single-pass scan of n elements may use: one per tile of the
// smallest tile any row uses, and one per group of 32 tiles (the two-level
// look-back of rows 10-12 puts its group descriptors after the tiles').
size_t scan_desc_count(size_t n) {
    const size_t tiles = (n + ss::kMinScanTile - 1) / ss::kMinScanTile;
    return tiles + (tiles + 31) / 32;
}

ss_status scan_lookback(Dtype dt, bool inclusive, const void* in, void* out, size_t n,
                        const void* carry_in, void* carry_out, cudaStream_t s) {
    const int cfg = effective_config(n);
    ss_status st = check_scan_args(in, out, n, ss::kMinScanTile);
    if (st != SS_OK) return st;
    if (n == 0) return SS_OK;
    const size_t tiles = (n + ss::kMinScanTile - 1) / ss::kMinScanTile;  // the most any kernel uses
    Workspace* w = nullptr;
    if (tiles > 1 || g_fault_tile.load() >= 0) {
        st = get_workspace(s, &w);
        if (st != SS_OK) return st;
        st = ensure_desc(w, scan_desc_count(n));
        if (st != SS_OK) return st;
    }
    cudaError_t e = ss::launch_scan_lookback(dt, inclusive, cfg, in, out, n, make_ws(w), carry_in,
                                             carry_out, s);
    if (e != cudaSuccess) return cuda_fail(e, "scan launch");
    return SS_OK;
}

// Scans with 64-bit sums: input element size 4 (widened) or 8 bytes, output
// 8 bytes.  in == out is allowed when both are 8 bytes wide.
ss_status scan_wide(ss::WideType type, bool inclusive, const void* in, void* out, size_t n, cudaStream_t s) {
    const size_t in_size = (type == ss::WideType::U32toU64 || type == ss::WideType::I32toI64) ? 4 : 8;
    if (n == 0) return SS_OK;
    if (in == nullptr || out == nullptr) return fail(SS_ERR_INVALID_ARG, "null pointer with n > 0");
    if ((reinterpret_cast<uintptr_t>(in) & (in_size - 1)) || (reinterpret_cast<uintptr_t>(out) & 7u))
        return fail(SS_ERR_INVALID_ARG, "in/out must be aligned to their element size");
    if (n / ss::kWideTile >= ((size_t)1 << 31) - 1 || n > SIZE_MAX / 16) return fail(SS_ERR_INVALID_ARG, "n too large");
    if (!(in_size == 8 && in == out) && overlaps(in, n * in_size, out, n * 8))
        return fail(SS_ERR_INVALID_ARG, in_size == 8 ? "in and out partially overlap"
                                                     : "a widened scan cannot overlap its input");
    const size_t tile = type == ss::WideType::F64 ? ss::kWideTileF64 : ss::kWideTile;
    const size_t tiles = (n + tile - 1) / tile;
    Workspace* w = nullptr;
    ss_status st = get_workspace(s, &w);
    if (st != SS_OK) return st;
    st = ensure_desc(w, 2 * tiles);  // two words per tile
    if (st != SS_OK) return st;
    cudaError_t e = ss::launch_scan_wide(type, inclusive, in, out, n, make_ws(w), s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "64-bit scan launch");
}

// The device address of a host buffer that the GPU can access directly
// (pinned and mapped, e.g. from cudaHostAlloc), or nullptr.
const void* mapped_device_ptr(const void* h) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        cudaGetLastError();  // not a pointer CUDA knows: clear the error and stage instead
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
    return a.devicePointer;
}

// The look-back scan on buffers that may live in host memory.  It runs the
// one-CTA-per-tile row of the configuration table, whose loads and stores
// are plain 16-byte accesses; the persistent rows stage tiles with bulk
// copies, which are kept to device memory.
ss_status scan_direct(Dtype dt, bool inclusive, const void* in, void* out, size_t n, cudaStream_t s) {
    constexpr int kDirectConfig = 1;
    const size_t tiles = (n + ss::kMinScanTile - 1) / ss::kMinScanTile;
    Workspace* w = nullptr;
    ss_status st = get_workspace(s, &w);
    if (st != SS_OK) return st;
    st = ensure_desc(w, tiles);
    if (st != SS_OK) return st;
    cudaError_t e = ss::launch_scan_lookback(dt, inclusive, kDirectConfig, in, out, n, make_ws(w), nullptr, nullptr, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "scan launch");
}

Dtype to_dtype(ss_dtype d) {
    return d == SS_F32 ? Dtype::F32 : (d == SS_U32 ? Dtype::U32 : Dtype::I32);
}

bool valid_dtype(ss_dtype d) { return d == SS_I32 || d == SS_U32 || d == SS_F32; }

ss::KeepRule positive_rule(ss_dtype dtype) {
    switch (dtype) {
        case SS_F32: return ss::KeepRule::PositiveF32;
        case SS_I32: return ss::KeepRule::PositiveI32;
        default: return ss::KeepRule::PositiveU32;
    }
}

// Every compaction entry point: argument checks, then the ordered
// (look-back) or the unordered (warp-aggregated atomic) kernel.  `flags` is
// used, and required, only under KeepRule::Flags.
ss_status compact_any(ss::KeepRule rule, const void* keys_v, const uint8_t* flags, void* out_v, uint64_t* d_count,
                      size_t n, bool unordered, cudaStream_t s) {
    const uint32_t* keys = static_cast<const uint32_t*>(keys_v);
    uint32_t* out = static_cast<uint32_t*>(out_v);
    const bool with_flags = rule == ss::KeepRule::Flags;
    if (d_count == nullptr) return fail(SS_ERR_INVALID_ARG, "d_count is null");
    if (reinterpret_cast<uintptr_t>(d_count) & 7u)
        return fail(SS_ERR_INVALID_ARG, "d_count must be 8-byte aligned");
    if (n > 0) {
        if (!keys || !out || (with_flags && !flags)) return fail(SS_ERR_INVALID_ARG, "null pointer with n > 0");
        if ((reinterpret_cast<uintptr_t>(keys) | reinterpret_cast<uintptr_t>(out)) & 3u)
            return fail(SS_ERR_INVALID_ARG, "keys/out must be 4-byte aligned");
        if (n > 0xffffffffull) return fail(SS_ERR_INVALID_ARG, "n must be < 2^32");
        if (overlaps(out, n * 4, keys, n * 4) || (with_flags && overlaps(out, n * 4, flags, n)))
            return fail(SS_ERR_INVALID_ARG, "out overlaps keys or flags");
        if (overlaps(d_count, 8, out, n * 4) || overlaps(d_count, 8, keys, n * 4) ||
            (with_flags && overlaps(d_count, 8, flags, n)))
            return fail(SS_ERR_INVALID_ARG, "d_count overlaps an array");
    }
    if (n == 0) {
        cudaError_t e = cudaMemsetAsync(d_count, 0, 8, s);
        return e == cudaSuccess ? SS_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (unordered) {
        cudaError_t e = ss::launch_compact_unordered(rule, keys, flags, out,
                                                     reinterpret_cast<unsigned long long*>(d_count), n, s);
        return e == cudaSuccess ? SS_OK : cuda_fail(e, "unordered compaction launch");
    }
    const size_t tiles = (n + ss::kCompactTile - 1) / ss::kCompactTile;
    Workspace* w = nullptr;
    if (tiles > 1 || g_fault_tile.load() >= 0) {
        ss_status st = get_workspace(s, &w);
        if (st != SS_OK) return st;
        st = ensure_desc(w, tiles);
        if (st != SS_OK) return st;
    }
    cudaError_t e = ss::launch_compact(rule, keys, flags, out, reinterpret_cast<unsigned long long*>(d_count), n,
                                       make_ws(w), s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "compaction launch");
}

// The caller-provided scratch of ss_scan_ws: a 256-byte header (the tile
// counter in word 0, the two status words in word 1), then the descriptors.
constexpr size_t kTempHeader = 256;

size_t temp_bytes_for(size_t n) { return n == 0 ? 0 : kTempHeader + scan_desc_count(n) * 8; }

// Reads and clears a status pair (device) on stream s, and maps it as
// ss_stream_status does.
ss_status read_status_words(uint32_t* d_status, cudaStream_t s, int64_t* failing_tile) {
    uint32_t words[2] = {0, 0};
    cudaError_t e = cudaMemcpyAsync(words, d_status, sizeof(words), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_status, 0, sizeof(words), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "status read-back");
    if (words[0] & ss::kErrCounter) return fail(SS_ERR_CUDA, "tile counter out of step with the launch");
    if (words[0] & ss::kErrBulkTimeout) return fail(SS_ERR_CUDA, "a bulk copy into shared memory did not complete in time");
    if (words[0] & ss::kErrLookbackTimeout) {
        if (failing_tile) *failing_tile = words[1] ? (int64_t)words[1] - 1 : -1;
        return fail(SS_ERR_LOOKBACK_TIMEOUT, "a look-back wait ran out");
    }
    return SS_OK;
}

}  // namespace

extern "C" {

ss_status scan_inclusive_i32(const int32_t* in, int32_t* out, size_t n, ss_stream_t stream) {
    return scan_lookback(Dtype::I32, true, in, out, n, nullptr, nullptr, (cudaStream_t)stream);
}
ss_status scan_exclusive_i32(const int32_t* in, int32_t* out, size_t n, ss_stream_t stream) {
    return scan_lookback(Dtype::I32, false, in, out, n, nullptr, nullptr, (cudaStream_t)stream);
}
ss_status scan_inclusive_u32(const uint32_t* in, uint32_t* out, size_t n, ss_stream_t stream) {
    return scan_lookback(Dtype::U32, true, in, out, n, nullptr, nullptr, (cudaStream_t)stream);
}
ss_status scan_exclusive_u32(const uint32_t* in, uint32_t* out, size_t n, ss_stream_t stream) {
    return scan_lookback(Dtype::U32, false, in, out, n, nullptr, nullptr, (cudaStream_t)stream);
}
ss_status scan_inclusive_f32(const float* in, float* out, size_t n, ss_stream_t stream) {
    return scan_lookback(Dtype::F32, true, in, out, n, nullptr, nullptr, (cudaStream_t)stream);
}
ss_status scan_exclusive_f32(const float* in, float* out, size_t n, ss_stream_t stream) {
    return scan_lookback(Dtype::F32, false, in, out, n, nullptr, nullptr, (cudaStream_t)stream);
}

ss_status ss_scan_seeded(ss_dtype dtype, int inclusive, const void* in, void* out, size_t n,
                         const void* d_carry_in, void* d_carry_out, ss_stream_t stream) {
    if (!valid_dtype(dtype)) return fail(SS_ERR_UNSUPPORTED, "unknown dtype");
    if (d_carry_in && (reinterpret_cast<uintptr_t>(d_carry_in) & 3u))
        return fail(SS_ERR_INVALID_ARG, "carry must be 4-byte aligned");
    if (d_carry_out && (reinterpret_cast<uintptr_t>(d_carry_out) & 3u))
        return fail(SS_ERR_INVALID_ARG, "carry must be 4-byte aligned");
    if (n == 0) {
        if (d_carry_out == nullptr) return SS_OK;
        cudaStream_t s = (cudaStream_t)stream;
        cudaError_t e = d_carry_in ? cudaMemcpyAsync(d_carry_out, d_carry_in, 4, cudaMemcpyDeviceToDevice, s)
                                   : cudaMemsetAsync(d_carry_out, 0, 4, s);
        return e == cudaSuccess ? SS_OK : cuda_fail(e, "carry copy");
    }
    return scan_lookback(to_dtype(dtype), inclusive != 0, in, out, n, d_carry_in, d_carry_out,
                         (cudaStream_t)stream);
}

ss_status ss_reduce_sum(ss_dtype dtype, const void* in, void* d_total, size_t n, ss_stream_t stream) {
    if (!valid_dtype(dtype)) return fail(SS_ERR_UNSUPPORTED, "unknown dtype");
    if (d_total == nullptr) return fail(SS_ERR_INVALID_ARG, "null total");
    if (reinterpret_cast<uintptr_t>(d_total) & 3u) return fail(SS_ERR_INVALID_ARG, "total must be 4-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    if (n == 0) {
        cudaError_t e = cudaMemsetAsync(d_total, 0, 4, s);
        return e == cudaSuccess ? SS_OK : cuda_fail(e, "total clear");
    }
    if (in == nullptr) return fail(SS_ERR_INVALID_ARG, "null pointer with n > 0");
    if (reinterpret_cast<uintptr_t>(in) & 3u) return fail(SS_ERR_INVALID_ARG, "in must be 4-byte aligned");
    if (n > SIZE_MAX / 8) return fail(SS_ERR_INVALID_ARG, "n too large");
    if (overlaps(in, n * 4, d_total, 4)) return fail(SS_ERR_INVALID_ARG, "the total overlaps the input");
    Workspace* w = nullptr;
    ss_status st = get_workspace(s, &w);
    if (st != SS_OK) return st;
    const uint32_t grid = ss::reduce_grid(device_sms(w->device));
    st = ensure_totals(w, (size_t)grid * 4);
    if (st != SS_OK) return st;
    cudaError_t e = ss::launch_reduce_sum(to_dtype(dtype), in, n, w->totals, ws_reduce_ticket(w), d_total, grid, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "reduction launch");
}

ss_status compact_u32(const uint32_t* keys, const uint8_t* flags, uint32_t* out, uint64_t* d_count,
                      size_t n, ss_stream_t stream) {
    return compact_any(ss::KeepRule::Flags, keys, flags, out, d_count, n, false, (cudaStream_t)stream);
}

ss_status compact_positive_f32(const float* in, float* out, uint64_t* d_count, size_t n, ss_stream_t stream) {
    return compact_any(ss::KeepRule::PositiveF32, in, nullptr, out, d_count, n, false, (cudaStream_t)stream);
}

ss_status ss_compact_positive(ss_dtype dtype, const void* in, void* out, uint64_t* d_count, size_t n,
                              ss_stream_t stream) {
    if (!valid_dtype(dtype)) return fail(SS_ERR_UNSUPPORTED, "unknown dtype");
    return compact_any(positive_rule(dtype), in, nullptr, out, d_count, n, false, (cudaStream_t)stream);
}

ss_status ss_compact_u32_unordered(const uint32_t* keys, const uint8_t* flags, uint32_t* out, uint64_t* d_count,
                                   size_t n, ss_stream_t stream) {
    return compact_any(ss::KeepRule::Flags, keys, flags, out, d_count, n, true, (cudaStream_t)stream);
}

ss_status ss_compact_positive_unordered(ss_dtype dtype, const void* in, void* out, uint64_t* d_count, size_t n,
                                        ss_stream_t stream) {
    if (!valid_dtype(dtype)) return fail(SS_ERR_UNSUPPORTED, "unknown dtype");
    return compact_any(positive_rule(dtype), in, nullptr, out, d_count, n, true, (cudaStream_t)stream);
}

ss_status scan_inclusive_u32_u64(const uint32_t* in, uint64_t* out, size_t n, ss_stream_t stream) {
    return scan_wide(ss::WideType::U32toU64, true, in, out, n, (cudaStream_t)stream);
}
ss_status scan_exclusive_u32_u64(const uint32_t* in, uint64_t* out, size_t n, ss_stream_t stream) {
    return scan_wide(ss::WideType::U32toU64, false, in, out, n, (cudaStream_t)stream);
}
ss_status scan_inclusive_i64(const int64_t* in, int64_t* out, size_t n, ss_stream_t stream) {
    return scan_wide(ss::WideType::I64, true, in, out, n, (cudaStream_t)stream);
}
ss_status scan_exclusive_i64(const int64_t* in, int64_t* out, size_t n, ss_stream_t stream) {
    return scan_wide(ss::WideType::I64, false, in, out, n, (cudaStream_t)stream);
}
ss_status scan_inclusive_f64(const double* in, double* out, size_t n, ss_stream_t stream) {
    return scan_wide(ss::WideType::F64, true, in, out, n, (cudaStream_t)stream);
}
ss_status scan_exclusive_f64(const double* in, double* out, size_t n, ss_stream_t stream) {
    return scan_wide(ss::WideType::F64, false, in, out, n, (cudaStream_t)stream);
}

ss_status ss_scan_wide(ss_wide_type type, int inclusive, const void* in, void* out, size_t n, ss_stream_t stream) {
    ss::WideType t;
    switch (type) {
        case SS_WIDE_U32_U64: t = ss::WideType::U32toU64; break;
        case SS_WIDE_I32_I64: t = ss::WideType::I32toI64; break;
        case SS_WIDE_I64: t = ss::WideType::I64; break;
        case SS_WIDE_F64: t = ss::WideType::F64; break;
        default: return fail(SS_ERR_UNSUPPORTED, "unknown 64-bit scan type");
    }
    return scan_wide(t, inclusive != 0, in, out, n, (cudaStream_t)stream);
}

ss_status ss_scan_rows(ss_dtype dtype, int inclusive, const void* in, void* out, size_t rows, size_t cols,
                       ss_stream_t stream) {
    if (!valid_dtype(dtype)) return fail(SS_ERR_UNSUPPORTED, "unknown dtype");
    cudaStream_t s = (cudaStream_t)stream;
    if (rows == 0 || cols == 0) return SS_OK;
    if (rows > SIZE_MAX / 8 / cols) return fail(SS_ERR_INVALID_ARG, "rows * cols too large");
    const size_t n = rows * cols;
    ss_status st = check_scan_args(in, out, n, ss::kMinScanTile);
    if (st != SS_OK) return st;
    if (cols >= kRowsFlat) {
        // Rows this long fill the GPU on their own: one flat single-pass scan
        // per row (the persistent kernel) beats tiles of every row in one launch.
        for (size_t r = 0; r < rows; ++r) {
            st = scan_lookback(to_dtype(dtype), inclusive != 0, static_cast<const uint32_t*>(in) + r * cols,
                               static_cast<uint32_t*>(out) + r * cols, cols, nullptr, nullptr, s);
            if (st != SS_OK) return st;
        }
        return SS_OK;
    }
    Workspace* w = nullptr;
    if (cols > ss::kRowsWarpMax) {
        const size_t tiles = rows * ((cols + ss::kRowsTile - 1) / ss::kRowsTile);  // the most either kernel uses
        if (tiles >= ((size_t)1 << 31)) return fail(SS_ERR_INVALID_ARG, "too many tiles");
        st = get_workspace(s, &w);
        if (st != SS_OK) return st;
        st = ensure_desc(w, tiles);
        if (st != SS_OK) return st;
    }
    cudaError_t e = ss::launch_scan_rows(to_dtype(dtype), inclusive != 0, in, out, rows, cols, make_ws(w), s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "batched scan launch");
}

ss_status ss_scan_segments(ss_dtype dtype, int inclusive, const void* in, void* out, size_t n,
                           const uint64_t* d_offsets, size_t num_segments, ss_stream_t stream) {
    if (!valid_dtype(dtype)) return fail(SS_ERR_UNSUPPORTED, "unknown dtype");
    cudaStream_t s = (cudaStream_t)stream;
    ss_status st = check_scan_args(in, out, n, ss::kMinScanTile);
    if (st != SS_OK) return st;
    if (n == 0) return SS_OK;
    if (num_segments > 0 && d_offsets == nullptr) return fail(SS_ERR_INVALID_ARG, "d_offsets is null");
    if (reinterpret_cast<uintptr_t>(d_offsets) & 7u) return fail(SS_ERR_INVALID_ARG, "d_offsets must be 8-byte aligned");
    if (num_segments > ((size_t)1 << 40)) return fail(SS_ERR_INVALID_ARG, "too many segments");
    if (num_segments > 0 && overlaps(d_offsets, (num_segments + 1) * 8, out, n * 4))
        return fail(SS_ERR_INVALID_ARG, "d_offsets overlaps out");
    const size_t tiles = (n + ss::kSegMinTile - 1) / ss::kSegMinTile;
    Workspace* w = nullptr;
    st = get_workspace(s, &w);
    if (st != SS_OK) return st;
    st = ensure_desc(w, tiles);
    if (st != SS_OK) return st;
    st = ensure_totals(w, ((n + 31) / 32) * 4);
    if (st != SS_OK) return st;
    cudaError_t e = ss::launch_scan_segments(to_dtype(dtype), inclusive != 0, in, out, n,
                                             reinterpret_cast<const unsigned long long*>(d_offsets), num_segments,
                                             static_cast<uint32_t*>(w->totals), make_ws(w), s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "segmented scan launch");
}

ss_status ss_moe_counts_offsets(const int32_t* topk_ids, size_t m, int32_t num_experts, uint32_t align,
                                uint32_t* d_counts, uint32_t* d_offsets, ss_stream_t stream) {
    cudaStream_t s = (cudaStream_t)stream;
    if (num_experts < 1 || num_experts > ss::kMoeMaxExperts)
        return fail(SS_ERR_INVALID_ARG, "num_experts must be in [1, 16384]");
    if (align < 1 || align > (1u << 20)) return fail(SS_ERR_INVALID_ARG, "align must be in [1, 2^20]");
    if (m > 0x7fffffffull) return fail(SS_ERR_INVALID_ARG, "m must be < 2^31");
    if ((uint64_t)m + (uint64_t)num_experts * (align - 1u) > 0xffffffffull)
        return fail(SS_ERR_INVALID_ARG, "the padded total does not fit in 32 bits");
    if (!d_counts || !d_offsets || (m > 0 && !topk_ids)) return fail(SS_ERR_INVALID_ARG, "null pointer");
    if ((reinterpret_cast<uintptr_t>(d_counts) | reinterpret_cast<uintptr_t>(d_offsets) |
         reinterpret_cast<uintptr_t>(topk_ids)) & 3u)
        return fail(SS_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
    const size_t cb = (size_t)num_experts * 4, ob = cb + 4;
    if (overlaps(d_counts, cb, d_offsets, ob) || (m > 0 && (overlaps(d_counts, cb, topk_ids, m * 4) ||
                                                            overlaps(d_offsets, ob, topk_ids, m * 4))))
        return fail(SS_ERR_INVALID_ARG, "counts, offsets and ids must not overlap");
    Workspace* w = nullptr;
    ss_status st = get_workspace(s, &w);
    if (st != SS_OK) return st;
    st = ensure_moe_acc(w, (size_t)num_experts);
    if (st != SS_OK) return st;
    const uint32_t grid = ss::moe_grid(m, device_sms(w->device));
    cudaError_t e = ss::launch_moe_counts_offsets(topk_ids, m, num_experts, align, d_counts, d_offsets, w->moe_acc,
                                                  ws_ticket(w), grid, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "MoE counts launch");
}

ss_status ss_scan(ss_dtype dtype, int inclusive, ss_algo algo, const void* in, void* out, size_t n,
                  ss_stream_t stream) {
    if (!valid_dtype(dtype)) return fail(SS_ERR_UNSUPPORTED, "unknown dtype");
    cudaStream_t s = (cudaStream_t)stream;
    if (algo == SS_ALGO_LOOKBACK)
        return scan_lookback(to_dtype(dtype), inclusive != 0, in, out, n, nullptr, nullptr, s);
    int tile_scan;
    switch (algo) {
        case SS_ALGO_REDUCE_THEN_SCAN: tile_scan = 0; break;
        case SS_ALGO_RTS_BLELLOCH: tile_scan = 1; break;
        case SS_ALGO_RTS_BLELLOCH_PAD32: tile_scan = 2; break;
        case SS_ALGO_RTS_BLELLOCH_PAD2: tile_scan = 3; break;
        default: return fail(SS_ERR_UNSUPPORTED, "unknown algorithm");
    }
    ss_status st = check_scan_args(in, out, n, ss::kRtsTile);
    if (st != SS_OK) return st;
    if (n == 0) return SS_OK;
    Workspace* w = nullptr;
    st = get_workspace(s, &w);
    if (st != SS_OK) return st;
    const size_t tiles = (n + ss::kRtsTile - 1) / ss::kRtsTile;
    st = ensure_totals(w, tiles * 4);
    if (st != SS_OK) return st;
    cudaError_t e = ss::launch_reduce_then_scan(to_dtype(dtype), inclusive != 0, tile_scan, in, out, n,
                                                w->totals, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "reduce-then-scan launch");
}

ss_status ss_scan_trace(int config, const uint32_t* in, uint32_t* out, size_t n, uint64_t* d_trace,
                        ss_stream_t stream) {
    cudaStream_t s = (cudaStream_t)stream;
    if (config < 0 || config >= ss::scan_config_count())
        return fail(SS_ERR_INVALID_ARG, "no such configuration");
    ss_status st = check_scan_args(in, out, n, ss::kMinScanTile);
    if (st != SS_OK) return st;
    if (n == 0) return SS_OK;
    if (d_trace == nullptr || (reinterpret_cast<uintptr_t>(d_trace) & 7u))
        return fail(SS_ERR_INVALID_ARG, "trace must be a non-null, 8-byte aligned device pointer");
    const ss::ScanConfig c = ss::scan_config(config);
    if (c.persistent && (n <= c.tile() || ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 15u)))
        return fail(SS_ERR_INVALID_ARG, "a persistent trace needs 16-byte aligned in/out and more than one tile");
    Workspace* w = nullptr;
    st = get_workspace(s, &w);
    if (st != SS_OK) return st;
    st = ensure_desc(w, scan_desc_count(n));
    if (st != SS_OK) return st;
    cudaError_t e = ss::launch_scan_trace(config, in, out, n, make_ws(w),
                                          reinterpret_cast<unsigned long long*>(d_trace), s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "trace launch");
}

ss_status ss_copy_u32(const uint32_t* in, uint32_t* out, size_t n, ss_stream_t stream) {
    ss_status st = check_scan_args(in, out, n, ss::scan_config(effective_config(n)).tile());
    if (st != SS_OK) return st;
    if (n == 0) return SS_OK;
    cudaError_t e = ss::launch_copy_probe(effective_config(n), in, out, n, (cudaStream_t)stream);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "copy launch");
}

ss_status ss_scan_temp_bytes(size_t n, size_t* bytes) {
    if (bytes == nullptr) return fail(SS_ERR_INVALID_ARG, "bytes is null");
    if (n > (SIZE_MAX / 8)) return fail(SS_ERR_INVALID_ARG, "n too large");
    *bytes = temp_bytes_for(n);
    return SS_OK;
}

ss_status ss_scan_ws(ss_dtype dtype, int inclusive, const void* in, void* out, size_t n, void* temp,
                     size_t temp_bytes, ss_stream_t stream) {
    if (dtype != SS_I32 && dtype != SS_U32 && dtype != SS_F32) return fail(SS_ERR_UNSUPPORTED, "unknown dtype");
    ss_status st = check_scan_args(in, out, n, ss::kMinScanTile);
    if (st != SS_OK) return st;
    if (n == 0) return SS_OK;
    const size_t need = temp_bytes_for(n);
    if (temp == nullptr) return fail(SS_ERR_INVALID_ARG, "temp is null");
    if (reinterpret_cast<uintptr_t>(temp) & 255u) return fail(SS_ERR_INVALID_ARG, "temp must be 256-byte aligned");
    if (temp_bytes < need) return fail(SS_ERR_INVALID_ARG, "temp_bytes is below ss_scan_temp_bytes(n)");
    if (overlaps(temp, need, in, n * 4) || overlaps(temp, need, out, n * 4))
        return fail(SS_ERR_INVALID_ARG, "temp overlaps in or out");
    cudaStream_t s = (cudaStream_t)stream;
    // The contents on entry are whatever the caller left there: clear what
    // this call uses (counter, status words, descriptors) on the stream.
    cudaError_t e = cudaMemsetAsync(temp, 0, need, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    unsigned long long* base = static_cast<unsigned long long*>(temp);
    ss::LookbackWs ws = make_ws(nullptr);
    ws.counter = base;
    ws.status = reinterpret_cast<uint32_t*>(base + 1);
    ws.desc = base + kTempHeader / 8;
    e = ss::launch_scan_lookback(to_dtype(dtype), inclusive != 0, effective_config(n), in, out, n, ws, nullptr,
                                 nullptr, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "scan launch");
}

ss_status ss_temp_status(void* temp, ss_stream_t stream, int64_t* failing_tile) {
    if (failing_tile) *failing_tile = -1;
    if (temp == nullptr || (reinterpret_cast<uintptr_t>(temp) & 255u))
        return fail(SS_ERR_INVALID_ARG, "temp must be a non-null, 256-byte aligned device pointer");
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return read_status_words(reinterpret_cast<uint32_t*>(static_cast<unsigned long long*>(temp) + 1), s,
                             failing_tile);
}

ss_status ss_stream_status(ss_stream_t stream, int64_t* failing_tile) {
    cudaStream_t s = (cudaStream_t)stream;
    if (failing_tile) *failing_tile = -1;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    Workspace* w = nullptr;
    {
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_ws.find(std::make_pair(dev, reinterpret_cast<uintptr_t>(s)));
        if (it != g_ws.end()) w = it->second;
    }
    if (w == nullptr) return SS_OK;
    uint32_t words[2] = {0, 0};
    e = cudaMemcpyAsync(words, ws_status(w), sizeof(words), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws_status(w), 0, sizeof(words), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "status read-back");
    if (words[0] & ss::kErrCounter) {
        // Start the workspace afresh: counter and every descriptor to zero.
        cudaMemsetAsync(ws_counter(w), 0, 8, s);
        if (w->desc) cudaMemsetAsync(w->desc, 0, w->desc_cap * 8, s);
        cudaStreamSynchronize(s);
        return fail(SS_ERR_CUDA, "tile counter out of step with the launch (concurrent use of one stream's workspace?)");
    }
    if (words[0] & ss::kErrBulkTimeout)
        return fail(SS_ERR_CUDA, "a bulk copy into shared memory did not complete in time");
    if (words[0] & ss::kErrLookbackTimeout) {
        if (failing_tile) *failing_tile = words[1] ? (int64_t)words[1] - 1 : -1;
        return fail(SS_ERR_LOOKBACK_TIMEOUT, "a look-back wait ran out");
    }
    return SS_OK;
}

static ss_status host_pipe_init(Workspace* w, size_t elems) {
    HostPipe& p = w->pipe;
    if (p.ready) return SS_OK;
    cudaError_t e;
    for (int b = 0; b < kHostBuffers; ++b) {
        e = cudaMalloc(&p.buf[b], elems * 4);
        if (e != cudaSuccess) return fail(SS_ERR_NO_MEMORY, "host pipeline buffers");
        if ((e = cudaEventCreateWithFlags(&p.ev_in[b], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.ev_scan[b], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.ev_out[b], cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "cudaEventCreate");
    }
    if ((e = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail(e, "cudaStreamCreate");
    p.ready = true;
    return SS_OK;
}

ss_status ss_set_host_mode(int mode) {
    if (mode < 0 || mode > 1) return fail(SS_ERR_INVALID_ARG, "host mode must be 0 or 1");
    g_host_mode.store(mode);
    return SS_OK;
}

ss_status ss_scan_host(ss_dtype dtype, int inclusive, const void* h_in, void* h_out, size_t n,
                       ss_stream_t stream) {
    if (!valid_dtype(dtype)) return fail(SS_ERR_UNSUPPORTED, "unknown dtype");
    if (n == 0) return SS_OK;
    if (h_in == nullptr || h_out == nullptr) return fail(SS_ERR_INVALID_ARG, "null pointer with n > 0");
    if (h_in != h_out && overlaps(h_in, n * 4, h_out, n * 4))
        return fail(SS_ERR_INVALID_ARG, "h_in and h_out partially overlap");
    cudaStream_t s = (cudaStream_t)stream;
    if (g_host_mode.load() == 0) {
        // Both buffers pinned and mapped: the kernel reads and writes host
        // memory directly (over NVLink-C2C on Grace), with no staging copies.
        const void* d_in = mapped_device_ptr(h_in);
        void* d_out = const_cast<void*>(mapped_device_ptr(h_out));
        if (d_in != nullptr && d_out != nullptr) {
            ss_status st = scan_direct(to_dtype(dtype), inclusive != 0, d_in, d_out, n, s);
            if (st != SS_OK) return st;
            cudaError_t e = cudaStreamSynchronize(s);
            return e == cudaSuccess ? SS_OK : cuda_fail(e, "cudaStreamSynchronize");
        }
    }
    Workspace* w = nullptr;
    ss_status st = get_workspace(s, &w);
    if (st != SS_OK) return st;
    std::lock_guard<std::mutex> lk(w->pipe_mu);
    st = host_pipe_init(w, kHostChunk);
    if (st != SS_OK) return st;
    HostPipe& p = w->pipe;
    void* carry = ws_carry(w);
    cudaError_t e = cudaMemsetAsync(carry, 0, 4, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    const size_t chunks = (n + kHostChunk - 1) / kHostChunk;
    const char* src = static_cast<const char*>(h_in);
    char* dst = static_cast<char*>(h_out);
    // The d2h stream must not start before earlier work on `s`; the h2d stream
    // must not overwrite a buffer before its previous results were copied out.
    cudaEvent_t start_ev = p.ev_scan[0];
    if ((e = cudaEventRecord(start_ev, s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    if ((e = cudaStreamWaitEvent(p.h2d, start_ev, 0)) != cudaSuccess) return cuda_fail(e, "wait");
    if ((e = cudaStreamWaitEvent(p.d2h, start_ev, 0)) != cudaSuccess) return cuda_fail(e, "wait");
    for (size_t c = 0; c < chunks; ++c) {
        const int b = (int)(c % kHostBuffers);
        const size_t off = c * kHostChunk;
        const size_t cnt = (n - off) < kHostChunk ? (n - off) : kHostChunk;
        if (c >= (size_t)kHostBuffers && (e = cudaStreamWaitEvent(p.h2d, p.ev_out[b], 0)) != cudaSuccess)
            return cuda_fail(e, "wait");
        if ((e = cudaMemcpyAsync(p.buf[b], src + off * 4, cnt * 4, cudaMemcpyHostToDevice, p.h2d)) != cudaSuccess)
            return cuda_fail(e, "cudaMemcpyAsync H2D");
        if ((e = cudaEventRecord(p.ev_in[b], p.h2d)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
        if ((e = cudaStreamWaitEvent(s, p.ev_in[b], 0)) != cudaSuccess) return cuda_fail(e, "wait");
        st = scan_lookback(to_dtype(dtype), inclusive != 0, p.buf[b], p.buf[b], cnt, carry, carry, s);
        if (st != SS_OK) return st;
        if ((e = cudaEventRecord(p.ev_scan[b], s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
        if ((e = cudaStreamWaitEvent(p.d2h, p.ev_scan[b], 0)) != cudaSuccess) return cuda_fail(e, "wait");
        if ((e = cudaMemcpyAsync(dst + off * 4, p.buf[b], cnt * 4, cudaMemcpyDeviceToHost, p.d2h)) != cudaSuccess)
            return cuda_fail(e, "cudaMemcpyAsync D2H");
        if ((e = cudaEventRecord(p.ev_out[b], p.d2h)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    }
    if ((e = cudaStreamSynchronize(p.d2h)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return SS_OK;
}

const char* ss_status_string(ss_status status) {
    switch (status) {
        case SS_OK: return "ok";
        case SS_ERR_INVALID_ARG: return "invalid argument";
        case SS_ERR_CUDA: return "CUDA error";
        case SS_ERR_LOOKBACK_TIMEOUT: return "look-back wait timed out";
        case SS_ERR_NO_MEMORY: return "out of device memory";
        case SS_ERR_UNSUPPORTED: return "unsupported";
    }
    return "unknown status";
}

const char* ss_last_error_detail(void) { return g_detail.c_str(); }

size_t ss_scan_tile_elems(void) { return ss::scan_config(effective_config(SIZE_MAX)).tile(); }

int ss_scan_config_count(void) { return ss::scan_config_count(); }

ss_status ss_set_scan_config(int config) {
    if (config < -1 || config >= ss::scan_config_count())
        return fail(SS_ERR_INVALID_ARG, "no such configuration");
    g_config.store(config);
    return SS_OK;
}

ss_status ss_set_compact_config(int config) {
    if (config < 0 || config >= ss::compact_kernel_count())
        return fail(SS_ERR_INVALID_ARG, "no such compaction configuration");
    ss::set_compact_kernel(config);
    return SS_OK;
}

ss_status ss_set_segments_config(int config) {
    if (config < 0 || config >= ss::segments_config_count())
        return fail(SS_ERR_INVALID_ARG, "no such segmented scan configuration");
    ss::set_segments_config(config);
    return SS_OK;
}

void ss_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : g_ws) {
        Workspace* w = kv.second;
        cudaSetDevice(w->device);
        cudaDeviceSynchronize();
        if (w->desc) cudaFree(w->desc);
        if (w->totals) cudaFree(w->totals);
        if (w->moe_acc) cudaFree(w->moe_acc);
        if (w->header) cudaFree(w->header);
        HostPipe& p = w->pipe;
        if (p.ready) {
            for (int b = 0; b < kHostBuffers; ++b) {
                cudaFree(p.buf[b]);
                cudaEventDestroy(p.ev_in[b]);
                cudaEventDestroy(p.ev_scan[b]);
                cudaEventDestroy(p.ev_out[b]);
            }
            cudaStreamDestroy(p.h2d);
            cudaStreamDestroy(p.d2h);
        }
        delete w;
    }
    g_ws.clear();
    cudaSetDevice(cur);
}

ss_status ss_debug_set_lookback_fault(int64_t tile, uint64_t timeout_ns) {
    if (tile < -1) return fail(SS_ERR_INVALID_ARG, "tile must be >= -1");
    g_fault_tile.store(tile);
    g_timeout_ns.store(timeout_ns);
    return SS_OK;
}

}  // extern "C"
