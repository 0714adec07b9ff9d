// internal.h -- launchers shared between the kernel files and the C ABI
// (api.cu).  Not installed; the public interface is include/streamscan.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ss {

enum class Dtype : int { I32 = 0, U32 = 1, F32 = 2 };

// Status word bits written by kernels and read back by ss_stream_status.
constexpr uint32_t kErrLookbackTimeout = 1u;
constexpr uint32_t kErrCounter = 2u;  // a CTA claimed a tile id past the grid

// Device pointers into a workspace for the single-pass kernels.
struct LookbackWs {
    unsigned long long* desc = nullptr;     // >= tiles descriptors
    unsigned long long* counter = nullptr;  // tile counter (epoch | count)
    uint32_t* status = nullptr;             // error bits, failing tile + 1
    uint64_t timeout_ns = 2000000000ull;    // look-back wait limit
    uint32_t max_polls = 1u << 22;          // backstop on polls per wait
    int64_t fault_tile = -1;                // test hook: tile that never publishes
};

// Tile geometry of a single-pass scan configuration.
struct ScanConfig {
    int threads;
    int items;  // per thread, a multiple of 4
    size_t tile() const { return (size_t)threads * (size_t)items; }
};

// Selectable scan configurations (index 0 is the default).
int scan_config_count();
ScanConfig scan_config(int idx);

// Single-pass decoupled look-back scan.  `carry_in` (device, may be null)
// seeds the prefix of element 0; `carry_out` (device, may be null) receives
// the inclusive total.  `in` may equal `out`.
cudaError_t launch_scan_lookback(Dtype dt, bool inclusive, int config, const void* in, void* out,
                                 size_t n, const LookbackWs& ws, const void* carry_in,
                                 void* carry_out, cudaStream_t s);

// Streaming copy with the scan's loader and storer (the bandwidth probe).
cudaError_t launch_copy_probe(int config, const void* in, void* out, size_t n, cudaStream_t s);

// Fused order-preserving compaction.
constexpr size_t kCompactTile = 4096;
cudaError_t launch_compact_u32(const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                               unsigned long long* d_count, size_t n, const LookbackWs& ws,
                               cudaStream_t s);

// Ablations (reduce-then-scan, three kernels).  `totals` holds one value
// per 4096-element tile.  tile_scan: 0 = register/shuffle tile scan,
// 1 = Blelloch tree unpadded, 2 = Blelloch padded i + i/32,
// 3 = Blelloch padded i + i/32 + i/1024.
constexpr size_t kRtsTile = 4096;
cudaError_t launch_reduce_then_scan(Dtype dt, bool inclusive, int tile_scan, const void* in,
                                    void* out, size_t n, void* totals, cudaStream_t s);

}  // namespace ss
