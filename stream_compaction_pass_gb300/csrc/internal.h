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
constexpr uint32_t kErrCounter = 2u;      // a CTA claimed a tile id past the grid
constexpr uint32_t kErrBulkTimeout = 4u;  // a bulk copy into shared memory never completed

// Device pointers into a workspace for the single-pass kernels.
struct LookbackWs {
    unsigned long long* desc = nullptr;     // >= tiles descriptors
    unsigned long long* counter = nullptr;  // tile counter (epoch | count)
    uint32_t* status = nullptr;             // error bits, failing tile + 1
    uint64_t timeout_ns = 2000000000ull;    // look-back wait limit
    uint32_t max_polls = 1u << 22;          // backstop on polls per wait
    int64_t fault_tile = -1;                // test hook: tile that never publishes
};

// Launch set-up of a kernel on the current device: SM count and resident CTAs
// per SM at `max_smem` bytes of dynamic shared memory, whose limit it also
// raises (launch.cu).  Done once per (kernel, device); thread-safe.
struct KernelSetup {
    int sms = 1;
    int blocks_per_sm = 1;
};
cudaError_t kernel_setup(const void* kern, int threads, size_t max_smem, KernelSetup* out);

// A single-pass scan configuration: which kernel, its tile geometry and
// its look-back window.
struct ScanConfig {
    int persistent;  // 0: one CTA per tile (scan.cu); 1: persistent, bulk-copy ring (scan_pipe.cu);
                     // 2: persistent and warp-specialised (scan_ws.cu; threads = data threads)
    int threads;
    int items;       // per thread, a multiple of 4
    int stages;      // ring depth of the persistent kernel
    int lookback_k;  // look-back window = 32 * lookback_k descriptors per poll
    size_t tile() const { return (size_t)threads * (size_t)items; }
};

// Selectable scan configurations.  Index 0 (one CTA per 4096-element tile,
// 32-descriptor window) is fixed; scan_default_config() is the one the
// library starts with.
int scan_config_count();
ScanConfig scan_config(int idx);
int scan_default_config();

// Smallest tile of any configuration: workspaces are sized with it, so a
// launch that falls back to a smaller tile still has a descriptor per tile.
constexpr size_t kMinScanTile = 4096;

// The persistent variant of launch_scan_lookback (scan_pipe.cu); `config`
// must name a persistent configuration and in/out must be 16-byte aligned.
cudaError_t launch_scan_lookback_pipe(Dtype dt, bool inclusive, int config, const void* in, void* out,
                                      size_t n, const LookbackWs& ws, const void* carry_in,
                                      void* carry_out, cudaStream_t s);

// Exclusive uint32 scan with a per-tile timing trace (8 x uint64 per tile,
// layout in scan_body.cuh).  Every row of the configuration table has a
// traced build.
cudaError_t launch_scan_trace(int config, const void* in, void* out, size_t n, const LookbackWs& ws,
                              unsigned long long* trace, cudaStream_t s);
cudaError_t launch_scan_trace_pipe(int config, const void* in, void* out, size_t n,
                                   const LookbackWs& ws, unsigned long long* trace, cudaStream_t s);
cudaError_t launch_scan_lookback_ws(Dtype dt, bool inclusive, int config, const void* in, void* out,
                                    size_t n, const LookbackWs& ws, const void* carry_in, void* carry_out,
                                    cudaStream_t s);
cudaError_t launch_scan_trace_ws(int config, const void* in, void* out, size_t n, const LookbackWs& ws,
                                 unsigned long long* trace, cudaStream_t s);

// Single-pass decoupled look-back scan.  `carry_in` (device, may be null)
// seeds the prefix of element 0; `carry_out` (device, may be null) receives
// the inclusive total.  `in` may equal `out`.
cudaError_t launch_scan_lookback(Dtype dt, bool inclusive, int config, const void* in, void* out,
                                 size_t n, const LookbackWs& ws, const void* carry_in,
                                 void* carry_out, cudaStream_t s);

// Streaming copy with the scan's loader and storer (the bandwidth probe).
cudaError_t launch_copy_probe(int config, const void* in, void* out, size_t n, cudaStream_t s);

// What a compaction keeps: keys whose flag byte is nonzero, or keys that
// satisfy "v > 0" in their own type (keep.cuh).
enum class KeepRule : int { Flags = 0, PositiveF32 = 1, PositiveI32 = 2, PositiveU32 = 3 };

// Fused order-preserving compaction.  `flags` is read only under
// KeepRule::Flags (null otherwise).
constexpr size_t kCompactTile = 4096;
cudaError_t launch_compact(KeepRule rule, const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                           unsigned long long* d_count, size_t n, const LookbackWs& ws, cudaStream_t s);

// Persistent form of the compaction (compact_pipe.cu): 16-byte aligned keys
// (and flags), n above one 16384-element tile.
cudaError_t launch_compact_pipe(KeepRule rule, const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                                unsigned long long* d_count, size_t n, const LookbackWs& ws, cudaStream_t s);

// Predicate compaction (compact_pred.cu): keys kept where the rule holds
// (PositiveF32/I32/U32), with a dedicated look-back warp and staged 16-byte
// stores; keys 16-byte aligned, n > 16384.
cudaError_t launch_compact_pred(KeepRule rule, const uint32_t* keys, uint32_t* out, unsigned long long* d_count,
                                size_t n, const LookbackWs& ws, cudaStream_t s);
int compact_kernel_count();
void set_compact_kernel(int k);

// Unordered compaction by warp-aggregated atomics (compact_unordered.cu):
// the kept keys in no fixed order, *d_count reset and counted on `s`.
cudaError_t launch_compact_unordered(KeepRule rule, const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                                     unsigned long long* d_count, size_t n, cudaStream_t s);

// Scans with 64-bit sums (scan_wide.cu): uint32 -> uint64, int32 -> int64,
// int64 (modulo 2^64; uint64 is the same bits) and fp64.  Descriptors are 16
// bytes, two 64-bit words per tile: the workspace holds one per kWideTile
// elements for the integer types (the smallest of their tiles), per
// kWideTileF64 for fp64.
enum class WideType : int { U32toU64 = 0, I32toI64 = 1, I64 = 2, F64 = 3 };
constexpr size_t kWideTile = 4096;
constexpr size_t kWideTileF64 = 4096;
cudaError_t launch_scan_wide(WideType type, bool inclusive, const void* in, void* out, size_t n,
                             const LookbackWs& ws, cudaStream_t s);

// Batched scans (scan_rows.cu): every row of a row-major rows x cols matrix
// scanned on its own.  Rows longer than kRowsWarpMax go through row-aligned
// kRowsTile-element tiles with the look-back (one descriptor per tile);
// shorter rows take one warp each and need no workspace.
constexpr size_t kRowsTile = 4096;
constexpr size_t kRowsWarpMax = 2048;
constexpr size_t kRowsPipeTile = 16384;  // persistent kernel for rows of at least kRowsPipeMin
constexpr size_t kRowsPipeMin = 16384;
cudaError_t launch_scan_rows(Dtype dt, bool inclusive, const void* in, void* out, size_t rows, size_t cols,
                             const LookbackWs& ws, cudaStream_t s);

// Segmented scans (scan_segments.cu): `bits` is a workspace bitmask of
// ceil(n / 32) words that the call zeroes and fills with the segment starts
// (offsets[0 .. num_segments-1]) before the scan.  Every form's tile is a
// multiple of kSegMinTile elements, so a descriptor per kSegMinTile elements
// covers any of them.
constexpr size_t kSegMinTile = 2048;
int segments_config_count();
void set_segments_config(int c);
cudaError_t launch_scan_segments(Dtype dt, bool inclusive, const void* in, void* out, size_t n,
                                 const unsigned long long* offsets, size_t num_segments, uint32_t* bits,
                                 const LookbackWs& ws, cudaStream_t s);

// MoE token counts and tile-aligned offsets (moe.cu).  `acc` holds
// num_experts uint32 and `ticket` one; both are zero on entry and the launch
// leaves them zero.
constexpr int32_t kMoeMaxExperts = 16384;
cudaError_t launch_moe_counts_offsets(const int32_t* ids, size_t m, int32_t num_experts, uint32_t align,
                                      uint32_t* counts, uint32_t* offsets, uint32_t* acc, uint32_t* ticket,
                                      uint32_t grid, cudaStream_t s);
uint32_t moe_grid(size_t m, int sms);

// Sum of a whole array (reduce.cu): int32/uint32 wrap modulo 2^32, fp32 in
// an order fixed by n and the grid.  `partials` holds `grid` values and
// `ticket` is zero on entry; the launch leaves it zero.
uint32_t reduce_grid(int sms);
cudaError_t launch_reduce_sum(Dtype dt, const void* in, size_t n, void* partials, uint32_t* ticket, void* total,
                              uint32_t grid, cudaStream_t s);

// Ablations (reduce-then-scan, three kernels).  `totals` holds one value
// per 4096-element tile.  tile_scan: 0 = register/shuffle tile scan,
// 1 = Blelloch tree unpadded, 2 = Blelloch padded i + i/32,
// 3 = Blelloch padded i + i/32 + i/1024.
constexpr size_t kRtsTile = 4096;
cudaError_t launch_reduce_then_scan(Dtype dt, bool inclusive, int tile_scan, const void* in,
                                    void* out, size_t n, void* totals, cudaStream_t s);

}  // namespace ss
