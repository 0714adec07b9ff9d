// scan.cu -- single-pass device-wide scan with decoupled look-back, and the
// copy probe that shares its loader and storer.
//
// One CTA per tile.  Each CTA (1) claims a tile id from the workspace
// counter, so a tile only ever waits on tiles whose CTAs are already running
// or done; (2) loads its tile with 16-byte coalesced loads; (3) scans it in
// registers and shuffles (tile.cuh); (4) publishes its aggregate, looks back
// over its predecessors' descriptors and publishes its inclusive prefix
// (lookback.cuh); (5) writes its outputs with 16-byte stores.  The input is
// read once and the output written once: 2 * n * sizeof(T) bytes of HBM
// traffic, against the three-pass scans' 4n ("Prefix sum and other parallel
// patterns", A device-level scan: scan then propagate, last paragraph;
// "7 Work-efficient Scan: Blelloch", last summary point).
//
// int32 and uint32 share the uint32 kernels: two's-complement addition and
// unsigned addition produce the same bits.
#include "internal.h"
#include "scan_body.cuh"

namespace ss {

template <typename T, bool INCLUSIVE, int THREADS, int VPT, int K, bool TRACE, bool GROUPED>
__global__ void __launch_bounds__(THREADS)
k_scan_lookback(const T* in, T* out, size_t n, uint32_t num_tiles, LookbackCtx ctx, bool aligned,
                const T* carry_in, T* carry_out, unsigned long long* trace) {
    constexpr size_t TILE = (size_t)THREADS * VPT * 4;
    constexpr size_t SEG = (size_t)32 * VPT * 4;  // elements per warp segment

    __shared__ ScanSmem<T, THREADS / 32> sm;
    __shared__ uint32_t s_tile, s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const unsigned long long t_begin = TRACE ? globaltimer_ns() : 0ull;

    if (threadIdx.x == 0) {
        uint32_t tile = 0, epoch = 0;
        if (num_tiles > 1) claim_tile(ctx.counter, num_tiles, &tile, &epoch);
        s_tile = tile;
        s_epoch = epoch;
    }
    __syncthreads();
    const uint32_t tile = s_tile;
    const uint32_t epoch = s_epoch;
    if (tile >= num_tiles) {  // counter out of step: never index past the descriptors
        if (threadIdx.x == 0) record_error(ctx.status, kErrCounter, tile);
        return;
    }
    unsigned long long* rec = TRACE ? trace + (size_t)tile * kTraceWords : nullptr;
    if (TRACE && threadIdx.x == 0) rec[0] = t_begin;

    const size_t seg = (size_t)tile * TILE + (size_t)warp * SEG;
    const bool fast = aligned && (seg + SEG <= n);
    T v[VPT][4];
    load_rows<T, VPT>(in, n, seg, lane, fast, v);
    scan_tile_body<T, INCLUSIVE, THREADS, VPT, K, TRACE, GROUPED>(v, out, n, seg, fast, tile, num_tiles, epoch,
                                                                  ctx, carry_in, carry_out, sm, rec);
}

template <int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS)
k_copy_probe(const uint32_t* in, uint32_t* out, size_t n, bool aligned) {
    constexpr size_t TILE = (size_t)THREADS * VPT * 4;
    constexpr size_t SEG = (size_t)32 * VPT * 4;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const size_t seg = (size_t)blockIdx.x * TILE + (size_t)warp * SEG;
    const bool fast = aligned && (seg + SEG <= n);
    uint32_t v[VPT][4];
    load_rows<uint32_t, VPT>(in, n, seg, lane, fast, v);
    store_rows<uint32_t, VPT>(out, n, seg, lane, fast, v);
}

// Configurations: {persistent, threads, items, stages, look-back K}.
static const ScanConfig kConfigs[] = {
    {0, 256, 16, 0, 1},  // 0: one CTA per 4096-element tile (the allocation-free entry point's kernel)
    {0, 256, 32, 0, 1},  // 1: one CTA per 8192-element tile (the fallback for unaligned or small inputs)
    {1, 512, 36, 3, 1},  // 2: persistent, 18432-element tiles, 3-stage ring (216 KB), single register buffer
    {1, 512, 32, 3, 1},  // 3: persistent, 16384, 3 stages (192 KB), single register buffer
    {1, 512, 16, 3, 1},  // 4: persistent, 8192, 3 stages (96 KB, two CTAs per SM)
    {2, 512, 32, 3, 1},  // 5: persistent and warp-specialised, 16384, 3 stages, look-back one tile late
    {1, 512, 32, 3, 1},  // 6: persistent, lean iteration (one barrier), 16384, 3 stages
    {1, 512, 32, 2, 1},  // 7: persistent, 16384, 2-stage ring (128 KB), double register buffer
    {1, 512, 36, 3, 1},  // 8: as row 2, each tile claimed from the counter when its copy starts -- the default
    {1, 512, 32, 3, 1},  // 9: as row 8 with 16384-element tiles
    {0, 256, 16, 0, 1},  // 10: one CTA per 4096-element tile, two-level look-back (groups of 32 tiles)
    {0, 256, 32, 0, 1},  // 11: the same with 8192-element tiles
    {0, 512, 16, 0, 1},  // 12: the same with 8192-element tiles of 512 threads
};
constexpr int kNumConfigs = sizeof(kConfigs) / sizeof(kConfigs[0]);
constexpr int kDefaultConfig = 8;

int scan_config_count() { return kNumConfigs; }
ScanConfig scan_config(int idx) { return kConfigs[(idx >= 0 && idx < kNumConfigs) ? idx : 0]; }
int scan_default_config() { return kDefaultConfig; }

static bool aligned16(const void* a, const void* b) {
    return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
}

template <typename T, bool INCL, int THREADS, int VPT, int K, bool TRACE = false, bool GROUPED = false>
static cudaError_t launch_one(const void* in, void* out, size_t n, const LookbackWs& ws,
                             const void* carry_in, void* carry_out, cudaStream_t s,
                             unsigned long long* trace = nullptr) {
    const size_t tile = (size_t)THREADS * VPT * 4;
    const uint32_t tiles = (uint32_t)((n + tile - 1) / tile);
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    k_scan_lookback<T, INCL, THREADS, VPT, K, TRACE, GROUPED><<<tiles, THREADS, 0, s>>>(
        static_cast<const T*>(in), static_cast<T*>(out), n, tiles, ctx, aligned16(in, out),
        static_cast<const T*>(carry_in), static_cast<T*>(carry_out), trace);
    return cudaGetLastError();
}

template <typename T, bool INCL>
static cudaError_t dispatch_config(int config, const void* in, void* out, size_t n,
                                   const LookbackWs& ws, const void* ci, void* co, cudaStream_t s) {
    switch (config) {
        case 1: return launch_one<T, INCL, 256, 8, 1>(in, out, n, ws, ci, co, s);
        case 10: return launch_one<T, INCL, 256, 4, 1, false, true>(in, out, n, ws, ci, co, s);
        case 11: return launch_one<T, INCL, 256, 8, 1, false, true>(in, out, n, ws, ci, co, s);
        case 12: return launch_one<T, INCL, 512, 4, 1, false, true>(in, out, n, ws, ci, co, s);
        default: return launch_one<T, INCL, 256, 4, 1>(in, out, n, ws, ci, co, s);
    }
}

// The persistent kernel needs 16-byte aligned in/out (bulk copies) and at
// least two tiles; anything else runs on the one-CTA-per-tile kernel of the
// same tile size, or on configuration 0.
static int per_tile_fallback(int config) {
    (void)config;
    return 1;  // 8192-element tiles, the fastest one-CTA-per-tile row
}

cudaError_t launch_scan_lookback(Dtype dt, bool inclusive, int config, const void* in, void* out,
                                 size_t n, const LookbackWs& ws, const void* carry_in,
                                 void* carry_out, cudaStream_t s) {
    const ScanConfig c = scan_config(config);
    if (c.persistent) {
        if (aligned16(in, out) && n > c.tile())
            return c.persistent == 2
                       ? launch_scan_lookback_ws(dt, inclusive, config, in, out, n, ws, carry_in, carry_out, s)
                       : launch_scan_lookback_pipe(dt, inclusive, config, in, out, n, ws, carry_in, carry_out, s);
        config = per_tile_fallback(config);
    }
    if (dt == Dtype::F32)
        return inclusive ? dispatch_config<float, true>(config, in, out, n, ws, carry_in, carry_out, s)
                         : dispatch_config<float, false>(config, in, out, n, ws, carry_in, carry_out, s);
    return inclusive ? dispatch_config<uint32_t, true>(config, in, out, n, ws, carry_in, carry_out, s)
                     : dispatch_config<uint32_t, false>(config, in, out, n, ws, carry_in, carry_out, s);
}

cudaError_t launch_scan_trace(int config, const void* in, void* out, size_t n, const LookbackWs& ws,
                              unsigned long long* trace, cudaStream_t s) {
    const ScanConfig c = scan_config(config);
    if (c.persistent) {
        if (!aligned16(in, out) || n <= c.tile()) return cudaErrorInvalidValue;
        return c.persistent == 2 ? launch_scan_trace_ws(config, in, out, n, ws, trace, s)
                                 : launch_scan_trace_pipe(config, in, out, n, ws, trace, s);
    }
    switch (config) {
        case 1: return launch_one<uint32_t, false, 256, 8, 1, true>(in, out, n, ws, nullptr, nullptr, s, trace);
        case 0: return launch_one<uint32_t, false, 256, 4, 1, true>(in, out, n, ws, nullptr, nullptr, s, trace);
        case 10: return launch_one<uint32_t, false, 256, 4, 1, true, true>(in, out, n, ws, nullptr, nullptr, s, trace);
        case 11: return launch_one<uint32_t, false, 256, 8, 1, true, true>(in, out, n, ws, nullptr, nullptr, s, trace);
        case 12: return launch_one<uint32_t, false, 512, 4, 1, true, true>(in, out, n, ws, nullptr, nullptr, s, trace);
        default: return cudaErrorInvalidValue;  // every row has a traced build
    }
}

template <int THREADS, int VPT>
static cudaError_t launch_copy(const void* in, void* out, size_t n, cudaStream_t s) {
    const size_t tile = (size_t)THREADS * VPT * 4;
    const uint32_t tiles = (uint32_t)((n + tile - 1) / tile);
    k_copy_probe<THREADS, VPT><<<tiles, THREADS, 0, s>>>(static_cast<const uint32_t*>(in),
                                                         static_cast<uint32_t*>(out), n,
                                                         aligned16(in, out));
    return cudaGetLastError();
}

cudaError_t launch_copy_probe(int config, const void* in, void* out, size_t n, cudaStream_t s) {
    (void)config;  // one geometry: 256 threads x 16 elements, the scan's default loader shape
    return launch_copy<256, 4>(in, out, n, s);
}

}  // namespace ss
