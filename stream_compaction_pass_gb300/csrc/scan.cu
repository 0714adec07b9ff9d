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
#include "tile.cuh"

namespace ss {

template <typename T, bool INCLUSIVE, int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS)
k_scan_lookback(const T* in, T* out, size_t n, uint32_t num_tiles, LookbackCtx ctx, bool aligned,
                const T* carry_in, T* carry_out) {
    constexpr int WARPS = THREADS / 32;
    constexpr size_t TILE = (size_t)THREADS * VPT * 4;
    constexpr size_t SEG = (size_t)32 * VPT * 4;  // elements per warp segment

    __shared__ T s_warp[WARPS];
    __shared__ T s_prefix;
    __shared__ uint32_t s_tile, s_epoch, s_fail;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

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

    const size_t tile_base = (size_t)tile * TILE;
    const size_t seg = tile_base + (size_t)warp * SEG;
    const bool fast = aligned && (seg + SEG <= n);

    T v[VPT][4];
    load_rows<T, VPT>(in, n, seg, lane, fast, v);

    T pre[VPT];
    const T warp_total = warp_rows_scan<T, VPT>(v, lane, pre);
    T warp_prefix, block_total;
    block_combine<T, WARPS>(warp_total, warp, lane, s_warp, &warp_prefix, &block_total);

    if (warp == 0) {
        T excl = T(0);
        bool failed = false;
        const bool dead = (int64_t)tile == ctx.fault_tile;  // test hook only
        if (tile == 0) {
            excl = carry_in ? *carry_in : T(0);
            if (num_tiles > 1 && lane == 0 && !dead)
                st_relaxed_u64(ctx.desc, pack_desc(epoch, kStateP, to_bits<T>(excl + block_total)));
            failed = dead;
        } else if (dead) {
            failed = true;  // publishes nothing, so successors must time out
        } else {
            if (lane == 0)
                st_relaxed_u64(ctx.desc + tile, pack_desc(epoch, kStateA, to_bits<T>(block_total)));
            excl = lookback<T>(ctx, tile, epoch, lane, &failed);
            if (lane == 0) {
                if (!failed) {
                    st_relaxed_u64(ctx.desc + tile,
                                   pack_desc(epoch, kStateP, to_bits<T>(excl + block_total)));
                } else {
                    st_relaxed_u64(ctx.desc + tile, pack_desc(epoch, kStatePoison, 0u));
                    record_error(ctx.status, kErrLookbackTimeout, tile);
                }
            }
        }
        if (lane == 0) {
            s_prefix = excl;
            s_fail = failed ? 1u : 0u;
        }
    }
    __syncthreads();
    if (s_fail) return;

    T y[VPT][4];
    rows_output<T, VPT, INCLUSIVE>(v, pre, s_prefix + warp_prefix, y);
    store_rows<T, VPT>(out, n, seg, lane, fast, y);

    if (carry_out != nullptr && tile == num_tiles - 1 && threadIdx.x == 0)
        *carry_out = s_prefix + block_total;
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

// Configurations: {threads, items per thread}.  Index 0 is the default.
static const ScanConfig kConfigs[] = {
    {256, 16},  // 4096-element tiles
    {256, 32},  // 8192
    {512, 16},  // 8192
    {128, 32},  // 4096
    {256, 24},  // 6144
};
constexpr int kNumConfigs = sizeof(kConfigs) / sizeof(kConfigs[0]);

int scan_config_count() { return kNumConfigs; }
ScanConfig scan_config(int idx) { return kConfigs[(idx >= 0 && idx < kNumConfigs) ? idx : 0]; }

static bool aligned16(const void* a, const void* b) {
    return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
}

template <typename T, bool INCL, int THREADS, int VPT>
static cudaError_t launch_one(const void* in, void* out, size_t n, const LookbackWs& ws,
                             const void* carry_in, void* carry_out, cudaStream_t s) {
    const size_t tile = (size_t)THREADS * VPT * 4;
    const uint32_t tiles = (uint32_t)((n + tile - 1) / tile);
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    k_scan_lookback<T, INCL, THREADS, VPT><<<tiles, THREADS, 0, s>>>(
        static_cast<const T*>(in), static_cast<T*>(out), n, tiles, ctx, aligned16(in, out),
        static_cast<const T*>(carry_in), static_cast<T*>(carry_out));
    return cudaGetLastError();
}

template <typename T, bool INCL>
static cudaError_t dispatch_config(int config, const void* in, void* out, size_t n,
                                   const LookbackWs& ws, const void* ci, void* co, cudaStream_t s) {
    switch (config) {
        case 1: return launch_one<T, INCL, 256, 8>(in, out, n, ws, ci, co, s);
        case 2: return launch_one<T, INCL, 512, 4>(in, out, n, ws, ci, co, s);
        case 3: return launch_one<T, INCL, 128, 8>(in, out, n, ws, ci, co, s);
        case 4: return launch_one<T, INCL, 256, 6>(in, out, n, ws, ci, co, s);
        default: return launch_one<T, INCL, 256, 4>(in, out, n, ws, ci, co, s);
    }
}

cudaError_t launch_scan_lookback(Dtype dt, bool inclusive, int config, const void* in, void* out,
                                 size_t n, const LookbackWs& ws, const void* carry_in,
                                 void* carry_out, cudaStream_t s) {
    if (dt == Dtype::F32)
        return inclusive ? dispatch_config<float, true>(config, in, out, n, ws, carry_in, carry_out, s)
                         : dispatch_config<float, false>(config, in, out, n, ws, carry_in, carry_out, s);
    return inclusive ? dispatch_config<uint32_t, true>(config, in, out, n, ws, carry_in, carry_out, s)
                     : dispatch_config<uint32_t, false>(config, in, out, n, ws, carry_in, carry_out, s);
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
    switch (config) {
        case 1: return launch_copy<256, 8>(in, out, n, s);
        case 2: return launch_copy<512, 4>(in, out, n, s);
        case 3: return launch_copy<128, 8>(in, out, n, s);
        case 4: return launch_copy<256, 6>(in, out, n, s);
        default: return launch_copy<256, 4>(in, out, n, s);
    }
}

}  // namespace ss
