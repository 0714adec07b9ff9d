// scan_body.cuh -- what one CTA does with one loaded tile of a single-pass
// scan: reduce, publish, look back, scan, store.  Shared by the one-CTA-per-
// tile kernel (scan.cu) and the persistent kernel (scan_pipe.cu), which only
// differ in how the tile reaches the registers.
//
// Order of work, chosen to shorten the chain of tiles waiting on each other:
//   1. the tile aggregate from a plain reduction (warp sums, then the block
//      combine of warp totals) -- all the look-back needs;
//   2. warp 0 publishes the aggregate and looks back while the other warps
//      run their detailed row scans, so the look-back's L2 round trips
//      overlap the scan arithmetic;
//   3. one barrier, then every thread adds the tile's prefix and stores.
#pragma once

#include "tile.cuh"

namespace ss {

// The prefix and the failure flag of a tile are handed from warp 0 to the
// other warps through shared memory.  A persistent kernel alternates two
// slots by tile parity: warp 0 may publish tile k+1's prefix (its last tile
// has no barrier before that) while a slower warp still reads tile k's.
template <typename T, int WARPS>
struct ScanSmem {
    T warp[WARPS];
    T prefix[2];
    uint32_t fail[2];
};

// Per-tile trace record (8 x uint64), written when a trace is taken:
//   [0] globaltimer when the CTA began this tile   [1] aggregate known
//   [2] aggregate published                        [3] look-back resolved
//   [4] outputs issued   [5] windows read   [6] polls that waited
//   [7] SM id (low 32 bits) and CTA index (high 32 bits)
constexpr int kTraceWords = 8;

__device__ __forceinline__ uint32_t sm_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

// Called by every thread of the CTA with its rows `v`.  Returns false
// (CTA-uniform) if the look-back failed; the tile's outputs are then not
// written and an error has been recorded.  With TRACE, thread 0 fills
// rec[1..7] (rec[0] is the caller's).
template <typename T, bool INCLUSIVE, int THREADS, int VPT, int K, bool TRACE = false, bool GROUPED = false>
__device__ __forceinline__ bool scan_tile_body(const T (&v)[VPT][4], T* out, size_t n, size_t seg,
                                               bool full, uint32_t tile, uint32_t num_tiles,
                                               uint32_t epoch, const LookbackCtx& ctx,
                                               const T* carry_in, T* carry_out,
                                               ScanSmem<T, THREADS / 32>& sm,
                                               unsigned long long* rec = nullptr) {
    constexpr int WARPS = THREADS / 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    T t = T(0);
#pragma unroll
    for (int j = 0; j < VPT; ++j) t += ((v[j][0] + v[j][1]) + v[j][2]) + v[j][3];
    T warp_prefix, block_total;
    block_combine<T, WARPS>(warp_sum(t), warp, lane, sm.warp, &warp_prefix, &block_total);
    if (TRACE && threadIdx.x == 0) rec[1] = globaltimer_ns();

    if (warp == 0) {
        LookbackStats stats{0u, 0u};
        T excl = T(0);
        bool failed = false;
        const bool dead = (int64_t)tile == ctx.fault_tile;  // test hook only
        if (tile == 0) {
            excl = carry_in ? *carry_in : T(0);
            if (num_tiles > 1 && lane == 0 && !dead)
                st_relaxed_u64(ctx.desc, pack_desc(epoch, kStateP, to_bits<T>(excl + block_total)));
            failed = dead;
        } else if (dead) {
            failed = true;  // publishes nothing, so its successors' waits run out
        } else {
            if (lane == 0)
                st_relaxed_u64(ctx.desc + tile, pack_desc(epoch, kStateA, to_bits<T>(block_total)));
            compiler_fence();  // publish before looking back
            if (TRACE && lane == 0) rec[2] = globaltimer_ns();
            if constexpr (GROUPED) {
                // group descriptors follow the launch's tile descriptors
                excl = lookback_two_level<T>(ctx, ctx.desc + num_tiles, tile, num_tiles, epoch, lane, block_total,
                                             &failed);
                if (TRACE) stats.windows = 1;
            } else {
                excl = lookback<T, K, TRACE>(ctx, tile, epoch, lane, &failed, &stats);
            }
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
            sm.prefix[0] = excl;
            sm.fail[0] = failed ? 1u : 0u;
            if (TRACE) {
                const unsigned long long now = globaltimer_ns();
                if (tile == 0) rec[2] = now;
                rec[3] = now;
                rec[5] = stats.windows;
                rec[6] = stats.waits;
                rec[7] = (unsigned long long)sm_id() | ((unsigned long long)blockIdx.x << 32);
            }
        }
    }

    T pre[VPT];
    warp_rows_scan<T, VPT>(v, lane, pre);
    __syncthreads();
    if (sm.fail[0]) return false;

    T y[VPT][4];
    rows_output<T, VPT, INCLUSIVE>(v, pre, sm.prefix[0] + warp_prefix, y);
    store_rows<T, VPT>(out, n, seg, lane, full, y);
    if (carry_out != nullptr && tile == num_tiles - 1 && threadIdx.x == 0)
        *carry_out = sm.prefix[0] + block_total;
    if (TRACE && threadIdx.x == 0) rec[4] = globaltimer_ns();
    return true;
}

}  // namespace ss
