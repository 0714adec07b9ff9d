// scan_rows.cu -- batched scans: a row-major rows x cols matrix, every row
// scanned on its own (the per-row cumulative sum over sorted probabilities
// in top-p sampling, "Prefix sum and other parallel patterns", In LLMs: MoE
// token dispatch, last paragraph).
//
// Two kernels, by row length:
//   - Rows longer than kRowsWarpMax elements are cut into 4096-element tiles
//     that never cross a row boundary.  Tiles are claimed in order from the
//     workspace counter, and each runs the single-pass look-back of the flat
//     scan ("A device-level scan: scan then propagate").  The row's first
//     tile publishes its inclusive prefix at once; the others look back no
//     further than it (the floor is the row's start, with prefix 0).  So the
//     rows' chains are independent, and one launch covers every row.
//   - Shorter rows take one warp each.  The warp walks its row in steps of
//     512 elements (four 128-element chunks, one 16-byte vector per lane
//     each).  Each chunk is a lane-local scan of 4 and a shuffle scan across
//     the warp; the running total carries from chunk to chunk.  No workspace
//     and no look-back.
// Rows whose start is not 16-byte aligned (cols not a multiple of 4, or an
// unaligned base) are read and written element by element with bounds checks.
#include "internal.h"
#include "scan_body.cuh"
#include "tile.cuh"

namespace ss {

namespace {

constexpr int kRThreads = 256;
constexpr int kRWarps = kRThreads / 32;
constexpr int kRVpt = 4;
constexpr size_t kRSeg = (size_t)32 * kRVpt * 4;   // 512 elements per warp
static_assert(kRSeg * kRWarps == kRowsTile, "tile geometry");
constexpr int kRSteps = 4;                          // chunks per warp step in the short-row kernel

}  // namespace

template <typename T, bool INCLUSIVE>
__global__ void __launch_bounds__(kRThreads)
k_scan_rows_tiles(const T* in, T* out, size_t cols, uint32_t tiles_per_row, uint32_t num_tiles, LookbackCtx ctx) {
    __shared__ ScanSmem<T, kRWarps> sm;
    __shared__ uint32_t s_tile, s_epoch;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        uint32_t tile, epoch;
        claim_tile(ctx.counter, num_tiles, &tile, &epoch);
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
    const size_t row = tile / tiles_per_row;
    const uint32_t j = tile % tiles_per_row;  // tile index inside the row
    const T* rin = in + row * cols;
    T* rout = out + row * cols;
    const size_t seg = (size_t)j * kRowsTile + (size_t)warp * kRSeg;
    const bool full = (size_t)j * kRowsTile + kRowsTile <= cols;

    T v[kRVpt][4];
    load_rows<T, kRVpt>(rin, cols, seg, lane, full && (reinterpret_cast<uintptr_t>(rin) & 15u) == 0, v);
    T t = T(0);
#pragma unroll
    for (int q = 0; q < kRVpt; ++q) t += ((v[q][0] + v[q][1]) + v[q][2]) + v[q][3];
    T warp_prefix, block_total;
    block_combine<T, kRWarps>(warp_sum(t), warp, lane, sm.warp, &warp_prefix, &block_total);

    if (warp == 0) {
        T excl = T(0);
        bool failed = false;
        const bool dead = (int64_t)tile == ctx.fault_tile;  // test hook only
        if (j == 0) {  // the row's first tile: its inclusive prefix is its own total
            if (tiles_per_row > 1 && lane == 0 && !dead)
                st_relaxed_u64(ctx.desc + tile, pack_desc(epoch, kStateP, to_bits<T>(block_total)));
            failed = dead;
        } else if (dead) {
            failed = true;  // publishes nothing, so its successors' waits run out
        } else {
            if (lane == 0) st_relaxed_u64(ctx.desc + tile, pack_desc(epoch, kStateA, to_bits<T>(block_total)));
            compiler_fence();  // publish before looking back
            const int64_t floor = (int64_t)(tile - j) - 1;  // just before the row's first tile, prefix 0
            excl = lookback<T, 1>(ctx, tile, epoch, lane, &failed, nullptr, floor, T(0));
            if (lane == 0) {
                if (!failed) {
                    st_relaxed_u64(ctx.desc + tile, pack_desc(epoch, kStateP, to_bits<T>(excl + block_total)));
                } else {
                    st_relaxed_u64(ctx.desc + tile, pack_desc(epoch, kStatePoison, 0u));
                    record_error(ctx.status, kErrLookbackTimeout, tile);
                }
            }
        }
        if (lane == 0) {
            sm.prefix[0] = excl;
            sm.fail[0] = failed ? 1u : 0u;
        }
    }
    T pre[kRVpt];
    warp_rows_scan<T, kRVpt>(v, lane, pre);
    __syncthreads();
    if (sm.fail[0]) return;
    T y[kRVpt][4];
    rows_output<T, kRVpt, INCLUSIVE>(v, pre, sm.prefix[0] + warp_prefix, y);
    store_rows<T, kRVpt>(rout, cols, seg, lane, full && (reinterpret_cast<uintptr_t>(rout) & 15u) == 0, y);
}

template <typename T, bool INCLUSIVE>
__global__ void __launch_bounds__(kRThreads)
k_scan_rows_warp(const T* in, T* out, size_t rows, size_t cols, bool vec) {
    const int lane = threadIdx.x & 31;
    const size_t gw = ((size_t)blockIdx.x * kRThreads + threadIdx.x) >> 5;
    const size_t nw = ((size_t)gridDim.x * kRThreads) >> 5;
    for (size_t r = gw; r < rows; r += nw) {  // warp-uniform
        const T* rin = in + r * cols;
        T* rout = out + r * cols;
        T carry = T(0);
        for (size_t c0 = 0; c0 < cols; c0 += (size_t)128 * kRSteps) {  // warp-uniform
            T v[kRSteps][4];
#pragma unroll
            for (int u = 0; u < kRSteps; ++u) {
                const size_t b = c0 + (size_t)u * 128 + (size_t)lane * 4;
                if (vec && b + 4 <= cols) {
                    const uint4 q = ld_vec(reinterpret_cast<const uint4*>(rin + b));
                    v[u][0] = from_bits<T>(q.x);
                    v[u][1] = from_bits<T>(q.y);
                    v[u][2] = from_bits<T>(q.z);
                    v[u][3] = from_bits<T>(q.w);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[u][e] = b + e < cols ? rin[b + e] : T(0);
                }
            }
#pragma unroll
            for (int u = 0; u < kRSteps; ++u) {
                const T s = ((v[u][0] + v[u][1]) + v[u][2]) + v[u][3];
                const T inc = warp_inclusive_scan<T>(s, lane);
                T run = carry + (inc - s);
                carry += __shfl_sync(kFullMask, inc, 31);
                T y[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (INCLUSIVE) {
                        run += v[u][e];
                        y[e] = run;
                    } else {
                        y[e] = run;
                        run += v[u][e];
                    }
                }
                const size_t b = c0 + (size_t)u * 128 + (size_t)lane * 4;
                if (vec && b + 4 <= cols) {
                    st_vec(reinterpret_cast<uint4*>(rout + b),
                           make_uint4(to_bits<T>(y[0]), to_bits<T>(y[1]), to_bits<T>(y[2]), to_bits<T>(y[3])));
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (b + e < cols) rout[b + e] = y[e];
                }
            }
        }
    }
}

template <typename T, bool INCL>
static cudaError_t launch_rows(const void* in, void* out, size_t rows, size_t cols, const LookbackWs& ws,
                               cudaStream_t s) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0, v = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        sms = v > 0 ? v : 1;
    }
    const T* pin = static_cast<const T*>(in);
    T* pout = static_cast<T*>(out);
    if (cols <= kRowsWarpMax) {
        const bool vec = cols % 4 == 0 && ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 15u) == 0;
        const size_t want = (rows + kRWarps - 1) / kRWarps;
        const size_t cap = (size_t)sms * (2048 / kRThreads);
        const unsigned grid = (unsigned)(want < cap ? want : cap);
        k_scan_rows_warp<T, INCL><<<grid, kRThreads, 0, s>>>(pin, pout, rows, cols, vec);
        return cudaGetLastError();
    }
    const uint32_t tpr = (uint32_t)((cols + kRowsTile - 1) / kRowsTile);
    const uint32_t tiles = (uint32_t)(rows * tpr);
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    k_scan_rows_tiles<T, INCL><<<tiles, kRThreads, 0, s>>>(pin, pout, cols, tpr, tiles, ctx);
    return cudaGetLastError();
}

cudaError_t launch_scan_rows(Dtype dt, bool inclusive, const void* in, void* out, size_t rows, size_t cols,
                             const LookbackWs& ws, cudaStream_t s) {
    if (dt == Dtype::F32)
        return inclusive ? launch_rows<float, true>(in, out, rows, cols, ws, s)
                         : launch_rows<float, false>(in, out, rows, cols, ws, s);
    return inclusive ? launch_rows<uint32_t, true>(in, out, rows, cols, ws, s)
                     : launch_rows<uint32_t, false>(in, out, rows, cols, ws, s);
}

}  // namespace ss
