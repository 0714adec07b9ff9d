// scan_rows.cu -- batched scans: a row-major rows x cols matrix, every row
// scanned on its own (the per-row cumulative sum over sorted probabilities
// in top-p sampling, "Prefix sum and other parallel patterns", In LLMs: MoE
// token dispatch, last paragraph).
//
// Three kernels, by row length:
//   - Rows of at least kRowsPipeMin elements (row starts 16-byte aligned)
//     run on a persistent grid with a bulk-copy ring, as the flat scan does
//     (k_scan_rows_pipe below).
//   - Other rows longer than kRowsWarpMax elements are cut into 4096-element tiles
//     that never cross a row boundary.  Tiles are claimed in order from the
//     workspace counter, and each runs the single-pass look-back of the flat
//     scan ("A device-level scan: scan then propagate").  The row's first
//     tile publishes its inclusive prefix at once; the others look back no
//     further than it (the floor is the row's start, with prefix 0).  So the
//     rows' chains are independent, and one launch covers every row.
//   - Rows of up to kRowsWarpMax elements take one warp each.  The warp
//     walks its row in steps of 512 elements (four 128-element chunks, one
//     16-byte vector per lane each).  Each chunk is a lane-local scan of 4
//     and a shuffle scan across the warp; the running total carries from
//     chunk to chunk.  Rows of at most 224 elements take one step instead,
//     several rows to a warp up to 128 elements (k_scan_rows_packed).  No
//     workspace and no look-back.
// Rows whose start is not 16-byte aligned (cols not a multiple of 4, or an
// unaligned base) are read and written element by element with bounds checks.
#include "bulk.cuh"
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
constexpr int kRPThreads = 512;                     // persistent long-row kernel

// store_rows for a segment that may run past n, when out + seg is 16-byte
// aligned: whole vectors inside n are stored as 16-byte vectors, only the
// one vector that straddles n element by element.  (Element-wise stores
// from a whole warp leave every 32-byte sector partly written per
// instruction, which measured several times slower than vector stores.)
template <typename T, int VPT>
__device__ __forceinline__ void store_rows_aligned_tail(T* out, size_t n, size_t seg, int lane,
                                                        const T (&y)[VPT][4]) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const size_t i0 = seg + (size_t)(32 * j + lane) * 4;
        if (i0 + 4 <= n) {
            st_vec(reinterpret_cast<uint4*>(out + i0), make_uint4(to_bits<T>(y[j][0]), to_bits<T>(y[j][1]),
                                                                  to_bits<T>(y[j][2]), to_bits<T>(y[j][3])));
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (i0 + k < n) out[i0 + k] = y[j][k];
        }
    }
}

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
    if ((reinterpret_cast<uintptr_t>(rout) & 15u) == 0)
        store_rows_aligned_tail<T, kRVpt>(rout, cols, seg, lane, y);
    else
        store_rows<T, kRVpt>(rout, cols, seg, lane, false, y);
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
                if (c0 + (size_t)u * 128 >= cols) break;  // past the row's end: a short row's last steps
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
                if (c0 + (size_t)u * 128 >= cols) break;
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

// Rows of at most 224 elements, packed: a row gets L lanes, each holding
// EPL / 4 16-byte vectors, with L * EPL the smallest power of two that
// covers the row; a warp takes 32 / L consecutive rows per step (they are
// contiguous in memory, so its loads stay coalesced).  Vector h of lane i in
// a group holds elements h * 4L + 4i .. h * 4L + 4i + 3, so that each load
// and store instruction covers whole 4L-element runs of a row.  The lane
// scan and a shuffle scan of width L per vector give every output, the
// first vector's group total carried into the second; no carry between
// steps, since a row fits in one step.
template <typename T, bool INCLUSIVE, int L, int EPL>
__global__ void __launch_bounds__(kRThreads)
k_scan_rows_packed(const T* in, T* out, size_t rows, size_t cols, bool vec) {
    static_assert(EPL == 4 || EPL == 8, "one or two 16-byte vectors per lane");
    constexpr int R = 32 / L;   // rows per warp step
    constexpr int H = EPL / 4;  // vectors per lane
    const int lane = threadIdx.x & 31;
    const int li = lane % L;    // lane inside its row's group
    const size_t gw = ((size_t)blockIdx.x * kRThreads + threadIdx.x) >> 5;
    const size_t nw = ((size_t)gridDim.x * kRThreads) >> 5;
    for (size_t rg = gw; rg * R < rows; rg += nw) {  // warp-uniform
        const size_t r = rg * R + (size_t)(lane / L);
        const bool live = r < rows;
        T v[H][4];
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const size_t bh = (size_t)h * 4 * L + (size_t)li * 4;  // first element of vector h in its row
            if (live && vec && bh + 4 <= cols) {
                const uint4 q = ld_vec(reinterpret_cast<const uint4*>(in + r * cols + bh));
                v[h][0] = from_bits<T>(q.x);
                v[h][1] = from_bits<T>(q.y);
                v[h][2] = from_bits<T>(q.z);
                v[h][3] = from_bits<T>(q.w);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[h][e] = live && bh + e < cols ? in[r * cols + bh + e] : T(0);
            }
        }
        T sum[H], inc[H];
#pragma unroll
        for (int h = 0; h < H; ++h) {
            sum[h] = ((v[h][0] + v[h][1]) + v[h][2]) + v[h][3];
            inc[h] = sum[h];
        }
#pragma unroll
        for (int d = 1; d < L; d <<= 1) {
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const T t = __shfl_up_sync(kFullMask, inc[h], d, L);
                if (li >= d) inc[h] += t;
            }
        }
        T carry = T(0);
#pragma unroll
        for (int h = 0; h < H; ++h) {
            T run = carry + (inc[h] - sum[h]);
            T y[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (INCLUSIVE) {
                    run += v[h][e];
                    y[e] = run;
                } else {
                    y[e] = run;
                    run += v[h][e];
                }
            }
            const size_t bh = (size_t)h * 4 * L + (size_t)li * 4;
            if (live && vec && bh + 4 <= cols) {
                st_vec(reinterpret_cast<uint4*>(out + r * cols + bh),
                       make_uint4(to_bits<T>(y[0]), to_bits<T>(y[1]), to_bits<T>(y[2]), to_bits<T>(y[3])));
            } else if (live) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (bh + e < cols) out[r * cols + bh + e] = y[e];
            }
            if (h + 1 < H) carry += __shfl_sync(kFullMask, inc[h], L - 1, L);  // the group's total of vector h
        }
    }
}

// Persistent form for long rows (at least 16384 elements, row starts
// 16-byte aligned).  It uses the single-register-buffer schedule of the flat
// scan (scan_pipe.cu): a rank per CTA, tiles rank + k*G, a three-stage
// bulk-copy ring, and the aggregate one iteration early.  A tile is VPT
// 16-byte vectors per lane (10240 to 18432 elements); the launcher picks VPT
// per call from the row length.
// Tiles are numbered row by row, and none crosses a row boundary:
//  - a row's last tile is shorter, and is fetched by a shorter bulk copy
//    (its byte count is a multiple of 16 because the row length is a
//    multiple of 4);
//  - lanes past the row's end read zeros and store nothing;
//  - a row's first tile publishes its inclusive prefix at once;
//  - every other tile looks back no further than the row's first tile, or
//    than this CTA's previous tile when that lies in the same row (its
//    inclusive prefix is then in hand).
template <typename T, bool INCLUSIVE, int VPT>
__global__ void __launch_bounds__(kRPThreads, 1)
k_scan_rows_pipe(const T* in, T* out, size_t cols, uint32_t tiles_per_row, uint32_t num_tiles, LookbackCtx ctx) {
    constexpr int STAGES = 3;
    constexpr int WARPS = kRPThreads / 32;
    constexpr uint32_t TILE = (uint32_t)kRPThreads * VPT * 4;
    static_assert(TILE >= kRowsTile, "descriptors are sized for kRowsTile-element tiles");
    constexpr uint32_t SEG = 32u * VPT * 4;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    T* ring = reinterpret_cast<T*>(smem_raw);
    __shared__ __align__(8) uint64_t bars[STAGES];
    __shared__ ScanSmem<T, WARPS> sm;
    __shared__ uint32_t s_rank, s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t G = gridDim.x;
    const uint64_t policy = policy_evict_first();

    if (threadIdx.x == 0) {
        uint32_t rank, epoch;
        claim_tile(ctx.counter, G, &rank, &epoch);
        s_rank = rank;
        s_epoch = epoch;
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_async_shared();
    }
    __syncthreads();
    const uint32_t rank = s_rank;
    const uint32_t epoch = s_epoch;
    if (rank >= G) {
        if (threadIdx.x == 0) record_error(ctx.status, kErrCounter, rank);
        return;
    }
    const uint32_t count = rank < num_tiles ? (num_tiles - rank + G - 1) / G : 0;
    uint32_t issued = 0, consumed = 0;  // thread 0

    // Tile geometry: element offset of tile t in the matrix, and its length.
    auto tile_base = [&](uint32_t t) {
        return (size_t)(t / tiles_per_row) * cols + (size_t)(t % tiles_per_row) * TILE;
    };
    auto tile_len = [&](uint32_t t) {
        const size_t start = (size_t)(t % tiles_per_row) * TILE;
        return (uint32_t)(cols - start < TILE ? cols - start : TILE);
    };
    auto issue = [&](uint32_t k) {
        const int s = (int)(k % STAGES);
        const uint32_t t = rank + k * G;
        const uint32_t bytes = tile_len(t) * (uint32_t)sizeof(T);  // a multiple of 16
        fence_async_shared();
        mbar_arrive_expect_tx(&bars[s], bytes);
        bulk_load(ring + (size_t)s * TILE, in + tile_base(t), bytes, &bars[s], policy);
        issued = k + 1;
    };
    auto read_rows = [&](uint32_t k, T (&v)[VPT][4]) {
        const uint32_t len = tile_len(rank + k * G);
        const T* src = ring + (size_t)(k % STAGES) * TILE + (size_t)warp * SEG + (size_t)lane * 4;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const uint32_t e0 = warp * SEG + (32u * j + lane) * 4;  // element index in the tile
            if (e0 < len) {  // len is a multiple of 4: a vector is all in or all out
                const uint4 r = lds_vec(src + 128 * j);
                v[j][0] = from_bits<T>(r.x);
                v[j][1] = from_bits<T>(r.y);
                v[j][2] = from_bits<T>(r.z);
                v[j][3] = from_bits<T>(r.w);
            } else {
                v[j][0] = v[j][1] = v[j][2] = v[j][3] = T(0);
            }
        }
    };
    auto reduce_publish = [&](uint32_t k, T* wp, T* agg) -> bool {
        const uint32_t t = rank + k * G;
        const bool ok = mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) record_error(ctx.status, kErrBulkTimeout, t);
            return false;
        }
        T v[VPT][4];
        read_rows(k, v);
        T x = T(0);
#pragma unroll
        for (int j = 0; j < VPT; ++j) x += ((v[j][0] + v[j][1]) + v[j][2]) + v[j][3];
        block_combine<T, WARPS>(warp_sum(x), warp, lane, sm.warp, wp, agg);
        if (threadIdx.x == 0 && (int64_t)t != ctx.fault_tile) {
            const bool first = t % tiles_per_row == 0;
            if (first) {
                if (tiles_per_row > 1) st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, to_bits<T>(*agg)));
            } else {
                st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateA, to_bits<T>(*agg)));
            }
        }
        compiler_fence();  // the aggregate just published stays ahead of the look-back
        return true;
    };

    T wp_cur = T(0), agg_cur = T(0), prev_incl = T(0);
    bool failed = false;
    uint32_t fail_at = 0;
    if (threadIdx.x == 0)
        for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);
    if (count > 0 && !reduce_publish(0, &wp_cur, &agg_cur)) failed = true;

    for (uint32_t k = 0; !failed && k < count; ++k) {
        const uint32_t t = rank + k * G;
        T wp_next = T(0), agg_next = T(0);
        if (k + 1 < count && !reduce_publish(k + 1, &wp_next, &agg_next)) {
            failed = true;
            fail_at = k;
            break;
        }
        if (warp == 0) {
            T excl = T(0);
            bool lb_failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            const uint32_t j = t % tiles_per_row;
            if (j == 0) {
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;
            } else {
                // The row's first tile, or this CTA's previous tile if it is in the same row.
                const uint32_t row_first = t - j;
                const bool prev_same_row = k > 0 && t - G >= row_first;
                const int64_t floor = prev_same_row ? (int64_t)t - (int64_t)G : (int64_t)row_first - 1;
                excl = lookback<T, 1>(ctx, t, epoch, lane, &lb_failed, nullptr, floor,
                                      prev_same_row ? prev_incl : T(0));
                if (lane == 0) {
                    if (!lb_failed) {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, to_bits<T>(excl + agg_cur)));
                    } else {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
                        record_error(ctx.status, kErrLookbackTimeout, t);
                    }
                }
            }
            prev_incl = excl + agg_cur;
            if (lane == 0) {
                sm.prefix[k & 1] = excl;
                sm.fail[k & 1] = lb_failed ? 1u : 0u;
            }
        }
        T v[VPT][4];
        read_rows(k, v);
        T pre[VPT];
        warp_rows_scan<T, VPT>(v, lane, pre);
        __syncthreads();  // tile k read by everyone; the prefix is in shared memory
        if (threadIdx.x == 0) {
            consumed = k + 1;
            if (k + STAGES < count) issue(k + STAGES);
        }
        if (sm.fail[k & 1]) {
            failed = true;
            fail_at = k;
            break;
        }
        rows_output_inplace<T, VPT, INCLUSIVE>(v, pre, sm.prefix[k & 1] + wp_cur);
        const uint32_t len = tile_len(t);
        uint4* dst = reinterpret_cast<uint4*>(out + tile_base(t) + (size_t)warp * SEG) + lane;
#pragma unroll
        for (int j = 0; j < VPT; ++j)  // 16-byte stores; a short tile's vectors are all in or all out
            if (warp * SEG + (32u * j + lane) * 4 < len)
                st_vec(dst + 32 * j, make_uint4(to_bits<T>(v[j][0]), to_bits<T>(v[j][1]), to_bits<T>(v[j][2]),
                                                to_bits<T>(v[j][3])));
        wp_cur = wp_next;
        agg_cur = agg_next;
    }

    if (failed && threadIdx.x == 0) {
        for (uint32_t j = fail_at + 1; j < count; ++j) {
            const uint32_t tt = rank + j * G;
            if ((int64_t)tt != ctx.fault_tile) st_relaxed_u64(ctx.desc + tt, pack_desc(epoch, kStatePoison, 0u));
        }
        for (uint32_t j = consumed; j < issued; ++j)
            mbar_wait_bounded(&bars[j % STAGES], (j / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
}

template <typename T, bool INCL, int VPT>
static cudaError_t launch_rows_pipe(const T* in, T* out, size_t rows, size_t cols, const LookbackWs& ws,
                                   cudaStream_t s) {
    constexpr size_t TILE = (size_t)kRPThreads * VPT * 4;
    constexpr size_t SMEM = 3 * TILE * sizeof(T);
    auto kern = k_scan_rows_pipe<T, INCL, VPT>;
    KernelSetup su;
    cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), kRPThreads, SMEM, &su);
    if (e != cudaSuccess) return e;
    const uint32_t tpr = (uint32_t)((cols + TILE - 1) / TILE);
    const uint32_t tiles = (uint32_t)(rows * tpr);
    const uint32_t grid = tiles < (uint32_t)su.sms ? tiles : (uint32_t)su.sms;
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    kern<<<grid, kRPThreads, SMEM, s>>>(in, out, cols, tpr, tiles, ctx);
    return cudaGetLastError();
}

template <typename T, bool INCL>
static cudaError_t launch_rows(const void* in, void* out, size_t rows, size_t cols, const LookbackWs& ws,
                               cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (sms <= 0) sms = 1;
    const T* pin = static_cast<const T*>(in);
    T* pout = static_cast<T*>(out);
    if (cols <= kRowsWarpMax) {
        const bool vec = cols % 4 == 0 && ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 15u) == 0;
        const size_t cap = (size_t)sms * (2048 / kRThreads);
        if (cols <= 224) {  // one step per row: several rows per warp up to 128 elements
            // lanes per row and elements per lane: 4 per lane up to 64 elements, then 8.
            // From about 224 elements on, the warp kernel is as fast.
            const int L = cols <= 4 ? 1 : cols <= 8 ? 2 : cols <= 16 ? 4 : cols <= 32 ? 8 : cols <= 64 ? 16
                        : cols <= 128 ? 16 : 32;
            const size_t per_cta = (size_t)kRWarps * (32 / L);
            const size_t want = (rows + per_cta - 1) / per_cta;
            const unsigned grid = (unsigned)(want < cap ? want : cap);
            if (cols <= 64) {
                switch (L) {
                    case 1: k_scan_rows_packed<T, INCL, 1, 4><<<grid, kRThreads, 0, s>>>(pin, pout, rows, cols, vec); break;
                    case 2: k_scan_rows_packed<T, INCL, 2, 4><<<grid, kRThreads, 0, s>>>(pin, pout, rows, cols, vec); break;
                    case 4: k_scan_rows_packed<T, INCL, 4, 4><<<grid, kRThreads, 0, s>>>(pin, pout, rows, cols, vec); break;
                    case 8: k_scan_rows_packed<T, INCL, 8, 4><<<grid, kRThreads, 0, s>>>(pin, pout, rows, cols, vec); break;
                    default: k_scan_rows_packed<T, INCL, 16, 4><<<grid, kRThreads, 0, s>>>(pin, pout, rows, cols, vec); break;
                }
            } else if (L == 16) {
                k_scan_rows_packed<T, INCL, 16, 8><<<grid, kRThreads, 0, s>>>(pin, pout, rows, cols, vec);
            } else {
                k_scan_rows_packed<T, INCL, 32, 8><<<grid, kRThreads, 0, s>>>(pin, pout, rows, cols, vec);
            }
            return cudaGetLastError();
        }
        const size_t want = (rows + kRWarps - 1) / kRWarps;
        const unsigned grid = (unsigned)(want < cap ? want : cap);
        k_scan_rows_warp<T, INCL><<<grid, kRThreads, 0, s>>>(pin, pout, rows, cols, vec);
        return cudaGetLastError();
    }
    if (cols >= kRowsPipeMin && cols % 4 == 0 &&
        ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 15u) == 0)
    {
        // Tiles of 10240, 14336, 16384 or 18432 elements (5, 7, 8 or 9 key
        // vectors per lane): the fewest tiles per row (fewer look-backs),
        // and among those the smallest tile (the least padding in a row's
        // short last tile, so less time per tile).
        auto tiles_of = [&](size_t vpt) { const size_t tile = (size_t)kRPThreads * vpt * 4; return (cols + tile - 1) / tile; };
        const size_t fewest = tiles_of(9);
        if (tiles_of(5) == fewest) return launch_rows_pipe<T, INCL, 5>(pin, pout, rows, cols, ws, s);
        if (tiles_of(7) == fewest) return launch_rows_pipe<T, INCL, 7>(pin, pout, rows, cols, ws, s);
        if (tiles_of(8) == fewest) return launch_rows_pipe<T, INCL, 8>(pin, pout, rows, cols, ws, s);
        return launch_rows_pipe<T, INCL, 9>(pin, pout, rows, cols, ws, s);
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
