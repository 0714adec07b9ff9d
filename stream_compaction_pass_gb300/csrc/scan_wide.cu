// scan_wide.cu -- single-pass scans with 64-bit sums: uint32 -> uint64 and
// int32 -> int64 (widened accumulation), int64 (wrapping modulo 2^64) and
// fp64.
//
// "Parallel Prefix Sum (Scan) for NVIDIA T4 (sm_75)", Key Features (64-bit
// indexing for large arrays): the sum of many 32-bit counts overflows 32
// bits, so it is carried and stored in 64 bits.  The method is the one of
// the 32-bit kernels ("Prefix sum and other parallel patterns", A
// device-level scan: scan then propagate, with decoupled look-back), on the
// schedule of the single-register-buffer persistent kernel (scan_pipe.cu):
//   - each CTA takes a rank and owns tiles rank, rank + G, ...;
//   - a three-stage ring receives each tile's input with one bulk copy;
//   - tile k+1 is summed and its aggregate published while tile k waits for
//     its look-back, which stops at this CTA's own previous tile;
//   - tile k is read again from the ring, scanned in registers and stored.
// The descriptors are 16 bytes (lookback_wide.cuh).
//
// A tile is 128 bytes of input per thread: 4096 elements of a 32-bit input
// in a 128-thread CTA (four per SM), 8192 of a 64-bit one in a 512-thread
// CTA (one per SM).  Each thread takes rows of 2 elements (16 rows or
// 8).  Warp w owns a contiguous segment; row j of it is 64 consecutive
// elements and lane l holds elements 2l and 2l+1.  So the scan order inside a
// warp is (row, lane, element), every output store of a warp is 512
// contiguous bytes (one 16-byte pair per lane), and every shared-memory read
// of a row is conflict-free (8 or 16 bytes per lane, consecutive).  The scan
// pass streams a 32-bit input's rows out of the ring four at a time, so its
// tile is never held whole in registers (a 64-bit input's eight rows are);
// the first group is scanned while warp 0 looks back.
//
// Inputs that are not 16-byte aligned, and the ragged last tile, are read
// and written element by element with bounds checks.
#include <type_traits>

#include "bulk.cuh"
#include "internal.h"
#include "lookback_wide.cuh"
#include "tensor_copy.cuh"

namespace ss {

namespace {

// Threads per CTA by input width, and 512 / threads CTAs per SM.  A tile is
// 128 bytes of input per thread: 4096 elements of a 32-bit input in 128
// threads, 8192 of a 64-bit one in 512.  Measured at n = 1e8 (fraction of
// the measured copy bandwidth; 512 / 256 / 128 threads): uint32 -> uint64
// inclusive 0.78 / 0.86 / 0.87, int64 exclusive 0.81 / 0.79 / 0.78.  The
// narrow CTAs hide each other's look-back when the input tile is small next
// to its output; a 64-bit input's tile, read whole into registers, gains
// nothing from them.
template <typename TI>
__host__ __device__ constexpr int wide_threads() {
    return sizeof(TI) == 4 ? 128 : 512;
}
template <typename TI>
__host__ __device__ constexpr uint32_t wide_tile() {
    return (uint32_t)wide_threads<TI>() * 128u / (uint32_t)sizeof(TI);
}
static_assert(wide_tile<uint32_t>() == kWideTile && wide_tile<double>() >= kWideTile,
              "the host sizes the descriptors for the smallest tile");

template <typename TI, typename TA> __device__ __forceinline__ TA widen(TI x);
template <> __device__ __forceinline__ unsigned long long widen<uint32_t, unsigned long long>(uint32_t x) {
    return (unsigned long long)x;
}
template <> __device__ __forceinline__ unsigned long long widen<int32_t, unsigned long long>(int32_t x) {
    return (unsigned long long)(long long)x;  // sign-extended; the adds are the same bits as int64's
}
template <> __device__ __forceinline__ unsigned long long widen<unsigned long long, unsigned long long>(
    unsigned long long x) {
    return x;
}

// A lane's two consecutive input elements from shared memory.
template <typename TI>
__device__ __forceinline__ void lds_pair(const void* p, TI (&x)[2]) {
    if constexpr (sizeof(TI) == 4) {
        uint32_t a, b;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(smem_u32(p)));
        x[0] = (TI)a;
        x[1] = (TI)b;
    } else {
        unsigned long long a, b;
        asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(smem_u32(p)));
        if constexpr (std::is_same<TI, double>::value) {
            x[0] = __longlong_as_double((long long)a);
            x[1] = __longlong_as_double((long long)b);
        } else {
            x[0] = a;
            x[1] = b;
        }
    }
}

__device__ __forceinline__ void st_v2_u64(void* p, unsigned long long a, unsigned long long b) {
    asm volatile("st.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

}  // namespace

template <typename TI, typename TA, bool INCLUSIVE>
__global__ void __launch_bounds__(wide_threads<TI>(), 512 / wide_threads<TI>())
k_scan_wide(const TI* in, TA* out, size_t n, uint32_t num_tiles, bool fast, LookbackCtx ctx) {
    constexpr int STAGES = 3;
    constexpr int THREADS = wide_threads<TI>();
    constexpr int WARPS = THREADS / 32;
    constexpr uint32_t TILE = (uint32_t)THREADS * 128u / (uint32_t)sizeof(TI);
    constexpr int EPV = 2;                                 // elements per lane per row
    constexpr int VPT = (int)TILE / (THREADS * EPV);     // rows per lane
    constexpr int GRP = sizeof(TI) == 8 ? VPT : 4;         // rows handled together
    static_assert(VPT % GRP == 0, "rows come in groups");
    constexpr uint32_t SEG = 32u * VPT * EPV;              // elements per warp segment
    constexpr uint32_t IN_BYTES = TILE * (uint32_t)sizeof(TI);
    static_assert(SEG * WARPS == TILE, "tile geometry");

    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[STAGES];
    // Warp totals, prefix and failure flag alternate between two slots by
    // tile parity, so a slot is never rewritten while a slower warp may still
    // read it.
    __shared__ TA s_warp[2][WARPS];
    __shared__ TA s_prefix[2];
    __shared__ uint32_t s_fail[2], s_rank, s_epoch;

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

    auto full_tile = [&](uint32_t k) { return fast && (size_t)(rank + k * G) * TILE + TILE <= n; };
    auto issue = [&](uint32_t k) {
        const int s = (int)(k % STAGES);
        if (full_tile(k)) {
            fence_async_shared();
            mbar_arrive_expect_tx(&bars[s], IN_BYTES);
            bulk_load(smem_raw + (size_t)s * IN_BYTES, in + (size_t)(rank + k * G) * TILE, IN_BYTES, &bars[s],
                      policy);
        } else {
            mbar_arrive(&bars[s]);  // read from global with bounds checks instead
        }
        issued = k + 1;
    };
    // This lane's rows g*GRP .. g*GRP+GRP-1 of tile k, widened.
    auto read_group = [&](uint32_t k, int g, TA (&v)[GRP][EPV]) {
        const size_t seg = (size_t)(rank + k * G) * TILE + (size_t)warp * SEG;
        if (full_tile(k)) {
            const unsigned char* src =
                smem_raw + (size_t)(k % STAGES) * IN_BYTES + ((size_t)warp * SEG + (size_t)lane * EPV) * sizeof(TI);
#pragma unroll
            for (int q = 0; q < GRP; ++q) {
                TI x[EPV];
                lds_pair<TI>(src + (size_t)(g * GRP + q) * 32 * EPV * sizeof(TI), x);
#pragma unroll
                for (int e = 0; e < EPV; ++e) v[q][e] = widen<TI, TA>(x[e]);
            }
        } else {
#pragma unroll
            for (int q = 0; q < GRP; ++q)
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    const size_t i = seg + (size_t)(32 * (g * GRP + q) + lane) * EPV + e;
                    v[q][e] = i < n ? widen<TI, TA>(in[i]) : TA(0);
                }
        }
    };
    // Waits for tile k, sums it, publishes its aggregate; false if the copy did not arrive.
    auto reduce_publish = [&](uint32_t k, TA* wp, TA* agg) -> bool {
        const uint32_t t = rank + k * G;
        const bool ok = mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) record_error(ctx.status, kErrBulkTimeout, t);
            return false;
        }
        TA x = TA(0);
#pragma unroll
        for (int g = 0; g < VPT / GRP; ++g) {
            TA v[GRP][EPV];
            read_group(k, g, v);
#pragma unroll
            for (int q = 0; q < GRP; ++q)
#pragma unroll
                for (int e = 0; e < EPV; ++e) x += v[q][e];
        }
        x = warp_sum(x);
        if (lane == 0) s_warp[k & 1][warp] = x;
        __syncthreads();
        // The warp totals scanned across the lanes of every warp (5 adds, not 16).
        const TA inc = warp_inclusive_scan<TA>(lane < WARPS ? s_warp[k & 1][lane] : TA(0), lane);
        const TA w = __shfl_sync(kFullMask, inc, warp > 0 ? warp - 1 : 0);
        *wp = warp > 0 ? w : TA(0);
        *agg = __shfl_sync(kFullMask, inc, WARPS - 1);
        const TA b = *agg;
        if (threadIdx.x == 0 && (int64_t)t != ctx.fault_tile) {
            if (t == 0) {
                if (num_tiles > 1) st_relaxed_desc16(ctx.desc, pack_desc16(epoch, kStateP, acc_bits<TA>(b)));
            } else {
                st_relaxed_desc16(ctx.desc + 2 * (size_t)t, pack_desc16(epoch, kStateA, acc_bits<TA>(b)));
            }
        }
        compiler_fence();  // the aggregate just published stays ahead of the look-back
        return true;
    };

    TA wp_cur = TA(0), agg_cur = TA(0), prev_incl = TA(0);
    bool failed = false;
    uint32_t fail_at = 0;
    if (threadIdx.x == 0)
        for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);
    if (count > 0 && !reduce_publish(0, &wp_cur, &agg_cur)) failed = true;

    for (uint32_t k = 0; !failed && k < count; ++k) {
        const uint32_t t = rank + k * G;
        TA wp_next = TA(0), agg_next = TA(0);
        if (k + 1 < count && !reduce_publish(k + 1, &wp_next, &agg_next)) {
            failed = true;
            fail_at = k;
            break;
        }
        if (warp == 0) {
            TA excl = TA(0);
            bool lb_failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;
            } else {
                const int64_t floor = k > 0 ? (int64_t)t - (int64_t)G : -1;
                excl = lookback_wide<TA>(ctx.desc, ctx, t, epoch, lane, &lb_failed, floor, prev_incl);
                if (lane == 0) {
                    if (!lb_failed) {
                        st_relaxed_desc16(ctx.desc + 2 * (size_t)t,
                                          pack_desc16(epoch, kStateP, acc_bits<TA>(excl + agg_cur)));
                    } else {
                        st_relaxed_desc16(ctx.desc + 2 * (size_t)t, pack_desc16(epoch, kStatePoison, 0ull));
                        record_error(ctx.status, kErrLookbackTimeout, t);
                    }
                }
            }
            prev_incl = excl + agg_cur;
            if (lane == 0) {
                s_prefix[k & 1] = excl;
                s_fail[k & 1] = lb_failed ? 1u : 0u;
            }
        }
        // Scan tile k group by group straight out of the ring: per row, the
        // lane's pair sum, a warp scan across lanes, the rows chained in
        // order.  The first group is scanned before the barrier, while warp 0
        // looks back.
        TA v[GRP][EPV];
        TA row_excl[GRP], row_tot[GRP];
        auto scan_group = [&](int g) {
            read_group(k, g, v);
#pragma unroll
            for (int q = 0; q < GRP; ++q) {
                const TA s = v[q][0] + v[q][1];
                const TA inc = warp_inclusive_scan<TA>(s, lane);
                const TA before = __shfl_up_sync(kFullMask, inc, 1);
                row_excl[q] = lane > 0 ? before : TA(0);
                row_tot[q] = __shfl_sync(kFullMask, inc, 31);
            }
        };
        scan_group(0);
        __syncthreads();  // the prefix is in shared memory
        if (s_fail[k & 1]) {
            failed = true;
            fail_at = k;
            break;
        }
        TA base = s_prefix[k & 1] + wp_cur;
        const size_t seg = (size_t)t * TILE + (size_t)warp * SEG;
        const bool full = full_tile(k);
#pragma unroll 1
        for (int g = 0; g < VPT / GRP; ++g) {
            if (g > 0) scan_group(g);
#pragma unroll
            for (int q = 0; q < GRP; ++q) {
                TA y0, y1;
                const TA r = base + row_excl[q];
                if (INCLUSIVE) {
                    y0 = r + v[q][0];
                    y1 = y0 + v[q][1];
                } else {
                    y0 = r;
                    y1 = r + v[q][0];
                }
                base += row_tot[q];
                const size_t i0 = seg + (size_t)(32 * (g * GRP + q) + lane) * EPV;
                if (full) {
                    st_v2_u64(out + i0, acc_bits<TA>(y0), acc_bits<TA>(y1));
                } else {
                    if (i0 < n) out[i0] = y0;
                    if (i0 + 1 < n) out[i0 + 1] = y1;
                }
            }
        }
        __syncthreads();  // tile k read by everyone
        if (threadIdx.x == 0) {
            consumed = k + 1;
            if (k + STAGES < count) issue(k + STAGES);
        }
        wp_cur = wp_next;
        agg_cur = agg_next;
    }

    if (failed && threadIdx.x == 0) {
        for (uint32_t k = fail_at + 1; k < count; ++k) {
            const uint32_t t = rank + k * G;
            if ((int64_t)t != ctx.fault_tile)
                st_relaxed_desc16(ctx.desc + 2 * (size_t)t, pack_desc16(epoch, kStatePoison, 0ull));
        }
        for (uint32_t k = consumed; k < issued; ++k)
            mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
}

template <typename TI, typename TA, bool INCL>
static cudaError_t launch_wide(const void* in, void* out, size_t n, const LookbackWs& ws, cudaStream_t s) {
    constexpr int THREADS = wide_threads<TI>();
    constexpr uint32_t TILE = (uint32_t)THREADS * 128u / (uint32_t)sizeof(TI);
    constexpr size_t SMEM = 3 * (size_t)TILE * sizeof(TI);
    auto kern = k_scan_wide<TI, TA, INCL>;
    KernelSetup su;
    cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), THREADS, SMEM, &su);
    if (e != cudaSuccess) return e;
    const uint32_t tiles = (uint32_t)((n + TILE - 1) / TILE);
    const uint32_t resident = (uint32_t)(su.sms * su.blocks_per_sm);
    const uint32_t grid = tiles < resident ? tiles : resident;
    const bool fast = ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 15u) == 0;
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    kern<<<grid, THREADS, SMEM, s>>>(static_cast<const TI*>(in), static_cast<TA*>(out), n, tiles, fast, ctx);
    return cudaGetLastError();
}

// fp64 form.  GB300 keeps little FP64 throughput (measured: about 528 G
// DADD/s for the chip, 1.7 per clock per SM; one warp per sub-partition
// already reaches it), so the fp64 scan is bound by its adds, not by HBM.
// This form needs about 2.3 adds per element, against 6.6 for the form above:
//  - Each lane owns 16 consecutive elements (blocked, not striped across
//    the warp).  It scans them in sequence (15 adds) while the tile is
//    summed, so the tile's aggregate is the last lane prefix of the block,
//    with no separate reduction.  One warp scan covers 16 elements.
//  - The lane's 16 prefixes stay in registers until the tile's output (the
//    next iteration), so a tile leaves the ring as soon as it is summed, and
//    two stages suffice.
//  - Outputs add the tile/warp/lane offset (one add each; warp 0 folds the
//    tile's prefix into the warp offsets).  They go through
//    a per-warp 4 KB area of shared memory, which one tensor store per warp
//    writes to global memory.
//  - A lane's 16 elements are one 128-byte row of shared memory.  Read or
//    written 16 bytes at a time in plain row-major order, the 8 lanes of a
//    quarter-warp would all hit the same 4 banks.  So the ring and the
//    output areas hold the rows with the 128-byte swizzle of the tensor
//    copies (chunk index XOR row index mod 8): tensor loads write the ring
//    that way and tensor stores read the output areas that way, and every
//    lane's 16-byte access of a quarter-warp falls in its own banks.
//  - Two 256-thread CTAs per SM (4096-element tiles): while one waits at a
//    barrier for its look-back, the other's adds keep the FP64 pipe busy.
template <bool INCLUSIVE, int THREADS>
__global__ void __launch_bounds__(THREADS, THREADS <= 128 ? 4 : (THREADS <= 256 ? 2 : 1))
k_scan_f64_blocked(const double* in, double* out, size_t n, uint32_t num_tiles, bool fast, LookbackCtx ctx,
                   const __grid_constant__ CUtensorMap map_in, const __grid_constant__ CUtensorMap map_out) {
    constexpr int STAGES = 2;
    constexpr int EPT = 16;                                // elements per thread
    constexpr int WARPS = THREADS / 32;
    constexpr uint32_t TILE = (uint32_t)THREADS * EPT;
    constexpr uint32_t SEG = 32u * EPT;                    // 512 elements per warp
    constexpr uint32_t IN_BYTES = TILE * 8;
    constexpr uint32_t ROWS = TILE / 16;                   // 128-byte rows per tile, one per thread
    constexpr uint32_t BOX_ROWS = ROWS < 256 ? ROWS : 256;  // rows per tensor load (at most 256)
    static_assert(SEG * WARPS == TILE && ROWS == THREADS && ROWS % BOX_ROWS == 0, "tile geometry");

    // STAGES x 64 KB ring, then the 64 KB output area.  The swizzled copies
    // want 1024-byte aligned areas: the start is rounded up here, into the
    // 1 KB of slack the launch adds.
    extern __shared__ __align__(128) unsigned char smem_raw[];
    double* ring = reinterpret_cast<double*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    double* stage_out = ring + (size_t)STAGES * TILE;
    __shared__ __align__(8) uint64_t bars[STAGES];
    __shared__ double s_wtot[2][WARPS];  // warp totals, their exclusive scan, then + the tile's prefix; by parity
    __shared__ double s_agg[2];
    __shared__ uint32_t s_fail[2], s_rank, s_epoch;

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

    auto full_tile = [&](uint32_t k) { return fast && (size_t)(rank + k * G) * TILE + TILE <= n; };
    auto issue = [&](uint32_t k) {
        const int s = (int)(k % STAGES);
        if (full_tile(k)) {
            fence_async_shared();
            mbar_arrive_expect_tx(&bars[s], IN_BYTES);
            const int32_t row0 = (int32_t)((size_t)(rank + k * G) * ROWS);
#pragma unroll
            for (uint32_t b = 0; b < ROWS / BOX_ROWS; ++b)
                tensor_load_2d(ring + (size_t)s * TILE + b * BOX_ROWS * 16, &map_in, 0, row0 + (int32_t)(b * BOX_ROWS),
                               &bars[s], policy);
        } else {
            mbar_arrive(&bars[s]);  // read from global with bounds checks instead
        }
        issued = k + 1;
    };
    // Waits for tile k, scans this lane's 16 elements into p, the lane
    // totals across the warp into *lane_excl, and (warp 0) the warp totals;
    // warp 0 publishes the tile's aggregate.  The tile's stage is free on
    // return.  False if the copy did not arrive.
    auto scan_in = [&](uint32_t k, double (&p)[EPT], double* lane_excl) -> bool {
        const uint32_t t = rank + k * G;
        const bool ok = mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) record_error(ctx.status, kErrBulkTimeout, t);
            return false;
        }
        const size_t e0 = (size_t)t * TILE + (size_t)threadIdx.x * EPT;
        if (full_tile(k)) {
            const uint32_t stage = smem_u32(ring + (size_t)(k % STAGES) * TILE);
#pragma unroll
            for (int q = 0; q < EPT; q += 2) {
                double a, b;
                asm volatile("ld.shared.v2.f64 {%0, %1}, [%2];"
                             : "=d"(a), "=d"(b)
                             : "r"(stage + swizzle128_offset(threadIdx.x, (uint32_t)q / 2)));
                p[q] = a;
                p[q + 1] = b;
            }
        } else {
#pragma unroll
            for (int q = 0; q < EPT; ++q) p[q] = e0 + q < n ? in[e0 + q] : 0.0;
        }
#pragma unroll
        for (int q = 1; q < EPT; ++q) p[q] += p[q - 1];
        const double inc = warp_inclusive_scan<double>(p[EPT - 1], lane);
        const double before = __shfl_up_sync(kFullMask, inc, 1);
        *lane_excl = lane > 0 ? before : 0.0;
        if (lane == 31) s_wtot[k & 1][warp] = inc;
        __syncthreads();  // warp totals are in; the stage has been read by everyone
        if (threadIdx.x == 0 && k + STAGES < count) issue(k + STAGES);
        if (warp == 0) {
            const double w = lane < WARPS ? s_wtot[k & 1][lane] : 0.0;
            const double winc = warp_inclusive_scan<double>(w, lane);
            const double agg = __shfl_sync(kFullMask, winc, WARPS - 1);
            if (lane < WARPS) s_wtot[k & 1][lane] = winc - w;  // exclusive; read after later barriers
            if (lane == 0) {
                s_agg[k & 1] = agg;
                if ((int64_t)t != ctx.fault_tile) {
                    if (t == 0) {
                        if (num_tiles > 1)
                            st_relaxed_desc16(ctx.desc, pack_desc16(epoch, kStateP, acc_bits<double>(agg)));
                    } else {
                        st_relaxed_desc16(ctx.desc + 2 * (size_t)t, pack_desc16(epoch, kStateA, acc_bits<double>(agg)));
                    }
                }
            }
            compiler_fence();  // the aggregate is published before this warp's look-back
        }
        return true;
    };

    double pc[EPT], pn[EPT];
    double lx_cur = 0.0, lx_next = 0.0, prev_incl = 0.0;
    bool failed = false;
    uint32_t fail_at = 0;
    if (threadIdx.x == 0)
        for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);
    if (count > 0 && !scan_in(0, pc, &lx_cur)) failed = true;

    // One iteration: scan tile k+1 into pn, look back for tile k, write tile k from pc.
    auto step = [&](uint32_t k, double (&p_cur)[EPT], double lx, double (&p_next)[EPT], double* lx_nx) -> bool {
        const uint32_t t = rank + k * G;
        if (k + 1 < count && !scan_in(k + 1, p_next, lx_nx)) {
            fail_at = k;
            return false;
        }
        if (warp == 0) {
            const double agg = s_agg[k & 1];
            double excl = 0.0;
            bool lb_failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;
            } else {
                const int64_t floor = k > 0 ? (int64_t)t - (int64_t)G : -1;
                excl = lookback_wide<double>(ctx.desc, ctx, t, epoch, lane, &lb_failed, floor, prev_incl);
                if (lane == 0) {
                    if (!lb_failed) {
                        st_relaxed_desc16(ctx.desc + 2 * (size_t)t,
                                          pack_desc16(epoch, kStateP, acc_bits<double>(excl + agg)));
                    } else {
                        st_relaxed_desc16(ctx.desc + 2 * (size_t)t, pack_desc16(epoch, kStatePoison, 0ull));
                        record_error(ctx.status, kErrLookbackTimeout, t);
                    }
                }
            }
            prev_incl = excl + agg;
            if (lane == 0) s_fail[k & 1] = lb_failed ? 1u : 0u;
            if (lane < WARPS) s_wtot[k & 1][lane] = excl + s_wtot[k & 1][lane];  // each warp's offset in the scan
        }
        __syncthreads();  // tile k's warp offsets, prefix included, are in shared memory
        if (s_fail[k & 1]) {
            fail_at = k;
            return false;
        }
        const double base = s_wtot[k & 1][warp] + lx;
        double y[EPT];
#pragma unroll
        for (int q = 0; q < EPT; ++q) {
            if (INCLUSIVE) y[q] = base + p_cur[q];
            else y[q] = q == 0 ? base : base + p_cur[q - 1];
        }
        const size_t e0 = (size_t)t * TILE + (size_t)threadIdx.x * EPT;
        if (full_tile(k)) {
            const double* area = stage_out + (size_t)warp * SEG;  // 32 rows, 1024-byte aligned
            if (lane == 0) bulk_wait_group_read0();  // this warp's previous store has read the area
            __syncwarp();
            const uint32_t mine = smem_u32(area);
#pragma unroll
            for (int q = 0; q < EPT; q += 2)
                asm volatile("st.shared.v2.f64 [%0], {%1, %2};" ::"r"(mine + swizzle128_offset(lane, (uint32_t)q / 2)),
                             "d"(y[q]), "d"(y[q + 1])
                             : "memory");
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
                tensor_store_2d(&map_out, 0, (int32_t)((size_t)t * ROWS + (size_t)warp * 32), area);
                bulk_commit_group();
            }
        } else {
#pragma unroll
            for (int q = 0; q < EPT; ++q)
                if (e0 + q < n) out[e0 + q] = y[q];
        }
        return true;
    };

    for (uint32_t k = 0; !failed && k < count; k += 2) {
        if (!step(k, pc, lx_cur, pn, &lx_next)) failed = true;
        else if (k + 1 < count && !step(k + 1, pn, lx_next, pc, &lx_cur)) failed = true;
    }

    if (failed && threadIdx.x == 0) {
        consumed = issued;  // every issued copy is waited for below
        for (uint32_t j = fail_at + 1; j < count; ++j) {
            const uint32_t tt = rank + j * G;
            if ((int64_t)tt != ctx.fault_tile)
                st_relaxed_desc16(ctx.desc + 2 * (size_t)tt, pack_desc16(epoch, kStatePoison, 0ull));
        }
        for (uint32_t j = fail_at + 1; j < issued; ++j)
            mbar_wait_bounded(&bars[j % STAGES], (j / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
    if (lane == 0) bulk_wait_group0();  // this warp's output stores are complete before the CTA leaves
    (void)consumed;
}

constexpr int kF64Threads = 256;
static_assert(kF64Threads * 16 == (int)kWideTileF64, "fp64 tile size shared with the host side");

template <bool INCL, int THREADS>
static cudaError_t launch_f64_blocked(const void* in, void* out, size_t n, const LookbackWs& ws, cudaStream_t s) {
    constexpr uint32_t TILE = (uint32_t)THREADS * 16;
    constexpr size_t SMEM = 3 * (size_t)TILE * 8 + 1024;  // two ring stages, the output area, alignment slack
    auto kern = k_scan_f64_blocked<INCL, THREADS>;
    KernelSetup su;
    cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), THREADS, SMEM, &su);
    if (e != cudaSuccess) return e;
    const uint32_t resident = (uint32_t)(su.sms * su.blocks_per_sm);  // the persistent grid
    const uint32_t tiles = (uint32_t)((n + TILE - 1) / TILE);
    const uint32_t grid = tiles < resident ? tiles : resident;
    // Full tiles go through the tensor copies: both buffers 16-byte aligned,
    // and every row coordinate within the copies' signed 32-bit range.
    const uint64_t rows = n / 16;
    const bool fast = ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 15u) == 0 &&
                      n >= TILE && rows <= (uint64_t)INT32_MAX;
    CUtensorMap map_in{}, map_out{};
    if (fast) {
        e = encode_rows128_f64(&map_in, in, rows, THREADS < 256 ? THREADS : 256);
        if (e == cudaSuccess) e = encode_rows128_f64(&map_out, out, rows, 32);
        if (e != cudaSuccess) return e;
    }
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    kern<<<grid, THREADS, SMEM, s>>>(static_cast<const double*>(in), static_cast<double*>(out), n, tiles, fast, ctx,
                                       map_in, map_out);
    return cudaGetLastError();
}

cudaError_t launch_scan_wide(WideType type, bool inclusive, const void* in, void* out, size_t n,
                             const LookbackWs& ws, cudaStream_t s) {
    using u64 = unsigned long long;
    switch (type) {
        case WideType::U32toU64:
            return inclusive ? launch_wide<uint32_t, u64, true>(in, out, n, ws, s)
                             : launch_wide<uint32_t, u64, false>(in, out, n, ws, s);
        case WideType::I32toI64:
            return inclusive ? launch_wide<int32_t, u64, true>(in, out, n, ws, s)
                             : launch_wide<int32_t, u64, false>(in, out, n, ws, s);
        case WideType::I64:
            return inclusive ? launch_wide<u64, u64, true>(in, out, n, ws, s)
                             : launch_wide<u64, u64, false>(in, out, n, ws, s);
        default:
            return inclusive ? launch_f64_blocked<true, kF64Threads>(in, out, n, ws, s)
                             : launch_f64_blocked<false, kF64Threads>(in, out, n, ws, s);
    }
}

}  // namespace ss
