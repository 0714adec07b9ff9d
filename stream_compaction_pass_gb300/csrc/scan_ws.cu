// scan_ws.cu -- the single-pass look-back scan, persistent and
// warp-specialised: sixteen data warps stream tiles through a bulk-copy ring
// and one look-back warp resolves tile prefixes in parallel with them.
//
// Per CTA (rank r from the workspace counter, tiles r, r + G, r + 2G, ...;
// see scan_pipe.cu for why this order guarantees progress):
//
//   data warps, iteration k (tile k is in ring stage k % STAGES):
//     1. wait for tile k+1's copy, sum it straight out of shared memory,
//        combine the warp sums (named barrier 1, data warps only) and publish
//        tile k+1's aggregate A; hand the aggregate to the look-back warp
//        (mbarrier agg_bar);
//     2. read tile k from the ring into registers and scan it (per-thread,
//        shuffle and block combine);
//     3. release tile k's stage and start the copy of tile k + STAGES;
//     4. wait for tile k's exclusive prefix from the look-back warp
//        (mbarrier pre_bar) and store tile k.
//   look-back warp, tile k: wait for tile k's aggregate, look back as far as
//     this CTA's previous tile (whose inclusive prefix it holds), publish P,
//     hand the prefix to the data warps.
//
// The look-back for tile k starts as soon as tile k's aggregate is known --
// during the data warps' iteration k-1 -- so its L2 round trips overlap a
// whole iteration of streaming instead of sitting on its critical path.
#include "bulk.cuh"
#include "internal.h"
#include "scan_body.cuh"

namespace ss {

namespace {

constexpr int kSlots = 2;  // aggregate / prefix hand-over slots

__device__ __forceinline__ void data_barrier(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// OR of `pred` over the data warps (named barrier 1).
__device__ __forceinline__ bool data_barrier_or(bool pred, int nthreads) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(nthreads)
        : "memory");
    return r != 0;
}

}  // namespace

template <typename T, bool INCLUSIVE, int DWARPS, int VPT, int STAGES, int K, bool LAG, bool TRACE>
__global__ void __launch_bounds__((DWARPS + 1) * 32, 1)
k_scan_ws(const T* in, T* out, size_t n, uint32_t num_tiles, LookbackCtx ctx, const T* carry_in,
          T* carry_out, unsigned long long* trace) {
    static_assert(STAGES >= 3, "the scan pass re-reads tile k while tile k+1 is summed");
    constexpr int DTHREADS = DWARPS * 32;
    constexpr uint32_t TILE = (uint32_t)DTHREADS * VPT * 4;
    constexpr uint32_t TILE_BYTES = TILE * (uint32_t)sizeof(T);
    constexpr uint32_t SEG = 32u * VPT * 4;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    T* ring = reinterpret_cast<T*>(smem_raw);
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t agg_bar[kSlots];
    __shared__ __align__(8) uint64_t pre_bar[kSlots];
    __shared__ T warp_tot[DWARPS];
    __shared__ T agg_slot[kSlots];
    __shared__ T pre_slot[kSlots];
    __shared__ uint32_t stop_slot[kSlots];  // data warps stopped: no aggregate follows
    __shared__ uint32_t fail_slot[kSlots];  // look-back failed: no prefix follows
    __shared__ uint32_t s_rank, s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t G = gridDim.x;

    if (threadIdx.x == 0) {
        uint32_t rank, epoch;
        claim_tile(ctx.counter, G, &rank, &epoch);  // one claim per CTA; the last resets the counter
        s_rank = rank;
        s_epoch = epoch;
        for (int s = 0; s < STAGES; ++s) mbar_init(&full_bar[s], 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&agg_bar[s], 1);
            mbar_init(&pre_bar[s], 1);
        }
        fence_async_shared();
    }
    __syncthreads();  // the only CTA-wide barrier
    const uint32_t rank = s_rank;
    const uint32_t epoch = s_epoch;
    if (rank >= G) {  // counter out of step: never index past the descriptors
        if (threadIdx.x == 0) record_error(ctx.status, kErrCounter, rank);
        return;
    }
    const uint32_t count = rank < num_tiles ? (num_tiles - rank + G - 1) / G : 0;
    if (count == 0) return;

    if (warp == DWARPS) {
        // ------------------------------------------------ look-back warp
        T prev_incl = T(0);
        for (uint32_t k = 0; k < count; ++k) {
            const uint32_t t = rank + k * G;
            const int slot = (int)(k % kSlots);
            // With LAG, start tile k's look-back once tile k+1's aggregate is
            // out too: by then the other CTAs have published theirs for the
            // tiles before tile k, and one window read usually suffices.
            const uint32_t gate = (LAG && k + 1 < count) ? k + 1 : k;
            const bool got = mbar_wait_bounded(&agg_bar[gate % kSlots], (gate / kSlots) & 1u, ctx.max_polls,
                                               ctx.timeout_ns);
            if (!__all_sync(kFullMask, got) || stop_slot[gate % kSlots]) break;
            if (gate != k && stop_slot[slot]) break;
            const T agg = agg_slot[slot];
            LookbackStats stats{0u, 0u};
            T excl = T(0);
            bool failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                excl = carry_in ? *carry_in : T(0);  // P of tile 0 was published with its aggregate
                failed = dead;
            } else if (dead) {
                failed = true;  // it published nothing, so its successors' waits run out
            } else {
                const int64_t floor = k > 0 ? (int64_t)t - (int64_t)G : -1;
                excl = lookback<T, K, TRACE>(ctx, t, epoch, lane, &failed, &stats, floor, prev_incl);
                if (lane == 0) {
                    if (!failed) {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, to_bits<T>(excl + agg)));
                    } else {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
                        record_error(ctx.status, kErrLookbackTimeout, t);
                    }
                }
            }
            prev_incl = excl + agg;
            if (lane == 0) {
                pre_slot[slot] = excl;
                fail_slot[slot] = failed ? 1u : 0u;
                if (TRACE) {
                    unsigned long long* rec = trace + (size_t)t * kTraceWords;
                    rec[3] = globaltimer_ns();
                    rec[5] = stats.windows;
                    rec[6] = stats.waits;
                    rec[7] = (unsigned long long)sm_id() | ((unsigned long long)blockIdx.x << 32);
                }
                mbar_arrive(&pre_bar[slot]);
            }
            if (failed) break;
        }
        return;
    }

    // ---------------------------------------------------- data warps
    const uint64_t policy = policy_evict_first();
    uint32_t issued = 0, consumed = 0;  // thread 0: copies started / stages released

    auto issue = [&](uint32_t k) {  // thread 0: start the copy of this CTA's k-th tile
        const int s = (int)(k % STAGES);
        const size_t base = (size_t)(rank + k * G) * TILE;
        if (base + TILE <= n) {
            fence_async_shared();  // earlier reads of this stage before the copy's writes
            mbar_arrive_expect_tx(&full_bar[s], TILE_BYTES);
            bulk_load(ring + (size_t)s * TILE, in + base, TILE_BYTES, &full_bar[s], policy);
        } else {
            mbar_arrive(&full_bar[s]);  // ragged last tile: read from global
        }
        issued = k + 1;
    };
    auto wait_full = [&](uint32_t k) -> bool {  // every data thread; uniform result
        const bool ok = mbar_wait_bounded(&full_bar[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        return !data_barrier_or(!ok, DTHREADS);
    };
    // This lane's rows of tile k: from the ring, or from global for the ragged tile.
    auto read_rows = [&](uint32_t k, T (&v)[VPT][4]) {
        const size_t tile_base = (size_t)(rank + k * G) * TILE;
        if (tile_base + TILE <= n) {
            const T* src = ring + (size_t)(k % STAGES) * TILE + (size_t)warp * SEG + (size_t)lane * 4;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const uint4 r = lds_vec(src + 128 * j);
                v[j][0] = from_bits<T>(r.x);
                v[j][1] = from_bits<T>(r.y);
                v[j][2] = from_bits<T>(r.z);
                v[j][3] = from_bits<T>(r.w);
            }
        } else {
            load_rows<T, VPT>(in, n, tile_base + (size_t)warp * SEG, lane, false, v);
        }
    };
    // Sums tile k, publishes its aggregate and hands it to the look-back warp;
    // returns this warp's prefix within the tile.
    auto reduce_publish = [&](uint32_t k) -> T {
        const uint32_t t = rank + k * G;
        if (TRACE && threadIdx.x == 0) trace[(size_t)t * kTraceWords] = globaltimer_ns();
        T v[VPT][4];
        read_rows(k, v);
        T x = T(0);
#pragma unroll
        for (int j = 0; j < VPT; ++j) x += ((v[j][0] + v[j][1]) + v[j][2]) + v[j][3];
        x = warp_sum(x);
        if (lane == 0) warp_tot[warp] = x;
        data_barrier(DTHREADS);
        T wp = T(0), agg = T(0);
#pragma unroll
        for (int w = 0; w < DWARPS; ++w) {
            const T tw = warp_tot[w];
            if (w < warp) wp += tw;
            agg += tw;
        }
        if (threadIdx.x == 0) {
            if ((int64_t)t != ctx.fault_tile) {
                if (t == 0) {
                    if (num_tiles > 1)
                        st_relaxed_u64(ctx.desc, pack_desc(epoch, kStateP,
                                                           to_bits<T>((carry_in ? *carry_in : T(0)) + agg)));
                } else {
                    st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateA, to_bits<T>(agg)));
                }
            }
            compiler_fence();
            if (TRACE) trace[(size_t)t * kTraceWords + 1] = trace[(size_t)t * kTraceWords + 2] = globaltimer_ns();
            const int slot = (int)(k % kSlots);
            agg_slot[slot] = agg;
            stop_slot[slot] = 0u;
            mbar_arrive(&agg_bar[slot]);
        }
        return wp;
    };
    auto stop_lookback = [&](uint32_t k) {  // thread 0: no aggregate for tile k will come
        const int slot = (int)(k % kSlots);
        stop_slot[slot] = 1u;
        mbar_arrive(&agg_bar[slot]);
    };

    if (threadIdx.x == 0)
        for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);

    bool failed = false;
    uint32_t fail_at = 0;
    T wp_cur = T(0);
    if (!wait_full(0)) {
        failed = true;
        if (threadIdx.x == 0) {
            record_error(ctx.status, kErrBulkTimeout, rank);
            stop_lookback(0);
        }
    } else {
        wp_cur = reduce_publish(0);
    }

    for (uint32_t k = 0; !failed && k < count; ++k) {
        const uint32_t t = rank + k * G;
        // 1. the next tile's aggregate
        T wp_next = T(0);
        if (k + 1 < count) {
            if (!wait_full(k + 1)) {
                failed = true;
                fail_at = k;
                if (threadIdx.x == 0) {
                    record_error(ctx.status, kErrBulkTimeout, t + G);
                    stop_lookback(k + 1);
                }
                break;
            }
            wp_next = reduce_publish(k + 1);
        }
        // 2. scan tile k in registers
        T v[VPT][4];
        read_rows(k, v);
        T pre[VPT];
        warp_rows_scan<T, VPT>(v, lane, pre);
        // 3. release tile k's stage
        data_barrier(DTHREADS);
        if (threadIdx.x == 0) {
            consumed = k + 1;
            if (k + STAGES < count) issue(k + STAGES);
        }
        // 4. tile k's prefix, then store
        const int slot = (int)(k % kSlots);
        const bool got = mbar_wait_bounded(&pre_bar[slot], (k / kSlots) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (data_barrier_or(!got || fail_slot[slot] != 0u, DTHREADS)) {
            failed = true;
            fail_at = k;
            if (threadIdx.x == 0 && !got) record_error(ctx.status, kErrLookbackTimeout, t);
            break;
        }
        const size_t tile_base = (size_t)t * TILE;
        rows_output_inplace<T, VPT, INCLUSIVE>(v, pre, pre_slot[slot] + wp_cur);
        store_rows<T, VPT>(out, n, tile_base + (size_t)warp * SEG, lane, tile_base + TILE <= n, v);
        if (carry_out != nullptr && t == num_tiles - 1 && threadIdx.x == 0)
            *carry_out = pre_slot[slot] + agg_slot[slot];
        if (TRACE && threadIdx.x == 0) trace[(size_t)t * kTraceWords + 4] = globaltimer_ns();
        wp_cur = wp_next;
    }

    if (failed && threadIdx.x == 0) {
        // Leaving early: poison this CTA's later tiles so their successors
        // fail fast; let copies in flight land (bounded waits).
        for (uint32_t k = fail_at + 1; k < count; ++k) {
            const uint32_t t = rank + k * G;
            if ((int64_t)t != ctx.fault_tile) st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
        }
        for (uint32_t k = consumed; k < issued; ++k)
            mbar_wait_bounded(&full_bar[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
}

template <typename T, bool INCL, int DWARPS, int VPT, int STAGES, int K, bool LAG, bool TRACE>
static cudaError_t launch_ws(const void* in, void* out, size_t n, const LookbackWs& ws, const void* carry_in,
                             void* carry_out, unsigned long long* trace, cudaStream_t s) {
    constexpr int THREADS = (DWARPS + 1) * 32;
    constexpr size_t TILE = (size_t)DWARPS * 32 * VPT * 4;
    constexpr size_t SMEM = (size_t)STAGES * TILE * sizeof(T);
    auto kern = k_scan_ws<T, INCL, DWARPS, VPT, STAGES, K, LAG, TRACE>;
    KernelSetup su;
    cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), THREADS, SMEM, &su);
    if (e != cudaSuccess) return e;
    const uint32_t tiles = (uint32_t)((n + TILE - 1) / TILE);
    const size_t resident = (size_t)su.sms * (size_t)su.blocks_per_sm;
    const uint32_t grid = (uint32_t)(tiles < resident ? tiles : resident);
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    kern<<<grid, THREADS, SMEM, s>>>(static_cast<const T*>(in), static_cast<T*>(out), n, tiles, ctx,
                                      static_cast<const T*>(carry_in), static_cast<T*>(carry_out), trace);
    return cudaGetLastError();
}

template <typename T, bool INCL, bool TRACE>
static cudaError_t dispatch_ws(int config, const void* in, void* out, size_t n, const LookbackWs& ws,
                               const void* ci, void* co, unsigned long long* tr, cudaStream_t s) {
    (void)config;  // row 5, the only warp-specialised row
    return launch_ws<T, INCL, 16, 8, 3, 1, true, TRACE>(in, out, n, ws, ci, co, tr, s);
}

cudaError_t launch_scan_lookback_ws(Dtype dt, bool inclusive, int config, const void* in, void* out,
                                    size_t n, const LookbackWs& ws, const void* carry_in, void* carry_out,
                                    cudaStream_t s) {
    if (dt == Dtype::F32)
        return inclusive ? dispatch_ws<float, true, false>(config, in, out, n, ws, carry_in, carry_out, nullptr, s)
                         : dispatch_ws<float, false, false>(config, in, out, n, ws, carry_in, carry_out, nullptr, s);
    return inclusive ? dispatch_ws<uint32_t, true, false>(config, in, out, n, ws, carry_in, carry_out, nullptr, s)
                     : dispatch_ws<uint32_t, false, false>(config, in, out, n, ws, carry_in, carry_out, nullptr, s);
}

cudaError_t launch_scan_trace_ws(int config, const void* in, void* out, size_t n, const LookbackWs& ws,
                                 unsigned long long* trace, cudaStream_t s) {
    return dispatch_ws<uint32_t, false, true>(config, in, out, n, ws, nullptr, nullptr, trace, s);
}

}  // namespace ss
