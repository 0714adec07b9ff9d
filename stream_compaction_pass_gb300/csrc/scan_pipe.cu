// scan_pipe.cu -- the single-pass look-back scan as a persistent kernel fed
// by the bulk-copy engine.
//
// The one-CTA-per-tile kernel (scan.cu) stops loading while a tile waits in
// its look-back, and with thousands of small tiles in flight each look-back
// walks far back to the last published inclusive prefix.  Here a grid of one
// or two CTAs per SM streams large tiles through a shared-memory ring: the
// bulk-copy engine (cp.async.bulk, one instruction per tile, completion
// counted on an mbarrier) fills the next STAGES-1 tiles while the CTA scans,
// looks back and stores the current one.
//
// Schedule, two forms (the configuration table in scan.cu picks one):
//  - fixed: each CTA takes a rank r from the workspace counter when it
//    starts, then processes tiles r, r + G, r + 2G, ... (G = grid size);
//  - claimed (the default row): each CTA claims its next tile from the
//    counter when it starts that tile's copy, so a faster SM takes more
//    tiles (k_scan_lookback_pipe_sb with DYN).
// Either way tiles are handed out in start (or claim) order, so the CTA
// owning the smallest unfinished tile has started and reaches that tile
// after finishing its own smaller ones: every look-back wait ends without
// relying on all CTAs being resident.  Consecutive tiles belong to
// different CTAs and are processed at about the same time.
//
// The per-tile arithmetic is the same as scan.cu's (scan_body.cuh).  Reading
// the ring back is conflict-free: lane l of a warp reads the l-th 16-byte
// vector of a 512-byte row.
#include <type_traits>

#include "bulk.cuh"
#include "internal.h"
#include "scan_body.cuh"

namespace ss {

template <typename T, bool INCLUSIVE, int THREADS, int VPT, int STAGES, int K, bool TRACE>
__global__ void __launch_bounds__(THREADS, 1)
k_scan_lookback_pipe(const T* in, T* out, size_t n, uint32_t num_tiles, LookbackCtx ctx,
                     const T* carry_in, T* carry_out, unsigned long long* trace) {
    static_assert(STAGES >= 2, "the ring needs two stages at least");
    constexpr int WARPS = THREADS / 32;
    constexpr uint32_t TILE = (uint32_t)THREADS * VPT * 4;
    constexpr uint32_t TILE_BYTES = TILE * (uint32_t)sizeof(T);
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
        claim_tile(ctx.counter, G, &rank, &epoch);  // one claim per CTA; the last resets the counter
        s_rank = rank;
        s_epoch = epoch;
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_async_shared();
    }
    __syncthreads();
    const uint32_t rank = s_rank;
    const uint32_t epoch = s_epoch;
    if (rank >= G) {  // counter out of step: never index past the descriptors
        if (threadIdx.x == 0) record_error(ctx.status, kErrCounter, rank);
        return;
    }
    // This CTA's tiles: rank + k*G for k = 0 .. count-1.
    const uint32_t count = rank < num_tiles ? (num_tiles - rank + G - 1) / G : 0;
    uint32_t issued = 0, fetched = 0;  // thread 0: copies started / tiles read from the ring

    auto issue = [&](uint32_t k) {  // thread 0: start the copy of this CTA's k-th tile
        const int s = (int)(k % STAGES);
        const size_t base = (size_t)(rank + k * G) * TILE;
        if (base + TILE <= n) {
            fence_async_shared();  // earlier reads of this stage before the copy's writes
            mbar_arrive_expect_tx(&bars[s], TILE_BYTES);
            bulk_load(ring + (size_t)s * TILE, in + base, TILE_BYTES, &bars[s], policy);
        } else {
            mbar_arrive(&bars[s]);  // ragged last tile: read from global by the consumers
        }
        issued = k + 1;
    };

    // Reads the k-th tile into v, frees its stage and starts the copy of tile
    // k + STAGES.  False (CTA-uniform) if the copy did not arrive in time.
    auto fetch = [&](uint32_t k, T (&v)[VPT][4]) -> bool {
        const uint32_t t = rank + k * G;
        const int s = (int)(k % STAGES);
        const size_t tile_base = (size_t)t * TILE;
        if (TRACE && threadIdx.x == 0) trace[(size_t)t * kTraceWords] = globaltimer_ns();
        const bool ok = mbar_wait_bounded(&bars[s], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) record_error(ctx.status, kErrBulkTimeout, t);
            return false;
        }
        if (tile_base + TILE <= n) {
            const T* src = ring + (size_t)s * TILE + (size_t)warp * SEG + (size_t)lane * 4;
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
        __syncthreads();  // stage s has been read
        if (threadIdx.x == 0) {
            fetched = k + 1;
            if (k + STAGES < count) issue(k + STAGES);
        }
        return true;
    };

    // Sums tile t (rows v) and publishes its aggregate at once: A, or P for
    // tile 0 (whose prefix is the seed).
    auto reduce_publish = [&](uint32_t t, const T (&v)[VPT][4], T* wp, T* agg) {
        T x = T(0);
#pragma unroll
        for (int j = 0; j < VPT; ++j) x += ((v[j][0] + v[j][1]) + v[j][2]) + v[j][3];
        block_combine<T, WARPS>(warp_sum(x), warp, lane, sm.warp, wp, agg);
        if (threadIdx.x == 0 && (int64_t)t != ctx.fault_tile) {
            if (t == 0) {
                if (num_tiles > 1)
                    st_relaxed_u64(ctx.desc, pack_desc(epoch, kStateP,
                                                       to_bits<T>((carry_in ? *carry_in : T(0)) + *agg)));
            } else {
                st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateA, to_bits<T>(*agg)));
            }
            if (TRACE) {
                unsigned long long* rec = trace + (size_t)t * kTraceWords;
                rec[1] = rec[2] = globaltimer_ns();
            }
        }
    };

    T wp_cur = T(0), agg_cur = T(0);  // warp prefix and aggregate of the current tile
    T prev_incl = T(0);               // warp 0: inclusive prefix through this CTA's previous tile
    uint32_t fail_at = 0xffffffffu;

    // One iteration: fetch + reduce + publish tile k+1, look back for tile
    // k and scan it, store it.  vc holds tile k, vn receives tile k+1.
    auto step = [&](uint32_t k, T (&vc)[VPT][4], T (&vn)[VPT][4]) -> bool {
        const uint32_t t = rank + k * G;
        T wp_next = T(0), agg_next = T(0);
        if (k + 1 < count) {
            if (!fetch(k + 1, vn)) {
                fail_at = k;
                return false;
            }
            reduce_publish(t + G, vn, &wp_next, &agg_next);
        }
        compiler_fence();  // the aggregate just published stays ahead of the look-back
        if (warp == 0) {
            LookbackStats stats{0u, 0u};
            T excl = T(0);
            bool failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                excl = carry_in ? *carry_in : T(0);
                failed = dead;
            } else if (dead) {
                failed = true;  // it published nothing, so its successors' waits run out
            } else {
                // The walk stops at this CTA's previous tile at the latest.
                const int64_t floor = k > 0 ? (int64_t)t - (int64_t)G : -1;
                excl = lookback<T, K, TRACE>(ctx, t, epoch, lane, &failed, &stats, floor, prev_incl);
                if (lane == 0) {
                    if (!failed) {
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
                sm.fail[k & 1] = failed ? 1u : 0u;
                if (TRACE) {
                    unsigned long long* rec = trace + (size_t)t * kTraceWords;
                    rec[3] = globaltimer_ns();
                    rec[5] = stats.windows;
                    rec[6] = stats.waits;
                    rec[7] = (unsigned long long)sm_id() | ((unsigned long long)blockIdx.x << 32);
                }
            }
        }
        T pre[VPT];
        warp_rows_scan<T, VPT>(vc, lane, pre);
        __syncthreads();
        if (sm.fail[k & 1]) {
            fail_at = k;
            return false;
        }
        const size_t tile_base = (size_t)t * TILE;
        rows_output_inplace<T, VPT, INCLUSIVE>(vc, pre, sm.prefix[k & 1] + wp_cur);
        store_rows<T, VPT>(out, n, tile_base + (size_t)warp * SEG, lane, tile_base + TILE <= n, vc);
        if (carry_out != nullptr && t == num_tiles - 1 && threadIdx.x == 0) *carry_out = sm.prefix[k & 1] + agg_cur;
        if (TRACE && threadIdx.x == 0) trace[(size_t)t * kTraceWords + 4] = globaltimer_ns();
        wp_cur = wp_next;
        agg_cur = agg_next;
        return true;
    };

    T va[VPT][4], vb[VPT][4];  // register double buffer: current and next tile
    bool failed = false;
    if (count > 0) {
        if (threadIdx.x == 0)
            for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);
        if (!fetch(0, va)) {
            failed = true;
            fail_at = 0;
        } else {
            reduce_publish(rank, va, &wp_cur, &agg_cur);
        }
        compiler_fence();
    }
    for (uint32_t k = 0; !failed && k < count; k += 2) {
        if (!step(k, va, vb)) {
            failed = true;
        } else if (k + 1 < count && !step(k + 1, vb, va)) {
            failed = true;
        }
    }

    if (failed && threadIdx.x == 0) {
        // Leaving early: poison this CTA's later tiles so that their
        // successors fail fast, and let its copies in flight land before the
        // shared memory goes away (bounded waits).
        for (uint32_t k = fail_at + 1; k < count; ++k) {
            const uint32_t t = rank + k * G;
            if ((int64_t)t != ctx.fault_tile) st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
        }
        for (uint32_t k = fetched; k < issued; ++k)
            mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
}

// Single-register-buffer form of the same schedule: the next tile is summed
// straight out of the ring (no registers held for it) and the current tile
// is read again for its scan, so a tile stays in the ring until its scan and
// the ring needs three stages.  Same arithmetic and look-back as above; it
// exists because the double register buffer does not fit 128 registers for
// every element type without spilling.
//
// DYN selects how tiles reach CTAs.  false: the fixed stride above (rank +
// k*G).  true: thread 0 claims each tile from the workspace counter when it
// starts that tile's copy, STAGES tiles ahead of its scan.  Claims are
// handed out in increasing order, so a CTA still processes its tiles in
// increasing order and its previous tile still bounds its look-back; what
// changes is that an SM that streams faster takes more tiles, instead of
// the look-back chain pacing every CTA at the slowest one's rate.  Each CTA
// stops at its first claim past the last tile, so a launch makes exactly
// num_tiles + G claims and the one that makes the last claim resets the
// counter for the next launch.  Every wait still ends: the CTA owning the
// smallest unfinished tile has claimed it, has finished its own earlier
// tiles, and finds every tile below it finished.
template <typename T, bool INCLUSIVE, int THREADS, int VPT, int STAGES, int K, bool TRACE, bool DYN>
__global__ void __launch_bounds__(THREADS, 1)
k_scan_lookback_pipe_sb(const T* in, T* out, size_t n, uint32_t num_tiles, LookbackCtx ctx,
                        const T* carry_in, T* carry_out, unsigned long long* trace) {
    static_assert(STAGES >= 3, "tile k stays in the ring while tile k+1 is summed");
    constexpr int WARPS = THREADS / 32;
    constexpr uint32_t TILE = (uint32_t)THREADS * VPT * 4;
    constexpr uint32_t TILE_BYTES = TILE * (uint32_t)sizeof(T);
    constexpr uint32_t SEG = 32u * VPT * 4;
    constexpr uint32_t kNoTile = 0xffffffffu;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    T* ring = reinterpret_cast<T*>(smem_raw);
    __shared__ __align__(8) uint64_t bars[STAGES];
    __shared__ ScanSmem<T, WARPS> sm;
    __shared__ uint32_t s_rank, s_epoch;
    __shared__ uint32_t s_tile[STAGES];  // DYN: the tile in each stage, kNoTile past the last

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t G = gridDim.x;
    const uint64_t policy = policy_evict_first();

    uint32_t issued = 0, consumed = 0;  // thread 0: copies started / stages read
    bool claims_done = false;           // thread 0 (DYN): a claim has come back past the last tile

    // DYN, thread 0: the next tile id from the counter, or kNoTile.
    auto claim_next = [&]() -> uint32_t {
        if (claims_done) return kNoTile;
        uint32_t id, ep;
        claim_tile(ctx.counter, num_tiles + G, &id, &ep);
        s_epoch = ep;
        if (id < num_tiles) return id;
        claims_done = true;
        return kNoTile;
    };

    if (threadIdx.x == 0) {
        if (!DYN) {
            uint32_t rank, epoch;
            claim_tile(ctx.counter, G, &rank, &epoch);
            s_rank = rank;
            s_epoch = epoch;
        } else {
            s_rank = 0;
        }
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_async_shared();
    }
    if (!DYN) __syncthreads();
    const uint32_t rank = DYN ? 0u : s_rank;
    if (!DYN && rank >= G) {
        if (threadIdx.x == 0) record_error(ctx.status, kErrCounter, rank);
        return;
    }
    const uint32_t count = DYN ? 0u : (rank < num_tiles ? (num_tiles - rank + G - 1) / G : 0);

    // The tile in this CTA's k-th slot.  DYN reads the id thread 0 stored
    // when it started that slot's copy; every reader is past a barrier that
    // follows the store, and the slot is only rewritten after a barrier that
    // follows every read.
    auto tile_of = [&](uint32_t k) -> uint32_t {
        if constexpr (DYN) return s_tile[k % STAGES];
        else return k < count ? rank + k * G : kNoTile;
    };

    auto issue = [&](uint32_t k) {  // thread 0
        const int s = (int)(k % STAGES);
        const uint32_t t = DYN ? claim_next() : rank + k * G;
        if (DYN) s_tile[s] = t;
        if (t != kNoTile) {
            const size_t base = (size_t)t * TILE;
            if (base + TILE <= n) {
                fence_async_shared();
                mbar_arrive_expect_tx(&bars[s], TILE_BYTES);
                bulk_load(ring + (size_t)s * TILE, in + base, TILE_BYTES, &bars[s], policy);
            } else {
                mbar_arrive(&bars[s]);
            }
        }
        issued = k + 1;
    };
    auto read_rows = [&](uint32_t k, uint32_t t, T (&v)[VPT][4]) {
        const size_t tile_base = (size_t)t * TILE;
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
    // Waits for slot k (tile t), sums it, publishes its aggregate; false if the copy did not arrive.
    auto reduce_publish = [&](uint32_t k, uint32_t t, T* wp, T* agg) -> bool {
        if (TRACE && threadIdx.x == 0) trace[(size_t)t * kTraceWords] = globaltimer_ns();
        const bool ok = mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) record_error(ctx.status, kErrBulkTimeout, t);
            return false;
        }
        T v[VPT][4];
        read_rows(k, t, v);
        T x = T(0);
#pragma unroll
        for (int j = 0; j < VPT; ++j) x += ((v[j][0] + v[j][1]) + v[j][2]) + v[j][3];
        block_combine<T, WARPS>(warp_sum(x), warp, lane, sm.warp, wp, agg);
        if (threadIdx.x == 0 && (int64_t)t != ctx.fault_tile) {
            if (t == 0) {
                if (num_tiles > 1)
                    st_relaxed_u64(ctx.desc, pack_desc(s_epoch, kStateP,
                                                       to_bits<T>((carry_in ? *carry_in : T(0)) + *agg)));
            } else {
                st_relaxed_u64(ctx.desc + t, pack_desc(s_epoch, kStateA, to_bits<T>(*agg)));
            }
            if (TRACE) trace[(size_t)t * kTraceWords + 1] = trace[(size_t)t * kTraceWords + 2] = globaltimer_ns();
        }
        compiler_fence();  // the aggregate just published stays ahead of the look-back
        return true;
    };

    if (threadIdx.x == 0) {
        if (DYN)
            for (uint32_t k = 0; k < (uint32_t)STAGES; ++k) issue(k);
        else
            for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);
    }
    if (DYN) __syncthreads();  // the first slots' tile ids and the epoch
    const uint32_t epoch = s_epoch;

    T wp_cur = T(0), agg_cur = T(0), prev_incl = T(0);
    int64_t prev_tile = -1;  // warp 0: this CTA's previous tile, whose inclusive prefix is prev_incl
    bool failed = false;
    uint32_t fail_at = 0;
    uint32_t t = tile_of(0);
    if (t != kNoTile && !reduce_publish(0, t, &wp_cur, &agg_cur)) failed = true;

    uint32_t k = 0;
    for (; !failed && t != kNoTile; ++k) {
        const uint32_t tn = tile_of(k + 1);
        T wp_next = T(0), agg_next = T(0);
        if (tn != kNoTile && !reduce_publish(k + 1, tn, &wp_next, &agg_next)) {
            failed = true;
            fail_at = k;
            break;
        }
        if (warp == 0) {
            LookbackStats stats{0u, 0u};
            T excl = T(0);
            bool lb_failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                excl = carry_in ? *carry_in : T(0);
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;
            } else {
                excl = lookback<T, K, TRACE>(ctx, t, epoch, lane, &lb_failed, &stats, prev_tile, prev_incl);
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
            prev_tile = t;
            if (lane == 0) {
                sm.prefix[k & 1] = excl;
                sm.fail[k & 1] = lb_failed ? 1u : 0u;
                if (TRACE) {
                    unsigned long long* rec = trace + (size_t)t * kTraceWords;
                    rec[3] = globaltimer_ns();
                    rec[5] = stats.windows;
                    rec[6] = stats.waits;
                    rec[7] = (unsigned long long)sm_id() | ((unsigned long long)blockIdx.x << 32);
                }
            }
        }
        T v[VPT][4];
        read_rows(k, t, v);
        T pre[VPT];
        warp_rows_scan<T, VPT>(v, lane, pre);
        __syncthreads();  // tile k read by everyone; the prefix is in shared memory
        if (threadIdx.x == 0) {
            consumed = k + 1;
            if (DYN || k + STAGES < count) issue(k + STAGES);
        }
        if (sm.fail[k & 1]) {
            failed = true;
            fail_at = k;
            break;
        }
        const size_t tile_base = (size_t)t * TILE;
        rows_output_inplace<T, VPT, INCLUSIVE>(v, pre, sm.prefix[k & 1] + wp_cur);
        store_rows<T, VPT>(out, n, tile_base + (size_t)warp * SEG, lane, tile_base + TILE <= n, v);
        if (carry_out != nullptr && t == num_tiles - 1 && threadIdx.x == 0) *carry_out = sm.prefix[k & 1] + agg_cur;
        if (TRACE && threadIdx.x == 0) trace[(size_t)t * kTraceWords + 4] = globaltimer_ns();
        wp_cur = wp_next;
        agg_cur = agg_next;
        t = tn;
    }

    if (failed && threadIdx.x == 0) {
        // Leaving early: poison this CTA's later tiles (DYN: the ones it has
        // claimed, then every claim up to its first one past the last tile,
        // which keeps the launch's claim count exact), and let its copies in
        // flight land before the shared memory goes away (bounded waits).
        for (uint32_t j = fail_at + 1; j < (DYN ? issued : count); ++j) {
            const uint32_t tt = DYN ? s_tile[j % STAGES] : rank + j * G;
            if (tt != kNoTile && (int64_t)tt != ctx.fault_tile)
                st_relaxed_u64(ctx.desc + tt, pack_desc(epoch, kStatePoison, 0u));
        }
        if (DYN)
            for (uint32_t tt = claim_next(); tt != kNoTile; tt = claim_next())
                if ((int64_t)tt != ctx.fault_tile) st_relaxed_u64(ctx.desc + tt, pack_desc(epoch, kStatePoison, 0u));
        for (uint32_t j = consumed; j < issued; ++j)
            if (!DYN || s_tile[j % STAGES] != kNoTile)
                mbar_wait_bounded(&bars[j % STAGES], (j / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
}

// Lean form: one CTA-wide barrier per iteration.
//  - Tile k+1's aggregate is formed without a barrier: each warp writes its
//    total to shared memory and bumps an arrival counter; the warp that
//    arrives last adds the totals up and publishes the aggregate.
//  - Warp 0 issues the first window of tile k's look-back before its own row
//    scan and consumes it afterwards, so that round trip overlaps the scan.
//  - The iteration's one barrier both hands warp 0's prefix to everyone and
//    tells the producer that tile k's stage has been read.
// Warp totals rotate through three slots and prefixes through two, so no
// slot is rewritten while a slower warp may still read it.
template <typename T, bool INCLUSIVE, int THREADS, int VPT, int STAGES, int K, bool TRACE>
__global__ void __launch_bounds__(THREADS, 1)
k_scan_lookback_lean(const T* in, T* out, size_t n, uint32_t num_tiles, LookbackCtx ctx,
                     const T* carry_in, T* carry_out, unsigned long long* trace) {
    static_assert(STAGES >= 3, "tile k stays in the ring while tile k+1 is summed");
    constexpr int WARPS = THREADS / 32;
    constexpr uint32_t TILE = (uint32_t)THREADS * VPT * 4;
    constexpr uint32_t TILE_BYTES = TILE * (uint32_t)sizeof(T);
    constexpr uint32_t SEG = 32u * VPT * 4;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    T* ring = reinterpret_cast<T*>(smem_raw);
    __shared__ __align__(8) uint64_t bars[STAGES];
    __shared__ T s_warp[3][WARPS];
    __shared__ T s_agg[3];
    __shared__ uint32_t s_arrive[3];
    __shared__ T s_prefix[2];
    __shared__ uint32_t s_fail[2];
    __shared__ uint32_t s_abort, s_rank, s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t G = gridDim.x;
    const uint64_t policy = policy_evict_first();

    if (threadIdx.x == 0) {
        uint32_t rank, epoch;
        claim_tile(ctx.counter, G, &rank, &epoch);
        s_rank = rank;
        s_epoch = epoch;
        s_abort = 0;
        for (int i = 0; i < 3; ++i) s_arrive[i] = 0;
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

    auto issue = [&](uint32_t k) {
        const int s = (int)(k % STAGES);
        const size_t base = (size_t)(rank + k * G) * TILE;
        if (base + TILE <= n) {
            fence_async_shared();
            mbar_arrive_expect_tx(&bars[s], TILE_BYTES);
            bulk_load(ring + (size_t)s * TILE, in + base, TILE_BYTES, &bars[s], policy);
        } else {
            mbar_arrive(&bars[s]);
        }
        issued = k + 1;
    };
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
    // Waits for tile k and sums it; the last warp to finish publishes the
    // aggregate.  A wait that runs out raises s_abort (seen after the barrier).
    auto reduce_publish = [&](uint32_t k) {
        const uint32_t t = rank + k * G;
        const int slot = (int)(k % 3);
        if (TRACE && threadIdx.x == 0) trace[(size_t)t * kTraceWords] = globaltimer_ns();
        if (!mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns)) {
            s_abort = 1u;
            record_error(ctx.status, kErrBulkTimeout, t);
        }
        T v[VPT][4];
        read_rows(k, v);
        T x = T(0);
#pragma unroll
        for (int j = 0; j < VPT; ++j) x += ((v[j][0] + v[j][1]) + v[j][2]) + v[j][3];
        x = warp_sum(x);
        if (lane == 0) {
            s_warp[slot][warp] = x;
            __threadfence_block();
            if (atomicAdd(&s_arrive[slot], 1u) == (uint32_t)WARPS - 1u) {
                __threadfence_block();
                T agg = T(0);
#pragma unroll
                for (int w = 0; w < WARPS; ++w) agg += *reinterpret_cast<volatile T*>(&s_warp[slot][w]);
                s_agg[slot] = agg;
                s_arrive[slot] = 0u;
                if ((int64_t)t != ctx.fault_tile) {
                    if (t == 0) {
                        if (num_tiles > 1)
                            st_relaxed_u64(ctx.desc, pack_desc(epoch, kStateP,
                                                               to_bits<T>((carry_in ? *carry_in : T(0)) + agg)));
                    } else {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateA, to_bits<T>(agg)));
                    }
                }
                if (TRACE) trace[(size_t)t * kTraceWords + 1] = trace[(size_t)t * kTraceWords + 2] = globaltimer_ns();
            }
        }
        compiler_fence();  // a publish by this warp stays ahead of its look-back
    };

    if (threadIdx.x == 0)
        for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);
    if (count > 0) reduce_publish(0);
    __syncthreads();  // tile 0's aggregate and warp totals are visible

    T prev_incl = T(0);  // warp 0
    uint32_t k = 0;
    bool failed = s_abort != 0u;
    for (; !failed && k < count; ++k) {
        const uint32_t t = rank + k * G;
        if (k + 1 < count) reduce_publish(k + 1);

        LookbackWindow<K> win;
        const T agg = s_agg[k % 3];  // formed in the previous iteration, visible since its barrier
        const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
        const int64_t floor = k > 0 ? (int64_t)t - (int64_t)G : -1;
        if (warp == 0 && t != 0 && !dead) win = lookback_prefetch<T, K>(ctx, t, epoch, lane, floor, prev_incl);

        T v[VPT][4];
        read_rows(k, v);
        T pre[VPT];
        warp_rows_scan<T, VPT>(v, lane, pre);

        if (warp == 0) {
            LookbackStats stats{0u, 0u};
            T excl = T(0);
            bool lb_failed = false;
            if (t == 0) {
                excl = carry_in ? *carry_in : T(0);
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;
            } else {
                excl = lookback<T, K, TRACE>(ctx, t, epoch, lane, &lb_failed, &stats, floor, prev_incl, &win);
                if (lane == 0) {
                    if (!lb_failed) {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, to_bits<T>(excl + agg)));
                    } else {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
                        record_error(ctx.status, kErrLookbackTimeout, t);
                    }
                }
            }
            prev_incl = excl + agg;
            if (lane == 0) {
                s_prefix[k & 1] = excl;
                s_fail[k & 1] = lb_failed ? 1u : 0u;
                if (TRACE) {
                    unsigned long long* rec = trace + (size_t)t * kTraceWords;
                    rec[3] = globaltimer_ns();
                    rec[5] = stats.windows;
                    rec[6] = stats.waits;
                    rec[7] = (unsigned long long)sm_id() | ((unsigned long long)blockIdx.x << 32);
                }
            }
        }
        __syncthreads();  // the prefix is out; tile k's stage has been read by everyone
        if (threadIdx.x == 0) {
            consumed = k + 1;
            if (k + STAGES < count) issue(k + STAGES);
        }
        if (s_abort != 0u || s_fail[k & 1] != 0u) {
            failed = true;
            break;
        }
        T wp = T(0);
#pragma unroll
        for (int w = 0; w < WARPS; ++w)
            if (w < warp) wp += s_warp[k % 3][w];
        const size_t tile_base = (size_t)t * TILE;
        rows_output_inplace<T, VPT, INCLUSIVE>(v, pre, s_prefix[k & 1] + wp);
        store_rows<T, VPT>(out, n, tile_base + (size_t)warp * SEG, lane, tile_base + TILE <= n, v);
        if (carry_out != nullptr && t == num_tiles - 1 && threadIdx.x == 0) *carry_out = s_prefix[k & 1] + agg;
        if (TRACE && threadIdx.x == 0) trace[(size_t)t * kTraceWords + 4] = globaltimer_ns();
    }

    if (failed && threadIdx.x == 0) {
        for (uint32_t j = k + 1; j < count; ++j) {
            const uint32_t tt = rank + j * G;
            if ((int64_t)tt != ctx.fault_tile) st_relaxed_u64(ctx.desc + tt, pack_desc(epoch, kStatePoison, 0u));
        }
        for (uint32_t j = consumed; j < issued; ++j)
            mbar_wait_bounded(&bars[j % STAGES], (j / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
}

template <typename T, bool INCL, int THREADS, int VPT, int STAGES, int K, bool TRACE, bool SB = false,
          bool LEAN = false, bool DYN = false>
static cudaError_t launch_pipe(const void* in, void* out, size_t n, const LookbackWs& ws,
                               const void* carry_in, void* carry_out, unsigned long long* trace,
                               cudaStream_t s) {
    constexpr size_t TILE = (size_t)THREADS * VPT * 4;
    constexpr size_t SMEM = (size_t)STAGES * TILE * sizeof(T);
    auto kern = [] {
        if constexpr (LEAN) return k_scan_lookback_lean<T, INCL, THREADS, VPT, STAGES, K, TRACE>;
        else if constexpr (SB) return k_scan_lookback_pipe_sb<T, INCL, THREADS, VPT, STAGES, K, TRACE, DYN>;
        else return k_scan_lookback_pipe<T, INCL, THREADS, VPT, STAGES, K, TRACE>;
    }();
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
static cudaError_t dispatch_pipe(int config, const void* in, void* out, size_t n, const LookbackWs& ws,
                                 const void* ci, void* co, unsigned long long* tr, cudaStream_t s) {
    switch (config) {  // the persistent rows of the configuration table (scan.cu)
        case 3: return launch_pipe<T, INCL, 512, 8, 3, 1, TRACE, true>(in, out, n, ws, ci, co, tr, s);
        case 4: return launch_pipe<T, INCL, 512, 4, 3, 1, TRACE>(in, out, n, ws, ci, co, tr, s);
        case 6: return launch_pipe<T, INCL, 512, 8, 3, 1, TRACE, false, true>(in, out, n, ws, ci, co, tr, s);
        case 7:  // the double register buffer spills for fp32 exclusive; that case takes the
                 // single-buffer kernel with the same 16384-element tiles (and a third stage)
            if constexpr (std::is_same<T, float>::value && !INCL)
                return launch_pipe<T, INCL, 512, 8, 3, 1, TRACE, true>(in, out, n, ws, ci, co, tr, s);
            else
                return launch_pipe<T, INCL, 512, 8, 2, 1, TRACE>(in, out, n, ws, ci, co, tr, s);
        case 8:  // 18432-element tiles claimed one at a time from the counter
            return launch_pipe<T, INCL, 512, 9, 3, 1, TRACE, true, false, true>(in, out, n, ws, ci, co, tr, s);
        case 9:  // the same with 16384-element tiles
            return launch_pipe<T, INCL, 512, 8, 3, 1, TRACE, true, false, true>(in, out, n, ws, ci, co, tr, s);
        default:  // 2: single register buffer, 18432-element tiles, three 72 KB stages
            return launch_pipe<T, INCL, 512, 9, 3, 1, TRACE, true>(in, out, n, ws, ci, co, tr, s);
    }
}

cudaError_t launch_scan_lookback_pipe(Dtype dt, bool inclusive, int config, const void* in, void* out,
                                      size_t n, const LookbackWs& ws, const void* carry_in,
                                      void* carry_out, cudaStream_t s) {
    if (dt == Dtype::F32)
        return inclusive ? dispatch_pipe<float, true, false>(config, in, out, n, ws, carry_in, carry_out, nullptr, s)
                         : dispatch_pipe<float, false, false>(config, in, out, n, ws, carry_in, carry_out, nullptr, s);
    return inclusive ? dispatch_pipe<uint32_t, true, false>(config, in, out, n, ws, carry_in, carry_out, nullptr, s)
                     : dispatch_pipe<uint32_t, false, false>(config, in, out, n, ws, carry_in, carry_out, nullptr, s);
}

cudaError_t launch_scan_trace_pipe(int config, const void* in, void* out, size_t n, const LookbackWs& ws,
                                   unsigned long long* trace, cudaStream_t s) {
    return dispatch_pipe<uint32_t, false, true>(config, in, out, n, ws, nullptr, nullptr, trace, s);
}

}  // namespace ss
