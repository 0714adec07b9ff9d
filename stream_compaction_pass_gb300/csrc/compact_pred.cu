// compact_pred.cu -- order-preserving compaction under a built-in predicate
// (keep keys[i] where keys[i] > 0 in its element type; no flag array).
// "Prefix sum and other parallel patterns", Stream compaction: compact.cu
// keeps v > 0; Exercise 1 fuses the flag pass into the compaction.
//
// A persistent CTA per SM takes a rank from the workspace counter and owns
// tiles rank, rank + G, ... (16384 keys each), which a three-stage
// shared-memory ring receives by bulk copies.  The CTA has 16 compute warps
// and one look-back warp:
//  - compute warps, iteration k: count the kept keys of tile k+1 (each warp
//    its own segment, no barrier: the last warp to finish adds the counts up
//    and publishes the tile's aggregate, one iteration early) and hand it to
//    the look-back warp; rank tile k's kept keys (per-row keep masks, the
//    rows' counts packed one byte per row and scanned across the warp, popc
//    inside a vector); take tile k's offsets from the look-back warp;
//    scatter.
//  - look-back warp: for each tile, as soon as it is handed over, walks the
//    predecessors' descriptors (no further than this CTA's previous tile),
//    publishes the inclusive count, and works out each warp's output
//    offset.  That is an iteration before the compute warps need them, so
//    the look-back's L2 round trips run beside their work instead of in
//    front of a barrier.
//  - scatter: a warp's kept keys form one contiguous run of the output.  Each
//    warp writes them, half a segment at a time, into its own staging area
//    at the output's 16-byte phase, then stores the run as aligned 16-byte
//    vectors (partial vectors at the two ends element by element).  Every
//    store instruction of a warp then covers 512 contiguous bytes, instead
//    of one 4-byte slot in every 16 bytes.
//  - sparse scatter: in a tile keeping fewer than 256 keys, none of whose
//    lanes keeps more than four, each lane reads only its kept keys from the
//    stage (before it is released) with their ranks, and stores them one by
//    one once the offsets are in.
// Named barriers hand each tile to the look-back warp and its offsets back.
// Each has two ids, by tile parity; each side must pass the other's barrier
// of tile k before it can arrive at the barrier of tile k + 2 with the same
// id, so neither side laps the other.
#include "bulk.cuh"
#include "internal.h"
#include "keep.cuh"
#include "tile.cuh"

namespace ss {

namespace {

constexpr int kPredComputeWarps = 16;
constexpr int kPredComputeThreads = kPredComputeWarps * 32;  // 512
constexpr int kPredThreads = kPredComputeThreads + 32;       // + the look-back warp
constexpr int kPredVpt = 8;                                  // 16-byte key vectors per lane per tile
constexpr int kPredStages = 3;
constexpr int kPredLookbackK = 1;  // descriptors per lane per look-back round
constexpr int kPredSlots = 4;      // sparse form: the most kept keys a lane may hold in a tile
// ... and fewer than this many in the tile.  Measured at n = 2^28 (ms): keep
// rate 0.001, sparse 0.240 against 0.267; 0.01 (164 keys a tile), 0.251
// against 0.272; 0.03 (492), 0.290 against 0.282.
constexpr uint32_t kPredSparseBelow = 256;
constexpr uint32_t kPredTile = (uint32_t)kPredComputeThreads * kPredVpt * 4;  // 16384
constexpr uint32_t kPredStageBytes = kPredTile * 4;
constexpr uint32_t kPredHalf = 32u * kPredVpt * 2;  // keys per staging pass: 4 rows of a warp segment
constexpr uint32_t kPredStgWords = kPredHalf + 4;   // + up to 3 words of phase, rounded to 16 bytes
constexpr size_t kPredSmem = (size_t)kPredStages * kPredStageBytes + (size_t)kPredComputeWarps * kPredStgWords * 4;
static_assert(kPredTile >= kCompactTile, "descriptors are sized for kCompactTile-element tiles");

// Named barriers (id 0 is __syncthreads).
constexpr uint32_t kBarCompute = 1;  // compute warps only
constexpr uint32_t kBarAgg = 2;      // + tile parity: the aggregate is in shared memory
constexpr uint32_t kBarPre = 4;      // + tile parity: the prefix is in shared memory

__device__ __forceinline__ void bar_sync_n(uint32_t id, uint32_t threads) {
    asm volatile("barrier.cta.sync.aligned %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void bar_arrive_n(uint32_t id, uint32_t threads) {
    asm volatile("barrier.cta.arrive.aligned %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void st_global_v4(uint32_t* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t vec_elem(const uint4& v, int s) {
    return s == 0 ? v.x : s == 1 ? v.y : s == 2 ? v.z : v.w;
}

// r[j] for a j known only at run time (0..7), by selects rather than a
// local-memory array.
__device__ __forceinline__ uint32_t select8(const uint32_t (&r)[8], uint32_t j) {
    const bool o = (j & 1u) != 0;
    const uint32_t a = o ? r[1] : r[0], b = o ? r[3] : r[2], c = o ? r[5] : r[4], d = o ? r[7] : r[6];
    const uint32_t ab = (j & 2u) ? b : a, cd = (j & 2u) ? d : c;
    return (j & 4u) ? cd : ab;
}

__device__ __forceinline__ uint32_t lds_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(smem_u32(p)) : "memory");
    return r;
}

}  // namespace

template <KeepRule RULE>
__global__ void __launch_bounds__(kPredThreads, 1)
k_compact_pred(const uint32_t* keys, uint32_t* out, unsigned long long* d_count, size_t n, uint32_t num_tiles,
               LookbackCtx ctx) {
    constexpr int VPT = kPredVpt;
    constexpr int STAGES = kPredStages;
    constexpr int CW = kPredComputeWarps;
    constexpr uint32_t CT = kPredComputeThreads;
    constexpr uint32_t ALL = kPredThreads;
    constexpr uint32_t TILE = kPredTile;
    constexpr uint32_t SEG = 32u * VPT * 4;  // keys per warp segment
    static_assert(VPT == 8, "two packed count words of four rows, one staging pass each");

    extern __shared__ __align__(128) unsigned char smem_raw[];  // ring, then the staging areas
    __shared__ __align__(8) uint64_t bars[STAGES];
    // By tile parity: the warps' counts; the counting warps' arrival tally and
    // timeout bits (reset by the last of them); the aggregate and the stop
    // flag (written once per tile by the last counting warp); each warp's
    // output offset, prefix included, and the look-back's failure flag
    // (written by the look-back warp).
    __shared__ uint32_t s_wsum[2][CW], s_base[2][CW];
    __shared__ uint32_t s_arrive[2], s_bad[2], s_agg[2], s_stop[2], s_fail[2], s_rank, s_epoch;
    // By tile parity: a counting warp had a lane keeping more than kPredSlots
    // keys (reset by the last of them), and the tile's form from that.
    __shared__ uint32_t s_crowded[2], s_sparse[2];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t G = gridDim.x;

    if (threadIdx.x == 0) {
        uint32_t rank, epoch;
        claim_tile(ctx.counter, G, &rank, &epoch);  // one claim per CTA; the last resets the counter
        s_rank = rank;
        s_epoch = epoch;
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_async_shared();
        for (int q = 0; q < 2; ++q) s_arrive[q] = s_bad[q] = s_stop[q] = s_fail[q] = s_crowded[q] = s_sparse[q] = 0u;
    }
    __syncthreads();
    const uint32_t rank = s_rank;
    const uint32_t epoch = s_epoch;
    if (rank >= G) {
        if (threadIdx.x == 0) record_error(ctx.status, kErrCounter, rank);
        return;
    }
    const uint32_t count = rank < num_tiles ? (num_tiles - rank + G - 1) / G : 0;

    if (warp == CW) {
        // ---- look-back warp ----
        uint32_t prev_incl = 0;  // inclusive count through this CTA's previous tile
        for (uint32_t k = 0; k < count; ++k) {
            const uint32_t t = rank + k * G;
            bar_sync_n(kBarAgg + (k & 1), ALL);
            if (s_stop[k & 1]) break;  // tile k's copy never arrived: the compute warps stop before its scatter
            const uint32_t agg = s_agg[k & 1];
            const uint32_t wc = lane < CW ? s_wsum[k & 1][lane] : 0u;
            const uint32_t wexcl = warp_inclusive_scan<uint32_t>(wc, lane) - wc;  // warp offsets inside the tile
            uint32_t excl = 0;
            bool lb_failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;  // it publishes nothing, so its successors' waits run out
            } else {
                const int64_t floor = k > 0 ? (int64_t)t - (int64_t)G : -1;
                excl = lookback<uint32_t, kPredLookbackK>(ctx, t, epoch, lane, &lb_failed, nullptr, floor, prev_incl);
                if (lane == 0) {
                    if (!lb_failed) {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, excl + agg));
                    } else {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
                        record_error(ctx.status, kErrLookbackTimeout, t);
                    }
                }
            }
            prev_incl = excl + agg;
            if (lane < CW) s_base[k & 1][lane] = excl + wexcl;
            if (lane == 0) {
                s_fail[k & 1] = lb_failed ? 1u : 0u;
                if (!lb_failed && t == num_tiles - 1) *d_count = (unsigned long long)excl + agg;
            }
            bar_arrive_n(kBarPre + (k & 1), ALL);
            if (lb_failed) {
                // The compute warps stop after this tile; they handed over
                // the next tile before they waited for this one's offsets.
                // Take that arrival, then leave.
                if (k + 1 < count) bar_sync_n(kBarAgg + ((k + 1) & 1), ALL);
                break;
            }
        }
        return;
    }

    // ---- compute warps ----
    const uint64_t policy = policy_evict_first();
    uint32_t issued = 0, consumed = 0;  // thread 0
    unsigned char* const ring = smem_raw;
    uint32_t* const stg = reinterpret_cast<uint32_t*>(smem_raw + (size_t)STAGES * kPredStageBytes) +
                          (size_t)warp * kPredStgWords;

    auto full = [&](uint32_t k) { return (size_t)(rank + k * G) * TILE + TILE <= n; };
    auto issue = [&](uint32_t k) {  // thread 0
        const int s = (int)(k % STAGES);
        if (full(k)) {
            fence_async_shared();
            mbar_arrive_expect_tx(&bars[s], kPredStageBytes);
            bulk_load(ring + (size_t)s * kPredStageBytes, keys + (size_t)(rank + k * G) * TILE, kPredStageBytes,
                      &bars[s], policy);
        } else {
            mbar_arrive(&bars[s]);  // ragged last tile: read from global with bounds checks
        }
        issued = k + 1;
    };
    // This lane's keys of tile k and their keep masks (bit e of m[j]: element e
    // of row j is kept).  Row j of a lane is the 16-byte vector j * 32 + lane
    // of its warp's segment.
    auto load_tile = [&](uint32_t k, uint32_t (&key)[VPT][4], uint32_t (&m)[VPT]) {
        const size_t seg = (size_t)(rank + k * G) * TILE + (size_t)warp * SEG;
        if (full(k)) {
            const unsigned char* kb =
                ring + (size_t)(k % STAGES) * kPredStageBytes + ((size_t)warp * SEG + (size_t)lane * 4) * 4;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const uint4 r = lds_vec(kb + 512 * j);
                key[j][0] = r.x;
                key[j][1] = r.y;
                key[j][2] = r.z;
                key[j][3] = r.w;
                m[j] = keep_mask4<RULE>(key[j]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                m[j] = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const size_t i = seg + (size_t)(32 * j + lane) * 4 + e;
                    key[j][e] = i < n ? keys[i] : 0u;
                    if (i < n && keep_bits<RULE>(key[j][e])) m[j] |= 1u << e;
                }
            }
        }
    };
    // The lane's key vectors of tile k that hold a kept key (rows with none
    // are left unread), given the masks from its count.
    auto load_kept = [&](uint32_t k, const uint32_t (&m)[VPT], uint32_t (&key)[VPT][4]) {
        const size_t seg = (size_t)(rank + k * G) * TILE + (size_t)warp * SEG;
        if (full(k)) {
            const unsigned char* kb =
                ring + (size_t)(k % STAGES) * kPredStageBytes + ((size_t)warp * SEG + (size_t)lane * 4) * 4;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                uint4 r = make_uint4(0u, 0u, 0u, 0u);
                if (m[j]) r = lds_vec(kb + 512 * j);
                key[j][0] = r.x;
                key[j][1] = r.y;
                key[j][2] = r.z;
                key[j][3] = r.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < VPT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const size_t i = seg + (size_t)(32 * j + lane) * 4 + e;
                    key[j][e] = ((m[j] >> e) & 1u) ? keys[i] : 0u;
                }
        }
    };
    // Waits for tile k and counts this warp's kept keys.  The last warp to
    // finish adds the counts up and publishes the tile's aggregate (or, if a
    // warp's copy wait ran out, publishes nothing and sets the tile's stop
    // flag).  No barrier: the warps meet through an arrival tally in shared
    // memory.
    auto count_tile = [&](uint32_t k, uint32_t (&m)[VPT]) {
        const uint32_t t = rank + k * G;
        const int par = (int)(k & 1);
        const bool ok = __all_sync(kFullMask, mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u,
                                                                ctx.max_polls, ctx.timeout_ns));
        uint32_t c = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) m[j] = 0u;
        if (ok) {
            uint32_t key[VPT][4];
            load_tile(k, key, m);
#pragma unroll
            for (int j = 0; j < VPT; ++j) c += (uint32_t)__popc(m[j]);
        }
        const bool crowded = __reduce_max_sync(kFullMask, c) > (uint32_t)kPredSlots;
        c = warp_sum(c);
        uint32_t last = 0;
        if (lane == 0) {
            s_wsum[par][warp] = c;
            if (crowded) atomicOr(&s_crowded[par], 1u);
            if (!ok) {
                atomicOr(&s_bad[par], 1u);
                record_error(ctx.status, kErrBulkTimeout, t);
            }
            __threadfence_block();  // the count (and bit) before the tally
            last = atomicAdd(&s_arrive[par], 1u) == (uint32_t)(CW - 1) ? 1u : 0u;
        }
        last = __shfl_sync(kFullMask, last, 0);
        if (last) {
            __syncwarp();
            __threadfence_block();  // every warp's count after the tally
            const uint32_t w = lane < CW ? *(volatile uint32_t*)&s_wsum[par][lane] : 0u;
            const uint32_t agg = warp_sum(w);
            if (lane == 0) {
                const uint32_t bad = *(volatile uint32_t*)&s_bad[par];
                if (!bad && (int64_t)t != ctx.fault_tile) {
                    if (t == 0) {
                        if (num_tiles > 1) st_relaxed_u64(ctx.desc, pack_desc(epoch, kStateP, agg));
                    } else {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateA, agg));
                    }
                }
                s_agg[par] = agg;
                s_stop[par] = bad;
                s_sparse[par] = (!*(volatile uint32_t*)&s_crowded[par] && agg < kPredSparseBelow) ? 1u : 0u;
                s_crowded[par] = 0u;
                s_bad[par] = 0u;
                s_arrive[par] = 0u;
            }
        }
    };
    // Writes this warp's kept keys of tile k, already ranked: row_run[j] is
    // the position of the lane's first kept key of row j in the warp's run,
    // c0 the count of rows 0..3, `start` the run's first output index.  Two
    // passes of four rows through the staging area; in each, key number i of
    // the pass goes to staging word i + a, where a puts the words at the
    // 16-byte phase of their output slots, so every full 16-byte vector of
    // the staging area is one aligned vector of the output.
    auto scatter = [&](const uint32_t (&key)[VPT][4], const uint32_t (&m)[VPT], const uint32_t (&row_run)[VPT],
                       uint32_t c0, uint32_t c_all, uint32_t start) {
        const uint32_t out_phase = (uint32_t)(reinterpret_cast<uintptr_t>(out) >> 2) & 3u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t first = h == 0 ? 0u : c0;                 // run position where the pass starts
            const uint32_t cnt = h == 0 ? c0 : c_all - c0;           // keys in the pass (warp-uniform)
            const size_t d0 = (size_t)start + first;                 // output index of the pass's first key
            const uint32_t a = (uint32_t)(d0 + out_phase) & 3u;      // its 16-byte phase, in words
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = 4 * h + q;
                const uint32_t base = row_run[j] - first + a;
                const uint32_t mj = m[j];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t idx = base + (uint32_t)__popc(mj & ((1u << e) - 1u));
                    if ((mj >> e) & 1u) stg[idx] = key[j][e];
                }
            }
            __syncwarp();
            const uint32_t tot = a + cnt;          // staging words in use, from word a
            uint32_t* const gbase = out + d0 - a;  // output slot of staging word 0 (16-byte aligned)
            for (uint32_t v = (uint32_t)lane; 4 * v < tot; v += 32) {
                const uint4 x = lds_vec(stg + 4 * v);
                if (4 * v >= a && 4 * v + 4 <= tot) {
                    st_global_v4(gbase + 4 * v, x);
                } else {
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint32_t w = 4 * v + (uint32_t)s;
                        if (w >= a && w < tot) gbase[w] = vec_elem(x, s);
                    }
                }
            }
            __syncwarp();  // the area is read before the next pass writes it
        }
    };

    if (threadIdx.x == 0)
        for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);

    bool failed = false;
    uint32_t poison_from = 0;  // first of this CTA's tiles (by k) left for thread 0 to poison on failure
    uint32_t m_cur[VPT], m_next[VPT];  // keep masks of tiles k and k+1, from their counts
#pragma unroll
    for (int j = 0; j < VPT; ++j) m_cur[j] = m_next[j] = 0u;
    if (count > 0) {
        count_tile(0, m_cur);
        bar_arrive_n(kBarAgg, ALL);  // tile 0 to the look-back warp
    }
    bar_sync_n(kBarCompute, CT);  // tile 0's stop flag is in shared memory
    if (count > 0 && s_stop[0]) {  // tile 0's copy did not arrive
        failed = true;
        poison_from = 0;
    }

    for (uint32_t k = 0; !failed && k < count; ++k) {
        if (k + 1 < count) {  // count tile k+1 and hand it to the look-back warp
            count_tile(k + 1, m_next);
            bar_arrive_n(kBarAgg + ((k + 1) & 1), ALL);
        }

        // Rank tile k's kept keys (masks from its count).
        uint32_t key[VPT][4], m[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) m[j] = m_cur[j];
        uint32_t row_run[VPT];
        uint32_t run = 0, c0 = 0;
#pragma unroll
        for (int w = 0; w < VPT / 4; ++w) {
            uint32_t packed = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) packed |= (uint32_t)__popc(m[4 * w + q]) << (8 * q);
            const uint32_t inc = warp_inclusive_scan<uint32_t>(packed, lane);
            const uint32_t exc = inc - packed;  // bytewise, no borrows (each byte <= 128)
            const uint32_t rows = __shfl_sync(kFullMask, inc, 31);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                row_run[4 * w + q] = run + ((exc >> (8 * q)) & 0xffu);
                run += (rows >> (8 * q)) & 0xffu;
            }
            if (w == 0) c0 = run;
        }
        // Sparse form, when the tile keeps fewer than kPredSparseBelow keys and
        // no lane more than kPredSlots (a tile-wide choice, made by its count:
        // a tile is as slow as its slowest warp): each lane reads just its kept keys from the stage now,
        // before the stage is released, with their positions in the warp's
        // run, and stores them once the run's offset is known.  Otherwise the
        // vectors holding a kept key are read again for the staged scatter.
        uint32_t packed = 0;  // bit 4j + e: element e of row j is kept
#pragma unroll
        for (int j = 0; j < VPT; ++j) packed |= m[j] << (4 * j);
        const uint32_t kept = (uint32_t)__popc(packed);
        const bool sparse = s_sparse[k & 1] != 0;
        uint32_t sp_key[kPredSlots], sp_pos[kPredSlots];
        if (sparse) {
            const size_t seg = (size_t)(rank + k * G) * TILE + (size_t)warp * SEG;
            const unsigned char* kb = ring + (size_t)(k % STAGES) * kPredStageBytes + (size_t)warp * SEG * 4;
            uint32_t rest = packed;
#pragma unroll
            for (int r = 0; r < kPredSlots; ++r) {
                if (!__any_sync(kFullMask, rest != 0)) break;
                if (rest) {
                    const uint32_t b = (uint32_t)__ffs(rest) - 1u;  // row b/4, element b%4
                    rest &= rest - 1u;
                    const uint32_t j = b >> 2;
                    const uint32_t elem = 128u * j + 4u * (uint32_t)lane + (b & 3u);  // index in the segment
                    sp_pos[r] = select8(row_run, j) + (uint32_t)__popc(packed & ((1u << b) - 1u) & (0xfu << (b & ~3u)));
                    sp_key[r] = full(k) ? lds_u32(kb + 4u * elem) : keys[seg + elem];
                }
            }
        } else {
            load_kept(k, m, key);  // only vectors with a kept key are read again
        }

        bar_sync_n(kBarPre + (k & 1), ALL);  // tile k's offsets; every compute warp has read tile k
        const bool lb_failed = s_fail[k & 1] != 0;
        const uint32_t base = s_base[k & 1][warp];
        if (threadIdx.x == 0) {
            consumed = k + 1;
            const bool next_stops = k + 1 < count && s_stop[(k + 1) & 1] != 0;
            if (!lb_failed && !next_stops && k + STAGES < count) issue(k + STAGES);
        }
        const bool next_stops = k + 1 < count && s_stop[(k + 1) & 1] != 0;
        if (lb_failed) {  // the look-back warp poisoned tile k
            failed = true;
            poison_from = k + 1;
            break;
        }
        if (sparse) {
#pragma unroll
            for (int r = 0; r < kPredSlots; ++r) {
                if (!__any_sync(kFullMask, kept > (uint32_t)r)) break;
                if (kept > (uint32_t)r) out[(size_t)base + sp_pos[r]] = sp_key[r];
            }
        } else {
            scatter(key, m, row_run, c0, run, base);
        }
        if (next_stops) {  // tile k+1's copy did not arrive; the look-back warp stops there too
            failed = true;
            poison_from = k + 1;
            break;
        }
#pragma unroll
        for (int j2 = 0; j2 < VPT; ++j2) m_cur[j2] = m_next[j2];
    }

    if (failed && threadIdx.x == 0) {
        // Later tiles of this CTA publish nothing else: poison them so that
        // their successors stop at once, then wait for the copies in flight.
        for (uint32_t k = poison_from; k < count; ++k) {
            const uint32_t t = rank + k * G;
            if ((int64_t)t != ctx.fault_tile) st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
        }
        for (uint32_t k = consumed; k < issued; ++k)
            mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
}

template <KeepRule RULE>
static cudaError_t launch_pred(const uint32_t* keys, uint32_t* out, unsigned long long* d_count, size_t n,
                               const LookbackWs& ws, cudaStream_t s) {
    auto kern = k_compact_pred<RULE>;
    KernelSetup su;
    cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), kPredThreads, kPredSmem, &su);
    if (e != cudaSuccess) return e;
    const uint32_t tiles = (uint32_t)((n + kPredTile - 1) / kPredTile);
    const uint32_t grid = tiles < (uint32_t)su.sms ? tiles : (uint32_t)su.sms;
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    kern<<<grid, kPredThreads, kPredSmem, s>>>(keys, out, d_count, n, tiles, ctx);
    return cudaGetLastError();
}

cudaError_t launch_compact_pred(KeepRule rule, const uint32_t* keys, uint32_t* out, unsigned long long* d_count,
                                size_t n, const LookbackWs& ws, cudaStream_t s) {
    switch (rule) {
        case KeepRule::PositiveF32: return launch_pred<KeepRule::PositiveF32>(keys, out, d_count, n, ws, s);
        case KeepRule::PositiveI32: return launch_pred<KeepRule::PositiveI32>(keys, out, d_count, n, ws, s);
        case KeepRule::PositiveU32: return launch_pred<KeepRule::PositiveU32>(keys, out, d_count, n, ws, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ss
