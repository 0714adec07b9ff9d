// compact_pipe.cu -- the fused order-preserving compaction as a persistent
// kernel fed by the bulk-copy engine.
//
// Same result as compact.cu (keep keys[i] where flags[i] != 0, in order;
// "Prefix sum and other parallel patterns", Stream compaction and Exercise
// 1; the built-in predicates run in compact_pred.cu), on the schedule of
// the persistent scan (scan_pipe.cu): each CTA takes a rank from the
// workspace counter and handles tiles rank, rank + G, ...; a shared-memory
// ring receives each tile's keys and flags with two bulk copies (the keys
// alone under a predicate).  Iteration k:
//   1. count the kept elements of tile k+1 from its flags (or keys) and
//      publish that count one iteration early (the tile's aggregate);
//   2. warp 0 looks back for tile k, no further than this CTA's previous
//      tile, while the other warps rank tile k's kept keys in registers
//      (per-row keep masks; the rows' counts packed one byte per row and
//      scanned across the warp; popc of the mask below an element inside a
//      vector);
//   3. the stage is released and the next copy started;
//   4. the kept keys go from registers to their output slots: a warp row's
//      kept keys form one contiguous run of the output.
// The default, chunked kernel (below) turns a tile's flags into words of
// keep bits when it counts them, and then uses the rest of the tile's stage
// to gather each warp's kept keys for 16-byte stores; tiles with few kept
// keys skip that and load and store just those keys.
#include <atomic>
#include <type_traits>

#include "bulk.cuh"
#include "internal.h"
#include "keep.cuh"
#include "tile.cuh"

namespace ss {

namespace {

// Bit 7 of each byte of the result is set iff that byte of w is nonzero:
// adding 0x7f to the low seven bits of a byte carries into bit 7 iff they are
// not all zero (and never out of the byte), and OR-ing w adds the byte's own
// bit 7.  Four flags in five operations.
__device__ __forceinline__ uint32_t nonzero_byte_bits(uint32_t w) {
    return (((w & 0x7f7f7f7fu) + 0x7f7f7f7fu) | w) & 0x80808080u;
}
// The keep mask of four flag bytes: bit e set iff byte e is nonzero.  The
// multiply by 2^21 + 2^14 + 2^7 + 1 moves bits 7, 15, 23 and 31 to bits 28..31
// (no other partial product reaches those bits, and none overlap below them,
// so nothing carries in).
__device__ __forceinline__ uint32_t byte_keep_mask(uint32_t w) {
    return (nonzero_byte_bits(w) * 0x00204081u) >> 28;
}
// The keep bits of 32 consecutive flag bytes (lo: bytes 0..15, hi: 16..31),
// bit i for byte i.
__device__ __forceinline__ uint32_t keep_bits32(uint4 lo, uint4 hi) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t m = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) m |= ((nonzero_byte_bits(w[q]) * 0x00204081u) >> (28 - 4 * q)) & (0xfu << (4 * q));
    return m;
}

// A 16-byte key vector through the read-only path: no L1 allocation, and a
// 256-byte L2 fetch around the miss (neighbouring vectors are usually wanted
// too when the flags are dense).
__device__ __forceinline__ uint4 ld_key_vec(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// One key through the read-only path, without the wider L2 fetch: with
// sparse flags the neighbouring keys are rarely wanted.
__device__ __forceinline__ uint32_t ld_key_u32(const uint32_t* p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t lds_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(smem_u32(p)) : "memory");
    return r;
}

}  // namespace

template <int THREADS, int VPT, int STAGES, KeepRule RULE>
__global__ void __launch_bounds__(THREADS, 1)
k_compact_pipe(const uint32_t* keys, const uint8_t* flags, uint32_t* out, unsigned long long* d_count,
               size_t n, uint32_t num_tiles, LookbackCtx ctx) {
    static_assert(VPT % 4 == 0, "rows are packed four to a word");
    constexpr int WARPS = THREADS / 32;
    constexpr int NW = VPT / 4;  // packed count words per lane
    constexpr uint32_t TILE = (uint32_t)THREADS * VPT * 4;
    constexpr uint32_t KEY_BYTES = TILE * 4;
    constexpr bool FLAGS = RULE == KeepRule::Flags;
    constexpr uint32_t STAGE_BYTES = KEY_BYTES + (FLAGS ? TILE : 0u);  // keys, then flags
    constexpr uint32_t SEG = 32u * VPT * 4;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[STAGES];
    __shared__ uint32_t s_warp[WARPS];
    __shared__ uint32_t s_prefix[2], s_fail[2], s_rank, s_epoch;  // prefix/fail alternate by tile parity

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
    if (rank >= G) {
        if (threadIdx.x == 0) record_error(ctx.status, kErrCounter, rank);
        return;
    }
    const uint32_t count = rank < num_tiles ? (num_tiles - rank + G - 1) / G : 0;
    uint32_t issued = 0, consumed = 0;  // thread 0

    auto stage_keys = [&](uint32_t k) -> unsigned char* { return smem_raw + (size_t)(k % STAGES) * STAGE_BYTES; };
    auto issue = [&](uint32_t k) {  // thread 0
        const int s = (int)(k % STAGES);
        const size_t base = (size_t)(rank + k * G) * TILE;
        if (base + TILE <= n) {
            fence_async_shared();
            mbar_arrive_expect_tx(&bars[s], STAGE_BYTES);
            bulk_load(stage_keys(k), keys + base, KEY_BYTES, &bars[s], policy);
            if constexpr (FLAGS) bulk_load(stage_keys(k) + KEY_BYTES, flags + base, TILE, &bars[s], policy);
        } else {
            mbar_arrive(&bars[s]);  // ragged last tile: read from global
        }
        issued = k + 1;
    };
    // This lane's key vectors of tile k (full tiles only).
    auto read_keys = [&](uint32_t k, uint32_t (&key)[VPT][4]) {
        const unsigned char* kb = stage_keys(k) + ((size_t)warp * SEG + (size_t)lane * 4) * 4;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const uint4 r = lds_vec(kb + 512 * j);
            key[j][0] = r.x;
            key[j][1] = r.y;
            key[j][2] = r.z;
            key[j][3] = r.w;
        }
    };
    // Keep masks of this lane's rows of tile k (bit e of m[j]: element e of row j is kept).
    auto read_masks = [&](uint32_t k, uint32_t (&m)[VPT]) {
        const size_t tile_base = (size_t)(rank + k * G) * TILE;
        const size_t seg = tile_base + (size_t)warp * SEG;
        if (!FLAGS && tile_base + TILE <= n) {
            uint32_t key[VPT][4];
            read_keys(k, key);
#pragma unroll
            for (int j = 0; j < VPT; ++j) m[j] = keep_mask4<RULE>(key[j]);
        } else if (!FLAGS) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                m[j] = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const size_t i = seg + (size_t)(32 * j + lane) * 4 + e;
                    if (i < n && keep_bits<RULE>(keys[i])) m[j] |= 1u << e;
                }
            }
        } else if (tile_base + TILE <= n) {
            const unsigned char* f = stage_keys(k) + KEY_BYTES + (size_t)warp * SEG + (size_t)lane * 4;
#pragma unroll
            for (int j = 0; j < VPT; ++j) m[j] = byte_keep_mask(lds_u32(f + 128 * j));
        } else {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                m[j] = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const size_t i = seg + (size_t)(32 * j + lane) * 4 + e;
                    if (i < n && flags[i] != 0) m[j] |= 1u << e;
                }
            }
        }
    };
    // Waits for tile k, counts its kept elements and publishes the count.
    auto count_publish = [&](uint32_t k, uint32_t* wp, uint32_t* agg) -> bool {
        const uint32_t t = rank + k * G;
        const bool ok = mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) record_error(ctx.status, kErrBulkTimeout, t);
            return false;
        }
        uint32_t m[VPT];
        read_masks(k, m);
        uint32_t c = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) c += (uint32_t)__popc(m[j]);
        block_combine<uint32_t, WARPS>(warp_sum(c), warp, lane, s_warp, wp, agg);
        if (threadIdx.x == 0 && (int64_t)t != ctx.fault_tile) {
            if (t == 0) {
                if (num_tiles > 1) st_relaxed_u64(ctx.desc, pack_desc(epoch, kStateP, *agg));
            } else {
                st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateA, *agg));
            }
        }
        compiler_fence();  // the count just published stays ahead of the look-back
        return true;
    };

    uint32_t wp_cur = 0, agg_cur = 0, prev_incl = 0;
    bool failed = false;
    uint32_t fail_at = 0;
    if (threadIdx.x == 0)
        for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);
    if (count > 0 && !count_publish(0, &wp_cur, &agg_cur)) failed = true;

    for (uint32_t k = 0; !failed && k < count; ++k) {
        const uint32_t t = rank + k * G;
        uint32_t wp_next = 0, agg_next = 0;
        if (k + 1 < count && !count_publish(k + 1, &wp_next, &agg_next)) {
            failed = true;
            fail_at = k;
            break;
        }
        if (warp == 0) {
            uint32_t excl = 0;
            bool lb_failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;
            } else {
                const int64_t floor = k > 0 ? (int64_t)t - (int64_t)G : -1;
                excl = lookback<uint32_t, 1>(ctx, t, epoch, lane, &lb_failed, nullptr, floor, prev_incl);
                if (lane == 0) {
                    if (!lb_failed) {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, excl + agg_cur));
                    } else {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
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
        // Rank tile k's kept keys.
        const size_t tile_base = (size_t)t * TILE;
        const size_t seg = tile_base + (size_t)warp * SEG;
        uint32_t m[VPT];
        uint32_t key[VPT][4];
        if (!FLAGS && tile_base + TILE <= n) {
            read_keys(k, key);
#pragma unroll
            for (int j = 0; j < VPT; ++j) m[j] = keep_mask4<RULE>(key[j]);
        } else if (tile_base + TILE <= n) {
            read_masks(k, m);
            read_keys(k, key);
        } else {
            read_masks(k, m);
#pragma unroll
            for (int j = 0; j < VPT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const size_t i = seg + (size_t)(32 * j + lane) * 4 + e;
                    key[j][e] = ((m[j] >> e) & 1u) ? keys[i] : 0u;
                }
        }
        uint32_t row_base[VPT];
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            uint32_t packed = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) packed |= (uint32_t)__popc(m[4 * w + q]) << (8 * q);
            const uint32_t inc = warp_inclusive_scan<uint32_t>(packed, lane);
            const uint32_t exc = inc - packed;  // bytewise, no borrows (each byte <= 128)
            const uint32_t rows = __shfl_sync(kFullMask, inc, 31);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                row_base[4 * w + q] = run + ((exc >> (8 * q)) & 0xffu);
                run += (rows >> (8 * q)) & 0xffu;
            }
        }
        __syncthreads();  // tile k read by everyone; the prefix is in shared memory
        if (threadIdx.x == 0) {
            consumed = k + 1;
            if (k + STAGES < count) issue(k + STAGES);
        }
        if (s_fail[k & 1]) {
            failed = true;
            fail_at = k;
            break;
        }
        uint32_t* dst = out + (size_t)s_prefix[k & 1] + wp_cur;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            uint32_t pos = row_base[j];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if ((m[j] >> e) & 1u) dst[pos++] = key[j][e];
            }
        }
        if (t == num_tiles - 1 && threadIdx.x == 0) *d_count = (unsigned long long)s_prefix[k & 1] + agg_cur;
        wp_cur = wp_next;
        agg_cur = agg_next;
    }

    if (failed && threadIdx.x == 0) {
        for (uint32_t k = fail_at + 1; k < count; ++k) {
            const uint32_t t = rank + k * G;
            if ((int64_t)t != ctx.fault_tile) st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
        }
        for (uint32_t k = consumed; k < issued; ++k)
            mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
}

// Selective-load form: only the flags go through the bulk-copy ring (one
// byte per element); each thread loads a 16-byte key vector only when one of
// its four flags is set, one tile ahead, into a second register buffer.  With
// sparse flags most key sectors are never read (at p = 0.01 about 8 % of the
// 32-byte sectors hold a kept key); with dense flags it moves the same bytes
// as the bulk-copy form.
template <int THREADS, int VPT, int STAGES>
__global__ void __launch_bounds__(THREADS, 1)
k_compact_sel(const uint32_t* keys, const uint8_t* flags, uint32_t* out, unsigned long long* d_count,
              size_t n, uint32_t num_tiles, LookbackCtx ctx) {
    static_assert(VPT % 4 == 0, "rows are packed four to a word");
    static_assert(STAGES >= 2, "the ring needs two stages at least");
    constexpr int WARPS = THREADS / 32;
    constexpr int NW = VPT / 4;
    constexpr uint32_t TILE = (uint32_t)THREADS * VPT * 4;
    constexpr uint32_t SEG = 32u * VPT * 4;

    extern __shared__ __align__(128) unsigned char smem_raw[];  // STAGES x TILE flag bytes
    __shared__ __align__(8) uint64_t bars[STAGES];
    __shared__ uint32_t s_warp[WARPS];
    __shared__ uint32_t s_prefix[2], s_fail[2], s_rank, s_epoch;  // prefix/fail alternate by tile parity

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
    if (rank >= G) {
        if (threadIdx.x == 0) record_error(ctx.status, kErrCounter, rank);
        return;
    }
    const uint32_t count = rank < num_tiles ? (num_tiles - rank + G - 1) / G : 0;
    uint32_t issued = 0, consumed = 0;  // thread 0

    auto issue = [&](uint32_t k) {  // thread 0: flags of this CTA's k-th tile
        const int s = (int)(k % STAGES);
        const size_t base = (size_t)(rank + k * G) * TILE;
        if (base + TILE <= n) {
            fence_async_shared();
            mbar_arrive_expect_tx(&bars[s], TILE);
            bulk_load(smem_raw + (size_t)s * TILE, flags + base, TILE, &bars[s], policy);
        } else {
            mbar_arrive(&bars[s]);  // ragged last tile: flags read from global
        }
        issued = k + 1;
    };
    // Waits for tile k's flags; this lane's keep masks, the tile's count and
    // this warp's prefix; publishes the count; starts the loads of the key
    // vectors that hold a kept element.  False if the copy did not arrive.
    auto prepare = [&](uint32_t k, uint32_t (&m)[VPT], uint32_t (&key)[VPT][4], uint32_t* wp,
                       uint32_t* agg) -> bool {
        const uint32_t t = rank + k * G;
        const size_t tile_base = (size_t)t * TILE;
        const size_t seg = tile_base + (size_t)warp * SEG;
        const bool ok = mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) record_error(ctx.status, kErrBulkTimeout, t);
            return false;
        }
        const bool full = tile_base + TILE <= n;
        if (full) {
            const unsigned char* f = smem_raw + (size_t)(k % STAGES) * TILE + (size_t)warp * SEG + (size_t)lane * 4;
#pragma unroll
            for (int j = 0; j < VPT; ++j) m[j] = byte_keep_mask(lds_u32(f + 128 * j));
            const uint4* kp = reinterpret_cast<const uint4*>(keys + seg) + lane;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                uint4 r = make_uint4(0u, 0u, 0u, 0u);
                if (m[j]) r = ld_vec(kp + 32 * j);
                key[j][0] = r.x;
                key[j][1] = r.y;
                key[j][2] = r.z;
                key[j][3] = r.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                m[j] = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const size_t i = seg + (size_t)(32 * j + lane) * 4 + e;
                    const bool keep = i < n && flags[i] != 0;
                    key[j][e] = keep ? keys[i] : 0u;
                    m[j] |= keep ? (1u << e) : 0u;
                }
            }
        }
        uint32_t c = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) c += (uint32_t)__popc(m[j]);
        block_combine<uint32_t, WARPS>(warp_sum(c), warp, lane, s_warp, wp, agg);  // also frees the stage
        if (threadIdx.x == 0) {
            if ((int64_t)t != ctx.fault_tile) {
                if (t == 0) {
                    if (num_tiles > 1) st_relaxed_u64(ctx.desc, pack_desc(epoch, kStateP, *agg));
                } else {
                    st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateA, *agg));
                }
            }
            consumed = k + 1;
            if (k + STAGES < count) issue(k + STAGES);
        }
        compiler_fence();  // the count just published stays ahead of the look-back
        return true;
    };

    uint32_t wp_cur = 0, agg_cur = 0, prev_incl = 0;
    uint32_t fail_at = 0;

    // One iteration: prepare tile k+1 into (mn, kn), look back for tile k
    // and write tile k from (mc, kc).
    auto step = [&](uint32_t k, uint32_t (&mc)[VPT], uint32_t (&kc)[VPT][4], uint32_t (&mn)[VPT],
                    uint32_t (&kn)[VPT][4]) -> bool {
        const uint32_t t = rank + k * G;
        uint32_t wp_next = 0, agg_next = 0;
        if (k + 1 < count && !prepare(k + 1, mn, kn, &wp_next, &agg_next)) {
            fail_at = k;
            return false;
        }
        if (warp == 0) {
            uint32_t excl = 0;
            bool lb_failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;
            } else {
                const int64_t floor = k > 0 ? (int64_t)t - (int64_t)G : -1;
                excl = lookback<uint32_t, 1>(ctx, t, epoch, lane, &lb_failed, nullptr, floor, prev_incl);
                if (lane == 0) {
                    if (!lb_failed) {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, excl + agg_cur));
                    } else {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
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
        uint32_t row_base[VPT];
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            uint32_t packed = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) packed |= (uint32_t)__popc(mc[4 * w + q]) << (8 * q);
            const uint32_t inc = warp_inclusive_scan<uint32_t>(packed, lane);
            const uint32_t exc = inc - packed;  // bytewise, no borrows (each byte <= 128)
            const uint32_t rows = __shfl_sync(kFullMask, inc, 31);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                row_base[4 * w + q] = run + ((exc >> (8 * q)) & 0xffu);
                run += (rows >> (8 * q)) & 0xffu;
            }
        }
        __syncthreads();  // the prefix is in shared memory
        if (s_fail[k & 1]) {
            fail_at = k;
            return false;
        }
        uint32_t* dst = out + (size_t)s_prefix[k & 1] + wp_cur;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            uint32_t pos = row_base[j];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if ((mc[j] >> e) & 1u) dst[pos++] = kc[j][e];
            }
        }
        if (t == num_tiles - 1 && threadIdx.x == 0) *d_count = (unsigned long long)s_prefix[k & 1] + agg_cur;
        wp_cur = wp_next;
        agg_cur = agg_next;
        return true;
    };

    uint32_t ma[VPT], mb[VPT];
    uint32_t ka[VPT][4], kb[VPT][4];
    bool failed = false;
    if (threadIdx.x == 0)
        for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);
    if (count > 0 && !prepare(0, ma, ka, &wp_cur, &agg_cur)) failed = true;
    for (uint32_t k = 0; !failed && k < count; k += 2) {
        if (!step(k, ma, ka, mb, kb)) failed = true;
        else if (k + 1 < count && !step(k + 1, mb, kb, ma, ka)) failed = true;
    }

    if (failed && threadIdx.x == 0) {
        for (uint32_t k = fail_at + 1; k < count; ++k) {
            const uint32_t t = rank + k * G;
            if ((int64_t)t != ctx.fault_tile) st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
        }
        for (uint32_t k = consumed; k < issued; ++k)
            mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
}

// Chunked form: one look-back per tile of four chunks (a chunk: 1024
// elements per warp; 32768-element tiles for 256 threads, 65536 for 512).  With sparse flags the work per element is small and
// a tile's fixed costs dominate: the wait for its flags, the barriers, and
// the look-back round trips.  A tile four times larger pays them once for
// four times the elements.
//  - Only the flags go through the ring: three stages of 64 KB.
//  - Counting tile k+1: lane l of a warp reads elements 32l .. 32l+31 of
//    each of its 1024-element (chunk, warp) shares and turns them into one
//    word of keep bits.  After a barrier the words overwrite the first 8 KB
//    of the tile's stage (its flags are no longer needed), and warp 0 scans
//    the 64 (chunk, warp) counts into offsets inside the tile and publishes
//    the tile's total.
//  - Warp 0 then looks back for tile k.  After a barrier, every warp writes
//    its share of each chunk of tile k at
//    prefix + offset(chunk, warp) + rank inside the share, in one of two
//    forms chosen per tile by its count:
//      dense: each row of 128 elements takes its keep masks from the words;
//        key vectors with a kept element are loaded one chunk ahead, and a
//        row's kept keys go to one contiguous run of the output;
//      sparse (fewer than `sparse_below` kept keys): each lane loads its
//        first few kept keys of every chunk before the next tile is counted,
//        so they arrive during that count and the look-back; after the
//        look-back it stores them, consecutive, with plain stores.
//  - Counts and offsets alternate between two slots by tile parity.
template <int THREADS, int STAGES>
__global__ void __launch_bounds__(THREADS, THREADS >= 512 ? 1 : 2)
k_compact_chunked(const uint32_t* keys, const uint8_t* flags, uint32_t* out, unsigned long long* d_count,
                  size_t n, uint32_t num_tiles, LookbackCtx ctx, uint32_t sparse_below) {
    constexpr int WARPS = THREADS / 32;
    constexpr int VPT = 8;                                // rows (16-byte key vectors) per lane per chunk
    constexpr int NW = VPT / 4;                           // packed count words per lane
    constexpr uint32_t SEG = 32u * VPT * 4;               // 1024 elements per warp per chunk
    constexpr uint32_t CHUNK = SEG * WARPS;               // 16384
    constexpr int CHUNKS = 4;
    constexpr uint32_t TILE = CHUNK * CHUNKS;             // 65536
    constexpr int kSlots = 4;                             // sparse form: kept keys per lane and chunk loaded early
    constexpr uint32_t kWordBytes = 4u * CHUNKS * WARPS * 32u;   // keep words at the start of a counted stage
    constexpr uint32_t kStageWarpBytes = 4u * (4u * 128u + 4u);  // a warp's staging: four rows and a shift
    static_assert(kWordBytes + WARPS * kStageWarpBytes <= TILE, "words and staging fit a stage");
    static_assert(kStageWarpBytes % 16u == 0u && kWordBytes % 16u == 0u, "staging areas are 16-byte aligned");
    constexpr int CPL = CHUNKS * WARPS / 32;  // (chunk, warp) counts per lane of warp 0
    static_assert(CPL == 1 || CPL == 2, "one or two (chunk, warp) counts per lane of warp 0");
    static_assert(SEG == 32u * 32u, "a lane's share of a chunk is one word of keep bits");
    static_assert(2 * CHUNKS <= VPT && kSlots <= 4, "the sparse slots fit the dense registers");

    extern __shared__ __align__(128) unsigned char smem_raw[];  // STAGES x TILE flag bytes
    __shared__ __align__(8) uint64_t bars[STAGES];
    __shared__ uint32_t s_cnt[2][CHUNKS * WARPS];   // count, then exclusive offset, of (chunk, warp)
    __shared__ uint32_t s_total[2];
    __shared__ uint32_t s_prefix[2], s_fail[2], s_rank, s_epoch;

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

    auto issue = [&](uint32_t k) {  // thread 0: flags of this CTA's k-th tile
        const int s = (int)(k % STAGES);
        const size_t base = (size_t)(rank + k * G) * TILE;
        if (base + TILE <= n) {
            fence_async_shared();
            mbar_arrive_expect_tx(&bars[s], TILE);
            bulk_load(smem_raw + (size_t)s * TILE, flags + base, TILE, &bars[s], policy);
        } else {
            mbar_arrive(&bars[s]);  // ragged last tile: flags read from global
        }
        issued = k + 1;
    };
    // The keep word of lane ln's share of chunk c, for a tile whose count has
    // turned its stage's first 8 KB into words.
    auto word_at = [&](uint32_t k, int c, int ln) -> uint32_t {
        return lds_u32(smem_raw + (size_t)(k % STAGES) * TILE + 4u * ((uint32_t)(c * WARPS + warp) * 32u + (uint32_t)ln));
    };
    // Keep masks of this lane's rows of chunk c: row j's four elements at lane
    // l are elements 128j + 4l .. 128j + 4l + 3 of the share, bits 4(l mod 8)
    // .. of the word of lane 4j + l/8.
    auto masks = [&](uint32_t k, int c, uint32_t (&m)[VPT]) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) m[j] = (word_at(k, c, 4 * j + (lane >> 3)) >> (4 * (lane & 7))) & 0xfu;
    };
    // Key vectors of chunk c of tile k that hold a kept element.
    auto load_keys = [&](uint32_t k, int c, const uint32_t (&m)[VPT], uint32_t (&key)[VPT][4]) {
        const size_t seg = (size_t)(rank + k * G) * TILE + (size_t)c * CHUNK + (size_t)warp * SEG;
        if (seg + SEG <= n) {
            const uint4* kp = reinterpret_cast<const uint4*>(keys + seg) + lane;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                uint4 r = make_uint4(0u, 0u, 0u, 0u);
                if (m[j]) r = ld_key_vec(kp + 32 * j);
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
    // Waits for tile k's flags, turns them into keep words (left in the
    // stage) and counts per (chunk, warp), turns the counts into offsets and
    // publishes the total.  False if the copy did not arrive.
    auto count_publish = [&](uint32_t k) -> bool {
        const uint32_t t = rank + k * G;
        const bool ok = mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) record_error(ctx.status, kErrBulkTimeout, t);
            return false;
        }
        uint32_t words[CHUNKS];
        const size_t t_base = (size_t)t * TILE;
        unsigned char* stage = smem_raw + (size_t)(k % STAGES) * TILE;
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) {
            uint32_t m = 0;
            if (t_base + TILE <= n) {
                const unsigned char* f = stage + (size_t)c * CHUNK + (size_t)warp * SEG + 32u * lane;
                // The two 16-byte halves in the order that puts each quarter-warp's
                // reads on distinct banks; the halves of the result swap back.
                const uint32_t h = (lane >> 2) & 1u;
                const uint32_t r = keep_bits32(lds_vec(f + 16u * h), lds_vec(f + 16u * (h ^ 1u)));
                m = h ? __funnelshift_l(r, r, 16) : r;
            } else {  // ragged last tile: flags from global memory
                const size_t seg = t_base + (size_t)c * CHUNK + (size_t)warp * SEG + 32u * lane;
                for (int i = 0; i < 32; ++i)
                    if (seg + i < n && flags[seg + i] != 0) m |= 1u << i;
            }
            words[c] = m;
            const uint32_t x = warp_sum((uint32_t)__popc(m));
            if (lane == 0) s_cnt[k & 1][c * WARPS + warp] = x;
        }
        __syncthreads();  // the tile's flags are read
        uint32_t* wst = reinterpret_cast<uint32_t*>(stage);
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) wst[(c * WARPS + warp) * 32 + lane] = words[c];
        fence_async_shared();  // these writes before the copy that later refills the stage
        if (warp == 0) {  // (chunk, warp) order is the elements' order
            const uint32_t a = s_cnt[k & 1][CPL * lane], b = CPL == 2 ? s_cnt[k & 1][CPL * lane + 1] : 0u;
            const uint32_t inc = warp_inclusive_scan<uint32_t>(a + b, lane);
            s_cnt[k & 1][CPL * lane] = inc - a - b;
            if (CPL == 2) s_cnt[k & 1][CPL * lane + 1] = inc - b;
            const uint32_t total = __shfl_sync(kFullMask, inc, 31);
            if (lane == 0) {
                s_total[k & 1] = total;
                if ((int64_t)t != ctx.fault_tile) {
                    if (t == 0) {
                        if (num_tiles > 1) st_relaxed_u64(ctx.desc, pack_desc(epoch, kStateP, total));
                    } else {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateA, total));
                    }
                }
            }
            compiler_fence();  // the count just published stays ahead of the look-back
        }
        return true;
    };

    uint32_t prev_incl = 0;  // warp 0
    uint32_t fail_at = 0;
    bool failed = false;
    if (threadIdx.x == 0)
        for (uint32_t k = 0; k < count && k < (uint32_t)STAGES; ++k) issue(k);
    if (count > 0 && !count_publish(0)) failed = true;

    for (uint32_t k = 0; !failed && k < count; ++k) {
        const uint32_t t = rank + k * G;
        if (k == 0) __syncthreads();  // tile 0's offsets and total are visible; later tiles' are by the
                                      // previous iteration's last barrier
        const uint32_t agg = s_total[k & 1];
        const bool sparse = agg < sparse_below;  // the same in every thread
        uint32_t ma[VPT], mb[VPT];
        uint32_t ka[VPT][4], kb[VPT][4];
        if (sparse) {
            // The slots live in the dense form's registers: ka[2c][r] holds slot r
            // of chunk c, ka[2c+1][0] the lane's count in chunk c, ma[c] its keep
            // bits past the slots and ma[4+c] the position of its first kept key in
            // the tile.
#pragma unroll
            for (int c = 0; c < CHUNKS; ++c) {
                uint32_t m = word_at(k, c, lane);
                const uint32_t cnt = (uint32_t)__popc(m);
                const uint32_t inc = warp_inclusive_scan<uint32_t>(cnt, lane);
                ma[4 + c] = s_cnt[k & 1][c * WARPS + warp] + inc - cnt;
                ka[2 * c + 1][0] = cnt;
                const uint32_t* kp = keys + (size_t)t * TILE + (size_t)c * CHUNK + (size_t)warp * SEG + 32u * lane;
#pragma unroll
                for (int r = 0; r < kSlots; ++r) {
                    if (!__any_sync(kFullMask, m != 0)) break;
                    if (m) {
                        ka[2 * c][r] = ld_key_u32(kp + (__ffs(m) - 1));
                        m &= m - 1;
                    }
                }
                ma[c] = m;
            }
        }
        if (k + 1 < count && !count_publish(k + 1)) {
            failed = true;
            fail_at = k;
            break;
        }
        if (warp == 0) {
            uint32_t excl = 0;
            bool lb_failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;
            } else {
                const int64_t floor = k > 0 ? (int64_t)t - (int64_t)G : -1;
                excl = lookback<uint32_t, 1>(ctx, t, epoch, lane, &lb_failed, nullptr, floor, prev_incl);
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
            if (lane == 0) {
                s_prefix[k & 1] = excl;
                s_fail[k & 1] = lb_failed ? 1u : 0u;
            }
        }
        // Dense form: masks and keys of chunk 0 load while warp 0 looks back.
        if (!sparse) {
            masks(k, 0, ma);
            load_keys(k, 0, ma, ka);
        }
        __syncthreads();  // the prefix is in shared memory
        if (s_fail[k & 1]) {
            failed = true;
            fail_at = k;
            break;
        }
        const uint32_t base = s_prefix[k & 1];
        if (sparse) {
            // A lane's kept keys of a chunk are consecutive in the output.
#pragma unroll
            for (int c = 0; c < CHUNKS; ++c) {
                uint32_t* dst = out + (size_t)base + ma[4 + c];
                const uint32_t cnt = ka[2 * c + 1][0];
#pragma unroll
                for (int r = 0; r < kSlots; ++r) {
                    if (!__any_sync(kFullMask, cnt > (uint32_t)r)) break;
                    if (cnt > (uint32_t)r) dst[r] = ka[2 * c][r];
                }
                const uint32_t* kp = keys + (size_t)t * TILE + (size_t)c * CHUNK + (size_t)warp * SEG + 32u * lane;
                uint32_t m = ma[c];
                for (uint32_t r = kSlots; m != 0; ++r, m &= m - 1) dst[r] = ld_key_u32(kp + (__ffs(m) - 1));
            }
        } else {
            // The warp's kept keys of one share, in two halves of four rows: each half
            // is gathered in order into this warp's staging area (in the tile's
            // stage, past the keep words) and written out with 16-byte stores.
            uint32_t* stg = reinterpret_cast<uint32_t*>(smem_raw + (size_t)(k % STAGES) * TILE + kWordBytes +
                                                        (size_t)warp * kStageWarpBytes);
            auto scatter = [&](int c, const uint32_t (&m)[VPT], const uint32_t (&key)[VPT][4]) {
                uint32_t* dst = out + (size_t)base + s_cnt[k & 1][c * WARPS + warp];
                uint32_t run = 0;  // kept keys of the share in the rows before this half
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    uint32_t packed = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) packed |= (uint32_t)__popc(m[4 * w + q]) << (8 * q);
                    const uint32_t inc = warp_inclusive_scan<uint32_t>(packed, lane);
                    const uint32_t exc = inc - packed;  // bytewise, no borrows (each byte <= 128)
                    const uint32_t rows = __shfl_sync(kFullMask, inc, 31);
                    // Staging index of the half's first key: its global address mod 16
                    // bytes, so that aligned vectors of the stage are aligned in memory.
                    uint32_t* g = dst + run;
                    const uint32_t s0 = (uint32_t)(reinterpret_cast<uintptr_t>(g) >> 2) & 3u;
                    uint32_t row_run = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = 4 * w + q;
                        uint32_t pos = s0 + row_run + ((exc >> (8 * q)) & 0xffu);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if ((m[j] >> e) & 1u) stg[pos++] = key[j][e];
                        row_run += (rows >> (8 * q)) & 0xffu;
                    }
                    __syncwarp();
                    uint32_t* ga = g - s0;  // 16-byte aligned; written only at [s0, s0 + row_run)
                    const uint32_t end = s0 + row_run;
                    for (uint32_t v = (uint32_t)lane; 4 * v < end; v += 32) {
                        const uint32_t lo = 4 * v;
                        if (lo >= s0 && lo + 4 <= end) {
                            st_vec(ga + lo, lds_vec(stg + lo));
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (lo + e >= s0 && lo + e < end) ga[lo + e] = stg[lo + e];
                        }
                    }
                    __syncwarp();
                    run += row_run;
                }
            };
            // Not unrolled: the two-chunk body is large, and one copy of it runs faster
            // when the flags are dense (measured at n = 2^28: 0.491 against 0.528 ms at
            // p = 0.99; 0.223 against 0.218 ms at p = 0.01).
#pragma unroll 1
            for (int c = 0; c < CHUNKS; c += 2) {
                masks(k, c + 1, mb);
                load_keys(k, c + 1, mb, kb);
                scatter(c, ma, ka);
                if (c + 2 < CHUNKS) {
                    masks(k, c + 2, ma);
                    load_keys(k, c + 2, ma, ka);
                }
                scatter(c + 1, mb, kb);
            }
            fence_async_shared();  // the staging writes before the copy that refills the stage
        }
        if (t == num_tiles - 1 && threadIdx.x == 0) *d_count = (unsigned long long)base + agg;
        __syncthreads();  // tile k's keep words read by everyone
        if (threadIdx.x == 0) {
            consumed = k + 1;
            if (k + STAGES < count) issue(k + STAGES);
        }
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

template <int THREADS, int VPT, int STAGES, bool SELECTIVE, KeepRule RULE = KeepRule::Flags>
static cudaError_t launch_compact_persistent(const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                                             unsigned long long* d_count, size_t n, const LookbackWs& ws,
                                             cudaStream_t s) {
    static_assert(!SELECTIVE || RULE == KeepRule::Flags, "selective key loads need a flag array");
    constexpr size_t TILE = (size_t)THREADS * VPT * 4;
    constexpr size_t SMEM = (size_t)STAGES * TILE * (SELECTIVE ? 1 : (RULE == KeepRule::Flags ? 5 : 4));
    auto kern = [] {
        if constexpr (SELECTIVE) return k_compact_sel<THREADS, VPT, STAGES>;
        else return k_compact_pipe<THREADS, VPT, STAGES, RULE>;
    }();
    KernelSetup su;
    cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), THREADS, SMEM, &su);
    if (e != cudaSuccess) return e;
    const uint32_t tiles = (uint32_t)((n + TILE - 1) / TILE);
    const size_t resident = (size_t)su.sms * (size_t)su.blocks_per_sm;
    const uint32_t grid = (uint32_t)(tiles < resident ? tiles : resident);
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    kern<<<grid, THREADS, SMEM, s>>>(keys, flags, out, d_count, n, tiles, ctx);
    return cudaGetLastError();
}

// 0: bulk-copied keys and flags; 1: bulk-copied flags, selective key loads;
// 2: the chunked kernel (one look-back per tile of four chunks) with two
// 256-thread CTAs per SM and 32768-element tiles (the default), each tile
// written in the sparse or the dense form by its count; 3 and 4: the same
// with every tile in the dense, or the sparse, form; 5, 6, 7: the same three
// with one 512-thread CTA per SM and 65536-element tiles.  Measured at
// n = 2^28 (ms at p = 0.01 / 0.5 / 0.99): two CTAs per SM 0.127 / 0.307 /
// 0.377, one 0.122 / 0.315 / 0.388: the second CTA's warps hide the dense
// form's key-load latency, and cost the sparse form a little.
static std::atomic<int> g_compact_kernel{2};  // read once per call; set from any thread
// Chunked rows 2..7: a tile keeping fewer keys than this takes the sparse
// form.  Measured at n = 2^28 with 65536-element tiles (all tiles in one
// form, ms): keep rate 0.01, sparse 0.122 against dense 0.221; 0.03, 0.173
// against 0.230; 0.05 (3277 keys a tile), 0.230 against 0.237; 0.1, 0.38
// against 0.26.  The 32768-element tiles take half the count.
static const uint32_t kCompactSparseBelow[] = {1728, 0, 65537, 3456, 0, 65537};

int compact_kernel_count() { return 2 + (int)(sizeof(kCompactSparseBelow) / sizeof(kCompactSparseBelow[0])); }

template <int THREADS>
static cudaError_t launch_compact_chunked(const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                                         unsigned long long* d_count, size_t n, const LookbackWs& ws,
                                         uint32_t sparse_below, cudaStream_t s) {
    constexpr int STAGES = 3;
    constexpr size_t TILE = (size_t)THREADS * 128;  // 65536 for 512 threads
    constexpr size_t SMEM = STAGES * TILE;
    auto kern = k_compact_chunked<THREADS, STAGES>;
    KernelSetup su;
    cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), THREADS, SMEM, &su);
    if (e != cudaSuccess) return e;
    const uint32_t tiles = (uint32_t)((n + TILE - 1) / TILE);
    const uint32_t resident = (uint32_t)(su.sms * su.blocks_per_sm);
    const uint32_t grid = tiles < resident ? tiles : resident;
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    kern<<<grid, THREADS, SMEM, s>>>(keys, flags, out, d_count, n, tiles, ctx, sparse_below);
    return cudaGetLastError();
}
void set_compact_kernel(int k) { g_compact_kernel.store(k, std::memory_order_relaxed); }

cudaError_t launch_compact_pipe(KeepRule rule, const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                                unsigned long long* d_count, size_t n, const LookbackWs& ws, cudaStream_t s) {
    // A predicate needs every key: its own kernel streams them all through the ring.
    if (rule != KeepRule::Flags) return launch_compact_pred(rule, keys, out, d_count, n, ws, s);
    const int cfg = g_compact_kernel.load(std::memory_order_relaxed);
    if (cfg == 0)
        return launch_compact_persistent<512, 8, 2, false>(keys, flags, out, d_count, n, ws, s);
    if (cfg >= 5 && n > (size_t)65536)
        return launch_compact_chunked<512>(keys, flags, out, d_count, n, ws, kCompactSparseBelow[cfg - 2], s);
    if (cfg >= 2 && cfg < 5 && n > (size_t)32768)
        return launch_compact_chunked<256>(keys, flags, out, d_count, n, ws, kCompactSparseBelow[cfg - 2], s);
    return launch_compact_persistent<512, 8, 3, true>(keys, flags, out, d_count, n, ws, s);
}

}  // namespace ss
