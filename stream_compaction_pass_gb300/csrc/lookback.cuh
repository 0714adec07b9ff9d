// lookback.cuh -- device building blocks shared by the single-pass kernels:
// the packed 64-bit tile-status descriptor, relaxed GPU-scope loads and
// stores in inline PTX, the shuffle warp scan, and the bounded decoupled
// look-back.
//
// The look-back follows the prose of "Prefix sum and other parallel
// patterns", section "A device-level scan: scan then propagate": a tile
// that knows its local sum publishes it ("local sum only"); it then reads the
// states earlier tiles published, summing local sums backwards until it meets
// a tile whose "inclusive prefix" is available, which gives its own offset;
// it then publishes its own inclusive prefix.  The page names two states; a
// reader also has to recognise a third, "nothing published yet" (X), and this
// build adds a fourth, POISON, published by a tile that gave up waiting so
// that its successors fail fast instead of each waiting out the limit.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"

namespace ss {

constexpr uint32_t kFullMask = 0xffffffffu;

// Descriptor: bits 63..32 = tag, bits 31..0 = value bits.
// tag = (epoch << 2) | state.  A descriptor whose epoch differs from the
// current launch's epoch reads as X, so descriptors never need clearing
// between launches.
constexpr uint32_t kStateX = 0;        // not yet published
constexpr uint32_t kStateA = 1;        // aggregate of this tile only
constexpr uint32_t kStateP = 2;        // inclusive prefix through this tile
constexpr uint32_t kStatePoison = 3;   // producer gave up (error path)

struct LookbackCtx {
    unsigned long long* desc;     // one descriptor per tile
    unsigned long long* counter;  // hi 32 bits epoch, lo 32 bits tiles claimed
    uint32_t* status;             // [0] error bits, [1] first failing tile + 1
    uint64_t timeout_ns;          // wait limit per look-back
    uint32_t max_polls;           // backstop on the number of polls
    int64_t fault_tile;           // test hook: this tile never publishes (-1: none)
};

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Compiler-only barrier: no instruction, but no memory access moves across
// it.  Placed after a descriptor is published so that the publishing store is
// emitted before the code that follows (a look-back loop in the same warp):
// without it the compiler was free to sink the store of a tile's aggregate
// below that tile's own look-back, which hides the aggregate from successors
// until the look-back ends and turns the decoupled chain back into a serial
// one (measured: 2.9x slower).
__device__ __forceinline__ void compiler_fence() { asm volatile("" ::: "memory"); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned long long pack_desc(uint32_t epoch, uint32_t state, uint32_t bits) {
    return ((unsigned long long)((epoch << 2) | state) << 32) | bits;
}

template <typename T> __device__ __forceinline__ uint32_t to_bits(T v);
template <> __device__ __forceinline__ uint32_t to_bits<uint32_t>(uint32_t v) { return v; }
template <> __device__ __forceinline__ uint32_t to_bits<float>(float v) { return __float_as_uint(v); }
template <typename T> __device__ __forceinline__ T from_bits(uint32_t b);
template <> __device__ __forceinline__ uint32_t from_bits<uint32_t>(uint32_t b) { return b; }
template <> __device__ __forceinline__ float from_bits<float>(uint32_t b) { return __uint_as_float(b); }

// Inclusive warp scan, 5 shuffle steps at offsets 1..16 ("Prefix sum and
// other parallel patterns", Warp scan and block scan).
template <typename T>
__device__ __forceinline__ T warp_inclusive_scan(T v, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        T t = __shfl_up_sync(kFullMask, v, off);
        if (lane >= off) v += t;
    }
    return v;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
    return v;
}

// Claims the next tile id for this CTA.  The counter's high word is the
// launch epoch; the CTA that claims the last id of the launch (`total_claims`
// claims in all) moves the counter to (epoch + 1, 0) for the next launch,
// which is safe because every other claim of this launch came before it.
__device__ __forceinline__ void claim_tile(unsigned long long* counter, uint32_t total_claims,
                                           uint32_t* tile, uint32_t* epoch) {
    unsigned long long old = atomicAdd(counter, 1ull);
    uint32_t cnt = (uint32_t)old;
    *epoch = (uint32_t)(old >> 32);
    *tile = cnt;
    if (cnt == total_claims - 1)
        atomicAdd(counter, (1ull << 32) - (unsigned long long)total_claims);
}

__device__ __forceinline__ void record_error(uint32_t* status, uint32_t bits, uint32_t tile) {
    if (status == nullptr) return;
    atomicOr(status, bits);
    atomicCAS(status + 1, 0u, tile + 1);
}

// Look-back for tile `tile` > 0, run by all 32 lanes of one warp after the
// tile's aggregate A was published.  Each poll reads a window of 32*K
// predecessors' descriptors in K coalesced loads: load q of lane l reads the
// tile at distance 32q + l + 1 (so each load instruction covers 32
// consecutive descriptors, 256 bytes), waits while any descriptor up to the
// nearest P is still X, and sums values back to and including that P; with
// no P in the window it sums the whole window and moves 32*K tiles further
// back.  Returns the tile's exclusive prefix in every lane; sets *failed
// (warp uniform) if the wait ran out or the nearest stop was poisoned.
// Counters one look-back fills in when a trace is taken.
struct LookbackStats {
    uint32_t windows;  // windows read
    uint32_t waits;    // polls that found an unpublished predecessor
};

// The first window of a look-back, loaded ahead of time: the loads are
// issued here and their values consumed by lookback(), so that their round
// trip overlaps whatever the warp does in between.
template <int K>
struct LookbackWindow {
    unsigned long long d[K];
};

template <typename T, int K>
__device__ __forceinline__ LookbackWindow<K> lookback_prefetch(const LookbackCtx& c, uint32_t tile, uint32_t epoch,
                                                               int lane, int64_t floor = -1,
                                                               T floor_value = T(0)) {
    LookbackWindow<K> w;
    const unsigned long long floor_desc = pack_desc(epoch, kStateP, to_bits<T>(floor_value));
    const int64_t pred = (int64_t)tile - 1;
#pragma unroll
    for (int q = 0; q < K; ++q) {
        const int64_t idx = pred - 32 * q - lane;
        w.d[q] = idx > floor ? ld_relaxed_u64(c.desc + idx) : floor_desc;
    }
    return w;
}

// Look-back for tile `tile` > 0 (see the description above LookbackStats).
// `floor` (optional) is a tile whose inclusive prefix `floor_value` the caller
// already knows (a persistent CTA's own previous tile); the walk treats it as
// a published P and never reads at or below it.  Without a floor, tile -1
// plays that role with value 0.  `window` (optional) is the first window,
// already loaded by lookback_prefetch() with the same tile and floor.
template <typename T, int K, bool TRACE = false>
__device__ __forceinline__ T lookback(const LookbackCtx& c, uint32_t tile, uint32_t epoch, int lane,
                                      bool* failed, LookbackStats* stats = nullptr,
                                      int64_t floor = -1, T floor_value = T(0),
                                      const LookbackWindow<K>* window = nullptr) {
    const uint32_t tag = epoch << 2;
    const unsigned long long floor_desc = pack_desc(epoch, kStateP, to_bits<T>(floor_value));
    if (TRACE) *stats = LookbackStats{0u, 0u};
    T acc = T(0);
    int64_t pred = (int64_t)tile - 1;
    uint32_t polls = 0;
    uint64_t t0 = 0;
    bool use_window = window != nullptr;
    *failed = false;
    while (true) {
        unsigned long long d[K];
        if (use_window) {
#pragma unroll
            for (int q = 0; q < K; ++q) d[q] = window->d[q];
            use_window = false;
        } else {
#pragma unroll
            for (int q = 0; q < K; ++q) {
                const int64_t idx = pred - 32 * q - lane;
                d[q] = idx > floor ? ld_relaxed_u64(c.desc + idx) : floor_desc;
            }
        }
        // Nearest stop (P or POISON) in distance order: load q, then lane.
        int qstop = K;     // load holding the nearest stop, K if none
        int first = 31;    // its lane
        bool x_before = false;  // an unpublished descriptor nearer than the stop
#pragma unroll
        for (int q = 0; q < K; ++q) {
            const uint32_t hi = (uint32_t)(d[q] >> 32);
            const uint32_t st = ((hi & ~3u) == tag) ? (hi & 3u) : kStateX;
            const uint32_t stops = __ballot_sync(kFullMask, st == kStateP || st == kStatePoison);
            const uint32_t xs = __ballot_sync(kFullMask, st == kStateX);
            if (qstop == K) {
                if (stops) {
                    qstop = q;
                    first = __ffs(stops) - 1;
                    if (xs & ((1u << first) - 1u)) x_before = true;
                } else if (xs) {
                    x_before = true;
                }
            }
        }
        if (TRACE) stats->windows += 1;
        if (x_before) {
            // A predecessor up to the nearest P has not published yet: wait.
            ++polls;
            if (TRACE) stats->waits += 1;
            if (polls == 1) t0 = globaltimer_ns();
            if (polls > 4) __nanosleep(polls < 16 ? 32 : (polls < 64 ? 128 : 256));
            bool give_up = polls >= c.max_polls || (globaltimer_ns() - t0) > c.timeout_ns;
            give_up = __shfl_sync(kFullMask, give_up, 0);
            if (give_up) {
                *failed = true;
                return T(0);
            }
            continue;
        }
        T v = T(0);
        bool poisoned = false;
#pragma unroll
        for (int q = 0; q < K; ++q) {
            if (q < qstop || (q == qstop && lane <= first)) v += from_bits<T>((uint32_t)d[q]);
            if (q == qstop && lane == first && (uint32_t)(d[q] >> 32) == (tag | kStatePoison)) poisoned = true;
        }
        if (__any_sync(kFullMask, poisoned)) {
            *failed = true;
            return T(0);
        }
        acc += warp_sum(v);
        if (qstop < K) return acc;
        pred -= 32 * K;
        polls = 0;
    }
}

// Two-level look-back, for kernels that run one CTA per tile: tiles form
// groups of 32 consecutive tiles, and group g has its own descriptor
// gdesc[g], published by the group's last tile -- first as A (the group's
// total), then as P (the inclusive prefix through the group).  A tile reads
// the descriptors of the tiles before it in its group (one load per lane):
// if one of them holds a P, the tile's prefix is that P plus the aggregates
// after it; otherwise their aggregates give the tile's offset inside the
// group, and a look-back over the group descriptors gives the group's
// prefix.  Tile t therefore needs about two round trips whatever t is,
// where the one-level look-back walks back t/32 windows while the tiles
// before it are still being resolved.  `agg` is the tile's aggregate (used
// for the group descriptors).  Returns the exclusive prefix in every lane;
// sets *failed (warp uniform) if a wait ran out or a predecessor was
// poisoned.  Tile 0 is not handled here (its prefix is the seed).
template <typename T>
__device__ __forceinline__ T lookback_two_level(const LookbackCtx& c, unsigned long long* gdesc, uint32_t tile,
                                                uint32_t num_tiles, uint32_t epoch, int lane, T agg,
                                                bool* failed) {
    const uint32_t tag = epoch << 2;
    const uint32_t g = tile >> 5;
    const uint32_t mate = (g << 5) + (uint32_t)lane;  // this lane's tile in the group
    const bool valid = mate < tile;
    const bool last_of_group = (tile & 31u) == 31u;
    *failed = false;
    uint32_t polls = 0;
    uint64_t t0 = 0;
    T in_group = T(0);
    bool have_p = false;
    while (true) {
        const unsigned long long d = valid ? ld_relaxed_u64(c.desc + mate) : 0ull;
        const uint32_t hi = (uint32_t)(d >> 32);
        const uint32_t st = ((hi & ~3u) == tag) ? (hi & 3u) : kStateX;
        const uint32_t pm = __ballot_sync(kFullMask, valid && (st == kStateP || st == kStatePoison));
        const int p = pm ? 31 - __clz(pm) : -1;                          // nearest stop: the highest such lane
        const uint32_t after = p >= 0 ? ~((2u << p) - 1u) : kFullMask;   // lanes nearer than the stop
        if (__ballot_sync(kFullMask, valid && st == kStateX) & after) {
            ++polls;
            if (polls == 1) t0 = globaltimer_ns();
            if (polls > 4) __nanosleep(polls < 16 ? 32 : (polls < 64 ? 128 : 256));
            bool give_up = polls >= c.max_polls || (globaltimer_ns() - t0) > c.timeout_ns;
            give_up = __shfl_sync(kFullMask, give_up, 0);
            if (give_up) {
                *failed = true;
                if (last_of_group && lane == 0) st_relaxed_u64(gdesc + g, pack_desc(epoch, kStatePoison, 0u));
                return T(0);
            }
            continue;
        }
        if (p >= 0 && __shfl_sync(kFullMask, st, p) == kStatePoison) {
            *failed = true;
            if (last_of_group && lane == 0) st_relaxed_u64(gdesc + g, pack_desc(epoch, kStatePoison, 0u));
            return T(0);
        }
        const bool take = valid && (int)lane >= p;
        in_group = warp_sum(take ? from_bits<T>((uint32_t)d) : T(0));
        have_p = p >= 0;
        break;
    }
    T excl = in_group;
    if (!have_p) {
        // No inclusive prefix before this tile in its group (g > 0: tile 0
        // always publishes one): in_group is the tile's offset in the group.
        if (last_of_group && lane == 0) st_relaxed_u64(gdesc + g, pack_desc(epoch, kStateA, to_bits<T>(in_group + agg)));
        compiler_fence();
        LookbackCtx gc = c;
        gc.desc = gdesc;
        const T gp = lookback<T, 1>(gc, g, epoch, lane, failed);
        if (*failed) {
            if (last_of_group && lane == 0) st_relaxed_u64(gdesc + g, pack_desc(epoch, kStatePoison, 0u));
            return T(0);
        }
        excl = gp + in_group;
    }
    if (last_of_group && lane == 0 && tile + 1 < num_tiles)
        st_relaxed_u64(gdesc + g, pack_desc(epoch, kStateP, to_bits<T>(excl + agg)));
    return excl;
}

}  // namespace ss
