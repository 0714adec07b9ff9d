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
// tile's aggregate A was published.  Reads predecessors' descriptors 32 at a
// time (lane i reads tile - 1 - i - 32k), waits while any descriptor up to
// the nearest P is still X, and sums values back to and including that P.
// Returns the tile's exclusive prefix in every lane; sets *failed (warp
// uniform) if the wait ran out or a predecessor was poisoned.
template <typename T>
__device__ __forceinline__ T lookback(const LookbackCtx& c, uint32_t tile, uint32_t epoch, int lane,
                                      bool* failed) {
    const uint32_t tag = epoch << 2;
    T acc = T(0);
    int64_t pred = (int64_t)tile - 1;
    uint32_t polls = 0;
    uint64_t t0 = 0;
    *failed = false;
    while (true) {
        const int64_t idx = pred - lane;
        unsigned long long d = idx >= 0 ? ld_relaxed_u64(c.desc + idx)
                                        : pack_desc(epoch, kStateP, 0u);
        const uint32_t hi = (uint32_t)(d >> 32);
        const uint32_t state = ((hi & ~3u) == tag) ? (hi & 3u) : kStateX;
        const uint32_t stop_mask = __ballot_sync(kFullMask, state == kStateP || state == kStatePoison);
        const int first = stop_mask ? __ffs(stop_mask) - 1 : 31;
        const uint32_t upto = (first == 31) ? kFullMask : ((2u << first) - 1u);
        const uint32_t x_mask = __ballot_sync(kFullMask, state == kStateX) & upto;
        if (x_mask) {
            // A predecessor up to the nearest P has not published yet: wait.
            ++polls;
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
        const uint32_t poison_mask = __ballot_sync(kFullMask, state == kStatePoison) & upto;
        if (poison_mask) {
            *failed = true;
            return T(0);
        }
        T v = (lane <= first) ? from_bits<T>((uint32_t)d) : T(0);
        acc += warp_sum(v);
        if (stop_mask) return acc;
        pred -= 32;
        polls = 0;
    }
}

}  // namespace ss
