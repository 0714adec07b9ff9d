// lookback_wide.cuh -- the decoupled look-back for 64-bit sums (uint64
// wraparound and fp64), on 16-byte tile descriptors.
//
// A 64-bit value and its state do not fit one 64-bit word, and a 16-byte
// access is not single-copy atomic as a whole; only its two 8-byte halves
// are.  So the descriptor is two words that carry the same tag
// (epoch << 2 | state) in their high halves and the value's low and high 32
// bits in their low halves:
//   w0 = tag << 32 | value[31:0],   w1 = tag << 32 | value[63:32].
// Both are written with one 16-byte relaxed store and read with one 16-byte
// relaxed load.  A reader accepts the descriptor only when both halves carry
// the same tag of the current epoch.  Each state is published at most once
// per tile and epoch, so two halves with equal tags come from the same
// publish.  A torn read (one half already A, the other still X, say) shows
// unequal tags and is treated as "not yet published", then polled again.
//
// The walk itself is the one of lookback.cuh ("Prefix sum and other
// parallel patterns", A device-level scan: scan then propagate): 32
// predecessors per poll, one per lane; sum back to the nearest P; bounded
// waits; POISON ends the walk with a failure; an optional floor tile whose
// inclusive prefix the caller already holds.
#pragma once

#include "lookback.cuh"

namespace ss {

template <typename TA> __device__ __forceinline__ unsigned long long acc_bits(TA v);
template <> __device__ __forceinline__ unsigned long long acc_bits<unsigned long long>(unsigned long long v) {
    return v;
}
template <> __device__ __forceinline__ unsigned long long acc_bits<double>(double v) {
    return (unsigned long long)__double_as_longlong(v);
}
template <typename TA> __device__ __forceinline__ TA acc_from_bits(unsigned long long b);
template <> __device__ __forceinline__ unsigned long long acc_from_bits<unsigned long long>(unsigned long long b) {
    return b;
}
template <> __device__ __forceinline__ double acc_from_bits<double>(unsigned long long b) {
    return __longlong_as_double((long long)b);
}

struct Desc16 {
    unsigned long long w0, w1;
};

__device__ __forceinline__ Desc16 pack_desc16(uint32_t epoch, uint32_t state, unsigned long long bits) {
    const unsigned long long tag = (unsigned long long)((epoch << 2) | state) << 32;
    return Desc16{tag | (bits & 0xffffffffull), tag | (bits >> 32)};
}

__device__ __forceinline__ void st_relaxed_desc16(unsigned long long* p, Desc16 d) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(d.w0), "l"(d.w1) : "memory");
}

__device__ __forceinline__ Desc16 ld_relaxed_desc16(const unsigned long long* p) {
    Desc16 d;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(d.w0), "=l"(d.w1) : "l"(p) : "memory");
    return d;
}

// `desc` holds two words per tile.  Returns the tile's exclusive prefix in
// every lane; sets *failed (warp uniform) when the wait ran out or the
// nearest stop was poisoned.
template <typename TA>
__device__ __forceinline__ TA lookback_wide(unsigned long long* desc, const LookbackCtx& c, uint32_t tile,
                                            uint32_t epoch, int lane, bool* failed, int64_t floor, TA floor_value) {
    const uint32_t tag = epoch << 2;
    TA acc = TA(0);
    int64_t pred = (int64_t)tile - 1;
    uint32_t polls = 0;
    uint64_t t0 = 0;
    *failed = false;
    while (true) {
        const int64_t idx = pred - lane;
        uint32_t st;
        TA val;
        if (idx > floor) {
            const Desc16 d = ld_relaxed_desc16(desc + 2 * idx);
            const uint32_t h0 = (uint32_t)(d.w0 >> 32), h1 = (uint32_t)(d.w1 >> 32);
            st = (h0 == h1 && (h0 & ~3u) == tag) ? (h0 & 3u) : kStateX;
            val = acc_from_bits<TA>((d.w0 & 0xffffffffull) | (d.w1 << 32));
        } else {
            st = kStateP;
            val = floor_value;
        }
        const bool stop = st == kStateP || st == kStatePoison;
        const uint32_t stop_mask = __ballot_sync(kFullMask, stop);
        const int first = stop_mask ? __ffs(stop_mask) - 1 : 31;
        const uint32_t upto = (first == 31) ? kFullMask : ((2u << first) - 1u);
        if (__ballot_sync(kFullMask, st == kStateX) & upto) {
            ++polls;
            if (polls == 1) t0 = globaltimer_ns();
            if (polls > 4) __nanosleep(polls < 16 ? 32 : (polls < 64 ? 128 : 256));
            bool give_up = polls >= c.max_polls || (globaltimer_ns() - t0) > c.timeout_ns;
            give_up = __shfl_sync(kFullMask, give_up, 0);
            if (give_up) {
                *failed = true;
                return TA(0);
            }
            continue;
        }
        if (stop_mask && ((__ballot_sync(kFullMask, st == kStatePoison) >> first) & 1u)) {
            *failed = true;
            return TA(0);
        }
        TA v = (stop_mask == 0 || lane <= first) ? val : TA(0);
        acc += warp_sum(v);
        if (stop_mask) return acc;
        pred -= 32;
        polls = 0;
    }
}

}  // namespace ss
