// keep.cuh -- which elements a compaction keeps.
//
// Two forms ("Prefix sum and other parallel patterns", Stream compaction and
// Exercise 1):
//   - Flags: a separate byte per element, nonzero keeps the key;
//   - a built-in predicate on the element itself, "v > 0" evaluated in the
//     element's own type: fp32 (so NaN, +0 and -0 are dropped, +inf is
//     kept), int32 (signed), uint32 (that is, nonzero).
// The predicate forms read no flag array: the keep decision is made from the
// value already loaded for the output, so flags and positions never reach
// device memory.
#pragma once

#include <cstdint>

#include "internal.h"

namespace ss {

template <KeepRule R>
__device__ __forceinline__ bool keep_bits(uint32_t bits) {
    if constexpr (R == KeepRule::PositiveF32) return __uint_as_float(bits) > 0.0f;
    else if constexpr (R == KeepRule::PositiveI32) return (int32_t)bits > 0;
    else return bits != 0u;  // PositiveU32
}

// Bit e set when element e of the 4-element vector v is kept.
template <KeepRule R>
__device__ __forceinline__ uint32_t keep_mask4(const uint32_t (&v)[4]) {
    return (keep_bits<R>(v[0]) ? 1u : 0u) | (keep_bits<R>(v[1]) ? 2u : 0u) | (keep_bits<R>(v[2]) ? 4u : 0u) |
           (keep_bits<R>(v[3]) ? 8u : 0u);
}

}  // namespace ss
