// compact_unordered.cu -- compaction by warp-aggregated atomics, the
// unordered counterpart of the fused single-pass compaction.
//
// "Prefix sum and other parallel patterns", Stream compaction: when the
// output order does not matter, a warp claims room for all of its kept
// elements with one atomic add on the global count, then writes each kept
// element at the claimed offset plus its rank among the warp's kept
// elements (ballot and popc).  That cuts the atomics to one per warp step.
//
// Here a warp's step is a 512-element batch (four 16-byte vectors per lane),
// so there is one atomic per 512 elements.  Inside a batch the kept keys keep
// their order: rows are ranked as in the ordered kernels, by the packed row
// counts scanned across the warp and a popc inside each vector.  The batches
// themselves land in whatever order their claims were served.  There is no
// look-back and no workspace.  *d_count is zeroed on the stream before the
// kernel and counts up.  What is left after the whole batches (fewer than 512
// elements), and all of an input that is not 16-byte aligned, goes 32
// elements per warp step through the page's own ballot form.
#include "internal.h"
#include "keep.cuh"
#include "tile.cuh"

namespace ss {

namespace {

constexpr int kUThreads = 256;
constexpr int kUVpt = 4;                         // 16-byte vectors per lane per batch
constexpr size_t kUBatch = (size_t)32 * kUVpt * 4;  // 512 elements

__device__ __forceinline__ unsigned long long claim(unsigned long long* d_count, uint32_t total, int lane) {
    unsigned long long start = 0;
    if (lane == 0 && total != 0u) start = atomicAdd(d_count, (unsigned long long)total);
    return __shfl_sync(kFullMask, start, 0);
}

__device__ __forceinline__ uint32_t nonzero_bytes(uint32_t w) {
    return ((w & 0x000000ffu) ? 1u : 0u) | ((w & 0x0000ff00u) ? 2u : 0u) |
           ((w & 0x00ff0000u) ? 4u : 0u) | ((w & 0xff000000u) ? 8u : 0u);
}

}  // namespace

template <KeepRule RULE>
__global__ void __launch_bounds__(kUThreads)
k_compact_unordered(const uint32_t* keys, const uint8_t* flags, uint32_t* out, unsigned long long* d_count,
                    size_t n, bool vec) {
    const int lane = threadIdx.x & 31;
    const size_t warp_id = ((size_t)blockIdx.x * kUThreads + threadIdx.x) >> 5;
    const size_t warps = ((size_t)gridDim.x * kUThreads) >> 5;
    const size_t body = vec ? (n / kUBatch) * kUBatch : 0;

    for (size_t b = warp_id * kUBatch; b < body; b += warps * kUBatch) {  // warp-uniform
        uint32_t m[kUVpt];
        uint32_t key[kUVpt][4];
        const uint4* kp = reinterpret_cast<const uint4*>(keys + b) + lane;
        if constexpr (RULE == KeepRule::Flags) {
            uint32_t fw[kUVpt];
#pragma unroll
            for (int j = 0; j < kUVpt; ++j)
                fw[j] = *reinterpret_cast<const uint32_t*>(flags + b + (size_t)(32 * j + lane) * 4);
#pragma unroll
            for (int j = 0; j < kUVpt; ++j) {
                m[j] = nonzero_bytes(fw[j]);
                uint4 r = make_uint4(0u, 0u, 0u, 0u);
                if (m[j]) r = ld_vec(kp + 32 * j);
                key[j][0] = r.x;
                key[j][1] = r.y;
                key[j][2] = r.z;
                key[j][3] = r.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kUVpt; ++j) {
                const uint4 r = ld_vec(kp + 32 * j);
                key[j][0] = r.x;
                key[j][1] = r.y;
                key[j][2] = r.z;
                key[j][3] = r.w;
                m[j] = keep_mask4<RULE>(key[j]);
            }
        }
        // Row counts, one byte per row (each at most 128), scanned across the warp at once.
        uint32_t packed = 0;
#pragma unroll
        for (int j = 0; j < kUVpt; ++j) packed |= (uint32_t)__popc(m[j]) << (8 * j);
        const uint32_t inc = warp_inclusive_scan<uint32_t>(packed, lane);
        const uint32_t exc = inc - packed;
        const uint32_t rows = __shfl_sync(kFullMask, inc, 31);
        uint32_t row_base[kUVpt];
        uint32_t total = 0;
#pragma unroll
        for (int j = 0; j < kUVpt; ++j) {
            row_base[j] = total + ((exc >> (8 * j)) & 0xffu);
            total += (rows >> (8 * j)) & 0xffu;
        }
        const unsigned long long start = claim(d_count, total, lane);
#pragma unroll
        for (int j = 0; j < kUVpt; ++j) {
            unsigned long long pos = start + row_base[j];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if ((m[j] >> e) & 1u) out[pos++] = key[j][e];
        }
    }

    for (size_t b = body + warp_id * 32; b < n; b += warps * 32) {  // warp-uniform
        const size_t i = b + lane;
        uint32_t key = 0;
        bool keep = false;
        if (i < n) {
            if constexpr (RULE == KeepRule::Flags) {
                keep = flags[i] != 0;
                if (keep) key = keys[i];
            } else {
                key = keys[i];
                keep = keep_bits<RULE>(key);
            }
        }
        const uint32_t mask = __ballot_sync(kFullMask, keep);
        const unsigned long long start = claim(d_count, (uint32_t)__popc(mask), lane);
        if (keep) out[start + (uint32_t)__popc(mask & ((1u << lane) - 1u))] = key;
    }
}

template <KeepRule RULE>
static cudaError_t launch_unordered(const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                                    unsigned long long* d_count, size_t n, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (sms <= 0) sms = 1;
    const bool vec = (reinterpret_cast<uintptr_t>(keys) & 15u) == 0 &&
                     (RULE != KeepRule::Flags || (reinterpret_cast<uintptr_t>(flags) & 3u) == 0);
    const size_t steps = vec ? (n + kUBatch - 1) / kUBatch : (n + 31) / 32;  // warp steps
    const size_t want = (steps + kUThreads / 32 - 1) / (kUThreads / 32);
    const size_t cap = (size_t)sms * (2048 / kUThreads);  // one full wave of 256-thread CTAs
    const unsigned grid = (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
    e = cudaMemsetAsync(d_count, 0, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return e;
    k_compact_unordered<RULE><<<grid, kUThreads, 0, s>>>(keys, flags, out, d_count, n, vec);
    return cudaGetLastError();
}

cudaError_t launch_compact_unordered(KeepRule rule, const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                                     unsigned long long* d_count, size_t n, cudaStream_t s) {
    switch (rule) {
        case KeepRule::Flags: return launch_unordered<KeepRule::Flags>(keys, flags, out, d_count, n, s);
        case KeepRule::PositiveF32: return launch_unordered<KeepRule::PositiveF32>(keys, flags, out, d_count, n, s);
        case KeepRule::PositiveI32: return launch_unordered<KeepRule::PositiveI32>(keys, flags, out, d_count, n, s);
        default: return launch_unordered<KeepRule::PositiveU32>(keys, flags, out, d_count, n, s);
    }
}

}  // namespace ss
