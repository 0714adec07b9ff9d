// compact.cu -- single-pass, order-preserving stream compaction.
//
// keep[i] = (flags[i] != 0), or a built-in predicate of keys[i] (keep.cuh);
// out[pos[i]] = keys[i] for kept i, where pos is
// the exclusive scan of keep; count = pos[n-1] + keep[n-1] ("Prefix sum and
// other parallel patterns", Stream compaction and Exercise 1).  The flag
// scan, the look-back and the scatter are fused into one pass, so neither
// the 0/1 flags nor the positions ever reach device memory (the "more
// efficient version" of that exercise, single pass like a DeviceSelect).
//
// Per tile of 4096 elements (256 threads, warp-striped rows of 4-element
// vectors as in tile.cuh):
//   1. load the flag bytes (one 32-bit word per 4 keys) and the key vectors;
//      a key vector whose four flags are all zero is not loaded (under a
//      predicate every key vector is loaded and tested instead);
//   2. per-row keep masks; the four rows' counts are packed into the bytes
//      of one 32-bit word and scanned across the warp in one shuffle scan
//      (each byte stays <= 128, so bytes never carry into each other); inside
//      a vector the rank comes from a popc of the mask below the element,
//      the vector counterpart of the page's ballot/popc warp rank;
//   3. block scan of the warp counts, then the decoupled look-back on counts
//      gives the tile's first output slot;
//   4. kept keys are staged in shared memory at their tile-local rank and
//      written out as one contiguous, coalesced run.
#include "internal.h"
#include "keep.cuh"
#include "tile.cuh"

namespace ss {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVpt = 4;                      // rows (4-key vectors) per lane
constexpr size_t kSeg = (size_t)32 * kVpt * 4;  // 512 elements per warp
static_assert(kSeg * kWarps == kCompactTile, "tile geometry");

__device__ __forceinline__ uint32_t ld_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// Bit k set when byte k of w is nonzero.
__device__ __forceinline__ uint32_t nonzero_byte_mask(uint32_t w) {
    return ((w & 0x000000ffu) ? 1u : 0u) | ((w & 0x0000ff00u) ? 2u : 0u) |
           ((w & 0x00ff0000u) ? 4u : 0u) | ((w & 0xff000000u) ? 8u : 0u);
}

}  // namespace

template <KeepRule RULE>
__global__ void __launch_bounds__(kThreads)
k_compact_u32(const uint32_t* keys, const uint8_t* flags, uint32_t* out,
              unsigned long long* d_count, size_t n, uint32_t num_tiles, LookbackCtx ctx,
              bool aligned) {
    __shared__ uint32_t s_keys[kCompactTile];
    __shared__ uint32_t s_warp[kWarps];
    __shared__ uint32_t s_prefix, s_tile, s_epoch, s_fail;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        uint32_t tile = 0, epoch = 0;
        if (num_tiles > 1) claim_tile(ctx.counter, num_tiles, &tile, &epoch);
        s_tile = tile;
        s_epoch = epoch;
    }
    __syncthreads();
    const uint32_t tile = s_tile;
    const uint32_t epoch = s_epoch;
    if (tile >= num_tiles) {  // counter out of step: never index past the descriptors
        if (threadIdx.x == 0) record_error(ctx.status, kErrCounter, tile);
        return;
    }

    const size_t seg = (size_t)tile * kCompactTile + (size_t)warp * kSeg;
    const bool fast = aligned && (seg + kSeg <= n);

    uint32_t m[kVpt];
    uint32_t key[kVpt][4];
    if (fast && RULE == KeepRule::Flags) {
        uint32_t fw[kVpt];
#pragma unroll
        for (int j = 0; j < kVpt; ++j) fw[j] = ld_u32(flags + seg + (size_t)(32 * j + lane) * 4);
        const uint4* kp = reinterpret_cast<const uint4*>(keys + seg) + lane;
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            m[j] = nonzero_byte_mask(fw[j]);
            uint4 r = make_uint4(0u, 0u, 0u, 0u);
            if (m[j]) r = ld_vec(kp + 32 * j);
            key[j][0] = r.x;
            key[j][1] = r.y;
            key[j][2] = r.z;
            key[j][3] = r.w;
        }
    } else if (fast) {  // predicate: every key vector is loaded and tested
        const uint4* kp = reinterpret_cast<const uint4*>(keys + seg) + lane;
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            const uint4 r = ld_vec(kp + 32 * j);
            key[j][0] = r.x;
            key[j][1] = r.y;
            key[j][2] = r.z;
            key[j][3] = r.w;
            m[j] = keep_mask4<RULE>(key[j]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            m[j] = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const size_t i = seg + (size_t)(32 * j + lane) * 4 + k;
                bool keep = false;
                key[j][k] = 0u;
                if (i < n) {
                    if constexpr (RULE == KeepRule::Flags) {
                        keep = flags[i] != 0;
                        if (keep) key[j][k] = keys[i];
                    } else {
                        key[j][k] = keys[i];
                        keep = keep_bits<RULE>(key[j][k]);
                    }
                }
                m[j] |= keep ? (1u << k) : 0u;
            }
        }
    }

    // Row counts packed one byte per row; one warp scan covers all rows.
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < kVpt; ++j) packed |= (uint32_t)__popc(m[j]) << (8 * j);
    const uint32_t inc = warp_inclusive_scan<uint32_t>(packed, lane);
    const uint32_t exc = inc - packed;              // bytewise: no borrows
    const uint32_t rows = __shfl_sync(kFullMask, inc, 31);  // row totals
    uint32_t row_base[kVpt];
    uint32_t warp_total = 0;
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
        row_base[j] = warp_total + ((exc >> (8 * j)) & 0xffu);
        warp_total += (rows >> (8 * j)) & 0xffu;
    }

    uint32_t warp_prefix, tile_count;
    block_combine<uint32_t, kWarps>(warp_total, warp, lane, s_warp, &warp_prefix, &tile_count);

    // Stage kept keys at their tile-local rank.
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
        uint32_t r = warp_prefix + row_base[j];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if ((m[j] >> k) & 1u) s_keys[r++] = key[j][k];
        }
    }

    if (warp == 0) {
        uint32_t excl = 0;
        bool failed = false;
        const bool dead = (int64_t)tile == ctx.fault_tile;  // test hook only
        if (tile == 0) {
            if (num_tiles > 1 && lane == 0 && !dead)
                st_relaxed_u64(ctx.desc, pack_desc(epoch, kStateP, tile_count));
            failed = dead;
        } else if (dead) {
            failed = true;
        } else {
            if (lane == 0) st_relaxed_u64(ctx.desc + tile, pack_desc(epoch, kStateA, tile_count));
            compiler_fence();  // publish before looking back
            excl = lookback<uint32_t, 1>(ctx, tile, epoch, lane, &failed);
            if (lane == 0) {
                if (!failed) {
                    st_relaxed_u64(ctx.desc + tile, pack_desc(epoch, kStateP, excl + tile_count));
                } else {
                    st_relaxed_u64(ctx.desc + tile, pack_desc(epoch, kStatePoison, 0u));
                    record_error(ctx.status, kErrLookbackTimeout, tile);
                }
            }
        }
        if (lane == 0) {
            s_prefix = excl;
            s_fail = failed ? 1u : 0u;
        }
    }
    __syncthreads();
    if (s_fail) return;

    uint32_t* dst = out + s_prefix;
    for (uint32_t r = threadIdx.x; r < tile_count; r += kThreads) dst[r] = s_keys[r];

    if (tile == num_tiles - 1 && threadIdx.x == 0)
        *d_count = (unsigned long long)s_prefix + tile_count;
}

template <KeepRule RULE>
static cudaError_t launch_per_tile(const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                                   unsigned long long* d_count, size_t n, const LookbackWs& ws, cudaStream_t s) {
    const uint32_t tiles = (uint32_t)((n + kCompactTile - 1) / kCompactTile);
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    const bool aligned = ((reinterpret_cast<uintptr_t>(keys) & 15u) == 0) &&
                         (RULE != KeepRule::Flags || (reinterpret_cast<uintptr_t>(flags) & 3u) == 0);
    k_compact_u32<RULE><<<tiles, kThreads, 0, s>>>(keys, flags, out, d_count, n, tiles, ctx, aligned);
    return cudaGetLastError();
}

cudaError_t launch_compact(KeepRule rule, const uint32_t* keys, const uint8_t* flags, uint32_t* out,
                           unsigned long long* d_count, size_t n, const LookbackWs& ws, cudaStream_t s) {
    // Large aligned inputs take the persistent kernel (bulk copies need
    // 16-byte aligned sources); the rest stay on one CTA per 4096-element tile.
    uintptr_t align = reinterpret_cast<uintptr_t>(keys);
    if (rule == KeepRule::Flags) align |= reinterpret_cast<uintptr_t>(flags);
    if ((align & 15u) == 0 && n > (size_t)16384) return launch_compact_pipe(rule, keys, flags, out, d_count, n, ws, s);
    switch (rule) {
        case KeepRule::Flags: return launch_per_tile<KeepRule::Flags>(keys, flags, out, d_count, n, ws, s);
        case KeepRule::PositiveF32: return launch_per_tile<KeepRule::PositiveF32>(keys, flags, out, d_count, n, ws, s);
        case KeepRule::PositiveI32: return launch_per_tile<KeepRule::PositiveI32>(keys, flags, out, d_count, n, ws, s);
        default: return launch_per_tile<KeepRule::PositiveU32>(keys, flags, out, d_count, n, ws, s);
    }
}

}  // namespace ss
