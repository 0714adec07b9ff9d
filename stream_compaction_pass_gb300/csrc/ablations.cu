// ablations.cu -- the measured alternatives to the single-pass scan.
//
// Reduce-then-scan, three kernels over 4096-element tiles:
//   K1 k_rts_reduce       each CTA sums one tile into totals[tile]  (reads n)
//   K2 k_rts_scan_totals  one CTA scans totals exclusively, looping over
//                         them with a running carry ("Prefix sum and other
//                         parallel patterns", scan_block_sums: one block,
//                         any number of tiles)
//   K3 k_rts_scan_tiles   each CTA rescans its tile seeded with its offset
//                         (reads n, writes n)
// 3n elements of traffic against the single pass's 2n.  The pages'
// three-pass variant scans first and propagates last (4n: "Prefix sum and
// other parallel patterns", A device-level scan; "The CUDA scan algorithm:
// the tree and the three kernels", One block scans 4,096); reduce-then-scan
// gives the same results with one pass less.
//
// K3's tile scan is either the register/shuffle scan of tile.cuh or the
// Blelloch tree in shared memory ("The CUDA scan algorithm: the tree and the
// three kernels", Two sweeps over one tree, and the up-sweep / down-sweep
// listing's index formulas a = (2k+1)*stride - 1, b = (2k+2)*stride - 1;
// "7 Work-efficient Scan: Blelloch", summary), with the tile's words either
// unpadded or padded by i/32 or i/32 + i/1024 to spread the tree's strided
// accesses over the 32 banks ("The stride doubles, and so does the
// conflict").  The Blelloch tile is 4096 words and 1024 threads, the page's
// geometry, so the page's request model applies to it unchanged.
#include "internal.h"
#include "tile.cuh"

namespace ss {

namespace {

constexpr int kRThreads = 256;
constexpr int kRVpt = 4;  // 256 * 16 = 4096 = kRtsTile
constexpr size_t kRSeg = (size_t)32 * kRVpt * 4;
static_assert(kRSeg * (kRThreads / 32) == kRtsTile, "tile geometry");

constexpr int kBThreads = 1024;
constexpr int kBPer = (int)kRtsTile / kBThreads;  // 4 words per thread

template <int PAD>
__device__ __forceinline__ int padded_word(int i) {
    if (PAD == 2) return i + (i >> 5);
    if (PAD == 3) return i + (i >> 5) + (i >> 10);
    return i;
}

template <int PAD>
constexpr int padded_words() {
    return PAD == 2 ? (int)kRtsTile + (int)kRtsTile / 32
                    : (PAD == 3 ? (int)kRtsTile + (int)kRtsTile / 32 + (int)kRtsTile / 1024
                                : (int)kRtsTile);
}

bool aligned16(const void* a, const void* b) {
    return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(kRThreads)
k_rts_reduce(const T* in, size_t n, T* totals, bool aligned) {
    __shared__ T s_warp[kRThreads / 32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const size_t seg = (size_t)blockIdx.x * kRtsTile + (size_t)warp * kRSeg;
    T v[kRVpt][4];
    load_rows<T, kRVpt>(in, n, seg, lane, aligned && seg + kRSeg <= n, v);
    T s = T(0);
#pragma unroll
    for (int j = 0; j < kRVpt; ++j) s += ((v[j][0] + v[j][1]) + v[j][2]) + v[j][3];
    s = warp_sum(s);
    T wp, total;
    block_combine<T, kRThreads / 32>(s, warp, lane, s_warp, &wp, &total);
    if (threadIdx.x == 0) totals[blockIdx.x] = total;
}

// One CTA of 1024 threads; 4 totals per thread per round, with a carry.
template <typename T>
__global__ void __launch_bounds__(1024)
k_rts_scan_totals(T* totals, uint32_t count) {
    __shared__ T s_warp[32];
    __shared__ T s_carry;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_carry = T(0);
    __syncthreads();
    for (uint32_t start = 0; start < count; start += 4096) {
        T v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t i = start + threadIdx.x * 4 + k;
            v[k] = i < count ? totals[i] : T(0);
        }
        const T s = ((v[0] + v[1]) + v[2]) + v[3];
        const T inc = warp_inclusive_scan<T>(s, lane);
        T ex = __shfl_up_sync(kFullMask, inc, 1);
        if (lane == 0) ex = T(0);
        T wp, total;
        block_combine<T, 32>(__shfl_sync(kFullMask, inc, 31), warp, lane, s_warp, &wp, &total);
        T r = s_carry + wp + ex;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t i = start + threadIdx.x * 4 + k;
            if (i < count) totals[i] = r;
            r += v[k];
        }
        __syncthreads();  // everyone has read s_carry and s_warp
        if (threadIdx.x == 0) s_carry = s_carry + total;
        __syncthreads();
    }
}

// K3 with the register/shuffle tile scan.
template <typename T, bool INCLUSIVE>
__global__ void __launch_bounds__(kRThreads)
k_rts_scan_tiles(const T* in, T* out, size_t n, const T* offsets, bool aligned) {
    __shared__ T s_warp[kRThreads / 32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const size_t seg = (size_t)blockIdx.x * kRtsTile + (size_t)warp * kRSeg;
    const bool fast = aligned && seg + kRSeg <= n;
    T v[kRVpt][4];
    load_rows<T, kRVpt>(in, n, seg, lane, fast, v);
    T pre[kRVpt];
    const T wt = warp_rows_scan<T, kRVpt>(v, lane, pre);
    T wp, total;
    block_combine<T, kRThreads / 32>(wt, warp, lane, s_warp, &wp, &total);
    T y[kRVpt][4];
    rows_output<T, kRVpt, INCLUSIVE>(v, pre, offsets[blockIdx.x] + wp, y);
    store_rows<T, kRVpt>(out, n, seg, lane, fast, y);
}

// K3 with the Blelloch tree.  PAD: 1 = unpadded, 2 = i + i/32,
// 3 = i + i/32 + i/1024.
template <typename T, bool INCLUSIVE, int PAD>
__global__ void __launch_bounds__(kBThreads)
k_rts_scan_tiles_blelloch(const T* in, T* out, size_t n, const T* offsets) {
    __shared__ T tile[padded_words<PAD>()];
    const int tid = threadIdx.x;
    const size_t base = (size_t)blockIdx.x * kRtsTile;
    T x[kBPer];
#pragma unroll
    for (int r = 0; r < kBPer; ++r) {
        const int i = tid + r * kBThreads;
        x[r] = base + i < n ? in[base + i] : T(0);
        tile[padded_word<PAD>(i)] = x[r];
    }
    __syncthreads();
    // Up-sweep: level `stride` has kRtsTile / (2 * stride) adds.
    for (int stride = 1; stride < (int)kRtsTile; stride <<= 1) {
        const int adds = (int)kRtsTile / (2 * stride);
        for (int k = tid; k < adds; k += kBThreads) {
            const int a = (2 * k + 1) * stride - 1;
            const int b = (2 * k + 2) * stride - 1;
            tile[padded_word<PAD>(b)] += tile[padded_word<PAD>(a)];
        }
        __syncthreads();
    }
    // Clear the root: the down-sweep then yields the exclusive scan.
    if (tid == 0) tile[padded_word<PAD>((int)kRtsTile - 1)] = T(0);
    __syncthreads();
    for (int stride = (int)kRtsTile / 2; stride > 0; stride >>= 1) {
        const int adds = (int)kRtsTile / (2 * stride);
        for (int k = tid; k < adds; k += kBThreads) {
            const int a = (2 * k + 1) * stride - 1;
            const int b = (2 * k + 2) * stride - 1;
            const T left = tile[padded_word<PAD>(a)];
            tile[padded_word<PAD>(a)] = tile[padded_word<PAD>(b)];
            tile[padded_word<PAD>(b)] += left;
        }
        __syncthreads();
    }
    const T off = offsets[blockIdx.x];
#pragma unroll
    for (int r = 0; r < kBPer; ++r) {
        const int i = tid + r * kBThreads;
        if (base + i < n) {
            const T ex = off + tile[padded_word<PAD>(i)];
            out[base + i] = INCLUSIVE ? ex + x[r] : ex;  // inclusive: one extra map
        }
    }
}

template <typename T, bool INCL>
static cudaError_t rts_typed(int tile_scan, const void* in_, void* out_, size_t n, void* totals_,
                             cudaStream_t s) {
    const T* in = static_cast<const T*>(in_);
    T* out = static_cast<T*>(out_);
    T* totals = static_cast<T*>(totals_);
    const uint32_t tiles = (uint32_t)((n + kRtsTile - 1) / kRtsTile);
    const bool al = aligned16(in, out);
    k_rts_reduce<T><<<tiles, kRThreads, 0, s>>>(in, n, totals, al);
    k_rts_scan_totals<T><<<1, 1024, 0, s>>>(totals, tiles);
    switch (tile_scan) {
        case 1: k_rts_scan_tiles_blelloch<T, INCL, 1><<<tiles, kBThreads, 0, s>>>(in, out, n, totals); break;
        case 2: k_rts_scan_tiles_blelloch<T, INCL, 2><<<tiles, kBThreads, 0, s>>>(in, out, n, totals); break;
        case 3: k_rts_scan_tiles_blelloch<T, INCL, 3><<<tiles, kBThreads, 0, s>>>(in, out, n, totals); break;
        default: k_rts_scan_tiles<T, INCL><<<tiles, kRThreads, 0, s>>>(in, out, n, totals, al); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_reduce_then_scan(Dtype dt, bool inclusive, int tile_scan, const void* in,
                                    void* out, size_t n, void* totals, cudaStream_t s) {
    if (dt == Dtype::F32)
        return inclusive ? rts_typed<float, true>(tile_scan, in, out, n, totals, s)
                         : rts_typed<float, false>(tile_scan, in, out, n, totals, s);
    return inclusive ? rts_typed<uint32_t, true>(tile_scan, in, out, n, totals, s)
                     : rts_typed<uint32_t, false>(tile_scan, in, out, n, totals, s);
}

}  // namespace ss
