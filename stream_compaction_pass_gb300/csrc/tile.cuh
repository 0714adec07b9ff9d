// tile.cuh -- the tile loader, the per-thread register scan, the warp scan
// of row sums and the block scan of warp totals, shared by the single-pass
// scan, the copy probe and the reduce-then-scan ablation.
//
// Data arrangement ("warp-striped rows"): a tile of THREADS * 4 * VPT
// elements is cut into one contiguous segment per warp; inside a warp's
// segment, row j (j = 0..VPT-1) is 128 consecutive elements and lane l holds
// elements 4l..4l+3 of every row as one 16-byte vector.  Every warp-wide
// load or store instruction therefore moves 512 contiguous bytes, and the
// scan order is (row, lane, element), so each row needs one warp scan of the
// lanes' 4-element sums.  This replaces the pages' "k consecutive items per
// thread" register scan ("Prefix sum and other parallel patterns",
// scan_tiles; "Parallel Prefix Sum (Scan) for NVIDIA T4 (sm_75)", How It
// Works steps 2-5) with an arrangement that needs no shared-memory transpose
// to keep loads coalesced.
#pragma once

#include "lookback.cuh"

namespace ss {

__device__ __forceinline__ uint4 ld_vec(const void* p) {
    uint4 r;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_vec(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Loads the warp's rows.  `fast`: the whole warp segment is in range and the
// pointer is 16-byte aligned; otherwise every element is guarded and the
// missing ones are the identity 0 ("CUDA prefix sum, the Hillis-Steele
// scan": the guard covers the load, zero is the identity).
template <typename T, int VPT>
__device__ __forceinline__ void load_rows(const T* in, size_t n, size_t seg, int lane, bool fast,
                                          T (&v)[VPT][4]) {
    if (fast) {
        const uint4* p = reinterpret_cast<const uint4*>(in + seg) + lane;
        uint4 r[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) r[j] = ld_vec(p + 32 * j);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            v[j][0] = from_bits<T>(r[j].x);
            v[j][1] = from_bits<T>(r[j].y);
            v[j][2] = from_bits<T>(r[j].z);
            v[j][3] = from_bits<T>(r[j].w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const size_t i = seg + (size_t)(32 * j + lane) * 4 + k;
                v[j][k] = i < n ? in[i] : T(0);
            }
    }
}

template <typename T, int VPT>
__device__ __forceinline__ void store_rows(T* out, size_t n, size_t seg, int lane, bool fast,
                                           const T (&y)[VPT][4]) {
    if (fast) {
        uint4* p = reinterpret_cast<uint4*>(out + seg) + lane;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
            st_vec(p + 32 * j, make_uint4(to_bits<T>(y[j][0]), to_bits<T>(y[j][1]),
                                          to_bits<T>(y[j][2]), to_bits<T>(y[j][3])));
    } else {
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const size_t i = seg + (size_t)(32 * j + lane) * 4 + k;
                if (i < n) out[i] = y[j][k];
            }
    }
}

// Per-thread row sums, one warp scan per row (the VPT scans interleaved for
// instruction-level parallelism), then the rows chained in order.
// pre[j] = sum of the warp segment's elements before this lane's row-j
// vector; returns the warp segment's total.
template <typename T, int VPT>
__device__ __forceinline__ T warp_rows_scan(const T (&v)[VPT][4], int lane, T (&pre)[VPT]) {
    T s[VPT], inc[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        s[j] = ((v[j][0] + v[j][1]) + v[j][2]) + v[j][3];
        inc[j] = s[j];
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            T t = __shfl_up_sync(kFullMask, inc[j], off);
            if (lane >= off) inc[j] += t;
        }
    }
    T run = T(0);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        T ex = __shfl_up_sync(kFullMask, inc[j], 1);
        if (lane == 0) ex = T(0);
        const T tot = __shfl_sync(kFullMask, inc[j], 31);
        pre[j] = run + ex;
        run += tot;
    }
    return run;
}

// Block scan of warp totals: every thread reads all warp totals from shared
// memory and sums them in warp order ("Prefix sum and other parallel
// patterns", block_exclusive_scan: each warp's last lane publishes its total,
// each warp adds the totals of the warps before it).
template <typename T, int WARPS>
__device__ __forceinline__ void block_combine(T warp_total, int warp, int lane, T* s_warp,
                                              T* warp_prefix, T* block_total) {
    if (lane == 0) s_warp[warp] = warp_total;
    __syncthreads();
    T wp = T(0), bt = T(0);
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        const T t = s_warp[w];
        if (w < warp) wp += t;
        bt += t;
    }
    *warp_prefix = wp;
    *block_total = bt;
}

// Outputs of one warp segment given the prefix of its first element.
template <typename T, int VPT, bool INCLUSIVE>
__device__ __forceinline__ void rows_output(const T (&v)[VPT][4], const T (&pre)[VPT], T base,
                                            T (&y)[VPT][4]) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        T r = base + pre[j];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (INCLUSIVE) {
                r += v[j][k];
                y[j][k] = r;
            } else {
                y[j][k] = r;
                r += v[j][k];
            }
        }
    }
}

// rows_output written over the rows themselves (saves a register copy).
template <typename T, int VPT, bool INCLUSIVE>
__device__ __forceinline__ void rows_output_inplace(T (&v)[VPT][4], const T (&pre)[VPT], T base) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        T r = base + pre[j];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const T x = v[j][k];
            if (INCLUSIVE) {
                r += x;
                v[j][k] = r;
            } else {
                v[j][k] = r;
                r += x;
            }
        }
    }
}

}  // namespace ss
