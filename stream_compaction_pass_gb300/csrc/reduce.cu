// reduce.cu -- the sum of a whole array, the first step of a scan split
// across devices.
//
// A scan split into P contiguous parts needs, before any part can be
// written, the sum of every part before it ("Prefix sum and other parallel
// patterns", A device-level scan: scan then propagate -- the block sums are
// scanned, then each block is offset by the sum of the blocks before it; here
// the blocks are whole devices' shares).  Each device reduces its part
// (n reads), the P totals are exchanged and exclusive-scanned, and each part
// is scanned seeded with its offset (2n), so 3n bytes move instead of the 4n
// of scanning first and adding the offset afterwards.
//
// One launch.  A grid of a few CTAs per SM strides over 16-byte vectors with
// several loads in flight per thread; each CTA's partial goes to the
// workspace, and the CTA that takes the last ticket adds the partials in CTA
// order and writes the total.  For a fixed n and grid the fp32 grouping is
// therefore the same on every run.  The ticket returns to zero at the end of
// every launch.
#include "internal.h"
#include "lookback.cuh"

namespace ss {

namespace {

constexpr int kReduceThreads = 512;
constexpr int kReduceUnroll = 4;  // 16-byte loads in flight per thread per step

template <typename T>
__device__ __forceinline__ T vec_sum(uint4 r) {
    return ((from_bits<T>(r.x) + from_bits<T>(r.y)) + from_bits<T>(r.z)) + from_bits<T>(r.w);
}

template <typename T>
__global__ void __launch_bounds__(kReduceThreads)
k_reduce_sum(const T* in, size_t n, T* partials, uint32_t* ticket, T* total, bool aligned) {
    constexpr int WARPS = kReduceThreads / 32;
    __shared__ T s_warp[WARPS];
    __shared__ bool s_last;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const size_t G = gridDim.x;
    T acc = T(0);
    if (aligned) {
        const size_t nv = n / 4;  // whole 16-byte vectors
        const uint4* v = reinterpret_cast<const uint4*>(in);
        const size_t stride = G * kReduceThreads;
        size_t i = (size_t)blockIdx.x * kReduceThreads + threadIdx.x;
        for (; i + (kReduceUnroll - 1) * stride < nv; i += kReduceUnroll * stride) {
            uint4 r[kReduceUnroll];
#pragma unroll
            for (int u = 0; u < kReduceUnroll; ++u) r[u] = __ldcs(v + i + u * stride);
#pragma unroll
            for (int u = 0; u < kReduceUnroll; ++u) acc += vec_sum<T>(r[u]);
        }
        for (; i < nv; i += stride) acc += vec_sum<T>(__ldcs(v + i));
        // the elements after the last whole vector
        for (size_t j = nv * 4 + (size_t)blockIdx.x * kReduceThreads + threadIdx.x; j < n; j += stride) acc += in[j];
    } else {
        for (size_t j = (size_t)blockIdx.x * kReduceThreads + threadIdx.x; j < n; j += G * kReduceThreads)
            acc += in[j];
    }
    acc = warp_sum(acc);
    if (lane == 0) s_warp[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        T b = T(0);
#pragma unroll
        for (int w = 0; w < WARPS; ++w) b += s_warp[w];
        partials[blockIdx.x] = b;
        __threadfence();  // the partial is visible before the ticket counts it
        s_last = atomicAdd(ticket, 1u) == (uint32_t)G - 1u;
    }
    __syncthreads();
    if (!s_last) return;
    // The last CTA: every other CTA's partial was written before its ticket.
    __threadfence();
    if (warp == 0) {
        T t = T(0);
        for (size_t b = 0; b < G; b += 32) {
            T p = (b + lane < G) ? *reinterpret_cast<volatile T*>(partials + b + lane) : T(0);
            t += warp_sum(p);  // a fixed tree per group of 32 partials, groups in order
        }
        if (lane == 0) {
            *total = t;
            *ticket = 0u;  // ready for the next launch on this workspace
        }
    }
}

}  // namespace

uint32_t reduce_grid(int sms) { return (uint32_t)(sms > 0 ? sms : 1) * 4u; }

cudaError_t launch_reduce_sum(Dtype dt, const void* in, size_t n, void* partials, uint32_t* ticket, void* total,
                              uint32_t grid, cudaStream_t s) {
    const bool aligned = (reinterpret_cast<uintptr_t>(in) & 15u) == 0;
    if (dt == Dtype::F32)
        k_reduce_sum<float><<<grid, kReduceThreads, 0, s>>>(static_cast<const float*>(in), n,
                                                            static_cast<float*>(partials), ticket,
                                                            static_cast<float*>(total), aligned);
    else
        k_reduce_sum<uint32_t><<<grid, kReduceThreads, 0, s>>>(static_cast<const uint32_t*>(in), n,
                                                               static_cast<uint32_t*>(partials), ticket,
                                                               static_cast<uint32_t*>(total), aligned);
    return cudaGetLastError();
}

}  // namespace ss
