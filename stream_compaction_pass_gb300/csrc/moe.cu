// moe.cu -- MoE token counts and tile-aligned expert offsets.
//
// "Prefix sum and other parallel patterns", In LLMs: MoE token dispatch
// (steps 1 and 2) and Exercise 2:
//   counts[e]    = number of ids equal to e            (histogram)
//   offsets[0]   = 0
//   offsets[e+1] = offsets[e] + align * ceil(counts[e] / align)
// so offsets[e] is where expert e's tokens start when every expert's segment
// is padded to whole GEMM tiles of `align` rows, and offsets[E] is the padded
// total.  An id outside [0, E) is not counted.
//
// One launch, following the exercise's outline:
//   1. each CTA counts its stretch of ids into a shared-memory histogram
//      (E bins) with shared atomics, 16-byte vector loads where aligned;
//   2. it adds its nonzero bins into a global accumulator of E words with
//      reductions (fire-and-forget atomics spread over E addresses), fences,
//      and takes a ticket;
//   3. the CTA that draws the last ticket reads the accumulator into
//      counts[E] and zeroes it again, rounds each count up to the tile, and
//      scans the rounded counts with one block scan (E is tens to thousands,
//      so one block suffices, as the exercise notes).  It then returns the
//      ticket to 0.  The accumulator and the ticket are left as they were
//      found, so the next launch on the stream needs no clearing.
// The last CTA reads the accumulator only after every CTA's reductions,
// fence and ticket.  No CTA waits for another, so nothing here can spin.
#include "internal.h"
#include "tile.cuh"

namespace ss {

namespace {

constexpr int kMoeThreads = 512;
constexpr int kMoeWarps = kMoeThreads / 32;

__device__ __forceinline__ void count_id(uint32_t* hist, int32_t id, int32_t num_experts) {
    if (id >= 0 && id < num_experts) atomicAdd(&hist[id], 1u);
}

__device__ __forceinline__ uint32_t ld_cg_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

}  // namespace

__global__ void __launch_bounds__(kMoeThreads)
k_moe_counts_offsets(const int32_t* ids, size_t m, int32_t num_experts, uint32_t align, size_t chunk,
                     bool vec, uint32_t* acc, uint32_t* ticket, uint32_t* counts, uint32_t* offsets) {
    extern __shared__ uint32_t hist[];  // num_experts bins
    __shared__ uint32_t s_warp[kMoeWarps];
    __shared__ uint32_t s_last;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t G = gridDim.x;

    for (int e = threadIdx.x; e < num_experts; e += kMoeThreads) hist[e] = 0u;
    __syncthreads();

    const size_t lo = (size_t)blockIdx.x * chunk;
    const size_t hi = lo + chunk < m ? lo + chunk : m;
    if (lo < hi) {
        if (vec) {  // chunk is a multiple of 4 and ids is 16-byte aligned
            const size_t nv = (hi - lo) / 4;
            const int4* v = reinterpret_cast<const int4*>(ids + lo);
            for (size_t i = threadIdx.x; i < nv; i += kMoeThreads) {
                const int4 q = v[i];
                count_id(hist, q.x, num_experts);
                count_id(hist, q.y, num_experts);
                count_id(hist, q.z, num_experts);
                count_id(hist, q.w, num_experts);
            }
            for (size_t i = lo + nv * 4 + threadIdx.x; i < hi; i += kMoeThreads) count_id(hist, ids[i], num_experts);
        } else {
            for (size_t i = lo + threadIdx.x; i < hi; i += kMoeThreads) count_id(hist, ids[i], num_experts);
        }
    }
    __syncthreads();

    for (int e = threadIdx.x; e < num_experts; e += kMoeThreads) {
        const uint32_t c = hist[e];
        if (c != 0u) atomicAdd(&acc[e], c);  // result unused: compiles to a reduction
    }
    __threadfence();  // this CTA's reductions are performed before its ticket
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1u) == G - 1u ? 1u : 0u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();  // every CTA's reductions are visible after the last ticket

    // Thread j owns the contiguous run of experts [j * per, (j + 1) * per).
    const int per = (num_experts + kMoeThreads - 1) / kMoeThreads;
    const int e0 = threadIdx.x * per;
    for (int e = threadIdx.x; e < num_experts; e += kMoeThreads) {  // coalesced pass over the accumulator
        const uint32_t c = ld_cg_u32(acc + e);
        acc[e] = 0u;  // left clean for the next launch
        counts[e] = c;
        hist[e] = c;
    }
    __syncthreads();
    uint32_t run_total = 0;
    for (int q = 0; q < per; ++q) {
        const int e = e0 + q;
        if (e >= num_experts) break;
        run_total += (hist[e] + align - 1u) / align * align;
    }
    uint32_t warp_prefix, block_total;
    const uint32_t lane_incl = warp_inclusive_scan<uint32_t>(run_total, lane);
    block_combine<uint32_t, kMoeWarps>(__shfl_sync(kFullMask, lane_incl, 31), warp, lane, s_warp, &warp_prefix,
                                       &block_total);
    uint32_t off = warp_prefix + lane_incl - run_total;
    for (int q = 0; q < per; ++q) {
        const int e = e0 + q;
        if (e >= num_experts) break;
        offsets[e] = off;
        off += (hist[e] + align - 1u) / align * align;
    }
    if (threadIdx.x == 0) {
        offsets[num_experts] = block_total;
        *ticket = 0u;  // ready for the next launch on this stream
    }
}

cudaError_t launch_moe_counts_offsets(const int32_t* ids, size_t m, int32_t num_experts, uint32_t align,
                                      uint32_t* counts, uint32_t* offsets, uint32_t* acc, uint32_t* ticket,
                                      uint32_t grid, cudaStream_t s) {
    const size_t smem = (size_t)num_experts * 4;
    if (smem > 0) {  // the limit is raised once per device, to the largest expert count
        KernelSetup su;
        cudaError_t e = kernel_setup(reinterpret_cast<const void*>(k_moe_counts_offsets), kMoeThreads,
                                     (size_t)kMoeMaxExperts * 4, &su);
        if (e != cudaSuccess) return e;
    }
    size_t chunk = (m + grid - 1) / grid;
    chunk = (chunk + 3) / 4 * 4;
    const bool vec = (reinterpret_cast<uintptr_t>(ids) & 15u) == 0;
    k_moe_counts_offsets<<<grid, kMoeThreads, smem, s>>>(ids, m, num_experts, align, chunk, vec, acc, ticket,
                                                         counts, offsets);
    return cudaGetLastError();
}

uint32_t moe_grid(size_t m, int sms) {
    const size_t per_cta = 8192;  // ids per CTA before another CTA pays off
    size_t g = (m + per_cta - 1) / per_cta;
    if (g < 1) g = 1;
    if (g > (size_t)sms) g = (size_t)sms;
    return (uint32_t)g;
}

}  // namespace ss
