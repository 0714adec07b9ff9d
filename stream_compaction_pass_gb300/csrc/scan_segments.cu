// scan_segments.cu -- segmented scans: every segment [offsets[s],
// offsets[s+1]) of a flat array scanned on its own.  This is the general form
// of the batched (per-row) scans: variable-length rows, as in a batch of
// sequences of different lengths ("Prefix sum and other parallel patterns",
// In LLMs: MoE token dispatch, last paragraph, the per-row cumulative sums).
//
// Two launches:
//   1. k_segment_heads marks every segment start in a bitmask over the
//      elements (one bit per element, zeroed just before on the stream).
//   2. k_scan_segments runs the persistent single-pass scan (the schedule of
//      scan_pipe.cu's single-register-buffer kernel, with each tile claimed
//      from the counter when its copy starts) with a segmented add, each
//      thread owning 32 consecutive elements (below).
//      The segmented add works on pairs (f, s): f says whether a segment
//      starts in the span, s is the sum since the last start in it, or over
//      the whole span if none.  (fa, sa) then (fb, sb) gives
//      (fa | fb, fb ? sb : sa + sb).  It replaces the plain add in the
//      thread, warp and block steps.  A tile publishes the s of its whole span:
//      - a tile that contains a start publishes it at once as its inclusive
//        prefix (P), because what follows its last start depends on no
//        predecessor;
//      - any other tile publishes it as its aggregate (A) and looks back as
//        usual.
//      So look-backs stop at the nearest tile holding a segment start.  The
//      prefix found by the look-back applies only up to the tile's first
//      start.
// The array's first element always starts a segment.
#include <atomic>

#include "bulk.cuh"
#include "internal.h"
#include "tensor_copy.cuh"
#include "tile.cuh"

namespace ss {

namespace {

constexpr int kSThreads = 512;
constexpr int kSWarps = kSThreads / 32;
constexpr int kSVpt = 8;                                        // row-striped form: rows of 4 elements per lane
constexpr uint32_t kSSeg = 32u * kSVpt * 4;                     // 1024 elements per warp
constexpr int kSEpt = 32;                                       // blocked form: elements per thread, one 128-byte row
constexpr uint32_t kSTile = (uint32_t)kSThreads * kSEpt;        // 16384, the row-striped form's tile
constexpr int kSStages = 3;
static_assert(kSSeg * kSWarps == kSTile, "one warp segment per warp");
// The blocked form's CTA width by mean segment length: 64 threads (eight
// CTAs per SM) below kSegNarrowBelowMean, else 128 (four CTAs per SM).
constexpr size_t kSegNarrowBelowMean = 2048;

// Rows per tensor load of the blocked form (a tile is one row per thread).
__host__ __device__ constexpr uint32_t blocked_box_rows(int threads) { return threads < 256 ? (uint32_t)threads : 256u; }

// Which form ss_scan_segments takes: 0 by mean segment length, 1 row-striped,
// 2 / 3 / 4 / 5 blocked with 256 / 128 / 512 / 64 threads a CTA.
std::atomic<int> g_seg_config{0};  // read once per call; set from any thread
static_assert(kSTile >= kSegMinTile, "the workspace holds a descriptor per kSegMinTile elements");

template <typename T>
struct SegPair {
    uint32_t f;
    T s;
};

// (a) then (b), in element order.
template <typename T>
__device__ __forceinline__ SegPair<T> seg_add(SegPair<T> a, SegPair<T> b) {
    return SegPair<T>{a.f | b.f, b.f ? b.s : a.s + b.s};
}

// 16-byte shared-memory accesses at a byte address of the shared window.
__device__ __forceinline__ uint4 lds_vec_at(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr)
                 : "memory");
    return r;
}
__device__ __forceinline__ void sts_vec_at(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Inclusive segmented scan across the 32 lanes of a warp.
template <typename T>
__device__ __forceinline__ SegPair<T> warp_seg_scan(SegPair<T> p, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const T s_up = __shfl_up_sync(kFullMask, p.s, off);
        const uint32_t f_up = __shfl_up_sync(kFullMask, p.f, off);
        if (lane >= off) {
            if (!p.f) p.s += s_up;
            p.f |= f_up;
        }
    }
    return p;
}

}  // namespace

// One bit per segment start.  Each thread takes four consecutive offsets
// (two 16-byte loads when the array is 16-byte aligned, so that more loads
// are in flight), ORs together the starts that share a 32-bit word (the
// offsets are sorted, so they are neighbours) and makes one atomic OR per
// word.
__global__ void k_segment_heads(const unsigned long long* offsets, size_t num_segments, size_t n, uint32_t* bits) {
    const size_t quads = (num_segments + 3) / 4;
    const bool vec = (reinterpret_cast<uintptr_t>(offsets) & 15u) == 0;
    for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < quads; q += (size_t)gridDim.x * blockDim.x) {
        const size_t s0 = q * 4;
        unsigned long long p[4];
        if (vec && s0 + 4 <= num_segments) {
            const ulonglong2 a = __ldg(reinterpret_cast<const ulonglong2*>(offsets + s0));
            const ulonglong2 b = __ldg(reinterpret_cast<const ulonglong2*>(offsets + s0 + 2));
            p[0] = a.x;
            p[1] = a.y;
            p[2] = b.x;
            p[3] = b.y;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) p[e] = s0 + e < num_segments ? offsets[s0 + e] : (unsigned long long)n;
        }
        unsigned long long word = ~0ull;
        uint32_t acc = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (p[e] >= n) continue;
            const unsigned long long w = p[e] >> 5;
            const uint32_t b = 1u << (p[e] & 31u);
            if (w == word) {
                acc |= b;
            } else {
                if (acc) atomicOr(bits + word, acc);
                word = w;
                acc = b;
            }
        }
        if (acc) atomicOr(bits + word, acc);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && n > 0) atomicOr(bits, 1u);  // the first element starts a segment
}

// Row-striped form (lane l of a warp holds 16-byte vector 32j + l of the
// warp's share as its row j): each row is joined across the warp by its
// own segmented scan, which makes it the dearer form when segments are
// short.  It stores straight from registers, with one 512-thread CTA per SM;
// taken only when selected (ss_set_segments_config).
template <typename T, bool INCLUSIVE>
__global__ void __launch_bounds__(kSThreads, 1)
k_scan_segments_rows(const T* in, T* out, size_t n, const uint32_t* bits, uint32_t num_tiles, bool fast,
                LookbackCtx ctx) {
    constexpr int STAGES = kSStages;
    constexpr uint32_t TILE_BYTES = kSTile * (uint32_t)sizeof(T);
    constexpr uint32_t HEAD_WORDS = kSTile / 32;  // the tile's head bits, one word per 32 elements
    constexpr int VPT = kSVpt;

    // The element ring, then one head-bit area per stage: a full tile's
    // elements and head words arrive by two bulk copies on one barrier.
    extern __shared__ __align__(128) unsigned char smem_raw[];
    T* ring = reinterpret_cast<T*>(smem_raw);
    uint32_t* heads = reinterpret_cast<uint32_t*>(smem_raw + (size_t)STAGES * TILE_BYTES);
    __shared__ __align__(8) uint64_t bars[STAGES];
    __shared__ T s_ws[2][kSWarps];         // warp summaries, by tile parity
    __shared__ uint32_t s_wf[2][kSWarps];
    __shared__ T s_prefix[2];
    __shared__ uint32_t s_fail[2], s_epoch;
    __shared__ uint32_t s_tile[STAGES];  // the tile in each stage, kNoTile past the last

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t G = gridDim.x;
    const uint64_t policy = policy_evict_first();
    constexpr uint32_t kNoTile = 0xffffffffu;

    // Tiles are claimed one at a time, when their copy starts (the scheme of
    // scan_pipe.cu's default row): claims come out in increasing order, each
    // CTA stops at its first claim past the last tile, so a launch makes
    // num_tiles + G claims and the last one resets the counter.
    uint32_t issued = 0, consumed = 0;  // thread 0
    bool claims_done = false;           // thread 0
    auto claim_next = [&]() -> uint32_t {
        if (claims_done) return kNoTile;
        uint32_t id, ep;
        claim_tile(ctx.counter, num_tiles + G, &id, &ep);
        s_epoch = ep;
        if (id < num_tiles) return id;
        claims_done = true;
        return kNoTile;
    };
    auto full_tile = [&](uint32_t t) { return fast && (size_t)t * kSTile + kSTile <= n; };
    auto issue = [&](uint32_t k) {  // thread 0
        const int s = (int)(k % STAGES);
        const uint32_t t = claim_next();
        s_tile[s] = t;
        if (t != kNoTile) {
            if (full_tile(t)) {
                fence_async_shared();
                mbar_arrive_expect_tx(&bars[s], TILE_BYTES + HEAD_WORDS * 4);
                bulk_load(ring + (size_t)s * kSTile, in + (size_t)t * kSTile, TILE_BYTES, &bars[s], policy);
                bulk_load(heads + (size_t)s * HEAD_WORDS, bits + (size_t)t * HEAD_WORDS, HEAD_WORDS * 4, &bars[s],
                          policy);
            } else {
                mbar_arrive(&bars[s]);  // read from global with bounds checks instead
            }
        }
        issued = k + 1;
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_async_shared();
        for (uint32_t k = 0; k < (uint32_t)STAGES; ++k) issue(k);
    }
    __syncthreads();  // the barriers, the first slots' tile ids and the epoch
    const uint32_t epoch = s_epoch;
    // The tile in this CTA's k-th slot: thread 0 stored it when it started
    // the slot's copy; every reader is past a barrier that follows the store,
    // and the slot is only rewritten after a barrier that follows every read.
    auto tile_of = [&](uint32_t k) -> uint32_t { return s_tile[k % STAGES]; };

    // This lane's rows of slot k (tile t).
    auto read_rows = [&](uint32_t k, uint32_t t, T (&v)[VPT][4]) {
        const size_t tile_base = (size_t)t * kSTile;
        const size_t seg = tile_base + (size_t)warp * kSSeg;
        if (full_tile(t)) {
            const T* src = ring + (size_t)(k % STAGES) * kSTile + (size_t)warp * kSSeg + (size_t)lane * 4;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const uint4 r = lds_vec(src + 128 * j);
                v[j][0] = from_bits<T>(r.x);
                v[j][1] = from_bits<T>(r.y);
                v[j][2] = from_bits<T>(r.z);
                v[j][3] = from_bits<T>(r.w);
            }
        } else {
            load_rows<T, VPT>(in, n, seg, lane, false, v);
        }
    };
    // The lane's segmented summary of its row-j vector.
    auto lane_pair = [&](const T (&x)[4], uint32_t h) {
        T r = T(0);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if ((h >> e) & 1u) r = T(0);
            r += x[e];
        }
        return SegPair<T>{h != 0u ? 1u : 0u, r};
    };
    // Waits for tile k, forms its warp summaries and its own; publishes the
    // tile's s as P (a segment starts in it) or A.  Leaves the warp
    // summaries in s_ws/s_wf[k & 1]; returns the tile summary and this
    // lane's head bits (nibble j = row j).  A warp with no segment start in
    // its span sums plainly.
    auto reduce_publish = [&](uint32_t k, uint32_t t, SegPair<T>* tile_pair, uint32_t* hb_out) -> bool {
        const bool ok = mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) record_error(ctx.status, kErrBulkTimeout, t);
            return false;
        }
        uint32_t hb = 0;
        const bool full = full_tile(t);
        const uint32_t* hw = heads + (size_t)(k % STAGES) * HEAD_WORDS;
        const size_t wbase = (size_t)t * HEAD_WORDS;  // the tile's first head word in `bits`
        const size_t nwords = (n + 31) / 32;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const uint32_t p = warp * kSSeg + (32u * j + lane) * 4;  // element index in the tile
            const uint32_t word = full ? hw[p >> 5] : (wbase + (p >> 5) < nwords ? bits[wbase + (p >> 5)] : 0u);
            hb |= ((word >> (p & 31u)) & 15u) << (4 * j);
        }
        *hb_out = hb;
        T v[VPT][4];
        read_rows(k, t, v);
        // The warp's summary: whether a segment starts in its span, and the
        // sum from its last start on (or of the whole span).  Element order
        // is (row, lane, element); the last start is found with one ballot
        // per row, and each lane adds its share past it, so a single plain
        // warp sum gives the summary (no segmented scan per row).
        SegPair<T> w{0u, T(0)};
        int last_row = -1;
        uint32_t last_lanes = 0u;
        if (__any_sync(kFullMask, hb != 0u)) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const uint32_t b = __ballot_sync(kFullMask, ((hb >> (4 * j)) & 15u) != 0u);
                if (b) {
                    last_row = j;
                    last_lanes = b;
                }
            }
        }
        const int last_lane = last_row >= 0 ? 31 - __clz(last_lanes) : -1;
        T x = T(0);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const T rs = ((v[j][0] + v[j][1]) + v[j][2]) + v[j][3];
            if (j > last_row) {
                x += rs;
            } else if (j == last_row) {
                if (lane > last_lane) {
                    x += rs;
                } else if (lane == last_lane) {  // from this lane's last start in the row on
                    const uint32_t h = (hb >> (4 * j)) & 15u;
                    const int e0 = 31 - __clz(h);
                    T r = v[j][3];
                    if (e0 <= 2) r = v[j][2] + r;
                    if (e0 <= 1) r = v[j][1] + r;
                    if (e0 <= 0) r = v[j][0] + r;
                    x += r;
                }
            }
        }
        w.s = warp_sum(x);
        w.f = last_row >= 0 ? 1u : 0u;
        if (lane == 0) {
            s_ws[k & 1][warp] = w.s;
            s_wf[k & 1][warp] = w.f;
        }
        __syncthreads();
        SegPair<T> tp{0u, T(0)};
#pragma unroll
        for (int q = 0; q < kSWarps; ++q) tp = seg_add(tp, SegPair<T>{s_wf[k & 1][q], s_ws[k & 1][q]});
        *tile_pair = tp;
        if (threadIdx.x == 0 && (int64_t)t != ctx.fault_tile) {
            if (tp.f || t == 0) {
                if (num_tiles > 1) st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, to_bits<T>(tp.s)));
            } else {
                st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateA, to_bits<T>(tp.s)));
            }
        }
        compiler_fence();  // the summary just published stays ahead of the look-back
        return true;
    };

    SegPair<T> tp_cur{0u, T(0)}, tp_next{0u, T(0)};
    uint32_t hb_cur = 0, hb_next = 0;
    T prev_incl = T(0);
    int64_t prev_tile = -1;  // warp 0: this CTA's previous tile, whose inclusive prefix is prev_incl
    bool failed = false;
    uint32_t fail_at = 0;
    uint32_t t = tile_of(0);
    if (t != kNoTile && !reduce_publish(0, t, &tp_cur, &hb_cur)) failed = true;

    for (uint32_t k = 0; !failed && t != kNoTile; ++k) {
        const uint32_t tn = tile_of(k + 1);
        if (tn != kNoTile && !reduce_publish(k + 1, tn, &tp_next, &hb_next)) {
            failed = true;
            fail_at = k;
            break;
        }
        if (warp == 0) {
            T excl = T(0);
            bool lb_failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;
            } else {
                excl = lookback<T, 1>(ctx, t, epoch, lane, &lb_failed, nullptr, prev_tile, prev_incl);
                if (lane == 0) {
                    if (lb_failed) {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
                        record_error(ctx.status, kErrLookbackTimeout, t);
                    } else if (!tp_cur.f) {  // a tile holding a start published its P already
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, to_bits<T>(excl + tp_cur.s)));
                    }
                }
            }
            prev_incl = tp_cur.f ? tp_cur.s : excl + tp_cur.s;
            prev_tile = t;
            if (lane == 0) {
                s_prefix[k & 1] = excl;
                s_fail[k & 1] = lb_failed ? 1u : 0u;
            }
        }
        // Tile k's rows: lane summaries, segmented warp scans per row (or
        // plain ones where this warp's span holds no segment start).
        T v[VPT][4];
        read_rows(k, t, v);
        const uint32_t hb = hb_cur;
        const bool seg_warp = __any_sync(kFullMask, hb != 0u);
        SegPair<T> ex[VPT], rt[VPT];  // per row: what the lanes before hold, and the row's total
        if (seg_warp) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const SegPair<T> inc = warp_seg_scan<T>(lane_pair(v[j], (hb >> (4 * j)) & 15u), lane);
                const T s_b = __shfl_up_sync(kFullMask, inc.s, 1);
                const uint32_t f_b = __shfl_up_sync(kFullMask, inc.f, 1);
                ex[j] = lane > 0 ? SegPair<T>{f_b, s_b} : SegPair<T>{0u, T(0)};
                rt[j] = SegPair<T>{__shfl_sync(kFullMask, inc.f, 31), __shfl_sync(kFullMask, inc.s, 31)};
            }
        } else {  // no start in this warp's span: plain scans, the flags all 0
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const T inc = warp_inclusive_scan<T>(((v[j][0] + v[j][1]) + v[j][2]) + v[j][3], lane);
                const T s_b = __shfl_up_sync(kFullMask, inc, 1);
                ex[j] = SegPair<T>{0u, lane > 0 ? s_b : T(0)};
                rt[j] = SegPair<T>{0u, __shfl_sync(kFullMask, inc, 31)};
            }
        }
        __syncthreads();  // tile k read by everyone; the prefix is in shared memory
        if (threadIdx.x == 0) {
            consumed = k + 1;
            issue(k + STAGES);
        }
        if (s_fail[k & 1]) {
            failed = true;
            fail_at = k;
            break;
        }
        // What comes before this warp's segment: the warps before it, in order.
        SegPair<T> run{0u, T(0)};
        for (int q = 0; q < warp; ++q) run = seg_add(run, SegPair<T>{s_wf[k & 1][q], s_ws[k & 1][q]});
        const T excl = s_prefix[k & 1];
        const size_t tile_base = (size_t)t * kSTile;
        {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const SegPair<T> before = seg_add(run, ex[j]);
                T r = before.f ? before.s : excl + before.s;
                const uint32_t h = (hb >> (4 * j)) & 15u;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if ((h >> e) & 1u) r = T(0);
                    const T x = v[j][e];
                    if (INCLUSIVE) {
                        r += x;
                        v[j][e] = r;
                    } else {
                        v[j][e] = r;
                        r += x;
                    }
                }
                run = seg_add(run, rt[j]);
            }
        }
        store_rows<T, VPT>(out, n, tile_base + (size_t)warp * kSSeg, lane, full_tile(t), v);
        tp_cur = tp_next;
        hb_cur = hb_next;
        t = tn;
    }

    if (failed && threadIdx.x == 0) {
        // Leaving early: poison the tiles this CTA has claimed and every later
        // claim up to its first one past the last tile (which keeps the
        // launch's claim count exact); let copies in flight land.
        for (uint32_t j = fail_at + 1; j < issued; ++j) {
            const uint32_t tt = s_tile[j % STAGES];
            if (tt != kNoTile && (int64_t)tt != ctx.fault_tile)
                st_relaxed_u64(ctx.desc + tt, pack_desc(epoch, kStatePoison, 0u));
        }
        for (uint32_t tt = claim_next(); tt != kNoTile; tt = claim_next())
            if ((int64_t)tt != ctx.fault_tile) st_relaxed_u64(ctx.desc + tt, pack_desc(epoch, kStatePoison, 0u));
        for (uint32_t j = consumed; j < issued; ++j)
            if (s_tile[j % STAGES] != kNoTile)
                mbar_wait_bounded(&bars[j % STAGES], (j / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
}

template <typename T, bool INCL>
static cudaError_t launch_segments_rows(const void* in, void* out, size_t n, const uint32_t* bits,
                                   const LookbackWs& ws, cudaStream_t s) {
    constexpr size_t SMEM = 3 * (size_t)kSTile * sizeof(T) + 3 * (size_t)(kSTile / 32) * 4;  // + head words
    auto kern = k_scan_segments_rows<T, INCL>;
    KernelSetup su;
    cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), kSThreads, SMEM, &su);
    if (e != cudaSuccess) return e;
    const uint32_t tiles = (uint32_t)((n + kSTile - 1) / kSTile);
    const uint32_t grid = tiles < (uint32_t)su.sms ? tiles : (uint32_t)su.sms;
    const bool fast = ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out) |
                        reinterpret_cast<uintptr_t>(bits)) & 15u) == 0;
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    kern<<<grid, kSThreads, SMEM, s>>>(static_cast<const T*>(in), static_cast<T*>(out), n, bits, tiles, fast, ctx);
    return cudaGetLastError();
}

// Blocked form, THREADS threads a CTA and 512 / THREADS CTAs per SM (tiles of
// THREADS * 32 elements).  Each thread owns 32 consecutive elements of the tile (one
// 128-byte row) and the tile's head word that covers exactly them, so a
// thread's segments run through its registers in element order: its
// summary and its outputs are sequential adds with resets at its own starts,
// and one segmented scan across the warp per tile joins the threads (the
// row-striped layout needs one per row of 128 elements).
//  - Tensor copies with the 128-byte swizzle bring each tile into the ring
//    (row r's 16-byte chunk c at chunk c ^ (r mod 8)), so the 8 threads of a
//    quarter-warp, each reading its own row 16 bytes at a time, hit distinct
//    banks.  The tile's head words ride the same barrier by a bulk copy.
//  - Iteration k sums tile k+1 and publishes its summary; warp 0 looks back
//    for tile k; then every thread reads its row of tile k again, writes its
//    outputs over it, and each warp stores its 32 rows with one tensor copy.
//    The stage is refilled in the next iteration, once those stores have
//    read it.
template <typename T, bool INCLUSIVE, int THREADS>
__global__ void __launch_bounds__(THREADS, 512 / THREADS)
k_scan_segments_blocked(const T* in, T* out, size_t n, const uint32_t* bits, uint32_t num_tiles, bool fast,
                        LookbackCtx ctx, const __grid_constant__ CUtensorMap map_in,
                const __grid_constant__ CUtensorMap map_out) {
    constexpr int STAGES = kSStages;
    constexpr int EPT = kSEpt;
    constexpr int WARPS = THREADS / 32;
    constexpr uint32_t TILE = (uint32_t)THREADS * EPT;
    constexpr uint32_t TILE_BYTES = TILE * (uint32_t)sizeof(T);
    constexpr uint32_t ROWS = TILE / EPT;                  // rows per tile, one per thread
    constexpr uint32_t BOX_ROWS = blocked_box_rows(THREADS);  // rows per tensor load
    constexpr uint32_t HEAD_WORDS = TILE / 32;             // one head word per row
    static_assert(sizeof(T) == 4 && ROWS == (uint32_t)THREADS && ROWS % BOX_ROWS == 0 && HEAD_WORDS == ROWS &&
                      TILE >= kSegMinTile,
                  "tile geometry");

    // The ring (1024-byte aligned for the swizzle, rounded up into the 1 KB
    // of slack the launch adds), then one head-word area per stage.
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* const sbase = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    T* const ring = reinterpret_cast<T*>(sbase);
    uint32_t* const heads = reinterpret_cast<uint32_t*>(sbase + (size_t)STAGES * TILE_BYTES);
    __shared__ __align__(8) uint64_t bars[STAGES];
    __shared__ T s_ws[2][WARPS];         // warp summaries, by tile parity
    __shared__ uint32_t s_wf[2][WARPS];
    __shared__ T s_prefix[2];
    __shared__ uint32_t s_fail[2], s_epoch;
    __shared__ uint32_t s_tile[STAGES];  // the tile in each stage, kNoTile past the last

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t G = gridDim.x;
    const uint64_t policy = policy_evict_first();
    constexpr uint32_t kNoTile = 0xffffffffu;

    // Tiles are claimed one at a time, when their copy starts (the scheme of
    // scan_pipe.cu's default row): claims come out in increasing order, each
    // CTA stops at its first claim past the last tile, so a launch makes
    // num_tiles + G claims and the last one resets the counter.
    uint32_t issued = 0, consumed = 0;  // thread 0
    bool claims_done = false;           // thread 0
    auto claim_next = [&]() -> uint32_t {
        if (claims_done) return kNoTile;
        uint32_t id, ep;
        claim_tile(ctx.counter, num_tiles + G, &id, &ep);
        s_epoch = ep;
        if (id < num_tiles) return id;
        claims_done = true;
        return kNoTile;
    };
    auto full_tile = [&](uint32_t t) { return fast && (size_t)t * TILE + TILE <= n; };
    auto issue = [&](uint32_t k) {  // thread 0
        const int s = (int)(k % STAGES);
        const uint32_t t = claim_next();
        s_tile[s] = t;
        if (t != kNoTile) {
            if (full_tile(t)) {
                fence_async_shared();
                mbar_arrive_expect_tx(&bars[s], TILE_BYTES + HEAD_WORDS * 4);
                const int32_t row0 = (int32_t)((size_t)t * ROWS);
#pragma unroll
                for (uint32_t b = 0; b < ROWS / BOX_ROWS; ++b)
                    tensor_load_2d(ring + (size_t)s * TILE + (size_t)b * BOX_ROWS * EPT, &map_in, 0,
                                   row0 + (int32_t)(b * BOX_ROWS), &bars[s], policy);
                bulk_load(heads + (size_t)s * HEAD_WORDS, bits + (size_t)t * HEAD_WORDS, HEAD_WORDS * 4, &bars[s],
                          policy);
            } else {
                mbar_arrive(&bars[s]);  // read from global with bounds checks instead
            }
        }
        issued = k + 1;
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_async_shared();
        for (uint32_t k = 0; k < (uint32_t)STAGES; ++k) issue(k);
    }
    __syncthreads();  // the barriers, the first slots' tile ids and the epoch
    const uint32_t epoch = s_epoch;
    // The tile in this CTA's k-th slot: thread 0 stored it when it started
    // the slot's copy; every reader is past a barrier that follows the store,
    // and the slot is only rewritten after a barrier that follows every read.
    auto tile_of = [&](uint32_t k) -> uint32_t { return s_tile[k % STAGES]; };

    // This thread's 32 elements of slot k (tile t) and their head word.
    auto read_row = [&](uint32_t k, uint32_t t, T (&x)[EPT]) {
        if (full_tile(t)) {
            const uint32_t row = smem_u32(ring + (size_t)(k % STAGES) * TILE);
#pragma unroll
            for (int c = 0; c < EPT / 4; ++c) {
                const uint4 r = lds_vec_at(row + swizzle128_offset(threadIdx.x, (uint32_t)c));
                x[4 * c] = from_bits<T>(r.x);
                x[4 * c + 1] = from_bits<T>(r.y);
                x[4 * c + 2] = from_bits<T>(r.z);
                x[4 * c + 3] = from_bits<T>(r.w);
            }
        } else {
            const size_t e0 = (size_t)t * TILE + (size_t)threadIdx.x * EPT;
#pragma unroll
            for (int q = 0; q < EPT; ++q) x[q] = e0 + q < n ? in[e0 + q] : T(0);
        }
    };
    auto head_word = [&](uint32_t k, uint32_t t) -> uint32_t {
        if (full_tile(t)) return heads[(size_t)(k % STAGES) * HEAD_WORDS + threadIdx.x];
        const size_t w = (size_t)t * HEAD_WORDS + threadIdx.x;
        return w < (n + 31) / 32 ? bits[w] : 0u;
    };
    // Waits for slot k (tile t); this thread's summary (whether a segment
    // starts in its row, and the sum from its last start on, or of the whole
    // row) goes to *mine, the warps' to s_ws/s_wf[k & 1], the tile's to
    // *tile_pair; publishes the tile's as P (a segment starts in it) or A.
    auto reduce_publish = [&](uint32_t k, uint32_t t, SegPair<T>* tile_pair, SegPair<T>* mine, uint32_t* h_out) -> bool {
        const bool ok = mbar_wait_bounded(&bars[k % STAGES], (k / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) record_error(ctx.status, kErrBulkTimeout, t);
            return false;
        }
        if (threadIdx.x == 0) consumed = k + 1;
        const uint32_t h = head_word(k, t);
        *h_out = h;
        T x[EPT];
        read_row(k, t, x);
        T suf = T(0);
#pragma unroll
        for (int q = 0; q < EPT; ++q) {
            if ((h >> q) & 1u) suf = T(0);
            suf += x[q];
        }
        *mine = SegPair<T>{h != 0u ? 1u : 0u, suf};
        // The warp's summary: after its last thread holding a start, every
        // thread's sum is its whole row's.
        const uint32_t starts = __ballot_sync(kFullMask, h != 0u);
        const int last = starts ? 31 - __clz(starts) : -1;
        const T ws = warp_sum(lane >= last ? suf : T(0));
        if (lane == 0) {
            s_ws[k & 1][warp] = ws;
            s_wf[k & 1][warp] = starts ? 1u : 0u;
        }
        __syncthreads();
        SegPair<T> tp{0u, T(0)};
#pragma unroll
        for (int q = 0; q < WARPS; ++q) tp = seg_add(tp, SegPair<T>{s_wf[k & 1][q], s_ws[k & 1][q]});
        *tile_pair = tp;
        if (threadIdx.x == 0 && (int64_t)t != ctx.fault_tile) {
            if (tp.f || t == 0) {
                if (num_tiles > 1) st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, to_bits<T>(tp.s)));
            } else {
                st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateA, to_bits<T>(tp.s)));
            }
        }
        compiler_fence();  // the summary just published stays ahead of the look-back
        return true;
    };

    SegPair<T> tp_cur{0u, T(0)}, tp_next{0u, T(0)}, me_cur{0u, T(0)}, me_next{0u, T(0)};
    uint32_t h_cur = 0, h_next = 0;
    T prev_incl = T(0);
    int64_t prev_tile = -1;  // warp 0: this CTA's previous tile, whose inclusive prefix is prev_incl
    bool failed = false;
    uint32_t fail_at = 0;
    uint32_t t = tile_of(0);
    if (t != kNoTile && !reduce_publish(0, t, &tp_cur, &me_cur, &h_cur)) failed = true;

    for (uint32_t k = 0; !failed && t != kNoTile; ++k) {
        if (lane == 0) bulk_wait_group_read0();  // this warp's store of slot k-1 has read its stage
        const uint32_t tn = tile_of(k + 1);
        if (tn != kNoTile && !reduce_publish(k + 1, tn, &tp_next, &me_next, &h_next)) {
            failed = true;
            fail_at = k;
            break;
        }
        // Slot k-1's stage is free (every warp waited for its store before the
        // barriers above): refill it.  With no tile in slot k+1 the claims are
        // over and this claims nothing.
        if (threadIdx.x == 0 && k >= 1) issue(k + STAGES - 1);
        if (warp == 0) {
            T excl = T(0);
            bool lb_failed = false;
            const bool dead = (int64_t)t == ctx.fault_tile;  // test hook only
            if (t == 0) {
                lb_failed = dead;
            } else if (dead) {
                lb_failed = true;
            } else {
                excl = lookback<T, 1>(ctx, t, epoch, lane, &lb_failed, nullptr, prev_tile, prev_incl);
                if (lane == 0) {
                    if (lb_failed) {
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStatePoison, 0u));
                        record_error(ctx.status, kErrLookbackTimeout, t);
                    } else if (!tp_cur.f) {  // a tile holding a start published its P already
                        st_relaxed_u64(ctx.desc + t, pack_desc(epoch, kStateP, to_bits<T>(excl + tp_cur.s)));
                    }
                }
            }
            prev_incl = tp_cur.f ? tp_cur.s : excl + tp_cur.s;
            prev_tile = t;
            if (lane == 0) {
                s_prefix[k & 1] = excl;
                s_fail[k & 1] = lb_failed ? 1u : 0u;
            }
        }
        // What precedes this thread's row inside the warp: the threads before
        // it, joined by one segmented scan across the warp.
        const SegPair<T> inc = warp_seg_scan<T>(me_cur, lane);
        const T ex_s = __shfl_up_sync(kFullMask, inc.s, 1);
        const uint32_t ex_f = __shfl_up_sync(kFullMask, inc.f, 1);
        __syncthreads();  // the prefix is in shared memory
        if (s_fail[k & 1]) {
            failed = true;
            fail_at = k;
            break;
        }
        SegPair<T> run{0u, T(0)};  // the warps before this one, in order
        for (int q = 0; q < warp; ++q) run = seg_add(run, SegPair<T>{s_wf[k & 1][q], s_ws[k & 1][q]});
        const SegPair<T> before = lane > 0 ? seg_add(run, SegPair<T>{ex_f, ex_s}) : run;
        T r = before.f ? before.s : s_prefix[k & 1] + before.s;
        T x[EPT];
        read_row(k, t, x);
        const uint32_t h = h_cur;
#pragma unroll
        for (int q = 0; q < EPT; ++q) {
            if ((h >> q) & 1u) r = T(0);
            if (INCLUSIVE) {
                r += x[q];
                x[q] = r;
            } else {
                const T v = x[q];
                x[q] = r;
                r += v;
            }
        }
        if (full_tile(t)) {  // over this thread's row of the stage, then the warp's 32 rows in one store
            const uint32_t row = smem_u32(ring + (size_t)(k % STAGES) * TILE);
#pragma unroll
            for (int c = 0; c < EPT / 4; ++c)
                sts_vec_at(row + swizzle128_offset(threadIdx.x, (uint32_t)c),
                           make_uint4(to_bits<T>(x[4 * c]), to_bits<T>(x[4 * c + 1]), to_bits<T>(x[4 * c + 2]),
                                      to_bits<T>(x[4 * c + 3])));
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
                tensor_store_2d(&map_out, 0, (int32_t)((size_t)t * ROWS + (size_t)warp * 32),
                                ring + (size_t)(k % STAGES) * TILE + (size_t)warp * 32 * EPT);
                bulk_commit_group();
            }
        } else {
            const size_t e0 = (size_t)t * TILE + (size_t)threadIdx.x * EPT;
#pragma unroll
            for (int q = 0; q < EPT; ++q)
                if (e0 + q < n) out[e0 + q] = x[q];
        }
        tp_cur = tp_next;
        me_cur = me_next;
        h_cur = h_next;
        t = tn;
    }

    if (failed && threadIdx.x == 0) {
        // Leaving early: poison the tiles this CTA has claimed and every later
        // claim up to its first one past the last tile (which keeps the
        // launch's claim count exact); let copies in flight land.
        for (uint32_t j = fail_at + 1; j < issued; ++j) {
            const uint32_t tt = s_tile[j % STAGES];
            if (tt != kNoTile && (int64_t)tt != ctx.fault_tile)
                st_relaxed_u64(ctx.desc + tt, pack_desc(epoch, kStatePoison, 0u));
        }
        for (uint32_t tt = claim_next(); tt != kNoTile; tt = claim_next())
            if ((int64_t)tt != ctx.fault_tile) st_relaxed_u64(ctx.desc + tt, pack_desc(epoch, kStatePoison, 0u));
        for (uint32_t j = consumed; j < issued; ++j)
            if (s_tile[j % STAGES] != kNoTile)
                mbar_wait_bounded(&bars[j % STAGES], (j / STAGES) & 1u, ctx.max_polls, ctx.timeout_ns);
    }
    if (lane == 0) bulk_wait_group0();  // this warp's output stores are complete before the CTA leaves
}

template <typename T, bool INCL, int THREADS>
static cudaError_t launch_segments_blocked(const void* in, void* out, size_t n, const uint32_t* bits,
                                           const LookbackWs& ws, cudaStream_t s) {
    constexpr size_t TILE = (size_t)THREADS * kSEpt;
    // the ring, the head words, alignment slack
    constexpr size_t SMEM = kSStages * TILE * sizeof(T) + kSStages * (TILE / 32) * 4 + 1024;
    auto kern = k_scan_segments_blocked<T, INCL, THREADS>;
    KernelSetup su;
    cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kern), THREADS, SMEM, &su);
    if (e != cudaSuccess) return e;
    const uint32_t tiles = (uint32_t)((n + TILE - 1) / TILE);
    const uint32_t resident = (uint32_t)(su.sms * su.blocks_per_sm);
    const uint32_t grid = tiles < resident ? tiles : resident;
    // Full tiles go through the tensor copies: every buffer 16-byte aligned,
    // at least one full tile, and every row coordinate in the copies' signed
    // 32-bit range.
    const uint64_t rows = n / 32;
    const bool fast = ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out) |
                        reinterpret_cast<uintptr_t>(bits)) & 15u) == 0 &&
                      n >= TILE && rows <= (uint64_t)INT32_MAX;
    CUtensorMap map_in{}, map_out{};
    if (fast) {
        e = encode_rows128_b32(&map_in, in, rows, blocked_box_rows(THREADS));
        if (e == cudaSuccess) e = encode_rows128_b32(&map_out, out, rows, 32);
        if (e != cudaSuccess) return e;
    }
    LookbackCtx ctx{ws.desc, ws.counter, ws.status, ws.timeout_ns, ws.max_polls, ws.fault_tile};
    kern<<<grid, THREADS, SMEM, s>>>(static_cast<const T*>(in), static_cast<T*>(out), n, bits, tiles, fast, ctx,
                                       map_in, map_out);
    return cudaGetLastError();
}

template <typename T, bool INCL>
static cudaError_t launch_segments_form(int form, const void* in, void* out, size_t n, const uint32_t* bits,
                                        const LookbackWs& ws, cudaStream_t s) {
    switch (form) {
        case 1: return launch_segments_rows<T, INCL>(in, out, n, bits, ws, s);
        case 2: return launch_segments_blocked<T, INCL, 256>(in, out, n, bits, ws, s);
        case 3: return launch_segments_blocked<T, INCL, 128>(in, out, n, bits, ws, s);
        case 4: return launch_segments_blocked<T, INCL, 512>(in, out, n, bits, ws, s);
        case 5: return launch_segments_blocked<T, INCL, 64>(in, out, n, bits, ws, s);
        default: return cudaErrorInvalidValue;
    }
}

int segments_config_count() { return 6; }
void set_segments_config(int c) { g_seg_config.store(c, std::memory_order_relaxed); }

cudaError_t launch_scan_segments(Dtype dt, bool inclusive, const void* in, void* out, size_t n,
                                 const unsigned long long* offsets, size_t num_segments, uint32_t* bits,
                                 const LookbackWs& ws, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(bits, 0, ((n + 31) / 32) * 4, s);
    if (e != cudaSuccess) return e;
    const size_t blocks = ((num_segments + 3) / 4 + 255) / 256;
    const unsigned grid = (unsigned)(blocks == 0 ? 1 : (blocks < 4096 ? blocks : 4096));
    k_segment_heads<<<grid, 256, 0, s>>>(offsets, num_segments, n, bits);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // The form by mean segment length (n / segments), measured at n = 1e8, fp32
    // inclusive, start marking included (ms; blocked with 64 / 128 / 256 / 512
    // threads a CTA, then row-striped): mean 4, 0.171 / 0.174 / 0.180 / 0.217
    // / 0.230; 100, 0.136 / 0.138 / 0.144 / 0.182 / 0.196; 1000, 0.133 / 0.134
    // / 0.140 / 0.178 / 0.186; 5000, 0.144 / 0.140 / 0.142 / 0.178 / 0.174;
    // 128,256, 0.158 / 0.153 / 0.158 / 0.187 / 0.173.  Narrow CTAs keep more
    // tiles in flight per SM; with short segments nearly every tile holds a
    // start, so its look-back ends at its predecessor.
    int form = g_seg_config.load(std::memory_order_relaxed);
    if (form == 0) form = num_segments > 0 && n / num_segments < kSegNarrowBelowMean ? 5 : 3;
    if (dt == Dtype::F32)
        return inclusive ? launch_segments_form<float, true>(form, in, out, n, bits, ws, s)
                         : launch_segments_form<float, false>(form, in, out, n, bits, ws, s);
    return inclusive ? launch_segments_form<uint32_t, true>(form, in, out, n, bits, ws, s)
                     : launch_segments_form<uint32_t, false>(form, in, out, n, bits, ws, s);
}

}  // namespace ss
