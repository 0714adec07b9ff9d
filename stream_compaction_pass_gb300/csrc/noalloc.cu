// noalloc.cu -- ss_scan_noalloc: the single-pass look-back scan for callers
// that may not allocate device memory.
//
// Some callers cannot call cudaMalloc: a host application that hands out
// every byte of device memory from its own pool and forbids other
// allocations (so that its accounting stays exact), or a latency-critical
// loop that must never pay for an allocation or the synchronisation that
// freeing can bring.  The regular entry points allocate a per-stream
// workspace on first use; this one never does.  Its scratch -- the tile
// counter, the status words and the tile descriptors -- lives in the
// file-scope device array below, which every GPU that loads the library
// holds until the process exits (2 MiB + 256 bytes per device).
//
// The scratch is shared by every call on a device and keeps the last call's
// contents.  Nothing has to be cleared between calls: the tile counter's
// count returns to zero at the end of every launch, and each launch tags its
// descriptors with a new epoch, so the previous call's descriptors read as
// "not yet published".  The whole array is zeroed once per device at set-up,
// and the descriptors again every 2^29 calls, before an epoch tag can come
// round.  Calls that overlap on the GPU (on different streams, or
// concurrent host threads with per-thread default streams) share the counter
// and descriptors and race; serialise them.
#include <cstdint>
#include <mutex>

#include "../../include/streamscan.h"
#include "internal.h"

namespace {

constexpr int kNoAllocConfig = 0;                  // 256 threads x 16 elements per tile
constexpr size_t kNoAllocTile = 4096;
constexpr size_t kNoAllocMaxTiles = (size_t)1 << 18;  // 2^18 tiles: n <= 2^30 elements
constexpr size_t kHeaderWords = 32;                 // 256 bytes: counter, status words
constexpr size_t kScratchWords = kHeaderWords + kNoAllocMaxTiles;
constexpr uint64_t kClearEvery = 1ull << 29;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned long long g_noalloc_scratch[kScratchWords];

std::mutex g_na_mu;
unsigned long long* g_na_ptr[kMaxDevices] = {};
uint64_t g_na_calls[kMaxDevices] = {};

// The returned status is this entry point's only error report; `why` names
// the reason for a reader of this file.
ss_status na_fail(ss_status st, const char* why) {
    (void)why;
    return st;
}

}  // namespace

// Test hook: sets the number of calls made so far on the current device, so
// that a test can reach the periodic descriptor clear without 2^29 calls.
extern "C" ss_status ss_debug_set_noalloc_calls(uint64_t calls) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return na_fail(SS_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return na_fail(SS_ERR_UNSUPPORTED, "device index too large");
    std::lock_guard<std::mutex> lk(g_na_mu);
    g_na_calls[dev] = calls;
    return SS_OK;
}

// The number of calls after which the descriptors are cleared (for tests).
extern "C" uint64_t ss_debug_noalloc_clear_period(void) { return kClearEvery; }

extern "C" ss_status ss_scan_noalloc(ss_dtype dtype, int inclusive, const void* in, void* out, size_t n,
                                     ss_stream_t stream) {
    if (dtype != SS_I32 && dtype != SS_U32 && dtype != SS_F32)
        return na_fail(SS_ERR_UNSUPPORTED, "unknown dtype");
    if (n == 0) return SS_OK;
    if (in == nullptr || out == nullptr) return na_fail(SS_ERR_INVALID_ARG, "null pointer with n > 0");
    if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 3u)
        return na_fail(SS_ERR_INVALID_ARG, "in/out must be 4-byte aligned");
    const size_t tiles = (n + kNoAllocTile - 1) / kNoAllocTile;
    if (tiles > kNoAllocMaxTiles)
        return na_fail(SS_ERR_INVALID_ARG, "n exceeds the no-alloc maximum of 2^30 elements");
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    if (a != b && a < b + n * 4 && b < a + n * 4)
        return na_fail(SS_ERR_INVALID_ARG, "in and out partially overlap");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return na_fail(SS_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return na_fail(SS_ERR_UNSUPPORTED, "device index too large");
    cudaStream_t s = (cudaStream_t)stream;
    // The scratch array is picked by the current device, so the stream must
    // belong to that device: a stream of another device would pair this
    // device's array with the other device's launch.
    int stream_dev = dev;
    e = cudaStreamGetDevice(s, &stream_dev);
    if (e != cudaSuccess) return na_fail(SS_ERR_CUDA, cudaGetErrorString(e));
    if (stream_dev != dev) return na_fail(SS_ERR_INVALID_ARG, "the stream belongs to another device than the current one");

    unsigned long long* scratch;
    {
        std::lock_guard<std::mutex> lk(g_na_mu);
        if (g_na_ptr[dev] == nullptr) {
            // Set-up, once per device with that device current.  The symbol's
            // host-side name is only a stand-in; the kernel needs the device
            // address.
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) return na_fail(SS_ERR_CUDA, cudaGetErrorString(e));
            e = cudaMemset(p, 0, sizeof(g_noalloc_scratch));
            if (e == cudaSuccess) e = cudaDeviceSynchronize();
            if (e != cudaSuccess) return na_fail(SS_ERR_CUDA, cudaGetErrorString(e));
            g_na_ptr[dev] = static_cast<unsigned long long*>(p);
        }
        scratch = g_na_ptr[dev];
        if (++g_na_calls[dev] % kClearEvery == 0) {
            e = cudaMemsetAsync(scratch + kHeaderWords, 0, kNoAllocMaxTiles * 8, s);
            if (e != cudaSuccess) return na_fail(SS_ERR_CUDA, cudaGetErrorString(e));
        }
    }

    ss::LookbackWs ws;
    ws.counter = scratch;
    ws.status = reinterpret_cast<uint32_t*>(scratch + 1);
    ws.desc = scratch + kHeaderWords;
    const ss::Dtype dt = dtype == SS_F32 ? ss::Dtype::F32 : (dtype == SS_U32 ? ss::Dtype::U32 : ss::Dtype::I32);
    e = ss::launch_scan_lookback(dt, inclusive != 0, kNoAllocConfig, in, out, n, ws, nullptr, nullptr, s);
    if (e != cudaSuccess) return na_fail(SS_ERR_CUDA, cudaGetErrorString(e));
    return SS_OK;
}
