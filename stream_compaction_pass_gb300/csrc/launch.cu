// launch.cu -- launch set-up shared by the kernel launchers: the dynamic
// shared-memory limit of a kernel and the number of its CTAs an SM holds,
// kept per (kernel, device).  The shared-memory attribute belongs to the
// device it was set on, so a process that launches on several devices sets
// it once on each; the table is locked so that host threads that launch at
// the same time on a new device set it up once.
#include <map>
#include <mutex>
#include <utility>

#include "internal.h"

namespace ss {

namespace {
std::mutex g_setup_mu;
std::map<std::pair<const void*, int>, KernelSetup> g_setup;
}  // namespace

cudaError_t kernel_setup(const void* kern, int threads, size_t max_smem, KernelSetup* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    const auto key = std::make_pair(kern, dev);
    auto it = g_setup.find(key);
    if (it != g_setup.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    KernelSetup k;
    if (max_smem > 0) {  // also at 48 KB and below: static shared memory counts against the default limit
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
        if (e != cudaSuccess) return e;
    }
    e = cudaDeviceGetAttribute(&k.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int b = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, threads, max_smem);
    if (e != cudaSuccess) return e;
    k.sms = k.sms > 0 ? k.sms : 1;
    k.blocks_per_sm = b > 0 ? b : 1;
    g_setup[key] = k;
    *out = k;
    return cudaSuccess;
}

}  // namespace ss
