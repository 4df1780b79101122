// launch_cache.cpp -- resident-CTA counts for the persistent decode grid.
//
// The grid is (SM count) x (CTAs of this kernel that fit on one SM at the
// call's shared-memory size).  Both numbers are queried once per (kernel,
// device, size) and kept for the life of the process; the kernel's dynamic
// shared-memory limit is raised once per (kernel, device) to the largest size
// any call can request.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

namespace lar {

namespace {

struct Entry {
    const void* kern;
    int dev;
    size_t smem;
    int occ;
    int sms;
};

std::mutex g_mu;
std::vector<Entry> g_cache;
std::vector<std::pair<const void*, int>> g_raised;  // (kernel, device) with the smem limit raised

}  // namespace

int cached_occupancy(const void* kern, int threads, size_t smem, size_t smem_max, int* sms_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    for (const Entry& e : g_cache)
        if (e.kern == kern && e.dev == dev && e.smem == smem) {
            *sms_out = e.sms;
            return e.occ;
        }
    bool raised = false;
    for (const auto& kd : g_raised) raised |= kd.first == kern && kd.second == dev;
    if (!raised) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem_max)) != cudaSuccess)
            return 0;
        g_raised.emplace_back(kern, dev);
    }
    int sms = 0, occ = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem) != cudaSuccess) return 0;
    g_cache.push_back({kern, dev, smem, occ, sms});
    *sms_out = sms;
    return occ;
}

}  // namespace lar
