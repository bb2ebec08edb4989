// Host-side caches of launch parameters that do not change between calls on a
// device (SM count, occupancy of a kernel, its shared-memory attribute), so a
// launch costs one driver call instead of several queries.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <tuple>

namespace convrot {

inline int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

inline std::mutex &launch_cache_mutex() {
    static std::mutex mu;
    return mu;
}

inline int sm_count() {
    static std::map<int, int> cache;
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(launch_cache_mutex());
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n;
    return n;
}

// Resident CTAs per SM of `kernel` with `threads` threads and `smem` dynamic bytes (at least 1).
inline int blocks_per_sm(const void *kernel, int threads, size_t smem) {
    static std::map<std::tuple<int, const void *, int, size_t>, int> cache;
    const auto key = std::make_tuple(current_device(), kernel, threads, smem);
    std::lock_guard<std::mutex> lock(launch_cache_mutex());
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    cache[key] = n;
    return n;
}

// Sets the dynamic shared-memory limit of `kernel` once per device.
inline cudaError_t ensure_smem_attr(const void *kernel, int bytes) {
    static std::map<std::tuple<int, const void *>, int> done;
    const auto key = std::make_tuple(current_device(), kernel);
    std::lock_guard<std::mutex> lock(launch_cache_mutex());
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[key] = bytes;
    return e;
}

}  // namespace convrot
