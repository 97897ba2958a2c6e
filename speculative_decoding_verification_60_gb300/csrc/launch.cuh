// Host-side launch helpers: grid sizing against the SM count, opt-in to
// large dynamic shared memory.
#pragma once

#include <cuda_runtime.h>

namespace sv {

// Make the device that owns `p` current for this library's CUDA runtime
// (the runtime is linked statically, so its current device is its own).
inline bool select_device_of(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return false;
    return cudaSetDevice(at.device) == cudaSuccess;
}

inline int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Persistent grid: min(work, SMs * resident CTAs per SM).  Sets the
// kernel's dynamic shared-memory limit first.
template <typename K>
inline bool launch_grid(K kernel, size_t dyn_smem, long long work, int* grid, int block = 512) {
    if (dyn_smem > 0 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_smem) != cudaSuccess)
        return false;
    // large shared-memory users ask for the whole carve-out, so that the
    // resident-CTA count below is what runs
    if (dyn_smem >= 48 * 1024 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return false;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, dyn_smem) != cudaSuccess) return false;
    const int sms = sm_count();
    if (per_sm < 1 || sms < 1) return false;
    long long g = (long long)sms * per_sm;
    if (work < g) g = work;
    *grid = (int)(g < 1 ? 1 : g);
    return true;
}

// Opt in to dyn_smem bytes of dynamic shared memory: static plus dynamic
// above 48 KiB needs it even when the dynamic part alone is smaller.
template <typename K>
inline bool set_dyn_smem(K kernel, size_t dyn_smem) {
    if (dyn_smem == 0) return true;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_smem) == cudaSuccess;
}

}  // namespace sv
