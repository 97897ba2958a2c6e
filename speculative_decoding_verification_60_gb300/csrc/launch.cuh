// Host-side launch helpers: the caller's current device kept across a call,
// grid sizing against the SM count, opt-in to large dynamic shared memory,
// both cached per (device, kernel, shared memory, block).
#pragma once

#include <cuda_runtime.h>

#include <mutex>

namespace sv {

// Puts back, when the scope ends, the device that was current when it
// began: the entry points make the logits' device current for their own
// launches and must not leave the caller on another device.
class DeviceGuard {
  public:
    DeviceGuard() {
        ok_ = cudaGetDevice(&prev_) == cudaSuccess;
        if (!ok_) cudaGetLastError();
    }
    ~DeviceGuard() {
        if (!ok_) return;
        int cur = -1;
        if (cudaGetDevice(&cur) == cudaSuccess && cur != prev_) cudaSetDevice(prev_);
    }
    DeviceGuard(const DeviceGuard&) = delete;
    DeviceGuard& operator=(const DeviceGuard&) = delete;

  private:
    int prev_ = 0;
    bool ok_ = false;
};

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

// Resident CTAs per SM and SM count of a kernel launch configuration on the
// current device, with the kernel's shared-memory attributes set.  The
// first call per (device, kernel, dyn_smem, block) queries and sets; later
// calls read the cache.
struct LaunchShape {
    int per_sm, sms;
};
inline bool launch_shape(const void* kernel, size_t dyn_smem, int block, LaunchShape* out) {
    struct Entry {
        const void* fn;
        int dev;
        size_t dyn;
        int block;
        LaunchShape shape;
    };
    constexpr int kEntries = 64;
    static std::mutex mu;
    static Entry table[kEntries];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (table[i].fn == kernel && table[i].dev == dev && table[i].dyn == dyn_smem && table[i].block == block) {
                *out = table[i].shape;
                return true;
            }
    }
    if (dyn_smem > 0 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_smem) != cudaSuccess)
        return false;
    // large shared-memory users ask for the whole carve-out, so that the
    // resident-CTA count below is what runs
    if (dyn_smem >= 48 * 1024 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return false;
    LaunchShape sh{0, 0};
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&sh.per_sm, kernel, block, dyn_smem) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&sh.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (sh.per_sm < 1 || sh.sms < 1) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (used < kEntries) table[used++] = Entry{kernel, dev, dyn_smem, block, sh};
    *out = sh;
    return true;
}

// Persistent grid: min(work, SMs * resident CTAs per SM).
template <typename K>
inline bool launch_grid(K kernel, size_t dyn_smem, long long work, int* grid, int block = 512) {
    LaunchShape sh;
    if (!launch_shape(reinterpret_cast<const void*>(kernel), dyn_smem, block, &sh)) return false;
    long long g = (long long)sh.sms * sh.per_sm;
    if (work < g) g = work;
    *grid = (int)(g < 1 ? 1 : g);
    return true;
}

// Opt in to dyn_smem bytes of dynamic shared memory (static plus dynamic
// above 48 KiB needs it even when the dynamic part alone is smaller); the
// attribute is set once per (device, kernel, size).
template <typename K>
inline bool set_dyn_smem(K kernel, size_t dyn_smem, int block) {
    if (dyn_smem == 0) return true;
    LaunchShape sh;
    return launch_shape(reinterpret_cast<const void*>(kernel), dyn_smem, block, &sh);
}

// Launch that may overlap its start with the end of the kernel before it on
// the stream (programmatic dependent launch): its CTAs are scheduled once
// every CTA of that kernel has started (each calls grid_dep_trigger first),
// and wait in grid_dep_wait, before reading anything it wrote, until it has
// completed.  After any other stream operation it is an ordinary launch.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t dyn_smem, cudaStream_t st,
                                    Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = dyn_smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace sv
