// api.cu -- status strings and the per-device fact cache.
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace fp8lin {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::atomic<bool> g_have[kMaxDevices];
std::mutex g_mu;
}  // namespace

fp8lin_status current_device(DeviceInfo *info) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8LIN_ERR_CUDA;
    if (!g_have[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_have[dev].load(std::memory_order_relaxed)) {
            DeviceInfo d;
            d.device = dev;
            if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
                return FP8LIN_ERR_CUDA;
            g_info[dev] = d;
            g_have[dev].store(true, std::memory_order_release);
        }
    }
    *info = g_info[dev];
    // The kernels are built for sm_103a only (tcgen05 tensor cores, TMA).
    if (info->cc_major != 10 || info->cc_minor != 3) return FP8LIN_ERR_UNSUPPORTED_DEVICE;
    return FP8LIN_OK;
}

namespace {
constexpr int kMaxCarveoutSlots = 80;  // amax 0, amax_rowcol 9, cast e4m3 1..4 and 21, cast e5m2 5..8 and 25,
                                       // block casts e4m3 33..39, e5m2 41..47, the casts without a
                                       // transposed copy at 48 more than their transposing form
std::atomic<bool> g_carveout_set[kMaxDevices][kMaxCarveoutSlots];
}  // namespace

fp8lin_status prefer_max_shared_carveout(const void *kernel, int device, int slot) {
    if (device < 0 || device >= kMaxDevices || slot < 0 || slot >= kMaxCarveoutSlots) return FP8LIN_ERR_CUDA;
    if (g_carveout_set[device][slot].load(std::memory_order_acquire)) return FP8LIN_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return FP8LIN_ERR_CUDA;
    g_carveout_set[device][slot].store(true, std::memory_order_release);
    return FP8LIN_OK;
}

}  // namespace fp8lin

extern "C" const char *fp8lin_status_str(fp8lin_status s) {
    switch (s) {
        case FP8LIN_OK: return "ok";
        case FP8LIN_ERR_INVALID_ARG: return "invalid argument (NULL pointer, negative size, bad format or fmt_max)";
        case FP8LIN_ERR_MISALIGNED: return "pointer not aligned as the call requires (16 bytes for tensors, 4 for scalars)";
        case FP8LIN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (dimensions must be multiples of 16 and at most 2^30)";
        case FP8LIN_ERR_CUDA: return "CUDA runtime error";
        case FP8LIN_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
        case FP8LIN_ERR_UNSUPPORTED_DEVICE: return "current device is not a compute capability 10.3 (sm_103a) GPU";
    }
    return "unknown status";
}
