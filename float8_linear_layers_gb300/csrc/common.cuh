// common.cuh -- host-side argument checks and per-device facts shared by the
// translation units of libfp8lin.  Device code lives with its kernel.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fp8lin.h"

namespace fp8lin {

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline bool dim_ok(int64_t d) { return d >= 0 && d <= FP8LIN_MAX_DIM; }

// Map the last CUDA error (launch configuration, invalid handle, ...) to a status.
inline fp8lin_status check_launch() {
    return cudaGetLastError() == cudaSuccess ? FP8LIN_OK : FP8LIN_ERR_CUDA;
}

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0;
    int cc_minor = 0;
};

// Facts about the current device, cached per device ordinal.
fp8lin_status current_device(DeviceInfo *info);

// Ask for the largest shared-memory carveout for `kernel` (once per device).
// The GEMM runs every SM at that carveout; an SM hosts CTAs of concurrently
// running kernels only when their carveouts agree, so the HBM-bound amax and
// cast kernels use the same setting to run beside a GEMM on another stream.
fp8lin_status prefer_max_shared_carveout(const void *kernel, int device, int slot);

// amax of n bf16 values into *amax (cleared first), on `stream`.  alone:
// nothing runs beside it, so the tensor's last 64 MB are loaded evict_last
// and the cast that follows (last rows first) finds them in L2.  Arguments
// are checked by the caller.
fp8lin_status launch_amax(const void *x, int64_t n, float *amax, cudaStream_t stream, bool alone);

// One tensor of a one-launch dynamic cast: n bf16 values, its own amax,
// scale and inverse-scale slots and its row-major FP8 copy.
struct QuantizeItem {
    const void *x;
    int64_t n;
    float *amax, *scale, *inv_scale;
    uint8_t *q;
};

// Dynamic per-tensor scaling of `count` tensors (1 .. FP8LIN_MAX_QUANTIZE_BATCH,
// one format) in one launch (quantize.cu); *launched says whether it ran (it
// declines fmt_max above 65504, tensors with nothing to read and devices
// without cooperative launch, and the caller then takes the two-kernel path
// per tensor).  Arguments are checked by the caller.
fp8lin_status launch_quantize_batch(const QuantizeItem *items, int count, fp8lin_fmt fmt, float fmt_max,
                                    cudaStream_t stream, bool *launched);

// Read and clear the device word in which quantize.cu's kernel records a
// bounded wait that ran out.
fp8lin_status take_quantize_error(unsigned int *bits);

}  // namespace fp8lin
