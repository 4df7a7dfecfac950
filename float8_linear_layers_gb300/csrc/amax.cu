// amax.cu -- amax = max |x| over one bf16 tensor (dynamic per-tensor scaling:
// the statistic is taken from the tensor itself every step; TorchTitan
// analysis page, section 3.3, "Mixed precision and Float8").
//
// HBM-bound: 2 bytes read per element, nothing else.  Design:
//  * grid sized to the SM count x resident blocks, grid-stride over 16-byte
//    vectors (8 bf16) with four independent loads in flight per thread;
//  * |x| is the bf16 pattern with the sign bit cleared; non-negative IEEE
//    patterns order like unsigned integers (NaN above Inf above finite, the
//    totalOrder of magnitudes), so the reduction runs on packed 16-bit
//    unsigned maxima (vmaxu2) and never converts to float;
//  * warp reduction with redux.sync, block reduction through shared memory,
//    one atomicMax per block on the fp32 bit pattern (bf16 << 16).
#include <cstdint>

#include "common.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_stream16(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t absmax4(uint32_t m, uint4 v) {
    const uint32_t k = 0x7FFF7FFFu;
    m = __vmaxu2(m, v.x & k);
    m = __vmaxu2(m, v.y & k);
    m = __vmaxu2(m, v.z & k);
    m = __vmaxu2(m, v.w & k);
    return m;
}

__global__ void __launch_bounds__(kThreads)
amax_bf16_kernel(const uint4 *__restrict__ x, int64_t nvec, const uint16_t *__restrict__ tail,
                 int ntail, unsigned int *__restrict__ amax_bits) {
    uint32_t m = 0;  // two packed 16-bit magnitudes
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < nvec; i += kUnroll * stride) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream16(x + i + u * stride);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) m = absmax4(m, v[u]);
    }
    for (; i < nvec; i += stride) m = absmax4(m, ld_stream16(x + i));
    uint32_t r = max(m & 0xFFFFu, m >> 16);
    if (blockIdx.x == 0 && threadIdx.x < ntail) r = max(r, (uint32_t)(tail[threadIdx.x] & 0x7FFFu));

    r = __reduce_max_sync(0xFFFFFFFFu, r);
    __shared__ uint32_t warp_max[kThreads / 32];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) warp_max[warp] = r;
    __syncthreads();
    if (warp == 0) {
        r = lane < kThreads / 32 ? warp_max[lane] : 0u;
        r = __reduce_max_sync(0xFFFFFFFFu, r);
        if (lane == 0 && r != 0) atomicMax(amax_bits, r << 16);
    }
}

}  // namespace

extern "C" fp8lin_status fp8lin_amax(const void *x, int64_t n, float *amax, cudaStream_t stream) {
    using namespace fp8lin;
    if (amax == nullptr || n < 0 || (n > 0 && x == nullptr)) return FP8LIN_ERR_INVALID_ARG;
    if (!aligned(amax, 4) || (n > 0 && !aligned(x, 16))) return FP8LIN_ERR_MISALIGNED;
    if (n > FP8LIN_MAX_DIM * FP8LIN_MAX_DIM) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo dev;
    fp8lin_status st = current_device(&dev);
    if (st != FP8LIN_OK) return st;
    if (cudaMemsetAsync(amax, 0, sizeof(float), stream) != cudaSuccess) return FP8LIN_ERR_CUDA;
    if (n == 0) return FP8LIN_OK;
    const int64_t nvec = n / 8;
    const int ntail = (int)(n % 8);
    const uint16_t *tail = static_cast<const uint16_t *>(x) + nvec * 8;
    int64_t want = (nvec + (int64_t)kThreads * kUnroll - 1) / ((int64_t)kThreads * kUnroll);
    int64_t cap = (int64_t)dev.sm_count * (2048 / kThreads);  // one full wave of resident blocks
    int grid = (int)(want < 1 ? 1 : (want < cap ? want : cap));
    amax_bf16_kernel<<<grid, kThreads, 0, stream>>>(static_cast<const uint4 *>(x), nvec, tail, ntail,
                                                    reinterpret_cast<unsigned int *>(amax));
    return check_launch();
}
