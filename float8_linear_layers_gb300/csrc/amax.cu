// amax.cu -- amax = max |x| over one bf16 tensor (dynamic per-tensor scaling:
// the statistic is taken from the tensor itself every step; TorchTitan
// analysis page, section 3.3, "Mixed precision and Float8").
//
// HBM-bound: 2 bytes read per element, nothing else.  Design:
//  * one block per 32 KB chunk (256 threads x eight 16-byte vectors), all
//    eight loads of a thread issued before any is used, so up to eight
//    resident blocks keep ~256 KB of reads in flight per SM;
//  * |x| is the bf16 pattern with the sign bit cleared; non-negative IEEE
//    patterns order like unsigned integers (NaN above Inf above finite, the
//    totalOrder of magnitudes), so the reduction runs on packed 16-bit
//    unsigned maxima (vmaxu2) and never converts to float;
//  * warp reduction with redux.sync, block reduction through shared memory;
//    a block issues its atomicMax on the fp32 bit pattern (bf16 << 16) only
//    when its maximum exceeds the value already there, so the thousands of
//    blocks of a large tensor do not serialise on one address.
#include <cstdint>

#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;                       // 16-byte vectors per thread
constexpr int kChunk = kThreads * kVec;       // vectors per block (32 KB)

__device__ __forceinline__ uint4 ld_stream16(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
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
    const int64_t base = (int64_t)blockIdx.x * kChunk + threadIdx.x;
    uint32_t m = 0;  // two packed 16-bit magnitudes
    if (base + (int64_t)(kVec - 1) * kThreads < nvec) {
        uint4 v[kVec];
#pragma unroll
        for (int u = 0; u < kVec; ++u) v[u] = ld_stream16(x + base + (int64_t)u * kThreads);
#pragma unroll
        for (int u = 0; u < kVec; ++u) m = absmax4(m, v[u]);
    } else {
        for (int u = 0; u < kVec; ++u) {
            const int64_t i = base + (int64_t)u * kThreads;
            if (i < nvec) m = absmax4(m, ld_stream16(x + i));
        }
    }
    uint32_t r = max(m & 0xFFFFu, m >> 16);
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x < ntail) r = max(r, (uint32_t)(tail[threadIdx.x] & 0x7FFFu));

    r = __reduce_max_sync(0xFFFFFFFFu, r);
    __shared__ uint32_t warp_max[kThreads / 32];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) warp_max[warp] = r;
    __syncthreads();
    if (warp == 0) {
        r = lane < kThreads / 32 ? warp_max[lane] : 0u;
        r = __reduce_max_sync(0xFFFFFFFFu, r);
        if (lane == 0 && r != 0) {
            const uint32_t bits = r << 16;
            // a relaxed read first: most blocks find a larger value already there
            if (bits > *reinterpret_cast<volatile unsigned int *>(amax_bits)) atomicMax(amax_bits, bits);
        }
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
    st = prefer_max_shared_carveout(reinterpret_cast<const void *>(&amax_bf16_kernel), dev.device, 0);
    if (st != FP8LIN_OK) return st;
    if (cudaMemsetAsync(amax, 0, sizeof(float), stream) != cudaSuccess) return FP8LIN_ERR_CUDA;
    if (n == 0) return FP8LIN_OK;
    const int64_t nvec = n / 8;
    const int ntail = (int)(n % 8);
    const uint16_t *tail = static_cast<const uint16_t *>(x) + nvec * 8;
    const int64_t blocks = (nvec + kChunk - 1) / kChunk;
    if (blocks > INT32_MAX) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    const int grid = blocks < 1 ? 1 : (int)blocks;
    amax_bf16_kernel<<<grid, kThreads, 0, stream>>>(static_cast<const uint4 *>(x), nvec, tail, ntail,
                                                    reinterpret_cast<unsigned int *>(amax));
    return check_launch();
}
