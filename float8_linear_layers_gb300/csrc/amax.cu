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
//  * loads are evict_first in L2 (a GEMM running beside keeps its operands),
//    except, for a tensor whose cast runs with nothing beside it
//    (fp8lin_quantize), its last 64 MB: evict_last, so the cast that follows
//    (last row block first) reads them from L2;
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
// Bytes at the end of the tensor the amax pass leaves in L2 for the cast.
#ifndef FP8LIN_AMAX_KEEP_MB
#define FP8LIN_AMAX_KEEP_MB 64
#endif
constexpr int64_t kKeepBytes = (int64_t)FP8LIN_AMAX_KEEP_MB << 20;

// Streaming 16-byte load: no L1 allocation, and first in line for L2
// eviction, so a GEMM running beside this kernel keeps its resident operand.
__device__ __forceinline__ uint4 ld_stream16(const uint4 *p) {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

// The same load, kept in L2 (evict_last): the tail of the tensor, which the
// cast that follows reads first (it visits its tiles last row block first,
// with evict_first loads that demote the lines once read).
__device__ __forceinline__ uint4 ld_keep16(const uint4 *p) {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
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
                 int ntail, unsigned int *__restrict__ amax_bits, int keep_from) {
    const int64_t base = (int64_t)blockIdx.x * kChunk + threadIdx.x;
    uint32_t m = 0;  // two packed 16-bit magnitudes
    if (base + (int64_t)(kVec - 1) * kThreads < nvec) {
        uint4 v[kVec];
        if ((int)blockIdx.x >= keep_from) {
#pragma unroll
            for (int u = 0; u < kVec; ++u) v[u] = ld_keep16(x + base + (int64_t)u * kThreads);
        } else {
#pragma unroll
            for (int u = 0; u < kVec; ++u) v[u] = ld_stream16(x + base + (int64_t)u * kThreads);
        }
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

// Row and column amax of a row-major bf16 [rows x cols] matrix (row-wise
// scaling's statistics).  A CTA walks a strip of kStrip 128 x 128 tiles
// along its 128 rows, with the next tile's loads in flight while the current
// one is reduced (the same coalesced 16-byte loads as the cast kernel: a
// one-tile-per-CTA version spent most of each CTA's life reducing with no
// loads in flight and read at half the per-tensor amax's rate).  Row maxima
// accumulate in registers over the strip and reduce once across the 16
// threads that share a row (shuffles): one atomicMax per row per strip.
// Column maxima reduce per tile over the thread's 8 rows, the lane 16 apart
// and the 8 warps (shared memory): one atomicMax per column per tile.  The
// atomics are fire-and-forget reductions on the fp32 bit patterns.
constexpr int kTile = 128;
constexpr int kStrip = 4;

__device__ __forceinline__ void load_tile(uint4 (&v)[8], const uint16_t *__restrict__ x, int rows, int cols,
                                          int r0, int c0, int row_base, int ch) {
    const bool col_in = (c0 + ch * 8) < cols;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = r0 + row_base + 16 * i;
        v[i] = (col_in && r < rows) ? ld_stream16(reinterpret_cast<const uint4 *>(x + (int64_t)r * cols + c0 + ch * 8))
                                    : make_uint4(0, 0, 0, 0);
    }
}

__global__ void __launch_bounds__(256)
amax_rowcol_kernel(const uint16_t *__restrict__ x, int rows, int cols, int strips_c, int tiles_c,
                   unsigned int *__restrict__ row_bits, unsigned int *__restrict__ col_bits) {
    __shared__ uint32_t col_part[8][kTile / 2];  // [warp][packed column pair]
    const int tr = blockIdx.x / strips_c, sc = blockIdx.x % strips_c;
    const int r0 = tr * kTile, tc0 = sc * kStrip;
    const int ntiles = min(kStrip, tiles_c - tc0);
    const int t = threadIdx.x, ch = t % 16, row_base = t / 16;
    const int warp = t / 32, lane = t % 32;
    const uint32_t k = 0x7FFF7FFFu;
    uint32_t rowm[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) rowm[i] = 0;
    uint4 v[8], nx[8];
    load_tile(v, x, rows, cols, r0, tc0 * kTile, row_base, ch);
    for (int s = 0; s < ntiles; ++s) {
        const int c0 = (tc0 + s) * kTile;
        if (s + 1 < ntiles) load_tile(nx, x, rows, cols, r0, c0 + kTile, row_base, ch);
        // columns: packed maxima of this thread's 8 columns over its 8 rows; rows: running maxima
        uint4 cm = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            cm.x = __vmaxu2(cm.x, v[i].x & k);
            cm.y = __vmaxu2(cm.y, v[i].y & k);
            cm.z = __vmaxu2(cm.z, v[i].z & k);
            cm.w = __vmaxu2(cm.w, v[i].w & k);
            const uint32_t m = absmax4(0u, v[i]);
            rowm[i] = max(rowm[i], max(m & 0xFFFFu, m >> 16));
        }
        if (col_bits != nullptr) {
            // lanes t and t ^ 16 hold the same columns for two row groups
            cm.x = __vmaxu2(cm.x, __shfl_xor_sync(0xFFFFFFFFu, cm.x, 16));
            cm.y = __vmaxu2(cm.y, __shfl_xor_sync(0xFFFFFFFFu, cm.y, 16));
            cm.z = __vmaxu2(cm.z, __shfl_xor_sync(0xFFFFFFFFu, cm.z, 16));
            cm.w = __vmaxu2(cm.w, __shfl_xor_sync(0xFFFFFFFFu, cm.w, 16));
            if (s > 0) __syncthreads();  // the previous tile's column maxima have been read
            if (lane < 16) {
                col_part[warp][4 * ch + 0] = cm.x;
                col_part[warp][4 * ch + 1] = cm.y;
                col_part[warp][4 * ch + 2] = cm.z;
                col_part[warp][4 * ch + 3] = cm.w;
            }
            __syncthreads();
            if (t < kTile / 2) {
                uint32_t m = 0;
#pragma unroll
                for (int w = 0; w < 8; ++w) m = __vmaxu2(m, col_part[w][t]);
                const int c = c0 + 2 * t;
                if (c < cols) {
                    const uint32_t lo = (m & 0xFFFFu) << 16, hi = m & 0xFFFF0000u;
                    if (lo != 0) atomicMax(col_bits + c, lo);
                    if (hi != 0) atomicMax(col_bits + c + 1, hi);
                }
            }
        }
        if (s + 1 < ntiles) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = nx[i];
        }
    }
    if (row_bits == nullptr) return;
    // rows: the 16 lanes sharing a row combine their maxima over the strip
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t m = rowm[i];
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const int r = r0 + row_base + 16 * i;
        if (ch == 0 && r < rows && m != 0) atomicMax(row_bits + r, m << 16);  // result unused: a reduction
    }
}

}  // namespace

extern "C" fp8lin_status fp8lin_amax_rowcol(const void *x, int64_t rows, int64_t cols, float *row_amax,
                                            float *col_amax, cudaStream_t stream) {
    using namespace fp8lin;
    if (rows < 0 || cols < 0) return FP8LIN_ERR_INVALID_ARG;
    const bool empty = rows == 0 || cols == 0;
    if (!empty && x == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if ((row_amax == nullptr && rows > 0 && col_amax == nullptr)) return FP8LIN_ERR_INVALID_ARG;
    if (!aligned(row_amax, 4) || !aligned(col_amax, 4) || (!empty && !aligned(x, 16))) return FP8LIN_ERR_MISALIGNED;
    if (!dim_ok(rows) || !dim_ok(cols) || rows % 16 || cols % 16) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo dev;
    fp8lin_status st = current_device(&dev);
    if (st != FP8LIN_OK) return st;
    st = prefer_max_shared_carveout(reinterpret_cast<const void *>(&amax_rowcol_kernel), dev.device, 9);
    if (st != FP8LIN_OK) return st;
    if (row_amax != nullptr && rows > 0 &&
        cudaMemsetAsync(row_amax, 0, (size_t)rows * sizeof(float), stream) != cudaSuccess)
        return FP8LIN_ERR_CUDA;
    if (col_amax != nullptr && cols > 0 &&
        cudaMemsetAsync(col_amax, 0, (size_t)cols * sizeof(float), stream) != cudaSuccess)
        return FP8LIN_ERR_CUDA;
    if (empty) return FP8LIN_OK;
    const int64_t tiles_r = (rows + kTile - 1) / kTile, tiles_c = (cols + kTile - 1) / kTile;
    const int64_t strips_c = (tiles_c + kStrip - 1) / kStrip;
    if (tiles_r * strips_c > INT32_MAX) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    amax_rowcol_kernel<<<(int)(tiles_r * strips_c), 256, 0, stream>>>(
        static_cast<const uint16_t *>(x), (int)rows, (int)cols, (int)strips_c, (int)tiles_c,
        reinterpret_cast<unsigned int *>(row_amax), reinterpret_cast<unsigned int *>(col_amax));
    return check_launch();
}

namespace fp8lin {

fp8lin_status launch_amax(const void *x, int64_t n, float *amax, cudaStream_t stream, bool alone) {
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
    // Beside a GEMM every load is evict_first (the GEMM's operands keep L2);
    // alone, the tail is kept for the cast.
    const int64_t keep_blocks = alone ? kKeepBytes / ((int64_t)kChunk * 16) : 0;
    const int keep_from = grid > keep_blocks ? (int)(grid - keep_blocks) : 0;
    amax_bf16_kernel<<<grid, kThreads, 0, stream>>>(static_cast<const uint4 *>(x), nvec, tail, ntail,
                                                    reinterpret_cast<unsigned int *>(amax), keep_from);
    return check_launch();
}

}  // namespace fp8lin

extern "C" fp8lin_status fp8lin_amax(const void *x, int64_t n, float *amax, cudaStream_t stream) {
    using namespace fp8lin;
    if (amax == nullptr || n < 0 || (n > 0 && x == nullptr)) return FP8LIN_ERR_INVALID_ARG;
    if (!aligned(amax, 4) || (n > 0 && !aligned(x, 16))) return FP8LIN_ERR_MISALIGNED;
    if (n > FP8LIN_MAX_DIM * FP8LIN_MAX_DIM) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    return launch_amax(x, n, amax, stream, false);
}
