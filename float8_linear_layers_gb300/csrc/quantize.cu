// quantize.cu -- dynamic per-tensor scaling of bf16 tensors in one launch:
// amax, scale and the saturating round-to-nearest-even cast to the row-major
// FP8 copy (TorchTitan analysis page, section 3.3, "Mixed precision and
// Float8": dynamic scaling takes the tensor's own statistic every step;
// Lecture 9 exercises: one factor per tensor).  For the casts a GEMM waits
// for, which run with nothing beside them.  One launch takes up to
// kMaxBatch tensors of one format (the X and W of a forward pass), each
// with its own amax, scale and inverse-scale slots and its own scale.
//
// HBM-bound: the two-kernel path (amax, then cast) reads a tensor twice.
// Here one persistent cooperative grid, one CTA per SM, reads the tensors
// once for their amax while keeping the last part of each CTA's slice in
// shared memory, meets at a grid barrier, then casts the staged part from
// shared memory and the rest of the slice last-read-first (so what L2 still
// holds is read before it is evicted).  The tensors are laid end to end as
// one range of 16-byte vectors (8 elements); element i of a tensor becomes
// byte i of its copy, and a CTA's slice is a contiguous part of that range,
// cut where it crosses from one tensor to the next.
//
// The grid barrier uses the call's own output slots, so the kernel needs no
// memory beyond its inputs and outputs: every slot is zero when it starts
// (the host clears them on the stream); every CTA publishes each tensor's
// maximum over its slice with atomicMax on that tensor's amax slot and then
// counts itself in on the first tensor's scale slot (atomicAdd on its
// bits); the CTA that arrives last reads the maxima, writes every other
// tensor's scale and inverse scale, overwrites the count with the first
// tensor's scale and publishes the first tensor's 1 / scale with release
// semantics; the others wait (acquire, at most kWaitLimitNs) until that slot
// is nonzero, then read the scales.  1 / scale is never zero: scale =
// fmt_max / max(amax, 1e-12) is finite for fmt_max <= 65504 (the host checks
// it), and a NaN or infinite amax gives a NaN or infinite inverse.  A wait
// that runs out records FP8LIN_ERR_TIMEOUT in this file's device error word
// (read by fp8lin_device_error) and the CTA skips its cast.
//
// Tensors of at most 1.5 MB in all take quantize_cluster_kernel instead
// (further down): one cluster of eight CTAs, no grid barrier and no
// clearing launch.
#include <atomic>
#include <cstdint>

#include "common.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 8;                       // 16-byte loads in flight per thread
#ifndef FP8LIN_QUANTIZE_STAGE_KB
#define FP8LIN_QUANTIZE_STAGE_KB 192
#endif
constexpr int kStageBytes = FP8LIN_QUANTIZE_STAGE_KB * 1024;   // slice tail kept in shared memory
constexpr int kStageVecs = kStageBytes / 16;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr int kMaxBatch = FP8LIN_MAX_QUANTIZE_BATCH;

__device__ unsigned int g_quantize_error = 0;

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint4 ld16(const uint4 *p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ void st_stream8(void *p, uint2 v, uint64_t policy) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "l"(policy)
                 : "memory");
}

__device__ __forceinline__ uint32_t absmax8(uint32_t m, uint4 v) {
    const uint32_t k = 0x7FFF7FFFu;
    m = __vmaxu2(m, v.x & k);
    m = __vmaxu2(m, v.y & k);
    m = __vmaxu2(m, v.z & k);
    m = __vmaxu2(m, v.w & k);
    return m;
}

template <int FMT>
__device__ __forceinline__ uint32_t cvt4(float a, float b, float c, float d) {
    // cvt packs its first source operand into the upper byte of each pair
    uint16_t lo, hi;
    if (FMT == FP8LIN_E4M3) {
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    } else {
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    }
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Eight codes sat_RNE(fp32(x) * s): one binary32 multiply, one conversion.
template <int FMT>
__device__ __forceinline__ uint2 cast8(uint4 v, float s) {
    uint2 r;
    r.x = cvt4<FMT>(__fmul_rn(bf16_lo(v.x), s), __fmul_rn(bf16_hi(v.x), s), __fmul_rn(bf16_lo(v.y), s),
                    __fmul_rn(bf16_hi(v.y), s));
    r.y = cvt4<FMT>(__fmul_rn(bf16_lo(v.z), s), __fmul_rn(bf16_hi(v.z), s), __fmul_rn(bf16_lo(v.w), s),
                    __fmul_rn(bf16_hi(v.w), s));
    return r;
}

// The tensors of one launch, end to end: tensor k holds vectors
// [begin(k), end[k]) of the range.
struct QBatch {
    const uint4 *x[kMaxBatch];
    uint2 *q[kMaxBatch];
    unsigned int *amax[kMaxBatch];
    float *scale[kMaxBatch];
    float *inv[kMaxBatch];
    int64_t end[kMaxBatch];
    int count;
    __device__ __forceinline__ int64_t begin(int k) const { return k == 0 ? 0 : end[k - 1]; }
};

// Maximum |x| (two packed 16-bit magnitudes) of vectors [lo, hi) of x, one
// thread's share: kUnroll loads in flight.
__device__ __forceinline__ uint32_t stream_max(const uint4 *__restrict__ x, int64_t lo, int64_t hi, int t,
                                               int threads, uint64_t policy) {
    uint32_t m = 0;
    int64_t i = lo + t;
    for (; i + (int64_t)(kUnroll - 1) * threads < hi; i += (int64_t)kUnroll * threads) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = ld16(x + i + (int64_t)u * threads, policy);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) m = absmax8(m, v[u]);
    }
    for (; i < hi; i += threads) m = absmax8(m, ld16(x + i, policy));
    return m;
}

// The same over [lo, hi), each vector also stored to stage[j - stage0].
__device__ __forceinline__ uint32_t stage_max(const uint4 *__restrict__ x, int64_t lo, int64_t hi, int t,
                                              int threads, uint64_t policy, uint4 *stage, int64_t stage0) {
    uint32_t m = 0;
    for (int64_t j = lo + t; j < hi; j += (int64_t)kUnroll * threads) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (j + (int64_t)u * threads < hi) v[u] = ld16(x + j + (int64_t)u * threads, policy);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (j + (int64_t)u * threads < hi) {
                stage[j + (int64_t)u * threads - stage0] = v[u];
                m = absmax8(m, v[u]);
            }
    }
    return m;
}

// fmt_max / max(amax, 1e-12) in binary32, from the amax slot's bits.
__device__ __forceinline__ float scale_of(unsigned int amax_bits, float fmt_max) {
    float a = __uint_as_float(amax_bits);
    a = (a < 1e-12f) ? 1e-12f : a;  // a NaN amax stays NaN
    return __fdiv_rn(fmt_max, a);
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1)
quantize_kernel(const QBatch b, float fmt_max) {
    extern __shared__ uint4 stage[];
    __shared__ uint32_t warp_max[kMaxBatch][kThreads / 32];
    __shared__ float s_shared[kMaxBatch];
    __shared__ int go;

    const int t = threadIdx.x;
    const int64_t nvec = b.end[b.count - 1];
    const int64_t per = (nvec + gridDim.x - 1) / gridDim.x;
    const int64_t v0 = min((int64_t)blockIdx.x * per, nvec);
    const int64_t v1 = min(v0 + per, nvec);
    const int64_t s0 = max(v0, v1 - (int64_t)kStageVecs);   // [s0, v1) stays in shared memory
    uint64_t normal, stream;   // phase 1 keeps what phase 2 re-reads; phase 2 and the stores stream
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(normal));
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(stream));

    // ---- phase 1: each tensor's amax over the slice; the slice's tail into shared memory
#pragma unroll
    for (int k = 0; k < kMaxBatch; ++k) {
        if (k >= b.count) break;
        const int64_t beg = b.begin(k), end = b.end[k];
        const uint4 *x = b.x[k] - beg;   // indexed by position in the whole range
        uint32_t m = 0;
        if (max(v0, beg) < min(s0, end)) m = stream_max(x, max(v0, beg), min(s0, end), t, kThreads, normal);
        if (max(s0, beg) < min(v1, end))   // packed maxima: combined lane by lane
            m = __vmaxu2(m, stage_max(x, max(s0, beg), min(v1, end), t, kThreads, stream, stage, s0));
        // packed maxima compare lane-wise; fold the two halves, then the warp
        const uint32_t r = __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
        if (t % 32 == 0) warp_max[k][t / 32] = r;
    }
    __syncthreads();

    // ---- grid barrier on the output slots (see the file comment)
    if (t < 32) {
        uint32_t r[kMaxBatch];
#pragma unroll
        for (int k = 0; k < kMaxBatch; ++k)
            r[k] = __reduce_max_sync(0xFFFFFFFFu, (k < b.count && t < kThreads / 32) ? warp_max[k][t] : 0u);
        if (t == 0) {
#pragma unroll
            for (int k = 0; k < kMaxBatch; ++k)
                if (k < b.count && r[k] != 0) atomicMax(b.amax[k], r[k] << 16);
            __threadfence();
            unsigned int *arrivals = reinterpret_cast<unsigned int *>(b.scale[0]);
            const unsigned int before = atomicAdd(arrivals, 1u);
            int arrived = 1;
            if (before == gridDim.x - 1) {
                __threadfence();
#pragma unroll
                for (int k = kMaxBatch - 1; k >= 1; --k) {
                    if (k >= b.count) continue;
                    const float s = scale_of(atomicOr(b.amax[k], 0u), fmt_max);
                    *b.scale[k] = s;
                    *b.inv[k] = __frcp_rn(s);
                    s_shared[k] = s;
                }
                const float s = scale_of(atomicOr(b.amax[0], 0u), fmt_max);
                *b.scale[0] = s;                // the count is complete: the slot takes the scale
                s_shared[0] = s;
                __threadfence();
                asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(b.inv[0]), "r"(__float_as_uint(__frcp_rn(s)))
                             : "memory");
            } else {
                const unsigned long long t0 = globaltimer();
                uint32_t flag = 0;
                while (true) {
                    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(flag) : "l"(b.inv[0]) : "memory");
                    if (flag != 0) break;
                    if (globaltimer() - t0 > kWaitLimitNs) {
                        atomicOr(&g_quantize_error, 1u << FP8LIN_ERR_TIMEOUT);
                        arrived = 0;
                        break;
                    }
                }
#pragma unroll
                for (int k = 0; k < kMaxBatch; ++k)
                    if (k < b.count) s_shared[k] = arrived ? *reinterpret_cast<volatile float *>(b.scale[k]) : 0.0f;
            }
            go = arrived;
        }
    }
    __syncthreads();
    if (!go) return;

    // ---- phase 2: the staged tail from shared memory, then the rest of the
    // slice last-read-first
#pragma unroll
    for (int k = 0; k < kMaxBatch; ++k) {
        if (k >= b.count) break;
        const int64_t beg = b.begin(k), lo = max(s0, beg), hi = min(v1, b.end[k]);
        const float s = s_shared[k];
        uint2 *q = b.q[k] - beg;
        for (int64_t j = lo + t; j < hi; j += kThreads) st_stream8(q + j, cast8<FMT>(stage[j - s0], s), stream);
    }
#pragma unroll
    for (int kk = 0; kk < kMaxBatch; ++kk) {
        const int k = kMaxBatch - 1 - kk;
        if (k >= b.count) continue;
        const int64_t beg = b.begin(k), lo = max(v0, beg), hi = min(s0, b.end[k]);
        if (lo >= hi) continue;
        const float s = s_shared[k];
        const uint4 *x = b.x[k] - beg;
        uint2 *q = b.q[k] - beg;
        const int64_t n_rest = hi - lo;
        int64_t i = t;
        for (; i + (int64_t)(kUnroll - 1) * kThreads < n_rest; i += (int64_t)kUnroll * kThreads) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) v[u] = ld16(x + (hi - 1 - i - (int64_t)u * kThreads), stream);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                st_stream8(q + (hi - 1 - i - (int64_t)u * kThreads), cast8<FMT>(v[u], s), stream);
        }
        for (; i < n_rest; i += kThreads) {
            const int64_t idx = hi - 1 - i;
            st_stream8(q + idx, cast8<FMT>(ld16(x + idx, stream), s), stream);
        }
    }
}

// Small batches (up to kSmallMaxVecs vectors in all, 1.5 MB of bf16): one
// cluster of kClusterCtas CTAs stages the whole range in shared memory, each
// CTA a contiguous slice.  The CTAs meet at a hardware cluster barrier, read
// the other CTAs' maxima from their shared memory (distributed shared
// memory), derive the same scales, and cast their staged slice.  The slots
// need no clearing and no global memory holds a partial result, so the
// launch needs no memset, and no wait is a spin: the barrier is the
// cluster's own, whose CTAs are resident together by construction.  A
// second barrier keeps every CTA resident until its peers have read its
// maxima.
constexpr int kClusterCtas = 8;
constexpr int kSmallThreads = 512;
constexpr int kSmallStageBytes = 192 * 1024;
constexpr int64_t kSmallMaxVecs = (int64_t)kClusterCtas * (kSmallStageBytes / 16);

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }

__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// A 32-bit word of peer CTA `rank`'s shared memory, at the address `local` has here.
__device__ __forceinline__ uint32_t ld_peer_u32(const uint32_t *local, uint32_t rank) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t remote, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

template <int FMT>
__global__ void __launch_bounds__(kSmallThreads, 1)
quantize_cluster_kernel(const QBatch b, int64_t per, float fmt_max) {
    extern __shared__ uint4 stage[];
    __shared__ uint32_t warp_max[kMaxBatch][kSmallThreads / 32];
    __shared__ uint32_t cta_max[kMaxBatch];

    const int t = threadIdx.x;
    const uint32_t rank = cluster_rank();
    const int64_t nvec = b.end[b.count - 1];
    const int64_t v0 = min((int64_t)rank * per, nvec);
    const int64_t v1 = min(v0 + per, nvec);
    uint64_t stream;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(stream));

    // ---- the slice into shared memory, and each tensor's maximum |x| over it
#pragma unroll
    for (int k = 0; k < kMaxBatch; ++k) {
        if (k >= b.count) break;
        const int64_t beg = b.begin(k), lo = max(v0, beg), hi = min(v1, b.end[k]);
        const uint32_t m = lo < hi ? stage_max(b.x[k] - beg, lo, hi, t, kSmallThreads, stream, stage, v0) : 0u;
        const uint32_t r = __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
        if (t % 32 == 0) warp_max[k][t / 32] = r;
    }
    __syncthreads();
    if (t < 32) {
#pragma unroll
        for (int k = 0; k < kMaxBatch; ++k) {
            const uint32_t r =
                __reduce_max_sync(0xFFFFFFFFu, (k < b.count && t < kSmallThreads / 32) ? warp_max[k][t] : 0u);
            if (t == 0) cta_max[k] = r;
        }
    }
    cluster_arrive();
    cluster_wait();   // every CTA's maxima are in its shared memory

    // ---- each tensor's maximum from every CTA's (each warp reads them), its scale
    const int lane = t % 32;
    float s[kMaxBatch];
#pragma unroll
    for (int k = 0; k < kMaxBatch; ++k) {
        uint32_t r = (k < b.count && lane < kClusterCtas) ? ld_peer_u32(&cta_max[k], (uint32_t)lane) : 0u;
        r = __reduce_max_sync(0xFFFFFFFFu, r);
        s[k] = scale_of(r << 16, fmt_max);
        if (k < b.count && rank == 0 && t == 0) {
            *b.amax[k] = r << 16;
            *b.scale[k] = s[k];
            *b.inv[k] = __frcp_rn(s[k]);
        }
    }
    cluster_arrive();   // this CTA is done reading its peers' shared memory

    // ---- the staged slice, cast
#pragma unroll
    for (int k = 0; k < kMaxBatch; ++k) {
        if (k >= b.count) break;
        const int64_t beg = b.begin(k), lo = max(v0, beg), hi = min(v1, b.end[k]);
        uint2 *q = b.q[k] - beg;
        for (int64_t j = lo + t; j < hi; j += kSmallThreads) st_stream8(q + j, cast8<FMT>(stage[j - v0], s[k]), stream);
    }
    cluster_wait();   // no CTA leaves while a peer may still read its maxima
}

std::atomic<int> g_grid[2][64];
std::atomic<int> g_small[2][64];   // 0 = not asked yet, 1 = the cluster path runs, -1 = it does not

// The small-batch path; *launched says whether it ran.
fp8lin_status launch_small(const QBatch &b, int64_t nvec, int f, float fmt_max, cudaStream_t stream, int device,
                           bool *launched) {
    auto kernel = f == 0 ? quantize_cluster_kernel<FP8LIN_E4M3> : quantize_cluster_kernel<FP8LIN_E5M2>;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = kClusterCtas;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterCtas);
    cfg.blockDim = dim3(kSmallThreads);
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int ok = g_small[f][device].load(std::memory_order_acquire);
    if (ok == 0) {
        int clusters = 0;
        cfg.dynamicSmemBytes = kSmallStageBytes;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallStageBytes) != cudaSuccess)
            return FP8LIN_ERR_CUDA;
        if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            clusters = 0;
        }
        ok = clusters >= 1 ? 1 : -1;
        g_small[f][device].store(ok, std::memory_order_release);
    }
    if (ok < 0) return FP8LIN_OK;
    const int64_t per = (nvec + kClusterCtas - 1) / kClusterCtas;
    cfg.dynamicSmemBytes = (size_t)per * 16;
    cfg.stream = stream;
    if (cudaLaunchKernelEx(&cfg, kernel, b, per, fmt_max) != cudaSuccess) return FP8LIN_ERR_CUDA;
    *launched = true;
    return fp8lin::check_launch();
}

}  // namespace

namespace fp8lin {

fp8lin_status launch_quantize_batch(const QuantizeItem *items, int count, fp8lin_fmt fmt, float fmt_max,
                                    cudaStream_t stream, bool *launched) {
    *launched = false;
    if (count < 1 || count > kMaxBatch || !(fmt_max <= 65504.0f)) return FP8LIN_OK;   // the two-kernel path
    QBatch b = {};
    int64_t nvec = 0;
    for (int k = 0; k < count; ++k) {
        if (items[k].n % 8 != 0) return FP8LIN_OK;
        nvec += items[k].n / 8;
        b.x[k] = static_cast<const uint4 *>(items[k].x);
        b.q[k] = reinterpret_cast<uint2 *>(items[k].q);
        b.amax[k] = reinterpret_cast<unsigned int *>(items[k].amax);
        b.scale[k] = items[k].scale;
        b.inv[k] = items[k].inv_scale;
        b.end[k] = nvec;
    }
    b.count = count;
    if (nvec == 0) return FP8LIN_OK;   // nothing to read: the two-kernel path publishes the floor scales
    DeviceInfo dev;
    fp8lin_status st = current_device(&dev);
    if (st != FP8LIN_OK) return st;
    if (dev.device >= 64) return FP8LIN_OK;
    const int f = fmt == FP8LIN_E4M3 ? 0 : 1;
    if (nvec <= kSmallMaxVecs) {
        st = launch_small(b, nvec, f, fmt_max, stream, dev.device, launched);
        if (st != FP8LIN_OK || *launched) return st;
    }
    auto kernel = f == 0 ? quantize_kernel<FP8LIN_E4M3> : quantize_kernel<FP8LIN_E5M2>;
    int grid = g_grid[f][dev.device].load(std::memory_order_acquire);
    if (grid == 0) {
        int coop = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev.device) != cudaSuccess)
            return FP8LIN_ERR_CUDA;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, kStageBytes) != cudaSuccess)
            return FP8LIN_ERR_CUDA;
        grid = (coop && per_sm >= 1) ? dev.sm_count : -1;   // one CTA per SM, all resident together
        g_grid[f][dev.device].store(grid, std::memory_order_release);
    }
    if (grid < 0) return FP8LIN_OK;
    const int g = nvec < grid ? (int)nvec : grid;
    // every slot starts at zero: the first tensor's count and flag, each tensor's maximum
    for (int k = 0; k < count; ++k) {
        const QuantizeItem &it = items[k];
        if (it.scale == it.amax + 1 && it.inv_scale == it.amax + 2) {
            if (cudaMemsetAsync(it.amax, 0, 3 * sizeof(float), stream) != cudaSuccess) return FP8LIN_ERR_CUDA;
        } else if (cudaMemsetAsync(it.amax, 0, sizeof(float), stream) != cudaSuccess ||
                   cudaMemsetAsync(it.scale, 0, sizeof(float), stream) != cudaSuccess ||
                   cudaMemsetAsync(it.inv_scale, 0, sizeof(float), stream) != cudaSuccess) {
            return FP8LIN_ERR_CUDA;
        }
    }
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeCooperative;
    attr.val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)g);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kStageBytes;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, b, fmt_max);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        // fewer SMs than the device reports are available to this context:
        // the caller takes the two-kernel path, now and from here on
        (void)cudaGetLastError();
        g_grid[f][dev.device].store(-1, std::memory_order_release);
        return FP8LIN_OK;
    }
    if (e != cudaSuccess) return FP8LIN_ERR_CUDA;
    *launched = true;
    return check_launch();
}

fp8lin_status take_quantize_error(unsigned int *bits) {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_quantize_error, sizeof v) != cudaSuccess) return FP8LIN_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_quantize_error, &zero, sizeof zero) != cudaSuccess) return FP8LIN_ERR_CUDA;
    *bits = v;
    return FP8LIN_OK;
}

}  // namespace fp8lin
