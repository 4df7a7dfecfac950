// gemm.cu -- the three scaled FP8 GEMMs of the Float8 linear layer on the
// sm_103a tensor cores (TorchTitan analysis page, section 3.3, "Mixed
// precision and Float8": Float8 applied to linear layers, composable with
// autograd, so forward, input gradient and weight gradient all run in FP8).
//
// Every GEMM is issued as C[P x Q] = A[P x R] . B[Q x R]^T with both operands
// stored contraction-contiguous ("K-major"); the cast kernel's transposed
// copies make that true for all three:
//     fwd   : Y [M x N]  = Xq   [M x K] . Wq  [N x K]^T    e4m3 x e4m3
//     dgrad : dX [M x K] = dYq  [M x N] . WqT [K x N]^T    e5m2 x e4m3
//     wgrad : dW [N x K] = dYqT [N x M] . XqT [K x M]^T    e5m2 x e4m3
// and the epilogue computes C = bf16_RN(acc_fp32 * (inv_a * inv_b)).
//
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0      TMA producer: 2-D tiled bulk-tensor loads of 128 x 128-byte
//               A and 256 x 128-byte B boxes, 128-byte swizzle, into a
//               4-stage shared-memory ring guarded by full/empty mbarriers;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32
//               accumulators); one thread issues tcgen05.mma kind::f8f6f4
//               (M = 128, N = 256, K = 32 per instruction, 4 per stage) and
//               tcgen05.commit frees each stage and publishes each finished
//               accumulator;
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns at a time, scale,
//               round to bf16, 16-byte stores; the accumulator is handed back
//               as soon as it is read, so the epilogue of tile i overlaps the
//               main loop of tile i + 1.
// Tiles are visited in groups of kGroupM row-blocks so that concurrently
// running CTAs share A and B panels in L2.
//
// Every mbarrier wait is bounded by wall-clock time (globaltimer).  A wait
// that runs out records FP8LIN_ERR_TIMEOUT in a device word, raises a
// shared abort flag that ends every role's loop, drains the copies and MMAs
// still in flight (again with bounded waits) and frees TMEM before exiting.
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kBM = 128;              // rows of A per tile (UMMA M)
constexpr int kBN = 256;              // rows of B per tile (UMMA N)
constexpr int kBK = 128;              // contraction bytes per stage (one 128-byte swizzle row)
constexpr int kUmmaK = 32;            // contraction elements per tcgen05.mma for 8-bit types
constexpr int kStages = 4;
constexpr int kAStage = kBM * kBK;    // 16 KB
constexpr int kBStage = kBN * kBK;    // 32 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 2 * kBN;    // two fp32 accumulators
constexpr int kGroupM = 16;
constexpr int kSmemBytes = kStages * (kAStage + kBStage) + 1024 /*barriers*/ + 1024 /*alignment*/;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr unsigned long long kDrainLimitNs = 200000000ull;  // 0.2 s per drain wait

static_assert(kBK == 128, "one stage is one 128-byte swizzle row of contraction");

__device__ unsigned int g_device_error = 0;

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of parity `parity` to complete, for at most `limit` ns.
// Gives up early once another role has raised the abort flag.  On running
// out, records the timeout and raises the flag.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                       unsigned long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit) {
            *abort_flag = 1;
            atomicOr(&g_device_error, 1u << FP8LIN_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms
// stacked along M/N (stride byte offset 1024).  The leading byte offset is
// unused for swizzled K-major layouts.  Bits 46..47 hold the descriptor
// version (1), bits 61..63 the layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void umma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// ------------------------------------------------------------- schedule

struct TileMap {
    int tiles_m, tiles_n;
    __device__ __forceinline__ void coords(int t, int &tm, int &tn) const {
        const int per_group = kGroupM * tiles_n;
        const int g = t / per_group;
        const int first_m = g * kGroupM;
        const int gm = min(tiles_m - first_m, kGroupM);
        const int r = t - g * per_group;
        tm = first_m + r % gm;
        tn = r / gm;
    }
};

// --------------------------------------------------------------- kernel

__global__ void __launch_bounds__(kThreads, 1)
fp8_gemm_tn_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   __nv_bfloat16 *__restrict__ C, int P, int Q, int R, const float *__restrict__ inv_a,
                   const float *__restrict__ inv_b, uint32_t idesc, TileMap tiles) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + kStages * kAStage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + kStages * kBStage);
    uint64_t *full = bars;                    // [kStages] TMA bytes landed
    uint64_t *empty = bars + kStages;         // [kStages] MMAs done reading the stage
    uint64_t *acc_full = bars + 2 * kStages;  // [2] accumulator finished
    uint64_t *acc_empty = acc_full + 2;       // [2] epilogue done reading the accumulator
    uint64_t *mma_done = acc_empty + 2;       // [1] drain of outstanding MMAs
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 4);  // one arrive per epilogue warp
        }
        mbar_init(smem_u32(mma_done), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_a);
        prefetch_tensormap(&map_b);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_tiles = tiles.tiles_m * tiles.tiles_n;
    const int num_kb = (R + kBK - 1) / kBK;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0;  // bit s: stage s has been armed at least once
            uint32_t armed_parity = 0;
            for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
                int tm, tn;
                tiles.coords(t, tm, tn);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) break;
                    const uint32_t fb = smem_u32(&full[stage]);
                    mbar_arrive_expect_tx(fb, kAStage + kBStage);
                    tma_load_2d(smem_u32(sA + stage * kAStage), &map_a, fb, kb * kBK, tm * kBM);
                    tma_load_2d(smem_u32(sB + stage * kBStage), &map_b, fb, kb * kBK, tn * kBN);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // Let every copy this thread started land before the CTA exits.
                for (int s = 0; s < kStages; ++s)
                    if (armed & (1u << s))
                        mbar_wait(smem_u32(&full[s]), (armed_parity >> s) & 1u, abort_flag, kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
                if (!mbar_wait(smem_u32(&acc_empty[acc]), acc_phase ^ 1u, abort_flag, kWaitLimitNs)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
                bool ok = true;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = sw128_kmajor_desc(smem_u32(sA + stage * kAStage));
                    const uint64_t b_desc = sw128_kmajor_desc(smem_u32(sB + stage * kBStage));
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        // advance the start address by k * 32 bytes inside the swizzle row
                        const uint64_t off = (uint64_t)((k * kUmmaK) >> 4);
                        umma_f8f6f4(d_tmem, a_desc + off, b_desc + off, idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&acc_full[acc]));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Every MMA issued above has completed once this arrives.
            umma_commit(smem_u32(mma_done));
            volatile int no_abort = 0;
            mbar_wait(smem_u32(mma_done), 0, &no_abort, kDrainLimitNs);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int sub = warp % 4;  // TMEM sub-partition this warp may read: lanes 32 sub .. 32 sub + 31
        const float sc = __fmul_rn(__ldg(inv_a), __ldg(inv_b));
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            const bool ok = mbar_wait(smem_u32(&acc_full[acc]), acc_phase, abort_flag, kWaitLimitNs);
            // reconverge: tcgen05.ld is warp-collective (.sync.aligned)
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            int tm, tn;
            tiles.coords(t, tm, tn);
            const int row = tm * kBM + sub * 32 + lane;
            __nv_bfloat16 *crow = C + (int64_t)row * Q;
            const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * kBN);
#pragma unroll 1
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), r);
                tmem_ld_wait();
                const int col0 = tn * kBN + c * 32;
                if (row < P) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (col0 + 8 * g < Q) {
                            uint4 o;
                            o.x = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * g + 0]), sc),
                                              __fmul_rn(__uint_as_float(r[8 * g + 1]), sc));
                            o.y = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * g + 2]), sc),
                                              __fmul_rn(__uint_as_float(r[8 * g + 3]), sc));
                            o.z = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * g + 4]), sc),
                                              __fmul_rn(__uint_as_float(r[8 * g + 5]), sc));
                            o.w = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * g + 6]), sc),
                                              __fmul_rn(__uint_as_float(r[8 * g + 7]), sc));
                            *reinterpret_cast<uint4 *>(crow + col0 + 8 * g) = o;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[acc]));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D map over a row-major [rows x inner] byte matrix, box = box_rows x 128 bytes.
bool make_operand_map(CUtensorMap *map, const void *base, int64_t rows, int64_t inner, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)inner};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4: fp32 accumulator
// (bits 4..5 = 1), A / B formats (bits 7..9 / 10..12: 0 = e4m3, 1 = e5m2),
// both operands K-major (bits 15, 16 = 0), N >> 3 at bits 17..22, M >> 4 at
// bits 24..28.
uint32_t make_idesc(fp8lin_fmt fa, fp8lin_fmt fb) {
    uint32_t d = 0;
    d |= 1u << 4;
    d |= (uint32_t)fa << 7;
    d |= (uint32_t)fb << 10;
    d |= (uint32_t)(kBN >> 3) << 17;
    d |= (uint32_t)(kBM >> 4) << 24;
    return d;
}

std::atomic<bool> g_smem_attr_set[64];

fp8lin_status gemm_tn(const uint8_t *A, fp8lin_fmt fa, const float *inv_a, const uint8_t *B, fp8lin_fmt fb,
                      const float *inv_b, void *C, int64_t P, int64_t Q, int64_t R, cudaStream_t stream) {
    using namespace fp8lin;
    if (inv_a == nullptr || inv_b == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (P < 0 || Q < 0 || R < 0) return FP8LIN_ERR_INVALID_ARG;
    const bool empty_out = P == 0 || Q == 0;
    if (!empty_out && C == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (!empty_out && R > 0 && (A == nullptr || B == nullptr)) return FP8LIN_ERR_INVALID_ARG;
    if (!aligned(inv_a, 4) || !aligned(inv_b, 4)) return FP8LIN_ERR_MISALIGNED;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16)) return FP8LIN_ERR_MISALIGNED;
    if (!dim_ok(P) || !dim_ok(Q) || !dim_ok(R) || P % 16 || Q % 16 || R % 16)
        return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo dev;
    fp8lin_status st = current_device(&dev);
    if (st != FP8LIN_OK) return st;
    if (empty_out) return FP8LIN_OK;
    if (R == 0) {  // empty contraction: C = 0
        return cudaMemsetAsync(C, 0, (size_t)P * (size_t)Q * 2, stream) == cudaSuccess ? FP8LIN_OK
                                                                                       : FP8LIN_ERR_CUDA;
    }
    const int64_t tiles_m = (P + kBM - 1) / kBM, tiles_n = (Q + kBN - 1) / kBN;
    if (tiles_m * tiles_n > INT32_MAX) return FP8LIN_ERR_UNSUPPORTED_SHAPE;

    CUtensorMap map_a, map_b;
    if (!make_operand_map(&map_a, A, P, R, kBM) || !make_operand_map(&map_b, B, Q, R, kBN))
        return FP8LIN_ERR_CUDA;

    if (dev.device >= 64) return FP8LIN_ERR_CUDA;
    if (!g_smem_attr_set[dev.device].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(fp8_gemm_tn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
            cudaSuccess)
            return FP8LIN_ERR_CUDA;
        g_smem_attr_set[dev.device].store(true, std::memory_order_release);
    }

    TileMap tm{(int)tiles_m, (int)tiles_n};
    const int num_tiles = (int)(tiles_m * tiles_n);
    const int grid = num_tiles < dev.sm_count ? num_tiles : dev.sm_count;
    fp8_gemm_tn_kernel<<<grid, kThreads, kSmemBytes, stream>>>(map_a, map_b, static_cast<__nv_bfloat16 *>(C),
                                                               (int)P, (int)Q, (int)R, inv_a, inv_b,
                                                               make_idesc(fa, fb), tm);
    return check_launch();
}

}  // namespace

extern "C" fp8lin_status fp8lin_fwd(const uint8_t *xq, const float *inv_x, const uint8_t *wq, const float *inv_w,
                                    void *y, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return gemm_tn(xq, FP8LIN_E4M3, inv_x, wq, FP8LIN_E4M3, inv_w, y, M, N, K, stream);
}

extern "C" fp8lin_status fp8lin_dgrad(const uint8_t *dyq, const float *inv_dy, const uint8_t *wqT,
                                      const float *inv_w, void *dx, int64_t M, int64_t N, int64_t K,
                                      cudaStream_t stream) {
    return gemm_tn(dyq, FP8LIN_E5M2, inv_dy, wqT, FP8LIN_E4M3, inv_w, dx, M, K, N, stream);
}

extern "C" fp8lin_status fp8lin_wgrad(const uint8_t *dyqT, const float *inv_dy, const uint8_t *xqT,
                                      const float *inv_x, void *dw, int64_t M, int64_t N, int64_t K,
                                      cudaStream_t stream) {
    return gemm_tn(dyqT, FP8LIN_E5M2, inv_dy, xqT, FP8LIN_E4M3, inv_x, dw, N, K, M, stream);
}

extern "C" fp8lin_status fp8lin_device_error(cudaStream_t stream, uint32_t *word) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP8LIN_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return FP8LIN_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) return FP8LIN_ERR_CUDA;
    if (word != nullptr) *word = v;
    return v == 0 ? FP8LIN_OK : FP8LIN_ERR_TIMEOUT;
}
