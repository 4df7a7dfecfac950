// gemm.cu -- the three scaled FP8 GEMMs of the Float8 linear layer on the
// sm_103a tensor cores (TorchTitan analysis page, section 3.3, "Mixed
// precision and Float8": Float8 applied to linear layers, composable with
// autograd, so forward, input gradient and weight gradient all run in FP8).
//
// Every GEMM is issued as C[P x Q] = A[P x R] . B[Q x R]^T.  Each operand is
// read either K-major (stored [rows x R], contraction contiguous) or MN-major
// (stored [R x rows], the row index contiguous): tcgen05 takes 8-bit operands
// in both majornesses, so the row-major FP8 copies the cast writes serve all
// three GEMMs and the transposed copies are optional:
//     fwd      : Y [M x N]  = Xq   [M x K] . Wq  [N x K]^T   both K-major
//     dgrad    : dX [M x K] = dYq  [M x N] . WqT [K x N]^T   both K-major
//     dgrad_mn : dX [M x K] = dYq  [M x N] . (Wq [N x K], read MN-major)
//     wgrad    : dW [N x K] = dYqT [N x M] . XqT [K x M]^T   both K-major
//     wgrad_mn : dW [N x K] = (dYq [M x N], MN-major) . (Xq [M x K], MN-major)
// (e4m3 x e4m3 forward, e5m2 x e4m3 backward) and the epilogue computes
// C = bf16_RN(acc_fp32 * (inv_a * inv_b)).  The two readings of the same
// bytes give bit-identical products.
//
// Kernel structure: clusters of two CTAs (one per SM of a pair), persistent,
// 192 threads per CTA.  A CTA pair owns a 256 x 256 output tile and computes
// it with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 32 per
// instruction): CTA r of the pair holds rows [128 r, 128 r + 128) of the A
// slab and rows [128 r, 128 r + 128) of the B slab in its own shared memory,
// and each SM's tensor core writes its 128 accumulator rows into its own
// TMEM.  Per CTA:
//   warp 0      TMA producer: 2-D tiled bulk-tensor loads of 128 x 128-byte A
//               and B boxes (128-byte swizzle) into a 6-stage ring; both
//               CTAs' loads complete on the leader CTA's full barrier;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators)
//               collectively with the peer CTA; in the leader CTA one thread
//               issues the MMAs (four per 128-byte slab) and multicasts each
//               tcgen05.commit to both CTAs' empty / accumulator barriers;
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns at a time, scale,
//               round to bf16, stage the 32 x 64-byte block in shared memory
//               (64-byte swizzle) and TMA-store it; each warp arrives on
//               the leader's accumulator-empty barrier once the last columns
//               are in registers, so the epilogue of tile i overlaps the
//               main loop of tile i + 1.
// Halving the B bytes per CTA (32 KB per slab instead of 48 KB for a
// 128 x 256 single-CTA tile) cuts the L2 -> SM traffic per flop by a third
// and leaves room for six stages.  Pair tiles are visited in groups of
// raster groups chosen from the operand sizes (see TileMap), so that the
// smaller operand is read from DRAM once when it fits in L2.
//
// The block-scaled GEMM (fp8_gemm_block_kernel, further down) runs on the
// same CTA pairs and 256 x 256 tiles and scales every 128-long contraction
// block's partial sums on the CUDA cores.
//
// Every mbarrier wait is bounded by wall-clock time (globaltimer).  A wait
// that runs out records FP8LIN_ERR_TIMEOUT in a device word, raises the
// CTA's abort flag, which ends every role's loop, drains the copies and MMAs
// still in flight (again with bounded waits), and the pair frees TMEM after
// a cluster barrier.
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kPairM = 256;           // output rows per CTA pair (UMMA M, cta_group::2)
constexpr int kPairN = 256;           // output columns per CTA pair (UMMA N)
constexpr int kBM = kPairM / 2;       // A rows held by each CTA
constexpr int kBN = kPairN / 2;       // B rows held by each CTA
constexpr int kBK = 128;              // contraction bytes per stage (one 128-byte swizzle row)
constexpr int kUmmaK = 32;            // contraction elements per tcgen05.mma for 8-bit types
#ifndef FP8LIN_GEMM_STAGES
#define FP8LIN_GEMM_STAGES 6
#endif
constexpr int kStages = FP8LIN_GEMM_STAGES;
constexpr int kAStage = kBM * kBK;    // 16 KB
constexpr int kBStage = kBN * kBK;    // 16 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 2 * kPairN; // two fp32 accumulators of 256 columns
constexpr int64_t kL2Resident = 40ll << 20;  // an operand up to this size is kept resident in L2
constexpr int kWaveGroup = 8;                 // otherwise: pair tiles per raster group
constexpr int kEpiCols = 32;                 // output columns per staged store: 64 bytes of bf16
constexpr int kEpiBuf = 32 * kEpiCols * 2;   // one epilogue warp's 32 rows x 64 bytes (2 KB)
constexpr int kEpiBytes = 4 * kEpiBuf;       // four epilogue warps, one buffer each
// The ring plus staging stays small enough that one cast / amax CTA (about
// 18 KB of shared memory) still fits beside a GEMM CTA on the same SM.
constexpr int kSmemBytes = kStages * (kAStage + kBStage) + kEpiBytes + 1024 /*barriers*/ + 1024 /*alignment*/;
#ifndef FP8LIN_WAIT_LIMIT_NS
#define FP8LIN_WAIT_LIMIT_NS 2000000000ull                  // 2 s per wait
#endif
constexpr unsigned long long kWaitLimitNs = FP8LIN_WAIT_LIMIT_NS;
constexpr unsigned long long kDrainLimitNs = 200000000ull;  // 0.2 s per drain wait

static_assert(kBK == 128, "one stage is one 128-byte swizzle row of contraction");
static_assert(kSmemBytes <= 232448, "shared memory per CTA is at most 227 KB");
static_assert(kPairN % kEpiCols == 0, "the epilogue stores whole 32-column blocks");
static_assert(kSmemBytes + 1024 + 18 * 1024 + 1024 <= 233472, "a cast CTA must fit beside a GEMM CTA");

__device__ unsigned int g_device_error = 0;

#ifdef FP8LIN_FAULT_INJECTION
// Test builds only (a library of its own, never the product one).  When
// g_withhold_slab >= 0, the producers of every CTA pair skip the copies of
// their g_withhold_slab-th slab (counted over the pair's tiles; for the
// power-of-two block-scaled GEMM, its stage of two slabs, scale atoms
// included) and the arrivals that would have expected them: nothing is ever
// in flight on that stage, so the MMA issuer's bounded wait on it runs out
// and the kernel takes its abort path.
__device__ int g_withhold_slab = -1;
#endif

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
// out, records the timeout and raises the flag.  The loop lives out of line;
// callers inline only the first try (mbar_wait below).
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
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

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned long long limit) {
    return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, abort_flag, limit);
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

// Start-address step, in 16-byte units, of the k-th K = 32 slice of a
// 128 x 128-byte slab.  K-major slab: rows are operand rows, so the slice
// starts 32 bytes further along each swizzled row.  MN-major slab: rows are
// contraction indices, so the slice starts 32 rows (4 KB) further down; the
// same descriptor (128-byte swizzle, 1024-byte stride between 8-row groups)
// describes both, with the majorness in the instruction descriptor.
template <bool MN>
__device__ __forceinline__ uint64_t kslice(int k) {
    return MN ? (uint64_t)((k * kUmmaK * 128) >> 4) : (uint64_t)((k * kUmmaK) >> 4);
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address, in the shared::cluster window, of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// Arrive on an mbarrier of either CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier of either CTA of the pair (the leader's, for the pair's MMA).
// `policy` is an L2 cache policy (createpolicy): the operand the raster
// holds in L2 is loaded evict_last, the one it streams with the normal policy.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t cluster_bar,
                                                 int c0, int c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// L2 policies of the two operands: the one the tile order holds (A unless
// the raster swaps the axes) evict_last, so the held panels outlive the
// streamed ones; the streamed operand keeps the normal policy (each of its
// panels is read by a whole wave of tiles that do not move through the
// contraction in lockstep, and evict_first lost slabs between readers).
__device__ __forceinline__ void operand_policies(int swap, uint64_t &pol_a, uint64_t &pol_b) {
    uint64_t keep, stream;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(stream));
    pol_a = swap ? stream : keep;
    pol_b = swap ? keep : stream;
}

// TMA store of one box from this CTA's shared memory, tracked in the
// issuing thread's bulk-async group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until none of this thread's committed bulk stores still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until all of this thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void umma_f8f6f4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on the mbarrier at this shared offset in every CTA of `mask`
// when all MMAs issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit_multicast(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

// Single-CTA forms (the block-scaled kernel): TMA completing on this CTA's
// barrier, MMA of one SM's tensor core, commit to this CTA's barrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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

// Pair tiles are visited in groups of `group` tiles along the "inner" axis
// (rows of A, or columns when `swap`), the inner index running fastest, so
// that the group's panels of that operand stay in L2 while the other
// operand's panels stream past them once per group.
struct TileMap {
    int tiles_m, tiles_n, group, swap;
    __device__ __forceinline__ void coords(int t, int &tm, int &tn) const {
        const int ti = swap ? tiles_n : tiles_m;   // inner axis
        const int to = swap ? tiles_m : tiles_n;   // outer axis
        const int per_group = group * to;
        const int g = t / per_group;
        const int first = g * group;
        const int gi = min(ti - first, group);
        const int r = t - g * per_group;
        const int i = first + r % gi, o = r / gi;
        tm = swap ? o : i;
        tn = swap ? i : o;
    }
};

// --------------------------------------------------------------- kernel

// VEC = false: inv_a, inv_b point to one float each (per-tensor scaling).
// VEC = true:  inv_a[P] and inv_b[Q] hold one inverse scale per row of A and
//              per row of B (row-wise scaling): C[p][q] = acc * (inv_a[p] * inv_b[q]).
// A_MN / B_MN: the operand is stored MN-major ([R x P] / [R x Q], the row
//              index contiguous) and loaded as 128 contraction rows x 128
//              bytes per slab; otherwise K-major ([P x R] / [Q x R]).
template <bool VEC, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1)
fp8_gemm_tn_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_c, int P, int Q, int R, const float *__restrict__ inv_a,
                   const float *__restrict__ inv_b, uint32_t idesc, TileMap tiles) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + kStages * kAStage;
    uint8_t *sC = sB + kStages * kBStage;     // epilogue staging: [4 warps][32 rows x 64 B], 64-byte swizzle
    uint64_t *bars = reinterpret_cast<uint64_t *>(sC + kEpiBytes);
    uint64_t *full = bars;                    // [kStages] both CTAs' slabs landed (leader's copy used)
    uint64_t *empty = bars + kStages;         // [kStages] the pair's MMAs are done with the slab
    uint64_t *acc_full = bars + 2 * kStages;  // [2] accumulator finished (arrived in both CTAs)
    uint64_t *acc_empty = acc_full + 2;       // [2] both CTAs' epilogues drained it (leader's copy used)
    uint64_t *mma_done = acc_empty + 2;       // [1] drain of outstanding MMAs (leader)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 8);  // four epilogue warps in each CTA of the pair
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
        // one warp of each CTA of the pair allocates collectively
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_tiles = tiles.tiles_m * tiles.tiles_n;
    const int num_kb = (R + kBK - 1) / kBK;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            uint64_t pol_a, pol_b;
            operand_policies(tiles.swap, pol_a, pol_b);
#ifdef FP8LIN_FAULT_INJECTION
            const int withhold = g_withhold_slab;
            int slab = 0;
#endif
            for (int t = pair; t < num_tiles && !*abort_flag; t += npairs) {
                int tm, tn;
                tiles.coords(t, tm, tn);
                const int a_row = tm * kPairM + (int)rank * kBM;
                const int b_row = tn * kPairN + (int)rank * kBN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) break;
                    bool issue = true;
#ifdef FP8LIN_FAULT_INJECTION
                    issue = slab++ != withhold;
#endif
                    if (issue) {
                        const uint32_t fb_local = smem_u32(&full[stage]);
                        if (leader) mbar_arrive_expect_tx(fb_local, 2 * (kAStage + kBStage));
                        const uint32_t fb = mapa_shared(fb_local, 0);
                        if (A_MN) tma_load_2d_pair(smem_u32(sA + stage * kAStage), &map_a, fb, a_row, kb * kBK, pol_a);
                        else      tma_load_2d_pair(smem_u32(sA + stage * kAStage), &map_a, fb, kb * kBK, a_row, pol_a);
                        if (B_MN) tma_load_2d_pair(smem_u32(sB + stage * kBStage), &map_b, fb, b_row, kb * kBK, pol_b);
                        else      tma_load_2d_pair(smem_u32(sB + stage * kBStage), &map_b, fb, kb * kBK, b_row, pol_b);
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (leader) {
                // Let every copy of the pair land before either CTA exits,
                // whether or not (or whenever) a wait ran out: both CTAs'
                // copies complete on the leader's full barriers.  A phase
                // the MMA issuer consumed has completed already.
                volatile int no_abort = 0;
                for (int s = 0; s < kStages; ++s)
                    if (armed & (1u << s))
                        mbar_wait(smem_u32(&full[s]), (armed_parity >> s) & 1u, &no_abort, kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader CTA)
        // Slabs are consumed two at a time: one pair of barrier waits, then
        // eight MMAs.  The tensor pipe keeps only a short queue of issued
        // MMAs, and the waits, fence and commits between groups must fit in
        // the time the queued ones take; four MMAs per wait leave the pipe
        // idle for part of every slab, eight do not.
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            // descriptors of slab 0; slab s starts s * 16 KB later (start-address field counts 16-byte units)
            const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(sA));
            const uint64_t b_desc0 = sw128_kmajor_desc(smem_u32(sB));
            for (int t = pair; t < num_tiles && !*abort_flag; t += npairs) {
                if (!mbar_wait(smem_u32(&acc_empty[acc]), acc_phase ^ 1u, abort_flag, kWaitLimitNs)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kPairN);
                bool ok = true;
                for (int kb = 0; kb < num_kb; kb += 2) {
                    const bool two = kb + 1 < num_kb;
                    const bool wrap = stage + 1 == kStages;
                    const int stage2 = wrap ? 0 : stage + 1;
                    const uint32_t phase2 = wrap ? phase ^ 1u : phase;
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs) ||
                        (two && !mbar_wait(smem_u32(&full[stage2]), phase2, abort_flag, kWaitLimitNs))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    {
                        const uint64_t a_desc = a_desc0 + (uint64_t)(stage * (kAStage >> 4));
                        const uint64_t b_desc = b_desc0 + (uint64_t)(stage * (kBStage >> 4));
#pragma unroll
                        for (int k = 0; k < kBK / kUmmaK; ++k) {
                            umma_f8f6f4_pair(d_tmem, a_desc + kslice<A_MN>(k), b_desc + kslice<B_MN>(k), idesc,
                                             (kb | k) != 0 ? 1u : 0u);
                        }
                        umma_commit_multicast(smem_u32(&empty[stage]), 0x3);
                    }
                    if (two) {
                        const uint64_t a_desc = a_desc0 + (uint64_t)(stage2 * (kAStage >> 4));
                        const uint64_t b_desc = b_desc0 + (uint64_t)(stage2 * (kBStage >> 4));
#pragma unroll
                        for (int k = 0; k < kBK / kUmmaK; ++k) {
                            umma_f8f6f4_pair(d_tmem, a_desc + kslice<A_MN>(k), b_desc + kslice<B_MN>(k), idesc, 1u);
                        }
                        umma_commit_multicast(smem_u32(&empty[stage2]), 0x3);
                    }
                    const int adv = two ? 2 : 1;
                    stage += adv;
                    if (stage >= kStages) {
                        stage -= kStages;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_multicast(smem_u32(&acc_full[acc]), 0x3);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Every MMA issued above has completed once this arrives.
            umma_commit_multicast(smem_u32(mma_done), 0x1);
            volatile int no_abort = 0;
            mbar_wait(smem_u32(mma_done), 0, &no_abort, kDrainLimitNs);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5, both CTAs)
        // Per 32-column block: tcgen05.ld, scale, round to bf16, write the
        // warp's 32 x 64-byte block into shared memory in the TMA 64-byte
        // swizzle (16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3):
        // conflict-free), and one lane issues a TMA store of the block.  The
        // accumulator is handed back as soon as its last columns are in
        // registers; the stores drain behind the next tile.
        const int sub = warp % 4;  // TMEM sub-partition this warp may read: lanes 32 sub .. 32 sub + 31
        uint8_t *stage_c = sC + (warp - 2) * kEpiBuf;
        uint8_t *dst = stage_c + lane * (kEpiCols * 2);
        const float sc = VEC ? 0.0f : __fmul_rn(__ldg(inv_a), __ldg(inv_b));
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = pair; t < num_tiles; t += npairs) {
            const bool ok = mbar_wait(smem_u32(&acc_full[acc]), acc_phase, abort_flag, kWaitLimitNs);
            // reconverge: tcgen05.ld is warp-collective (.sync.aligned)
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            int tm, tn;
            tiles.coords(t, tm, tn);
            const int row0 = tm * kPairM + (int)rank * kBM + sub * 32;  // first of this warp's rows
            const int row = row0 + lane;
            const uint32_t tbase = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(acc * kPairN);
            const float sa = (VEC && row < P) ? __ldg(inv_a + row) : 0.0f;
#pragma unroll 1
            for (int blk = 0; blk < kPairN / kEpiCols; ++blk) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(blk * kEpiCols), r);
                const int col0 = tn * kPairN + blk * kEpiCols;
                float f[32];
                if (VEC) {
                    // one inverse scale per output column: the same 32 floats for every lane
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        const float4 b4 = (col0 + 4 * g < Q) ? __ldg(reinterpret_cast<const float4 *>(inv_b + col0) + g)
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                        f[4 * g + 0] = __fmul_rn(sa, b4.x);
                        f[4 * g + 1] = __fmul_rn(sa, b4.y);
                        f[4 * g + 2] = __fmul_rn(sa, b4.z);
                        f[4 * g + 3] = __fmul_rn(sa, b4.w);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) f[j] = sc;
                }
                tmem_ld_wait();
                if (blk == kPairN / kEpiCols - 1) {
                    // every column of the accumulator is in registers: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[acc]), 0));
                }
                // the previous block's store must have read the staging buffer
                if (lane == 0) bulk_wait_read_0();
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 o;
                    o.x = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * c + 0]), f[8 * c + 0]),
                                      __fmul_rn(__uint_as_float(r[8 * c + 1]), f[8 * c + 1]));
                    o.y = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * c + 2]), f[8 * c + 2]),
                                      __fmul_rn(__uint_as_float(r[8 * c + 3]), f[8 * c + 3]));
                    o.z = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * c + 4]), f[8 * c + 4]),
                                      __fmul_rn(__uint_as_float(r[8 * c + 5]), f[8 * c + 5]));
                    o.w = pack_bf16x2(__fmul_rn(__uint_as_float(r[8 * c + 6]), f[8 * c + 6]),
                                      __fmul_rn(__uint_as_float(r[8 * c + 7]), f[8 * c + 7]));
                    *reinterpret_cast<uint4 *>(dst + ((c ^ ((lane >> 1) & 3)) << 4)) = o;
                }
                // make the generic-proxy writes visible to the TMA engine, then store
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0 && row0 < P && col0 < Q) {
                    tma_store_2d(&map_c, smem_u32(stage_c), col0, row0);
                    bulk_commit_group();
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA frees TMEM or exits while the pair still uses its shared memory
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------- block-scaled kernel

// mbar_wait entirely inline, for code after setmaxnreg: a call there would
// have to follow the caller's changed register budget.
__device__ __forceinline__ bool mbar_wait_inl(uint32_t bar, uint32_t parity, volatile int *abort_flag,
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

// mbar_arrive_cluster without release semantics, for a consumer that hands back
// TMEM it has finished reading (tcgen05.wait::ld has returned and
// tcgen05.fence::before_thread_sync orders the reads before the arrival):
// it publishes no memory, and a release at cluster scope costs the arriving
// warp hundreds of cycles.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Wait until at most one of this thread's committed bulk stores still reads
// shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// tcgen05.wait::ld tied to the registers a load wrote (32 or 64 columns), so
// that no use of them can be scheduled above it while another load is in
// flight.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
                 "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
                 "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                 "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
                 "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
                 "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
                 "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
                 "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait_regs64(uint32_t (&r)[64]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                 "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]),
                 "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]),
                 "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]),
                 "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]),
                 "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
                 :
                 : "memory");
}

// Asynchronous global -> shared copies (the scale ring of the block-scaled
// GEMM): 16 bytes, of which the first src_bytes are read and the rest
// zero-filled; 4 bytes; and an arrival on an mbarrier once every copy this
// thread issued before it has landed (counted in the barrier's init count).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }


// Block scaling along the contraction: C[p][q] = sum over 128-long
// contraction blocks j of (sum_{k in j} A[p][k] B[q][k])_fp32 * ia(p, j) * ib(q, j),
// with ia(p, j) = inv_a[j * sa_r + p] and ib(q, j) = inv_b[(q / 128) * sb_q +
// j * sb_r], or inv_b[j * sb_r + q] when B_COLS (one scale per row of B, i.e.
// per output column).
//
// The tensor cores cannot accumulate across contraction blocks (every
// block's partial sum needs its own scales), so each block's MMAs write a
// fresh fp32 partial into TMEM and the CUDA cores promote it: scale and add
// into accumulators held in registers.  Clusters of two CTAs, persistent
// over 256 x 256 output tiles as the per-tensor kernel (cta_group::2 MMAs of
// M 256, N 256, K 32: half the shared-memory and L2 traffic per flop of a
// one-SM 128 x 128 tile), 384 threads per CTA:
//   warpgroup 0 (40 registers after setmaxnreg.dec)
//     warp 0    TMA producer: this CTA's A and B slabs of each block into a
//               6-stage ring, completing on the leader's barrier;
//     warp 1    allocates 512 TMEM columns with the peer: two 128 x 256 fp32
//               partial buffers; in the leader one thread issues each
//               block's four MMAs into a free buffer and multicasts the
//               commits to both CTAs;
//     warp 2    scale loader: per block this CTA's 128 row scales of A and
//               the tile's two B scales (or 256 column scales) into an
//               8-deep ring, with asynchronous copies;
//     warp 3    idle;
//   warpgroups 1, 2 (232 registers after setmaxnreg.inc)
//     warps 4..11 promotion: warp w reads TMEM lanes 32 (w % 4) .. + 31,
//               columns 128 ((w - 4) / 4) .. + 127 of the buffer (64 columns
//               per load, or with column scales 32 with the next 32 in
//               flight), scales them and adds them to 128 fp32 accumulators
//               (two columns per fma.rn.f32x2); hands the buffer back to the
//               leader once its last columns are in registers, with a
//               relaxed arrival (a release at cluster scope costs each warp
//               more than the block's arithmetic); after the tile's last
//               block, rounds to bf16 and TMA-stores as the per-tensor
//               epilogue does.
// The register split is 128 x 40 + 256 x 232 = 64512 = 384 x 168, the
// registers the CTA is launched with (the host checks the compiled count
// before launching).  The two partial buffers let the MMAs of block j + 1 run
// while block j is promoted.
constexpr int kBlk = 128;                             // contraction block and scale block of the recipe
constexpr int kBlkThreads = 384;
constexpr int kBlkLaunchRegs = 168;
constexpr int kBlkLowRegs = 40;
constexpr int kBlkHighRegs = 232;
static_assert(128 * kBlkLowRegs + 256 * kBlkHighRegs == kBlkThreads * kBlkLaunchRegs,
              "the register split must add up to the launch allocation");
constexpr int kBlkPromoWarps = 8;
constexpr int kBlkWarpCols = 128;                     // columns each promotion warp owns
constexpr int kBlkTmemCols = 2 * kPairN;
constexpr int kBlkStages = 5;                         // slab ring: about five blocks of lookahead
constexpr int kBlkEpiBytes = kBlkPromoWarps * 2 * kEpiBuf;  // two staging buffers per promotion warp
constexpr int kBlkScaleSlots = 8;                     // contraction blocks of scales in flight
constexpr int kBlkSlotFloats = kBM + kPairN;          // this CTA's row scales of A, then B's scales
constexpr int kBlkScaleBytes = kBlkScaleSlots * kBlkSlotFloats * 4;
constexpr int kBlkSmemBytes =
    kBlkStages * (kAStage + kBStage) + kBlkEpiBytes + kBlkScaleBytes + 1024 /*barriers*/ + 1024 /*alignment*/;
static_assert(kBlkSmemBytes <= 232448, "shared memory per CTA is at most 227 KB");
static_assert(kBK == kBlk && kBlkWarpCols == kBlk, "a slab is one contraction block; a warp's columns one B block");

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Two lanes of fp32 at once (fma.rn.f32x2 / mul.rn.f32x2: each lane rounded
// once, as the scalar instructions): acc += p * s, and p * c.
__device__ __forceinline__ void fma2(float &acc0, float &acc1, float p0, float p1, float s0, float s1) {
    asm("{\n\t.reg .b64 a, p, s;\n\t"
        "mov.b64 a, {%0, %1};\n\t"
        "mov.b64 p, {%2, %3};\n\t"
        "mov.b64 s, {%4, %5};\n\t"
        "fma.rn.f32x2 a, p, s, a;\n\t"
        "mov.b64 {%0, %1}, a;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "f"(p0), "f"(p1), "f"(s0), "f"(s1));
}
__device__ __forceinline__ void mul2(float &r0, float &r1, float p0, float p1, float c0, float c1) {
    asm("{\n\t.reg .b64 r, p, c;\n\t"
        "mov.b64 p, {%2, %3};\n\t"
        "mov.b64 c, {%4, %5};\n\t"
        "mul.rn.f32x2 r, p, c;\n\t"
        "mov.b64 {%0, %1}, r;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(p0), "f"(p1), "f"(c0), "f"(c1));
}

// The promotion of 32 partial sums of one row: acc += p * sab, or with
// per-column scales acc += (p * col[j]) * sab; two columns per instruction.
template <bool B_COLS>
__device__ __forceinline__ void promote32(float *acc, const uint32_t (&p)[32], float sab, const float *col) {
    if (B_COLS) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const float4 b = reinterpret_cast<const float4 *>(col)[g];
            float q0, q1, q2, q3;
            mul2(q0, q1, __uint_as_float(p[4 * g + 0]), __uint_as_float(p[4 * g + 1]), b.x, b.y);
            mul2(q2, q3, __uint_as_float(p[4 * g + 2]), __uint_as_float(p[4 * g + 3]), b.z, b.w);
            fma2(acc[4 * g + 0], acc[4 * g + 1], q0, q1, sab, sab);
            fma2(acc[4 * g + 2], acc[4 * g + 3], q2, q3, sab, sab);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; j += 2)
            fma2(acc[j], acc[j + 1], __uint_as_float(p[j]), __uint_as_float(p[j + 1]), sab, sab);
    }
}

template <bool B_COLS>
__device__ __forceinline__ void promote64(float *acc, const uint32_t (&p)[64], float sab, const float *col) {
    promote32<B_COLS>(acc, reinterpret_cast<const uint32_t (&)[32]>(p[0]), sab, col);
    promote32<B_COLS>(acc + 32, reinterpret_cast<const uint32_t (&)[32]>(p[32]), sab, col + 32);
}

template <bool A_MN, bool B_MN, bool B_COLS>
__global__ void __launch_bounds__(kBlkThreads, 1)
fp8_gemm_block_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                      const __grid_constant__ CUtensorMap map_c, int P, int Q, int R,
                      const float *__restrict__ inv_a, long long sa_r, const float *__restrict__ inv_b,
                      long long sb_q, long long sb_r, uint32_t idesc, TileMap tiles) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = smem;                                 // [stages][128 x 128 B]
    uint8_t *sB = smem + kBlkStages * kAStage;          // [stages][128 x 128 B]
    uint8_t *sC = sB + kBlkStages * kBStage;            // epilogue staging: [8 warps][2][32 rows x 64 B]
    float *sScale = reinterpret_cast<float *>(sC + kBlkEpiBytes);  // [slots][A rows 128, B 256 (or 2)]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sScale + kBlkScaleSlots * kBlkSlotFloats);
    uint64_t *full = bars;                              // [stages] both CTAs' slabs landed (leader's copy used)
    uint64_t *empty = bars + kBlkStages;                // [stages] the pair's MMAs are done with the slabs
    uint64_t *pfull = bars + 2 * kBlkStages;               // [2] a partial buffer is complete (in both CTAs)
    uint64_t *pempty = pfull + 2;                       // [2] both CTAs' promotion warps read it (leader's copy)
    uint64_t *sfull = pempty + 2;                       // [slots] a block's scales landed
    uint64_t *sempty = sfull + kBlkScaleSlots;          // [slots] the promotion warps are done with them
    uint64_t *mma_done = sempty + kBlkScaleSlots;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kBlkStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&pfull[b]), 1);
            mbar_init(smem_u32(&pempty[b]), 2 * kBlkPromoWarps);  // eight warps in each CTA of the pair
        }
        for (int s = 0; s < kBlkScaleSlots; ++s) {
            mbar_init(smem_u32(&sfull[s]), 32);         // one asynchronous arrival per loader lane
            mbar_init(smem_u32(&sempty[s]), kBlkPromoWarps);
        }
        mbar_init(smem_u32(mma_done), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_a);
        prefetch_tensormap(&map_b);
        prefetch_tensormap(&map_c);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kBlkTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_tiles = tiles.tiles_m * tiles.tiles_n;
    const int num_kb = (R + kBK - 1) / kBK;

    if (warp < 4) {
        setmaxnreg_dec<kBlkLowRegs>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            uint64_t pol_a, pol_b;
            operand_policies(tiles.swap, pol_a, pol_b);
#ifdef FP8LIN_FAULT_INJECTION
            const int withhold = g_withhold_slab;
            int slab = 0;
#endif
            for (int t = pair; t < num_tiles && !*abort_flag; t += npairs) {
                int tm, tn;
                tiles.coords(t, tm, tn);
                const int a_row = tm * kPairM + (int)rank * kBM;
                const int b_row = tn * kPairN + (int)rank * kBN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_inl(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) break;
                    bool issue = true;
#ifdef FP8LIN_FAULT_INJECTION
                    issue = slab++ != withhold;
#endif
                    if (issue) {
                        const uint32_t fb_local = smem_u32(&full[stage]);
                        if (leader) mbar_arrive_expect_tx(fb_local, 2 * (kAStage + kBStage));
                        const uint32_t fb = mapa_shared(fb_local, 0);
                        if (A_MN) tma_load_2d_pair(smem_u32(sA + stage * kAStage), &map_a, fb, a_row, kb * kBK, pol_a);
                        else      tma_load_2d_pair(smem_u32(sA + stage * kAStage), &map_a, fb, kb * kBK, a_row, pol_a);
                        if (B_MN) tma_load_2d_pair(smem_u32(sB + stage * kBStage), &map_b, fb, b_row, kb * kBK, pol_b);
                        else      tma_load_2d_pair(smem_u32(sB + stage * kBStage), &map_b, fb, kb * kBK, b_row, pol_b);
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == kBlkStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (leader) {
                // let every copy of the pair land before either CTA exits, abort or not
                volatile int no_abort = 0;
                for (int s = 0; s < kBlkStages; ++s)
                    if (armed & (1u << s))
                        mbar_wait_inl(smem_u32(&full[s]), (armed_parity >> s) & 1u, &no_abort, kDrainLimitNs);
            }
        } else if (warp == 1 && lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (leader CTA)
            int stage = 0;
            uint32_t phase = 0;
            int pb = 0;
            uint32_t pphase = 0;
            const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(sA));
            const uint64_t b_desc0 = sw128_kmajor_desc(smem_u32(sB));
            bool ok = true;
            for (int t = pair; t < num_tiles && ok && !*abort_flag; t += npairs) {
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait_inl(smem_u32(&pempty[pb]), pphase ^ 1u, abort_flag, kWaitLimitNs) ||
                        !mbar_wait_inl(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = a_desc0 + (uint64_t)(stage * (kAStage >> 4));
                    const uint64_t b_desc = b_desc0 + (uint64_t)(stage * (kBStage >> 4));
                    const uint32_t d_tmem = tmem_base + (uint32_t)(pb * kPairN);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k)
                        umma_f8f6f4_pair(d_tmem, a_desc + kslice<A_MN>(k), b_desc + kslice<B_MN>(k), idesc,
                                         k != 0 ? 1u : 0u);
                    umma_commit_multicast(smem_u32(&empty[stage]), 0x3);
                    umma_commit_multicast(smem_u32(&pfull[pb]), 0x3);
                    if (++stage == kBlkStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++pb == 2) {
                        pb = 0;
                        pphase ^= 1u;
                    }
                }
            }
            // every MMA issued above has completed once this arrives
            umma_commit_multicast(smem_u32(mma_done), 0x1);
            volatile int no_abort = 0;
            mbar_wait_inl(smem_u32(mma_done), 0, &no_abort, kDrainLimitNs);
        } else if (warp == 2) {
            // ------------------------------------------------ scale loader (both CTAs)
            // Lane l copies this CTA's rows 4l .. 4l + 3 of the tile (16
            // bytes; rows past P zero-filled without a read) and, with
            // B_COLS, columns 4l .. 4l + 3 and 128 + 4l .. 128 + 4l + 3;
            // otherwise lanes 0, 1 copy the scales of the tile's two B blocks
            // (the last block of B repeated past Q, where every partial sum
            // is zero).
            int slot = 0;
            uint32_t sphase = 0;
            bool ok = true;
            const long long last_qb = (long long)(Q - 1) / kBlk;
            for (int t = pair; t < num_tiles && ok; t += npairs) {
                int tm, tn;
                tiles.coords(t, tm, tn);
                const int r = tm * kPairM + (int)rank * kBM + 4 * lane, c = tn * kPairN + 4 * lane;
                const bool r_in = r < P, c0_in = c < Q, c1_in = c + kBlk < Q;
                const long long qb = min((long long)(2 * tn + (lane & 1)), last_qb);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait_inl(smem_u32(&sempty[slot]), sphase ^ 1u, abort_flag,
                                                               kWaitLimitNs))) {
                        ok = false;
                        break;
                    }
                    const uint32_t s = smem_u32(sScale + slot * kBlkSlotFloats);
                    cp_async_16(s + 16u * lane, r_in ? inv_a + (long long)kb * sa_r + r : inv_a, r_in ? 16u : 0u);
                    if (B_COLS) {
                        const float *b = inv_b + (long long)kb * sb_r + c;
                        cp_async_16(s + 4u * kBM + 16u * lane, c0_in ? b : inv_b, c0_in ? 16u : 0u);
                        cp_async_16(s + 4u * (kBM + kBlk) + 16u * lane, c1_in ? b + kBlk : inv_b, c1_in ? 16u : 0u);
                    } else if (lane < 2) {
                        cp_async_4(s + 4u * (kBM + lane), inv_b + qb * sb_q + (long long)kb * sb_r);
                    }
                    cp_async_arrive_noinc(smem_u32(&sfull[slot]));
                    if (++slot == kBlkScaleSlots) {
                        slot = 0;
                        sphase ^= 1u;
                    }
                }
            }
            cp_async_wait_all();
        }
    } else {
        setmaxnreg_inc<kBlkHighRegs>();
        // ------------------------------------------------ promotion + epilogue (warps 4..11, both CTAs)
        const int sub = warp % 4;          // TMEM lanes 32 sub .. 32 sub + 31: this warp's 32 rows
        const int cw = (warp - 4) / 4;     // which 128-column half of the pair tile
        const int srow = sub * 32 + lane;  // this thread's row within the CTA's 128
        uint8_t *stage_c = sC + (warp - 4) * 2 * kEpiBuf;  // two buffers, alternate 32-column blocks
        const uint32_t pempty_leader0 = mapa_shared(smem_u32(&pempty[0]), 0);
        const uint32_t pempty_leader1 = mapa_shared(smem_u32(&pempty[1]), 0);
        const uint32_t tlane = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(cw * kBlkWarpCols);
        int pb = 0, slot = 0;
        uint32_t pphase = 0, sphase = 0;
        bool ok = true;
        // Partial sums come out of TMEM 64 columns per load, or, with column
        // scales (whose shared-memory reads need registers of their own), 32
        // at a time with the next 32 in flight.
        uint32_t x[32], y[32];
        uint32_t x64[64];
        // A block's scales, read from the ring one block ahead of their use:
        // sab = row scale (times the B block's scale), col = column scales.
        auto scales = [&](int slot_, float &sab_, const float *&col_) -> bool {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_inl(smem_u32(&sfull[slot_]), sphase ^ (slot_ < slot ? 1u : 0u),
                                                       abort_flag, kWaitLimitNs)))
                return false;
            const float *sc = sScale + slot_ * kBlkSlotFloats;
            sab_ = B_COLS ? sc[srow] : __fmul_rn(sc[srow], sc[kBM + cw]);
            col_ = sc + kBM + cw * kBlkWarpCols;
            return true;
        };
        for (int t = pair; t < num_tiles && ok; t += npairs) {
            int tm, tn;
            tiles.coords(t, tm, tn);
            const int row0 = tm * kPairM + (int)rank * kBM + sub * 32;
            const int col_base = tn * kPairN + cw * kBlkWarpCols;   // first output column of this warp
            float acc[kBlkWarpCols];
#pragma unroll
            for (int j = 0; j < kBlkWarpCols; ++j) acc[j] = 0.0f;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_inl(smem_u32(&pfull[pb]), pphase, abort_flag, kWaitLimitNs))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if constexpr (B_COLS) {
                tmem_ld_32x32b_x32(tlane + (uint32_t)(pb * kPairN), x);
                float sab;
                const float *col;
                ok = scales(slot, sab, col);
                tmem_ld_wait_regs(x);
                if (!ok) break;
                for (int kb = 0; kb < num_kb; ++kb) {
                    // x holds columns 0..31 of block kb's buffer; sab, col its scales
                    const uint32_t tb = tlane + (uint32_t)(pb * kPairN);
                    tmem_ld_32x32b_x32(tb + 32u, y);
                    promote32<B_COLS>(acc, x, sab, col);
                    tmem_ld_wait_regs(y);
                    tmem_ld_32x32b_x32(tb + 64u, x);
                    promote32<B_COLS>(acc + 32, y, sab, col + 32);
                    tmem_ld_wait_regs(x);
                    tmem_ld_32x32b_x32(tb + 96u, y);
                    promote32<B_COLS>(acc + 64, x, sab, col + 64);
                    tmem_ld_wait_regs(y);
                    // the warp's part of the buffer is in registers: hand it back to the leader
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(pb ? pempty_leader1 : pempty_leader0);
                    if (++pb == 2) {
                        pb = 0;
                        pphase ^= 1u;
                    }
                    const bool more = kb + 1 < num_kb;
                    const int next_slot = slot + 1 == kBlkScaleSlots ? 0 : slot + 1;
                    float sab_n = 0.0f;
                    const float *col_n = col;
                    if (more) {
                        if (!__all_sync(0xFFFFFFFFu,
                                        mbar_wait_inl(smem_u32(&pfull[pb]), pphase, abort_flag, kWaitLimitNs)) ||
                            !scales(next_slot, sab_n, col_n)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        tmem_ld_32x32b_x32(tlane + (uint32_t)(pb * kPairN), x);
                    }
                    promote32<B_COLS>(acc + 96, y, sab, col + 96);
                    __syncwarp();
                    if (lane == 0) mbar_arrive_local(smem_u32(&sempty[slot]));
                    slot = next_slot;
                    if (slot == 0) sphase ^= 1u;
                    sab = sab_n;
                    col = col_n;
                    if (more) tmem_ld_wait_regs(x);
                }
            } else {
                tmem_ld_32x32b_x64(tlane + (uint32_t)(pb * kPairN), x64);
                float sab;
                const float *col;
                ok = scales(slot, sab, col);
                tmem_ld_wait_regs64(x64);
                if (!ok) break;
                for (int kb = 0; kb < num_kb; ++kb) {
                    // x64 holds columns 0..63 of block kb's buffer; sab, col its scales
                    const uint32_t tb = tlane + (uint32_t)(pb * kPairN);
                    promote64<B_COLS>(acc, x64, sab, col);
                    tmem_ld_32x32b_x64(tb + 64u, x64);
                    tmem_ld_wait_regs64(x64);
                    // the warp's part of the buffer is in registers: hand it back to the leader
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(pb ? pempty_leader1 : pempty_leader0);
                    if (++pb == 2) {
                        pb = 0;
                        pphase ^= 1u;
                    }
                    const bool more = kb + 1 < num_kb;
                    const int next_slot = slot + 1 == kBlkScaleSlots ? 0 : slot + 1;
                    float sab_n = 0.0f;
                    const float *col_n = col;
                    promote64<B_COLS>(acc + 64, x64, sab, col + 64);
                    if (more) {
                        if (!__all_sync(0xFFFFFFFFu,
                                        mbar_wait_inl(smem_u32(&pfull[pb]), pphase, abort_flag, kWaitLimitNs)) ||
                            !scales(next_slot, sab_n, col_n)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        tmem_ld_32x32b_x64(tlane + (uint32_t)(pb * kPairN), x64);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive_local(smem_u32(&sempty[slot]));
                    slot = next_slot;
                    if (slot == 0) sphase ^= 1u;
                    sab = sab_n;
                    col = col_n;
                    if (more) tmem_ld_wait_regs64(x64);
                }
            }
            if (!ok) break;
            // epilogue: round to bf16 and TMA-store 32 columns at a time from
            // two alternating staging buffers; the blocks past the output's
            // edge (a suffix of the four) are neither staged nor stored
            if (lane == 0) bulk_wait_read_0();   // the previous tile's stores are done reading
#pragma unroll
            for (int c = 0; c < kBlkWarpCols / kEpiCols; ++c) {
                const int col0 = col_base + c * kEpiCols;
                if (row0 >= P || col0 >= Q) break;
                uint8_t *buf = stage_c + (c & 1) * kEpiBuf;
                if (c >= 2 && lane == 0) bulk_wait_read_1();   // the store of block c - 2 (same buffer) has read it
                __syncwarp();
                uint8_t *dst = buf + lane * (kEpiCols * 2);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int j = c * kEpiCols + 8 * g;
                    uint4 o;
                    o.x = pack_bf16x2(acc[j + 0], acc[j + 1]);
                    o.y = pack_bf16x2(acc[j + 2], acc[j + 3]);
                    o.z = pack_bf16x2(acc[j + 4], acc[j + 5]);
                    o.w = pack_bf16x2(acc[j + 6], acc[j + 7]);
                    *reinterpret_cast<uint4 *>(dst + ((g ^ ((lane >> 1) & 3)) << 4)) = o;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&map_c, smem_u32(buf), col0, row0);
                    bulk_commit_group();
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA frees TMEM or exits while the pair still uses its shared memory
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kBlkTmemCols)
                     : "memory");
    }
}

// ------------------------------------- power-of-two block-scaled kernel

// Block scaling with power-of-two scales, applied by the tensor cores:
// tcgen05.mma kind::mxf8f6f4.block_scale multiplies every 32-long run of the
// contraction by the scale bytes (unsigned exponents, 2^(byte - 127)) of its
// A row and B row and accumulates in fp32 across the whole contraction, so
// the MMAs accumulate in TMEM as in the per-tensor kernel and nothing is
// promoted on the CUDA cores.  The scales of a 128-long slab (this CTA's 128
// A rows and the tile's 256 B rows: 512 + 1024 bytes, stored by the cast as
// the "atoms" described at fp8lin_cast_mx) ride in the slab's stage.  The
// MMA reads them from TMEM: row p's four bytes (one per 32-run of the slab,
// picked by the scale IDs of the instruction descriptor) in lane p, column
// p / 32 of the A region; column n's in column n / 32 of the B region, in
// every lane quarter (each quarter's datapath reads its own copy), and in
// each CTA of the pair its own TMEM for all 256 B rows.
//
// The scales go into TMEM with tcgen05.st from a warpgroup of their own
// (one warp per lane quarter, each writing the same 16 + 32 bytes per lane),
// not with tcgen05.cp: a copy issued between the MMAs occupies the tensor
// pipe (about 50 cycles per 512-byte atom, three per 512-cycle slab, where
// the writes from registers run beside the MMAs).  Once the four writer
// warps' stores have completed, one thread per CTA hands the slot to the
// leader's MMA issuer through an mbarrier.
//
// A stage holds two slabs (256 contraction elements): one barrier round,
// one MMA commit and one scale hand-over per two slabs, since each commit
// and each copy issued between MMAs costs tensor-pipe time.
//
// TMEM: one 256-column fp32 accumulator (columns 0..255) and a 32-column
// scale slot per stage from column 256.  With one accumulator the epilogue
// frees it as soon as it is in registers: eight epilogue warps (two per
// lane quarter, 128 columns each) load their columns, hand the accumulator
// back to the leader, then round, stage and TMA-store while the next tile's
// MMAs run.  512 threads:
//   warpgroup 0 (56 registers after setmaxnreg)
//     warp 0    TMA producer: A and B slabs (completing on the leader's
//               barrier) and the slab's scale atoms (completing on this
//               CTA's own barrier);
//     warp 1    TMEM allocation; in the leader one thread issues the MMAs,
//               two slabs per round of barrier waits;
//     warps 2-3 idle;
//   warpgroups 1, 2 (200 registers): epilogue;
//   warpgroup 3 (56 registers): scale writers.
// 128 x 56 + 256 x 200 + 128 x 56 = 65536 = 512 x 128, the registers the
// CTA is launched with (the host checks the compiled count).
constexpr int kMxSlabs = 2;                          // 128-long slabs per stage
constexpr int kMxStages = 3;                         // stages: six slabs in flight
constexpr int kMxThreads = 512;
constexpr int kMxLaunchRegs = 128;
constexpr int kMxLowRegs = 56;
constexpr int kMxHighRegs = 200;
static_assert(2 * 128 * kMxLowRegs + 256 * kMxHighRegs <= kMxThreads * kMxLaunchRegs,
              "the register split must fit in the launch allocation");
constexpr int kMxSfa = 512;                          // this CTA's A scales per slab
constexpr int kMxSfb = 1024;                         // the tile's B scales per slab (both 128-row blocks)
constexpr int kMxEpiBytes = kBlkPromoWarps * kEpiBuf;  // one staging buffer per epilogue warp
constexpr int kMxSmemBytes =
    kMxStages * kMxSlabs * (kAStage + kBStage + kMxSfa + kMxSfb) + kMxEpiBytes + 1024 + 1024;
constexpr int kMxSfCol = kPairN;                     // first TMEM column of the scale slots
constexpr int kMxSfSlotCols = 32;                    // per stage: A 2 x 4 columns, B 2 x 8 columns
static_assert(kMxSmemBytes <= 232448, "shared memory per CTA is at most 227 KB");
static_assert(kMxSfCol + kMxStages * kMxSfSlotCols <= 512, "scale slots fit in the allocated TMEM");
static_assert(kMxSlabs == 2 && kMxSlabs * (4 + 8) <= kMxSfSlotCols, "a stage's scales fit in its slot");
static_assert((kMxStages * kMxSlabs * (kAStage + kBStage)) % 1024 == 0 && kMxEpiBytes % 1024 == 0,
              "the epilogue staging (64-byte swizzle) and the scale atoms start on aligned offsets");

__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, uint4 a, uint4 b) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// AND of v over the 128 threads of the scale-writer warpgroup (named barrier 1).
__device__ __forceinline__ bool writers_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void umma_mx_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kMxThreads, 1)
fp8_gemm_mx_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CUtensorMap map_sfa,
                   const __grid_constant__ CUtensorMap map_sfb, int P, int Q, int R, int pb_a, int pb_b,
                   uint32_t idesc, TileMap tiles) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = smem;                                   // [stages][2 slabs][128 x 128 B]
    uint8_t *sB = sA + kMxStages * kMxSlabs * kAStage;    // [stages][2 slabs][128 x 128 B]
    uint8_t *sC = sB + kMxStages * kMxSlabs * kBStage;    // epilogue staging: [8 warps][32 rows x 64 B]
    uint8_t *sSfa = sC + kMxEpiBytes;                     // [stages][2 slabs][512 B]
    uint8_t *sSfb = sSfa + kMxStages * kMxSlabs * kMxSfa; // [stages][2 slabs][1024 B]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sSfb + kMxStages * kMxSlabs * kMxSfb);
    uint64_t *full = bars;                                // [stages] both CTAs' A and B slabs landed (leader)
    uint64_t *empty = bars + kMxStages;                   // [stages] the pair's MMAs are done with the stage
    uint64_t *sf_full = bars + 2 * kMxStages;             // [stages] this CTA's scale atoms landed
    uint64_t *sf_ready = bars + 3 * kMxStages;            // [stages] both CTAs' scales are in TMEM (leader)
    uint64_t *acc_full = bars + 4 * kMxStages;            // the tile's accumulator is complete (both CTAs)
    uint64_t *acc_empty = acc_full + 1;                   // both CTAs' epilogues hold it in registers (leader)
    uint64_t *mma_done = acc_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kMxStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
            mbar_init(smem_u32(&sf_full[s]), 1);
            mbar_init(smem_u32(&sf_ready[s]), 2);    // one arrival from each CTA of the pair
        }
        mbar_init(smem_u32(acc_full), 1);
        mbar_init(smem_u32(acc_empty), 2 * kBlkPromoWarps);  // eight warps in each CTA of the pair
        mbar_init(smem_u32(mma_done), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_a);
        prefetch_tensormap(&map_b);
        prefetch_tensormap(&map_c);
        prefetch_tensormap(&map_sfa);
        prefetch_tensormap(&map_sfb);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kBlkTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_tiles = tiles.tiles_m * tiles.tiles_n;
    const int num_kb = (R + kBK - 1) / kBK;
    const int num_st = (num_kb + kMxSlabs - 1) / kMxSlabs;   // stages per tile (the last may hold one slab)

    if (warp < 4) {
        setmaxnreg_dec<kMxLowRegs>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            uint64_t pol_a, pol_b;
            operand_policies(tiles.swap, pol_a, pol_b);
#ifdef FP8LIN_FAULT_INJECTION
            const int withhold = g_withhold_slab;   // counted in stages (two slabs each) here
            int stage_count = 0;
#endif
            for (int t = pair; t < num_tiles && !*abort_flag; t += npairs) {
                int tm, tn;
                tiles.coords(t, tm, tn);
                const int a_row = tm * kPairM + (int)rank * kBM;
                const int b_row = tn * kPairN + (int)rank * kBN;
                for (int ks = 0; ks < num_st; ++ks) {
                    if (!mbar_wait_inl(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) break;
#ifdef FP8LIN_FAULT_INJECTION
                    if (stage_count++ == withhold) {
                        // neither this stage's slabs nor its scale atoms are copied
                        if (++stage == kMxStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
#endif
                    const uint32_t fb_local = smem_u32(&full[stage]);
                    if (leader) mbar_arrive_expect_tx(fb_local, 2 * kMxSlabs * (kAStage + kBStage));
                    const uint32_t sb = smem_u32(&sf_full[stage]);
                    mbar_arrive_expect_tx(sb, kMxSlabs * (kMxSfa + kMxSfb));
                    const uint32_t fb = mapa_shared(fb_local, 0);
                    // both slabs are loaded even past the contraction's end (zero-filled,
                    // scales past the last atom read as zero), so every stage moves the same bytes
#pragma unroll
                    for (int h = 0; h < kMxSlabs; ++h) {
                        const int kb = ks * kMxSlabs + h;
                        const int sl = stage * kMxSlabs + h;
                        if (A_MN) tma_load_2d_pair(smem_u32(sA + sl * kAStage), &map_a, fb, a_row, kb * kBK, pol_a);
                        else      tma_load_2d_pair(smem_u32(sA + sl * kAStage), &map_a, fb, kb * kBK, a_row, pol_a);
                        if (B_MN) tma_load_2d_pair(smem_u32(sB + sl * kBStage), &map_b, fb, b_row, kb * kBK, pol_b);
                        else      tma_load_2d_pair(smem_u32(sB + sl * kBStage), &map_b, fb, kb * kBK, b_row, pol_b);
                        // scale atoms: this CTA's 128 A rows; both 128-row blocks of the tile's B rows
                        tma_load_2d(smem_u32(sSfa + sl * kMxSfa), &map_sfa, sb, 0, kb * pb_a + 2 * tm + (int)rank);
                        tma_load_2d(smem_u32(sSfb + sl * kMxSfb), &map_sfb, sb, 0, kb * pb_b + 2 * tn);
                    }
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == kMxStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            {
                // let every copy land before either CTA exits, abort or not
                volatile int no_abort = 0;
                for (int s = 0; s < kMxStages; ++s)
                    if (armed & (1u << s)) {
                        if (leader)
                            mbar_wait_inl(smem_u32(&full[s]), (armed_parity >> s) & 1u, &no_abort, kDrainLimitNs);
                        mbar_wait_inl(smem_u32(&sf_full[s]), (armed_parity >> s) & 1u, &no_abort, kDrainLimitNs);
                    }
            }
        } else if (warp == 1 && lane == 0 && leader) {
            // ------------------------------------------------ scale copies + MMA issuer (leader CTA)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_phase = 0;
            const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(sA));
            const uint64_t b_desc0 = sw128_kmajor_desc(smem_u32(sB));
            bool ok = true;
            // slab h of stage st: its scales at columns 4h (A) and 8 + 8h (B) of the slot
            auto issue_slab = [&](int st, int h, bool first) {
                const uint32_t sf = tmem_base + (uint32_t)(kMxSfCol + st * kMxSfSlotCols);
                const int sl = st * kMxSlabs + h;
                const uint64_t a_desc = a_desc0 + (uint64_t)(sl * (kAStage >> 4));
                const uint64_t b_desc = b_desc0 + (uint64_t)(sl * (kBStage >> 4));
#pragma unroll
                for (int k = 0; k < kBK / kUmmaK; ++k)
                    umma_mx_pair(tmem_base, a_desc + kslice<A_MN>(k), b_desc + kslice<B_MN>(k),
                                 idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29), sf + 4 * h, sf + 8 + 8 * h,
                                 (first && k == 0) ? 0u : 1u);
            };
            for (int t = pair; t < num_tiles && ok && !*abort_flag; t += npairs) {
                if (!mbar_wait_inl(smem_u32(acc_empty), acc_phase ^ 1u, abort_flag, kWaitLimitNs)) break;
                tc_fence_after();
                for (int ks = 0; ks < num_st; ++ks) {
                    if (!mbar_wait_inl(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs) ||
                        !mbar_wait_inl(smem_u32(&sf_ready[stage]), phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_slab(stage, 0, ks == 0);
                    if (ks * kMxSlabs + 1 < num_kb) issue_slab(stage, 1, false);
                    umma_commit_multicast(smem_u32(&empty[stage]), 0x3);
                    if (++stage == kMxStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_multicast(smem_u32(acc_full), 0x3);
                acc_phase ^= 1u;
            }
            // every MMA issued above has completed once this arrives
            umma_commit_multicast(smem_u32(mma_done), 0x1);
            volatile int no_abort = 0;
            mbar_wait_inl(smem_u32(mma_done), 0, &no_abort, kDrainLimitNs);
        }
    } else if (warp >= 12) {
        setmaxnreg_dec<kMxLowRegs>();
        // ------------------------------------------------ scale writers (warps 12..15, both CTAs)
        // Warp 12 + q writes lane quarter q: lane r holds the 16 bytes of atom
        // row r (rows r, r + 32, r + 64, r + 96, one per column) for A and
        // for each of B's two 128-row blocks -- the same bytes in every quarter.
        const int q = warp - 12;
        const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)kMxSfCol;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = pair; t < num_tiles && ok; t += npairs) {
            for (int ks = 0; ks < num_st; ++ks) {
                // the four writer warps agree on going on (every one of them reaches this
                // barrier on every slab, so none is left waiting at the one below)
                if (!writers_all(__all_sync(0xFFFFFFFFu, mbar_wait_inl(smem_u32(&sf_full[stage]), phase,
                                                                        abort_flag, kWaitLimitNs)))) {
                    ok = false;
                    break;
                }
                // slot columns: A of slab 0, A of slab 1 (4 each), B of slab 0, B of slab 1 (8 each)
                const uint32_t a_sm = smem_u32(sSfa + stage * kMxSlabs * kMxSfa + 16 * lane);
                const uint32_t b_sm = smem_u32(sSfb + stage * kMxSlabs * kMxSfb + 16 * lane);
                const uint4 a0 = lds128(a_sm), a1 = lds128(a_sm + kMxSfa);
                const uint4 b00 = lds128(b_sm), b01 = lds128(b_sm + 512);
                const uint4 b10 = lds128(b_sm + kMxSfb), b11 = lds128(b_sm + kMxSfb + 512);
                const uint32_t slot = tq + (uint32_t)(stage * kMxSfSlotCols);
                tmem_st_32x32b_x8(slot, a0, a1);
                tmem_st_32x32b_x8(slot + 8, b00, b01);
                tmem_st_32x32b_x8(slot + 16, b10, b11);
                tmem_st_wait();
                tc_fence_before();
                // the four writer warps meet; one thread per CTA then tells the
                // leader's issuer.  The stores have completed (tcgen05.wait::st) and
                // the fence orders them before the arrival, and nothing in generic
                // memory is published, so the peer CTA arrives without release
                // semantics (a release at cluster scope costs hundreds of cycles per
                // arrival, more than a slab's MMAs leave).
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (q == 0 && lane == 0) {
                    if (leader) mbar_arrive_local(smem_u32(&sf_ready[stage]));
                    else        mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&sf_ready[stage]), 0));
                }
                if (++stage == kMxStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        setmaxnreg_inc<kMxHighRegs>();
        // ------------------------------------------------ epilogue (warps 4..11, both CTAs)
        const int sub = warp % 4;          // TMEM lanes 32 sub .. 32 sub + 31: this warp's 32 rows
        const int cw = (warp - 4) / 4;     // which 128-column half of the pair tile
        uint8_t *stage_c = sC + (warp - 4) * kEpiBuf;      // this warp's staging buffer
        const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);
        const uint32_t tlane = tmem_base + ((uint32_t)(sub * 32) << 16) + (uint32_t)(cw * kBlkWarpCols);
        uint32_t acc_phase = 0;
        uint32_t lo[64], hi[64];
        for (int t = pair; t < num_tiles; t += npairs) {
            int tm, tn;
            tiles.coords(t, tm, tn);
            const int row0 = tm * kPairM + (int)rank * kBM + sub * 32;
            const int col_base = tn * kPairN + cw * kBlkWarpCols;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_inl(smem_u32(acc_full), acc_phase, abort_flag, kWaitLimitNs)))
                break;
            acc_phase ^= 1u;
            tc_fence_after();
            tmem_ld_32x32b_x64(tlane, lo);
            tmem_ld_32x32b_x64(tlane + 64u, hi);
            tmem_ld_wait_regs64(lo);
            tmem_ld_wait_regs64(hi);
            // the warp's part of the accumulator is in registers: hand it back to the leader
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_leader);
            // round to bf16 and TMA-store 32 columns at a time through the staging
            // buffer; blocks past the output's edge are neither staged nor stored
            if (lane == 0) bulk_wait_read_0();   // the previous tile's stores are done reading
#pragma unroll
            for (int c = 0; c < kBlkWarpCols / kEpiCols; ++c) {
                const int col0 = col_base + c * kEpiCols;
                if (row0 >= P || col0 >= Q) break;
                uint8_t *buf = stage_c;
                if (c >= 1 && lane == 0) bulk_wait_read_0();   // the store of block c - 1 has read the buffer
                __syncwarp();
                uint8_t *dst = buf + lane * (kEpiCols * 2);
                const uint32_t *src = c < 2 ? lo + 32 * c : hi + 32 * (c - 2);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int j = 8 * g;
                    uint4 o;
                    o.x = pack_bf16x2(__uint_as_float(src[j + 0]), __uint_as_float(src[j + 1]));
                    o.y = pack_bf16x2(__uint_as_float(src[j + 2]), __uint_as_float(src[j + 3]));
                    o.z = pack_bf16x2(__uint_as_float(src[j + 4]), __uint_as_float(src[j + 5]));
                    o.w = pack_bf16x2(__uint_as_float(src[j + 6]), __uint_as_float(src[j + 7]));
                    *reinterpret_cast<uint4 *>(dst + ((g ^ ((lane >> 1) & 3)) << 4)) = o;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&map_c, smem_u32(buf), col0, row0);
                    bulk_commit_group();
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA frees TMEM or exits while the pair still uses its shared memory
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kBlkTmemCols)
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

// 2-D map over the row-major bf16 output [rows x cols]; box = 32 rows x 32
// columns (64 bytes), 64-byte swizzle, as the epilogue stages it.
bool make_output_map(CUtensorMap *map, void *base, int64_t rows, int64_t cols) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kEpiCols, 32u};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over an operand read MN-major: logically [P x R], stored as the
// row-major [R x P] byte matrix (P contiguous); box = 128 contraction rows x
// box_cols bytes.
bool make_operand_map_mn(CUtensorMap *map, const void *base, int64_t P, int64_t R, int box_cols) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)P, (cuuint64_t)R};
    cuuint64_t strides[1] = {(cuuint64_t)P};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)kBK};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
// A / B majorness (bits 15 / 16: 0 = K-major, 1 = MN-major), N >> 3 at bits
// 17..22, M >> 4 at bits 24..28; M and N are the pair's (256 x 256), or the
// single CTA's (128 x 128) for the block-scaled kernel.
uint32_t make_idesc(fp8lin_fmt fa, fp8lin_fmt fb, bool a_mn, bool b_mn, int m = kPairM, int n = kPairN) {
    uint32_t d = 0;
    d |= 1u << 4;
    d |= (uint32_t)fa << 7;
    d |= (uint32_t)fb << 10;
    d |= (uint32_t)a_mn << 15;
    d |= (uint32_t)b_mn << 16;
    d |= (uint32_t)(n >> 3) << 17;
    d |= (uint32_t)(m >> 4) << 24;
    return d;
}

// Per kernel instance (scale mode x A majorness x B majorness) and device:
// attributes set, co-resident clusters.
std::atomic<bool> g_smem_attr_set[8][64];
std::atomic<int> g_max_clusters[8][64];

template <bool VEC, bool A_MN, bool B_MN>
constexpr int instance() {
    return VEC * 4 + A_MN * 2 + B_MN;
}

cudaLaunchConfig_t launch_config(int grid, cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    attr->id = cudaLaunchAttributeClusterDimension;
    attr->val.clusterDim.x = 2;
    attr->val.clusterDim.y = 1;
    attr->val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Raster: keep the smaller operand resident in L2 (up to kL2Resident: a
// panel set read by SMs of both dies is cached in each die's half of the L2)
// and stream the larger one once.  If neither fits, the tiles
// running at once move through the contraction together, so L2 only has to
// hold their current slabs: group kWaveGroup tiles along one axis (a wave
// covers a compact block of tiles, each panel read once per group),
// choosing the orientation with the fewest modelled DRAM bytes.  Either way
// the producers load the held operand evict_last (operand_policies).
TileMap raster(int64_t P, int64_t Q, int64_t R, int64_t tiles_m, int64_t tiles_n) {
    const int64_t bytes_a = P * R, bytes_b = Q * R;
    TileMap tm{(int)tiles_m, (int)tiles_n, 1, 0};
    if (bytes_a <= kL2Resident && bytes_a <= bytes_b) {
        tm.group = (int)tiles_m;                      // all of A per column of tiles
    } else if (bytes_b <= kL2Resident) {
        tm.group = (int)tiles_n;                      // all of B per row of tiles
        tm.swap = 1;
    } else {
        const int64_t g = kWaveGroup;
        const int64_t gm = g < tiles_m ? g : tiles_m, gn = g < tiles_n ? g : tiles_n;
        const int64_t traffic_m = bytes_a + bytes_b * ((tiles_m + gm - 1) / gm);   // A panels held
        const int64_t traffic_n = bytes_b + bytes_a * ((tiles_n + gn - 1) / gn);   // B panels held
        if (traffic_n < traffic_m) {
            tm.group = (int)gn;
            tm.swap = 1;
        } else {
            tm.group = (int)gm;
        }
    }
    return tm;
}

// Checks shared by every GEMM entry point.
fp8lin_status gemm_checks(const uint8_t *A, const float *inv_a, const uint8_t *B, const float *inv_b, void *C,
                          int64_t P, int64_t Q, int64_t R) {
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
    return FP8LIN_OK;
}

template <bool VEC, bool A_MN, bool B_MN>
fp8lin_status gemm_tn(const uint8_t *A, fp8lin_fmt fa, const float *inv_a, const uint8_t *B, fp8lin_fmt fb,
                      const float *inv_b, void *C, int64_t P, int64_t Q, int64_t R, cudaStream_t stream) {
    using namespace fp8lin;
    fp8lin_status st = gemm_checks(A, inv_a, B, inv_b, C, P, Q, R);
    if (st != FP8LIN_OK) return st;
    if (VEC && (!aligned(inv_a, 16) || !aligned(inv_b, 16))) return FP8LIN_ERR_MISALIGNED;
    const bool empty_out = P == 0 || Q == 0;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != FP8LIN_OK) return st;
    if (empty_out) return FP8LIN_OK;
    if (R == 0) {  // empty contraction: C = 0
        return cudaMemsetAsync(C, 0, (size_t)P * (size_t)Q * 2, stream) == cudaSuccess ? FP8LIN_OK
                                                                                       : FP8LIN_ERR_CUDA;
    }
    const int64_t tiles_m = (P + kPairM - 1) / kPairM, tiles_n = (Q + kPairN - 1) / kPairN;
    if (tiles_m * tiles_n > INT32_MAX) return FP8LIN_ERR_UNSUPPORTED_SHAPE;

    CUtensorMap map_a, map_b, map_c;
    const bool ok_a = A_MN ? make_operand_map_mn(&map_a, A, P, R, kBM) : make_operand_map(&map_a, A, P, R, kBM);
    const bool ok_b = B_MN ? make_operand_map_mn(&map_b, B, Q, R, kBN) : make_operand_map(&map_b, B, Q, R, kBN);
    if (!ok_a || !ok_b ||
        !make_output_map(&map_c, C, P, Q))
        return FP8LIN_ERR_CUDA;

    if (dev.device >= 64) return FP8LIN_ERR_CUDA;
    if (!g_smem_attr_set[instance<VEC, A_MN, B_MN>()][dev.device].load(std::memory_order_acquire)) {
        auto kernel = fp8_gemm_tn_kernel<VEC, A_MN, B_MN>;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
                cudaSuccess ||
            cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return FP8LIN_ERR_CUDA;
        // pairs that can be resident at once (a GPC with an odd number of free SMs leaves one idle)
        int clusters = 0;
        cudaLaunchAttribute attr;
        cudaLaunchConfig_t cfg = launch_config(2 * (dev.sm_count / 2), nullptr, &attr);
        if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters < 1)
            clusters = dev.sm_count / 2;
        g_max_clusters[instance<VEC, A_MN, B_MN>()][dev.device].store(clusters, std::memory_order_relaxed);
        g_smem_attr_set[instance<VEC, A_MN, B_MN>()][dev.device].store(true, std::memory_order_release);
    }

    const TileMap tm = raster(P, Q, R, tiles_m, tiles_n);
    const int num_tiles = (int)(tiles_m * tiles_n);
    const int max_pairs = g_max_clusters[instance<VEC, A_MN, B_MN>()][dev.device].load(std::memory_order_relaxed);
    const int pairs = num_tiles < max_pairs ? num_tiles : max_pairs;
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = launch_config(2 * pairs, stream, &attr);
    const int p = (int)P, q = (int)Q, r = (int)R;
    const uint32_t idesc = make_idesc(fa, fb, A_MN, B_MN);
    if (cudaLaunchKernelEx(&cfg, fp8_gemm_tn_kernel<VEC, A_MN, B_MN>, map_a, map_b, map_c, p, q, r, inv_a, inv_b,
                           idesc, tm) !=
        cudaSuccess)
        return FP8LIN_ERR_CUDA;
    return check_launch();
}

std::atomic<bool> g_blk_attr_set[8][64];
std::atomic<int> g_blk_ctas[8][64];

// The block-scaled GEMM (see fp8_gemm_block_kernel): inverse scales of A at
// inv_a[j * sa_r + p], of B at inv_b[(q / 128) * sb_q + j * sb_r] (or
// [j * sb_r + q] when B_COLS); sizes are the caller's to guarantee.  The
// scale loader copies four consecutive rows' (columns') scales at a time, so
// those vectors are 16-byte aligned with strides that are multiples of 4.
template <bool A_MN, bool B_MN, bool B_COLS>
fp8lin_status gemm_block(const uint8_t *A, fp8lin_fmt fa, const float *inv_a, int64_t sa_r, const uint8_t *B,
                         fp8lin_fmt fb, const float *inv_b, int64_t sb_q, int64_t sb_r, void *C, int64_t P,
                         int64_t Q, int64_t R, cudaStream_t stream) {
    using namespace fp8lin;
    fp8lin_status st = gemm_checks(A, inv_a, B, inv_b, C, P, Q, R);
    if (st != FP8LIN_OK) return st;
    if (!aligned(inv_a, 16) || sa_r % 4 || (B_COLS && (!aligned(inv_b, 16) || sb_r % 4)))
        return FP8LIN_ERR_MISALIGNED;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != FP8LIN_OK) return st;
    if (P == 0 || Q == 0) return FP8LIN_OK;
    if (R == 0) {
        return cudaMemsetAsync(C, 0, (size_t)P * (size_t)Q * 2, stream) == cudaSuccess ? FP8LIN_OK
                                                                                       : FP8LIN_ERR_CUDA;
    }
    const int64_t tiles_m = (P + kPairM - 1) / kPairM, tiles_n = (Q + kPairN - 1) / kPairN;
    if (tiles_m * tiles_n > INT32_MAX) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    CUtensorMap map_a, map_b, map_c;
    const bool ok_a = A_MN ? make_operand_map_mn(&map_a, A, P, R, kBM) : make_operand_map(&map_a, A, P, R, kBM);
    const bool ok_b = B_MN ? make_operand_map_mn(&map_b, B, Q, R, kBN) : make_operand_map(&map_b, B, Q, R, kBN);
    if (!ok_a || !ok_b || !make_output_map(&map_c, C, P, Q)) return FP8LIN_ERR_CUDA;
    if (dev.device >= 64) return FP8LIN_ERR_CUDA;
    constexpr int inst = A_MN * 4 + B_MN * 2 + B_COLS;
    auto kernel = fp8_gemm_block_kernel<A_MN, B_MN, B_COLS>;
    cudaLaunchAttribute attr;
    auto config = [&](int grid, cudaStream_t s) {
        cudaLaunchConfig_t cfg = launch_config(grid, s, &attr);
        cfg.blockDim = dim3(kBlkThreads, 1, 1);
        cfg.dynamicSmemBytes = kBlkSmemBytes;
        return cfg;
    };
    if (!g_blk_attr_set[inst][dev.device].load(std::memory_order_acquire)) {
        // The register split assumes the compiled count; with any other
        // count setmaxnreg.inc could wait forever, so never launch it then.
        cudaFuncAttributes fa_attr;
        if (cudaFuncGetAttributes(&fa_attr, kernel) != cudaSuccess) return FP8LIN_ERR_CUDA;
        if (fa_attr.numRegs != kBlkLaunchRegs) return FP8LIN_ERR_CUDA;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBlkSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return FP8LIN_ERR_CUDA;
        int clusters = 0;
        cudaLaunchConfig_t cfg = config(2 * (dev.sm_count / 2), nullptr);
        if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters < 1)
            return FP8LIN_ERR_CUDA;
        g_blk_ctas[inst][dev.device].store(clusters, std::memory_order_relaxed);
        g_blk_attr_set[inst][dev.device].store(true, std::memory_order_release);
    }
    const TileMap tm = raster(P, Q, R, tiles_m, tiles_n);
    const int num_tiles = (int)(tiles_m * tiles_n);
    const int max_pairs = g_blk_ctas[inst][dev.device].load(std::memory_order_relaxed);
    const int pairs = num_tiles < max_pairs ? num_tiles : max_pairs;
    cudaLaunchConfig_t cfg = config(2 * pairs, stream);
    const uint32_t idesc = make_idesc(fa, fb, A_MN, B_MN);
    if (cudaLaunchKernelEx(&cfg, kernel, map_a, map_b, map_c, (int)P, (int)Q, (int)R, inv_a, (long long)sa_r, inv_b,
                           (long long)sb_q, (long long)sb_r, idesc, tm) != cudaSuccess)
        return FP8LIN_ERR_CUDA;
    return check_launch();
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

std::atomic<bool> g_mx_attr_set[4][64];
std::atomic<int> g_mx_ctas[4][64];

// 2-D map over scale atoms: [atom_rows x 128] 32-bit words (512 bytes per
// atom), box = box_rows atoms; atoms past the end read as zero.
bool make_sf_map(CUtensorMap *map, const void *base, int64_t atom_rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {128, (cuuint64_t)atom_rows};
    cuuint64_t strides[1] = {512};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Instruction descriptor of tcgen05.mma kind::mxf8f6f4.block_scale: A / B
// formats (bits 7..9 / 10..12), majorness (bits 15 / 16), N >> 3 at bits
// 17..22, unsigned-exponent scales (bit 23), M >> 4 at bits 24..28; the scale
// IDs (bits 4..5 for B, 29..30 for A: which byte of the scale words, i.e.
// which 32-run of the slab) are or-ed in per MMA.
uint32_t make_idesc_mx(fp8lin_fmt fa, fp8lin_fmt fb, bool a_mn, bool b_mn) {
    uint32_t d = 0;
    d |= (uint32_t)fa << 7;
    d |= (uint32_t)fb << 10;
    d |= (uint32_t)a_mn << 15;
    d |= (uint32_t)b_mn << 16;
    d |= (uint32_t)(kPairN >> 3) << 17;
    d |= 1u << 23;
    d |= (uint32_t)(kPairM >> 4) << 24;
    return d;
}

// The power-of-two block-scaled GEMM (see fp8_gemm_mx_kernel): C = A . B^T
// with the scale atoms of A (operand rows P, contraction R) and of B
// (operand rows Q); sizes are the caller's to guarantee.
template <bool A_MN, bool B_MN>
fp8lin_status gemm_mx(const uint8_t *A, fp8lin_fmt fa, const uint8_t *sfa, const uint8_t *B, fp8lin_fmt fb,
                      const uint8_t *sfb, void *C, int64_t P, int64_t Q, int64_t R, cudaStream_t stream) {
    using namespace fp8lin;
    if (P < 0 || Q < 0 || R < 0) return FP8LIN_ERR_INVALID_ARG;
    const bool empty_out = P == 0 || Q == 0;
    if (!empty_out && C == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (!empty_out && R > 0 && (A == nullptr || B == nullptr || sfa == nullptr || sfb == nullptr))
        return FP8LIN_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(sfa, 16) || !aligned(sfb, 16))
        return FP8LIN_ERR_MISALIGNED;
    if (!dim_ok(P) || !dim_ok(Q) || !dim_ok(R) || P % 16 || Q % 16 || R % 16) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo dev;
    fp8lin_status st = current_device(&dev);
    if (st != FP8LIN_OK) return st;
    if (empty_out) return FP8LIN_OK;
    if (R == 0) {
        return cudaMemsetAsync(C, 0, (size_t)P * (size_t)Q * 2, stream) == cudaSuccess ? FP8LIN_OK
                                                                                       : FP8LIN_ERR_CUDA;
    }
    const int64_t tiles_m = (P + kPairM - 1) / kPairM, tiles_n = (Q + kPairN - 1) / kPairN;
    const int64_t pb_a = ceil_div(P, 128), pb_b = ceil_div(Q, 128), nkb = ceil_div(R, 128);
    if (tiles_m * tiles_n > INT32_MAX || nkb * (pb_a + 2) > INT32_MAX || nkb * (pb_b + 2) > INT32_MAX)
        return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    CUtensorMap map_a, map_b, map_c, map_sfa, map_sfb;
    const bool ok_a = A_MN ? make_operand_map_mn(&map_a, A, P, R, kBM) : make_operand_map(&map_a, A, P, R, kBM);
    const bool ok_b = B_MN ? make_operand_map_mn(&map_b, B, Q, R, kBN) : make_operand_map(&map_b, B, Q, R, kBN);
    if (!ok_a || !ok_b || !make_output_map(&map_c, C, P, Q) || !make_sf_map(&map_sfa, sfa, nkb * pb_a, 1) ||
        !make_sf_map(&map_sfb, sfb, nkb * pb_b, 2))
        return FP8LIN_ERR_CUDA;
    if (dev.device >= 64) return FP8LIN_ERR_CUDA;
    constexpr int inst = A_MN * 2 + B_MN;
    auto kernel = fp8_gemm_mx_kernel<A_MN, B_MN>;
    cudaLaunchAttribute attr;
    auto config = [&](int grid, cudaStream_t s) {
        cudaLaunchConfig_t cfg = launch_config(grid, s, &attr);
        cfg.blockDim = dim3(kMxThreads, 1, 1);
        cfg.dynamicSmemBytes = kMxSmemBytes;
        return cfg;
    };
    if (!g_mx_attr_set[inst][dev.device].load(std::memory_order_acquire)) {
        // the register split assumes the compiled count (see gemm_block)
        cudaFuncAttributes fa_attr;
        if (cudaFuncGetAttributes(&fa_attr, kernel) != cudaSuccess) return FP8LIN_ERR_CUDA;
        if (fa_attr.numRegs != kMxLaunchRegs) return FP8LIN_ERR_CUDA;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return FP8LIN_ERR_CUDA;
        int clusters = 0;
        cudaLaunchConfig_t cfg = config(2 * (dev.sm_count / 2), nullptr);
        if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters < 1)
            return FP8LIN_ERR_CUDA;
        g_mx_ctas[inst][dev.device].store(clusters, std::memory_order_relaxed);
        g_mx_attr_set[inst][dev.device].store(true, std::memory_order_release);
    }
    const TileMap tm = raster(P, Q, R, tiles_m, tiles_n);
    const int num_tiles = (int)(tiles_m * tiles_n);
    const int max_pairs = g_mx_ctas[inst][dev.device].load(std::memory_order_relaxed);
    const int pairs = num_tiles < max_pairs ? num_tiles : max_pairs;
    cudaLaunchConfig_t cfg = config(2 * pairs, stream);
    const uint32_t idesc = make_idesc_mx(fa, fb, A_MN, B_MN);
    if (cudaLaunchKernelEx(&cfg, kernel, map_a, map_b, map_c, map_sfa, map_sfb, (int)P, (int)Q, (int)R, (int)pb_a,
                           (int)pb_b, idesc, tm) != cudaSuccess)
        return FP8LIN_ERR_CUDA;
    return check_launch();
}


}  // namespace

// Block scaling: X and dY in 1 x 128 / 128 x 1 blocks, W in 128 x 128 blocks
// (fp8lin_cast_blockwise); the GEMM scales each 128-long contraction block.
extern "C" fp8lin_status fp8lin_fwd_block(const uint8_t *xq, const float *inv_x, const uint8_t *wq,
                                          const float *inv_w, void *y, int64_t M, int64_t N, int64_t K,
                                          cudaStream_t stream) {
    // A = Xq (row blocks, inv_x [KB x M]), B = Wq (tiles, inv_w [NB x KB]); contraction K
    const int64_t kb = ceil_div(K, kBlk);
    return gemm_block<false, false, false>(xq, FP8LIN_E4M3, inv_x, M, wq, FP8LIN_E4M3, inv_w, kb, 1, y, M, N,
                                           K, stream);
}

extern "C" fp8lin_status fp8lin_dgrad_block(const uint8_t *dyq, const float *inv_dy, const uint8_t *wq,
                                            const float *inv_w, void *dx, int64_t M, int64_t N, int64_t K,
                                            cudaStream_t stream) {
    // A = dYq (row blocks, inv_dy [NB x M]), B = Wq read MN-major: row k of B,
    // contraction block j scaled by inv_w[j][k / 128]; contraction N
    const int64_t kb = ceil_div(K, kBlk);
    return gemm_block<false, true, false>(dyq, FP8LIN_E5M2, inv_dy, M, wq, FP8LIN_E4M3, inv_w, 1, kb, dx, M, K,
                                          N, stream);
}

extern "C" fp8lin_status fp8lin_wgrad_block(const uint8_t *dyq, const float *inv_dy, const uint8_t *xq,
                                            const float *inv_x, void *dw, int64_t M, int64_t N, int64_t K,
                                            cudaStream_t stream) {
    // A = dYq read MN-major (column blocks: row n of A, block j at inv_dy[j][n]),
    // B = Xq read MN-major (column blocks: row k of B, block j at inv_x[j][k]); contraction M
    return gemm_block<true, true, true>(dyq, FP8LIN_E5M2, inv_dy, N, xq, FP8LIN_E4M3, inv_x, 1, K, dw, N, K, M,
                                        stream);
}

// Power-of-two block scaling (fp8lin_cast_mx): the tensor cores apply the
// scales of every 32-long run of the contraction.
extern "C" fp8lin_status fp8lin_fwd_mx(const uint8_t *xq, const uint8_t *sf_x, const uint8_t *wq,
                                       const uint8_t *sf_w, void *y, int64_t M, int64_t N, int64_t K,
                                       cudaStream_t stream) {
    // A = Xq row copy [M x K], B = Wq row copy [N x K], both K-major; contraction K
    return gemm_mx<false, false>(xq, FP8LIN_E4M3, sf_x, wq, FP8LIN_E4M3, sf_w, y, M, N, K, stream);
}

extern "C" fp8lin_status fp8lin_dgrad_mx(const uint8_t *dyq, const uint8_t *sf_dy, const uint8_t *wq,
                                         const uint8_t *sf_w, void *dx, int64_t M, int64_t N, int64_t K,
                                         cudaStream_t stream) {
    // A = dYq row copy [M x N] (K-major), B = Wq column copy [N x K] read MN-major; contraction N
    return gemm_mx<false, true>(dyq, FP8LIN_E5M2, sf_dy, wq, FP8LIN_E4M3, sf_w, dx, M, K, N, stream);
}

extern "C" fp8lin_status fp8lin_wgrad_mx(const uint8_t *dyq, const uint8_t *sf_dy, const uint8_t *xq,
                                         const uint8_t *sf_x, void *dw, int64_t M, int64_t N, int64_t K,
                                         cudaStream_t stream) {
    // A = dYq column copy [M x N] read MN-major, B = Xq column copy [M x K] read MN-major; contraction M
    return gemm_mx<true, true>(dyq, FP8LIN_E5M2, sf_dy, xq, FP8LIN_E4M3, sf_x, dw, N, K, M, stream);
}

extern "C" fp8lin_status fp8lin_fwd(const uint8_t *xq, const float *inv_x, const uint8_t *wq, const float *inv_w,
                                    void *y, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return gemm_tn<false, false, false>(xq, FP8LIN_E4M3, inv_x, wq, FP8LIN_E4M3, inv_w, y, M, N, K, stream);
}

extern "C" fp8lin_status fp8lin_dgrad(const uint8_t *dyq, const float *inv_dy, const uint8_t *wqT,
                                      const float *inv_w, void *dx, int64_t M, int64_t N, int64_t K,
                                      cudaStream_t stream) {
    return gemm_tn<false, false, false>(dyq, FP8LIN_E5M2, inv_dy, wqT, FP8LIN_E4M3, inv_w, dx, M, K, N, stream);
}

extern "C" fp8lin_status fp8lin_wgrad(const uint8_t *dyqT, const float *inv_dy, const uint8_t *xqT,
                                      const float *inv_x, void *dw, int64_t M, int64_t N, int64_t K,
                                      cudaStream_t stream) {
    return gemm_tn<false, false, false>(dyqT, FP8LIN_E5M2, inv_dy, xqT, FP8LIN_E4M3, inv_x, dw, N, K, M, stream);
}

// The backward GEMMs on the row-major FP8 copies the cast writes as q.
extern "C" fp8lin_status fp8lin_dgrad_mn(const uint8_t *dyq, const float *inv_dy, const uint8_t *wq,
                                         const float *inv_w, void *dx, int64_t M, int64_t N, int64_t K,
                                         cudaStream_t stream) {
    return gemm_tn<false, false, true>(dyq, FP8LIN_E5M2, inv_dy, wq, FP8LIN_E4M3, inv_w, dx, M, K, N, stream);
}

extern "C" fp8lin_status fp8lin_wgrad_mn(const uint8_t *dyq, const float *inv_dy, const uint8_t *xq,
                                         const float *inv_x, void *dw, int64_t M, int64_t N, int64_t K,
                                         cudaStream_t stream) {
    return gemm_tn<false, true, true>(dyq, FP8LIN_E5M2, inv_dy, xq, FP8LIN_E4M3, inv_x, dw, N, K, M, stream);
}

extern "C" fp8lin_status fp8lin_fwd_rowwise(const uint8_t *xq, const float *inv_x_rows, const uint8_t *wq,
                                            const float *inv_w_rows, void *y, int64_t M, int64_t N, int64_t K,
                                            cudaStream_t stream) {
    return gemm_tn<true, false, false>(xq, FP8LIN_E4M3, inv_x_rows, wq, FP8LIN_E4M3, inv_w_rows, y, M, N, K, stream);
}

extern "C" fp8lin_status fp8lin_dgrad_rowwise(const uint8_t *dyq, const float *inv_dy_rows, const uint8_t *wqT,
                                              const float *inv_w_cols, void *dx, int64_t M, int64_t N, int64_t K,
                                              cudaStream_t stream) {
    return gemm_tn<true, false, false>(dyq, FP8LIN_E5M2, inv_dy_rows, wqT, FP8LIN_E4M3, inv_w_cols, dx, M, K, N, stream);
}

extern "C" fp8lin_status fp8lin_wgrad_rowwise(const uint8_t *dyqT, const float *inv_dy_cols, const uint8_t *xqT,
                                              const float *inv_x_cols, void *dw, int64_t M, int64_t N, int64_t K,
                                              cudaStream_t stream) {
    return gemm_tn<true, false, false>(dyqT, FP8LIN_E5M2, inv_dy_cols, xqT, FP8LIN_E4M3, inv_x_cols, dw, N, K, M, stream);
}

namespace {

// One bounded wait on an mbarrier that nothing arrives on: the same wait the
// GEMM kernels use, made to run out so that its timeout path can be checked.
__global__ void bounded_wait_probe_kernel(unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, limit_ns);
}

}  // namespace

extern "C" fp8lin_status fp8lin_selftest_bounded_wait(uint64_t limit_ns, cudaStream_t stream) {
    using namespace fp8lin;
    if (limit_ns < 1000ull || limit_ns > 1000000000ull) return FP8LIN_ERR_INVALID_ARG;
    DeviceInfo dev;
    fp8lin_status st = current_device(&dev);
    if (st != FP8LIN_OK) return st;
    bounded_wait_probe_kernel<<<1, 32, 0, stream>>>((unsigned long long)limit_ns);
    return check_launch();
}

extern "C" fp8lin_status fp8lin_device_error(cudaStream_t stream, uint32_t *word) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP8LIN_ERR_CUDA;
    unsigned int v = 0, zero = 0, vq = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return FP8LIN_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) return FP8LIN_ERR_CUDA;
    if (fp8lin::take_quantize_error(&vq) != FP8LIN_OK) return FP8LIN_ERR_CUDA;   // the one-launch cast's word
    v |= vq;
    if (word != nullptr) *word = v;
    return v == 0 ? FP8LIN_OK : FP8LIN_ERR_TIMEOUT;
}

#ifdef FP8LIN_FAULT_INJECTION
// Test builds only: choose the slab (the stage, for the power-of-two
// block-scaled GEMM) whose copies every GEMM's producers withhold (-1:
// none).  Synchronous; takes effect from the next launch on the current
// device.
extern "C" fp8lin_status fp8lin_test_withhold_slab(int slab) {
    if (slab < -1) return FP8LIN_ERR_INVALID_ARG;
    if (cudaMemcpyToSymbol(g_withhold_slab, &slab, sizeof slab) != cudaSuccess) return FP8LIN_ERR_CUDA;
    return cudaDeviceSynchronize() == cudaSuccess ? FP8LIN_OK : FP8LIN_ERR_CUDA;
}
#endif
