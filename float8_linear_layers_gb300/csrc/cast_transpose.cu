// cast_transpose.cu -- scale one bf16 matrix and cast it to FP8 (the Float8
// derived dtype; TorchTitan analysis page, section 3.3, "Mixed precision and
// Float8"), writing the row-major copy and, when asked for, the transposed
// copy in the same pass (the tensor cores read 8-bit operands either way, so
// per-tensor scaling needs only the row-major copy).  Per-tensor, delayed,
// static and row-wise scales here; block scales with fp32 scales
// (cast_block_kernel) and with power-of-two scales laid out for the tensor
// cores (cast_mx_kernel), below, in one pass with no amax call: persistent
// kernels fed by a per-thread cp.async ring (TileRing).
//
// HBM-bound: per element 2 bytes read, 1 (+ 1) bytes written.  In the
// per-tensor cast one CTA owns a 128 x 128 tile:
//  * phase 1: coalesced 16-byte loads (16 threads per 256-byte tile row, all
//    eight loads of a thread issued before any use), fp32 product with the
//    scale, cvt.rn.satfinite into packed FP8 pairs; the row-major copy is
//    stored straight from registers (8 bytes per thread, 128-byte rows);
//    with a transposed copy the bytes also go to a 16 KB shared tile whose
//    4-byte words are XOR swizzled by row group so that phase 2 reads are
//    bank-conflict free (without one, the kernel is instantiated with no
//    tile at all, so that two CTAs fit beside a GEMM CTA);
//  * phase 2: each thread gathers a 16-row x 4-column block as 16 words,
//    transposes 4 x 4 byte blocks with byte permutes and stores four 16-byte
//    chunks of the transposed copy; eight lanes cover one 128-byte row of
//    the transposed copy, so every warp store writes four full 128-byte rows.
// The scale is derived in every CTA from the device amax (IEEE division), so
// no separate launch and no host round trip is needed; CTA 0 publishes it.
// Tiles are visited from the last row block to the first, so that the part of
// the tensor the preceding amax pass read last is re-read from L2.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda_bf16.h>

#include "common.cuh"

namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;

// Word index of (row, word) in the swizzled shared tile: bits 2..4 of the
// word index are XORed with the row's 16-row group.
__device__ __forceinline__ int swz(int row, int word) { return word ^ (((row >> 4) & 7) << 2); }

template <int FMT>
__device__ __forceinline__ uint32_t cvt4(float a, float b, float c, float d) {
    // cvt packs its first source operand into the upper byte of each pair.
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

// Streaming 16-byte load that does not allocate in L1 (the data is used once;
// at the shared-memory-heavy carveout L1 is small).
__device__ __forceinline__ uint4 ld_stream16(const void *p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

// L2 policy for data touched once: first in line for eviction, so a GEMM
// running beside this kernel keeps its resident operand in L2.
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void st_stream8(void *p, uint2 v, uint64_t policy) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void st_stream16(void *p, uint4 v, uint64_t policy) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int FMT>
__device__ __forceinline__ uint2 cast8(uint4 v, float s) {
    uint2 r;
    r.x = cvt4<FMT>(__fmul_rn(bf16_lo(v.x), s), __fmul_rn(bf16_hi(v.x), s),
                    __fmul_rn(bf16_lo(v.y), s), __fmul_rn(bf16_hi(v.y), s));
    r.y = cvt4<FMT>(__fmul_rn(bf16_lo(v.z), s), __fmul_rn(bf16_hi(v.z), s),
                    __fmul_rn(bf16_lo(v.w), s), __fmul_rn(bf16_hi(v.w), s));
    return r;
}

// Eight elements with one scale per element (row-wise scaling's qT codes:
// the scale of each column).
template <int FMT>
__device__ __forceinline__ uint2 cast8_each(uint4 v, const float (&sc)[8]) {
    uint2 r;
    r.x = cvt4<FMT>(__fmul_rn(bf16_lo(v.x), sc[0]), __fmul_rn(bf16_hi(v.x), sc[1]),
                    __fmul_rn(bf16_lo(v.y), sc[2]), __fmul_rn(bf16_hi(v.y), sc[3]));
    r.y = cvt4<FMT>(__fmul_rn(bf16_lo(v.z), sc[4]), __fmul_rn(bf16_hi(v.z), sc[5]),
                    __fmul_rn(bf16_lo(v.w), sc[6]), __fmul_rn(bf16_hi(v.w), sc[7]));
    return r;
}

// Where the scale comes from.
enum ScaleMode : int {
    kDynamic = 0,  // scale = fmt_max / max(amax, 1e-12), amax of this tensor (computed beforehand)
    kStatic = 1,   // scale given by the caller
    kDelayed = 2,  // scale = fmt_max / max(max of the amax history except `slot`, 1e-12)
    kRowwise = 3,  // one scale per row of q (from row amax) and per row of qT (from column amax)
};

__device__ __forceinline__ float scale_from_amax(float a, float fmt_max) {
    a = (a < 1e-12f) ? 1e-12f : a;  // a NaN amax stays NaN
    return __fdiv_rn(fmt_max, a);
}

// Largest of n non-negative fp32 values (their bit patterns order the same
// way; a NaN ranks above everything), skipping index `skip`.  Warp-parallel.
__device__ __forceinline__ float history_max(const float *__restrict__ h, int n, int skip) {
    const int lane = threadIdx.x % 32;
    uint32_t m = 0;
    for (int i = lane; i < n; i += 32)
        if (i != skip) m = max(m, __float_as_uint(__ldg(h + i)) & 0x7FFFFFFFu);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    return __uint_as_float(m);
}

// Packed 16-bit magnitude maximum of eight bf16 values.
__device__ __forceinline__ uint32_t absmax8(uint32_t m, uint4 v) {
    const uint32_t k = 0x7FFF7FFFu;
    m = __vmaxu2(m, v.x & k);
    m = __vmaxu2(m, v.y & k);
    m = __vmaxu2(m, v.z & k);
    m = __vmaxu2(m, v.w & k);
    return m;
}

// TRANS = false: no transposed copy (qT is NULL), so no shared tile either:
// beside a GEMM CTA, whose shared memory leaves room for one 16 KB tile per
// SM, the registers then fit two CTAs of this kernel instead of one.
template <int FMT, int MODE, bool RECORD, bool TRANS>
__global__ void __launch_bounds__(kThreads)
cast_transpose_kernel(const uint16_t *__restrict__ x, int rows, int cols, int tiles_c, int num_tiles,
                      float fmt_max, const float *__restrict__ scale_src, int hist_len, int slot,
                      float *__restrict__ scale_out, float *__restrict__ inv_out, uint8_t *__restrict__ q,
                      uint8_t *__restrict__ qT, unsigned int *__restrict__ amax_record,
                      const float *__restrict__ col_src, float *__restrict__ col_inv_out) {
    __shared__ __align__(16) uint32_t tile[TRANS ? kTile : 1][kTile / 4];
    __shared__ uint32_t warp_max[kThreads / 32];
    __shared__ float srow[MODE == kRowwise ? kTile : 1], scol[MODE == kRowwise ? kTile : 1];

    float s = 0.0f;
    if (MODE == kRowwise) {
        // per-row / per-column scales are formed below, per element
    } else if (MODE == kStatic) {
        s = __ldg(scale_src);
    } else {
        // scale = fmt_max / max(amax, 1e-12): binary32, round to nearest even.
        float a = (MODE == kDynamic) ? __ldg(scale_src) : history_max(scale_src, hist_len, slot);
        a = (a < 1e-12f) ? 1e-12f : a;  // a NaN amax stays NaN
        s = __fdiv_rn(fmt_max, a);
    }
    if (MODE != kRowwise && blockIdx.x == 0 && threadIdx.x == 0) {
        if (scale_out != nullptr) *scale_out = s;
        *inv_out = __frcp_rn(s);
    }
    if ((int)blockIdx.x >= num_tiles) return;

    // Tiles run last-row-block first: the amax pass that precedes this kernel
    // read the tensor front to back, so its tail is what L2 still holds.
    const int tile_id = num_tiles - 1 - (int)blockIdx.x;
    const int tr = tile_id / tiles_c, tc = tile_id % tiles_c;
    const int r0 = tr * kTile, c0 = tc * kTile;
    const int t = threadIdx.x;

    // ---- phase 1: 128 rows x 16 chunks of 8 elements = 2048 chunks, 8 per thread
    const int ch = t % 16;          // chunk within the row (8 columns)
    const int row_base = t / 16;    // rows row_base + 16 i
    const bool col_in = (c0 + ch * 8) < cols;
    const uint64_t pol = evict_first_policy();
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = r0 + row_base + 16 * i;
        if (col_in && r < rows)
            v[i] = ld_stream16(x + (int64_t)r * cols + c0 + ch * 8, pol);
        else
            v[i] = make_uint4(0, 0, 0, 0);
    }
    if (RECORD) {
        // this tile's max |x| (zero padding never raises it), one conditional
        // atomicMax per CTA on the fp32 bit pattern (bf16 << 16)
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = absmax8(m, v[i]);
        uint32_t r = __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
        if (t % 32 == 0) warp_max[t / 32] = r;
        __syncthreads();
        if (t < 32) {
            r = __reduce_max_sync(0xFFFFFFFFu, t < kThreads / 32 ? warp_max[t] : 0u);
            if (t == 0 && r != 0) {
                const uint32_t bits = r << 16;
                if (bits > *reinterpret_cast<volatile unsigned int *>(amax_record)) atomicMax(amax_record, bits);
            }
        }
    }
    if (MODE == kRowwise) {
        // q: the scale of each row; qT: the scale of each column (a row of
        // x^T).  The tile's 128 + 128 scales are formed once, one per thread.
        if (t < kTile) {
            const int r = r0 + t;
            const bool ok = q != nullptr && r < rows;
            const float rs = ok ? scale_from_amax(__ldg(scale_src + r), fmt_max) : 0.0f;
            srow[t] = rs;
            if (ok && tc == 0) inv_out[r] = __frcp_rn(rs);
        } else {
            const int c = c0 + t - kTile;
            const bool ok = qT != nullptr && c < cols;
            const float cs = ok ? scale_from_amax(__ldg(col_src + c), fmt_max) : 0.0f;
            scol[t - kTile] = cs;
            if (ok && tr == 0) col_inv_out[c] = __frcp_rn(cs);
        }
        __syncthreads();
        float csc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) csc[j] = scol[ch * 8 + j];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int lr = row_base + 16 * i;
            const int r = r0 + lr;
            if (q != nullptr && col_in && r < rows)
                st_stream8(q + (int64_t)r * cols + c0 + ch * 8, cast8<FMT>(v[i], srow[lr]), pol);
            if (TRANS) *reinterpret_cast<uint2 *>(&tile[lr][swz(lr, 2 * ch)]) = cast8_each<FMT>(v[i], csc);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int lr = row_base + 16 * i;
            const int r = r0 + lr;
            const uint2 p = cast8<FMT>(v[i], s);
            if (q != nullptr && col_in && r < rows)
                st_stream8(q + (int64_t)r * cols + c0 + ch * 8, p, pol);
            if (TRANS) *reinterpret_cast<uint2 *>(&tile[lr][swz(lr, 2 * ch)]) = p;
        }
    }
    if constexpr (!TRANS) {
        return;
    } else {
        __syncthreads();

        // ---- phase 2: warp w owns columns 16w..16w+15; lane (rc, cq) owns rows
        // 16 rc .. 16 rc + 15 of columns 16 w + 4 cq .. + 3.
        const int w = t / 32, lane = t % 32;
        const int rc = lane % 8, cq = lane / 8;
        const int word = 4 * w + cq;
        uint32_t rw[16];
    #pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int lr = 16 * rc + i;
            rw[i] = tile[lr][swz(lr, word)];
        }
        // out[j][k]: column j, rows 4k .. 4k+3 (byte b = row 4k+b)
        uint32_t out[4][4];
    #pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t a0 = rw[4 * k], a1 = rw[4 * k + 1], a2 = rw[4 * k + 2], a3 = rw[4 * k + 3];
            const uint32_t t0 = __byte_perm(a0, a1, 0x5140);  // a0.b0 a1.b0 a0.b1 a1.b1
            const uint32_t t1 = __byte_perm(a2, a3, 0x5140);  // a2.b0 a3.b0 a2.b1 a3.b1
            const uint32_t t2 = __byte_perm(a0, a1, 0x7362);  // a0.b2 a1.b2 a0.b3 a1.b3
            const uint32_t t3 = __byte_perm(a2, a3, 0x7362);  // a2.b2 a3.b2 a2.b3 a3.b3
            out[0][k] = __byte_perm(t0, t1, 0x5410);
            out[1][k] = __byte_perm(t0, t1, 0x7632);
            out[2][k] = __byte_perm(t2, t3, 0x5410);
            out[3][k] = __byte_perm(t2, t3, 0x7632);
        }
        const int rr = r0 + 16 * rc;
        if (rr < rows) {
    #pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = c0 + 16 * w + 4 * cq + j;
                if (c < cols)
                    st_stream16(qT + (int64_t)c * rows + rr, make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]), pol);
            }
        }
    }
}

// One launch of the cast, with or without the transposed copy.
template <int FMT, int MODE, bool REC>
void launch_cast(int grid, cudaStream_t stream, const uint16_t *x, int rows, int cols, int tiles_c, int num_tiles,
                 float fmt_max, const float *src, int hist_len, int slot, float *scale, float *inv, uint8_t *q,
                 uint8_t *qT, unsigned int *rec, const float *col_src, float *col_inv) {
    if (qT != nullptr)
        cast_transpose_kernel<FMT, MODE, REC, true><<<grid, kThreads, 0, stream>>>(
            x, rows, cols, tiles_c, num_tiles, fmt_max, src, hist_len, slot, scale, inv, q, qT, rec, col_src,
            col_inv);
    else
        cast_transpose_kernel<FMT, MODE, REC, false><<<grid, kThreads, 0, stream>>>(
            x, rows, cols, tiles_c, num_tiles, fmt_max, src, hist_len, slot, scale, inv, q, qT, rec, col_src,
            col_inv);
}

template <int FMT>
void launch_mode(int mode, bool record, int grid, cudaStream_t stream, const uint16_t *x, int rows, int cols,
                 int tiles_c, int num_tiles, float fmt_max, const float *src, int hist_len, int slot,
                 float *scale, float *inv, uint8_t *q, uint8_t *qT, unsigned int *rec, const float *col_src,
                 float *col_inv) {
    auto launch = [&](auto fn) {
        fn(grid, stream, x, rows, cols, tiles_c, num_tiles, fmt_max, src, hist_len, slot, scale, inv, q, qT, rec,
           col_src, col_inv);
    };
    if (mode == kRowwise)
        launch(launch_cast<FMT, kRowwise, false>);
    else if (mode == kDynamic)
        launch(launch_cast<FMT, kDynamic, false>);
    else if (mode == kStatic && !record)
        launch(launch_cast<FMT, kStatic, false>);
    else if (mode == kStatic)
        launch(launch_cast<FMT, kStatic, true>);
    else
        launch(launch_cast<FMT, kDelayed, true>);
}

// The max-shared carveout for both forms (with and without the transposed
// copy) of one mode; carveout slots `slot` and `slot` + 48.
template <int FMT, int MODE, bool REC>
fp8lin_status carveout_pair(int device, int slot) {
    fp8lin_status st = fp8lin::prefer_max_shared_carveout(
        reinterpret_cast<const void *>(&cast_transpose_kernel<FMT, MODE, REC, true>), device, slot);
    if (st != FP8LIN_OK) return st;
    return fp8lin::prefer_max_shared_carveout(
        reinterpret_cast<const void *>(&cast_transpose_kernel<FMT, MODE, REC, false>), device, slot + 48);
}

template <int FMT>
fp8lin_status set_carveouts(int device) {
    const int base = FMT == FP8LIN_E4M3 ? 1 : 5;
    fp8lin_status st = carveout_pair<FMT, kDynamic, false>(device, base);
    if (st == FP8LIN_OK) st = carveout_pair<FMT, kStatic, false>(device, base + 1);
    if (st == FP8LIN_OK) st = carveout_pair<FMT, kStatic, true>(device, base + 2);
    if (st == FP8LIN_OK) st = carveout_pair<FMT, kDelayed, true>(device, base + 3);
    if (st == FP8LIN_OK) st = carveout_pair<FMT, kRowwise, false>(device, base + 20);
    return st;
}

// The load ring of the persistent block casts: every thread copies its own
// 8 x 16 bytes of a 128 x 128 tile into its own slots of a shared-memory
// ring (cp.async) and reads back only those, so the ring needs no barrier
// and no spin-wait (cp.async.wait_group covers it): a CTA keeps the next
// kRingStages - 1 tiles in flight while it reduces and casts the current
// one, and its registers hold one tile.
constexpr int kRingStages = 3;
constexpr int kRingStageBytes = 8 * kThreads * 16;             // one 128 x 128 bf16 tile
constexpr int kRingSmem = kRingStages * kRingStageBytes;   // dynamic shared memory
constexpr int kRingCtasPerSm = 2;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
                 : "memory");
    return v;
}


// This thread's view of the ring over x [rows x cols]: it owns the 16-byte
// chunk ch of rows row_base + 16 i (i < 8) of every tile, in slot i of a
// stage at ((8 stage + i) kThreads + t) 16 bytes.
struct TileRing {
    const uint16_t *x;
    int rows, cols, tiles_c, num_tiles;
    int ch, row_base;
    uint32_t slots;   // shared address of this thread's slot 0 of stage 0

    __device__ __forceinline__ TileRing(const uint16_t *x_, int rows_, int cols_, int tiles_r, int tiles_c_,
                                        uint8_t *ring)
        : x(x_), rows(rows_), cols(cols_), tiles_c(tiles_c_), num_tiles(tiles_r * tiles_c_),
          ch((int)threadIdx.x % 16), row_base((int)threadIdx.x / 16),
          slots((uint32_t)__cvta_generic_to_shared(ring) + 16u * threadIdx.x) {}

    __device__ __forceinline__ uint32_t slot(int s, int i) const {
        return slots + (uint32_t)((8 * s + i) * kThreads * 16);
    }
    // Copies of tile `tile` into stage s: one commit group even when the tile
    // does not exist, so that group n is always tile n of this CTA.
    __device__ __forceinline__ void issue(int tile, int s) const {
        if (tile < num_tiles) {
            const int r0 = (tile / tiles_c) * kTile, c0 = (tile % tiles_c) * kTile;
            if (c0 + ch * 8 < cols) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = r0 + row_base + 16 * i;
                    if (r < rows) cp_async16(slot(s, i), x + (int64_t)r * cols + c0 + ch * 8);
                }
            }
        }
        cp_async_commit();
    }
    // This thread's 8 x 8 elements of a tile from stage s (zero past the edge).
    __device__ __forceinline__ void read(int r0, int c0, int s, uint4 (&v)[8]) const {
        const bool col_in = c0 + ch * 8 < cols;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = r0 + row_base + 16 * i;
            v[i] = (col_in && r < rows) ? lds128(slot(s, i)) : make_uint4(0, 0, 0, 0);
        }
    }
};

// ------------------------------------------------------------ block scaling

// Block scaling: every block is scaled like a tensor of its own (amax of the
// block, scale = fmt_max / max(amax, 1e-12), saturating RNE cast).  Every
// 1 x 128, 128 x 1 and 128 x 128 block lies inside one 128 x 128 tile, so one
// pass over x makes any of
//   ROW : 1 x 128 blocks (a scale per row of the tile)     q_row, inv_row [tiles_c x rows]
//   COL : 128 x 1 blocks (a scale per column of the tile)  q_col, inv_col [tiles_r x cols]
//   TILE: the 128 x 128 block                              q_tile, inv_tile [tiles_r x tiles_c]
// (each copy row-major like x), with no separate amax pass: 2 bytes read and
// 1 byte written per element and copy.  Row maxima reduce over the 16 lanes
// that share a row (two rows per shuffle; one lane per row divides for its
// scale and the others read it); column maxima over the thread's 8 rows, the lane pair
// 16 apart, then the 8 warps through shared memory.  A persistent kernel
// whose loads come through the TileRing.
template <int FMT, bool ROW, bool COL, bool TILE>
__global__ void __launch_bounds__(kThreads, kRingCtasPerSm)
cast_block_kernel(const uint16_t *__restrict__ x, int rows, int cols, int tiles_r, int tiles_c, float fmt_max,
                  uint8_t *__restrict__ q_row, float *__restrict__ inv_row, uint8_t *__restrict__ q_col,
                  float *__restrict__ inv_col, uint8_t *__restrict__ q_tile, float *__restrict__ inv_tile) {
    extern __shared__ __align__(16) uint8_t ring_smem[];                 // [stages][8][kThreads][16 B]
    __shared__ uint32_t col_part[COL ? kThreads / 32 : 1][kTile / 2];   // per-warp column maxima, packed pairs
    __shared__ __align__(16) float col_scale[COL ? kTile : 1];
    __shared__ uint32_t warp_max[2][kThreads / 32];                      // by tile parity

    const int t = threadIdx.x, lane = t % 32, warp = t / 32;
    const int ch = t % 16;        // 8-column chunk of the tile row
    const int row_base = t / 16;  // rows row_base + 16 i
    const TileRing ring(x, rows, cols, tiles_r, tiles_c, ring_smem);
    const int num_tiles = ring.num_tiles;
    const int step = (int)gridDim.x;
    const uint64_t pol = evict_first_policy();
#pragma unroll
    for (int s = 0; s < kRingStages - 1; ++s) ring.issue((int)blockIdx.x + s * step, s);

    int stage = 0, parity = 0;
    for (int tile = (int)blockIdx.x; tile < num_tiles; tile += step) {
        ring.issue(tile + (kRingStages - 1) * step, stage == 0 ? kRingStages - 1 : stage - 1);
        cp_async_wait<kRingStages - 1>();
        const int tr = tile / tiles_c, tc = tile % tiles_c;
        const int r0 = tr * kTile, c0 = tc * kTile;
        const bool col_in = (c0 + ch * 8) < cols;
        uint4 v[8];
        ring.read(r0, c0, stage, v);
        stage = stage + 1 == kRingStages ? 0 : stage + 1;

        // magnitudes as bf16 bit patterns without the sign: their unsigned order
        // is the order of |x| (a NaN above everything); zero padding never wins
        const uint32_t k = 0x7FFF7FFFu;
        uint32_t rowm[8];
        uint32_t colm2[4] = {0, 0, 0, 0};  // packed pairs: columns 2j, 2j + 1 of this thread's chunk
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t a = v[i].x & k, b = v[i].y & k, c = v[i].z & k, d = v[i].w & k;
            const uint32_t m = __vmaxu2(__vmaxu2(a, b), __vmaxu2(c, d));
            rowm[i] = max(m & 0xFFFFu, m >> 16);
            colm2[0] = __vmaxu2(colm2[0], a);
            colm2[1] = __vmaxu2(colm2[1], b);
            colm2[2] = __vmaxu2(colm2[2], c);
            colm2[3] = __vmaxu2(colm2[3], d);
        }
        float srow[8];  // the rows' scales (ROW)
        if (ROW) {
            // the row maxima over the 16 lanes sharing the rows, two rows per word
            uint32_t pm[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pm[j] = rowm[2 * j] | (rowm[2 * j + 1] << 16);
#pragma unroll
                for (int o = 8; o >= 1; o >>= 1) pm[j] = __vmaxu2(pm[j], __shfl_xor_sync(0xFFFFFFFFu, pm[j], o));
                rowm[2 * j] = pm[j] & 0xFFFFu;
                rowm[2 * j + 1] = pm[j] >> 16;
            }
            // lane ch % 8 of the 16 divides for row ch % 8; the others read it
            const int c = ch & 7;
            const uint32_t pc = (c >> 1) == 0 ? pm[0] : ((c >> 1) == 1 ? pm[1] : ((c >> 1) == 2 ? pm[2] : pm[3]));
            const float sc = scale_from_amax(__uint_as_float(((pc >> (16 * (c & 1))) & 0xFFFFu) << 16), fmt_max);
#pragma unroll
            for (int r = 0; r < 8; ++r) srow[r] = __shfl_sync(0xFFFFFFFFu, sc, (lane & 16) | r);
        }
        if (COL) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t m = __vmaxu2(colm2[j], __shfl_xor_sync(0xFFFFFFFFu, colm2[j], 16));
                if (lane < 16) col_part[warp][ch * 4 + j] = m;
            }
        }
        if (TILE) {
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = max(m, rowm[i]);
            m = __reduce_max_sync(0xFFFFFFFFu, m);
            if (lane == 0) warp_max[parity][warp] = m;
        }
        if (COL || TILE) __syncthreads();
        if (COL) {
            if (t < kTile) {
                uint32_t m = 0;
#pragma unroll
                for (int w = 0; w < kThreads / 32; ++w) m = max(m, (col_part[w][t / 2] >> (16 * (t % 2))) & 0xFFFFu);
                const float s = scale_from_amax(__uint_as_float(m << 16), fmt_max);
                col_scale[t] = s;
                if (c0 + t < cols) inv_col[(int64_t)tr * cols + c0 + t] = __frcp_rn(s);
            }
            __syncthreads();
        }
        float s_tile = 0.0f;
        if (TILE) {
            uint32_t m = 0;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) m = max(m, warp_max[parity][w]);
            s_tile = scale_from_amax(__uint_as_float(m << 16), fmt_max);
            if (t == 0) inv_tile[(int64_t)tr * tiles_c + tc] = __frcp_rn(s_tile);
        }
        parity ^= 1;
        float csc[8];
        if (COL) {
            const float4 lo = *reinterpret_cast<const float4 *>(&col_scale[ch * 8]);
            const float4 hi = *reinterpret_cast<const float4 *>(&col_scale[ch * 8 + 4]);
            csc[0] = lo.x, csc[1] = lo.y, csc[2] = lo.z, csc[3] = lo.w;
            csc[4] = hi.x, csc[5] = hi.y, csc[6] = hi.z, csc[7] = hi.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = r0 + row_base + 16 * i;
            const bool ok = col_in && r < rows;
            const int64_t off = (int64_t)r * cols + c0 + ch * 8;
            if (ROW) {
                if (ok) st_stream8(q_row + off, cast8<FMT>(v[i], srow[i]), pol);
                if (ch == 0 && r < rows) inv_row[(int64_t)tc * rows + r] = __frcp_rn(srow[i]);
            }
            if (COL && ok) st_stream8(q_col + off, cast8_each<FMT>(v[i], csc), pol);
            if (TILE && ok) st_stream8(q_tile + off, cast8<FMT>(v[i], s_tile), pol);
        }
    }
    cp_async_wait<0>();   // no copy outlives the CTA (the tail's groups are empty)
}

// Persistent grid: min(tiles, CTAs per SM x SMs), the attributes set once
// per kernel and device.
template <typename Kernel>
fp8lin_status ring_grid(Kernel kernel, std::atomic<int> (&ctas_per_sm)[64], int device, int sm_count, int num_tiles,
                        int *grid) {
    if (device < 0 || device >= 64) return FP8LIN_ERR_CUDA;
    int per_sm = ctas_per_sm[device].load(std::memory_order_acquire);
    if (per_sm == 0) {
        const void *k = reinterpret_cast<const void *>(kernel);
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmem) != cudaSuccess ||
            cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, kRingSmem) != cudaSuccess ||
            per_sm < 1)
            return FP8LIN_ERR_CUDA;
        ctas_per_sm[device].store(per_sm, std::memory_order_release);
    }
    const int64_t slots = (int64_t)per_sm * sm_count;
    *grid = (int)(num_tiles < slots ? num_tiles : slots);
    return FP8LIN_OK;
}

template <int FMT, bool ROW, bool COL, bool TILE>
fp8lin_status launch_block(int device, int sm_count, int num_tiles, cudaStream_t stream, const uint16_t *x, int rows,
                           int cols, int tiles_r, int tiles_c, float fmt_max, uint8_t *q_row, float *inv_row,
                           uint8_t *q_col, float *inv_col, uint8_t *q_tile, float *inv_tile) {
    static std::atomic<int> ctas_per_sm[64];
    int grid = 0;
    const fp8lin_status st =
        ring_grid(&cast_block_kernel<FMT, ROW, COL, TILE>, ctas_per_sm, device, sm_count, num_tiles, &grid);
    if (st != FP8LIN_OK) return st;
    cast_block_kernel<FMT, ROW, COL, TILE><<<grid, kThreads, kRingSmem, stream>>>(
        x, rows, cols, tiles_r, tiles_c, fmt_max, q_row, inv_row, q_col, inv_col, q_tile, inv_tile);
    return FP8LIN_OK;
}

template <int FMT>
fp8lin_status launch_block_any(int device, int sm_count, int which, int num_tiles, cudaStream_t stream,
                               const uint16_t *x, int rows, int cols, int tiles_r, int tiles_c, float fmt_max,
                               uint8_t *qr, float *ir, uint8_t *qc, float *ic, uint8_t *qt, float *it) {
#define FP8LIN_BLOCK_LAUNCH(R, C, T) \
    launch_block<FMT, R, C, T>(device, sm_count, num_tiles, stream, x, rows, cols, tiles_r, tiles_c, fmt_max, qr, ir, qc, ic, qt, it)
    switch (which) {
        case 1: return FP8LIN_BLOCK_LAUNCH(true, false, false);
        case 2: return FP8LIN_BLOCK_LAUNCH(false, true, false);
        case 3: return FP8LIN_BLOCK_LAUNCH(true, true, false);
        case 4: return FP8LIN_BLOCK_LAUNCH(false, false, true);
        case 5: return FP8LIN_BLOCK_LAUNCH(true, false, true);
        case 6: return FP8LIN_BLOCK_LAUNCH(false, true, true);
        default: return FP8LIN_BLOCK_LAUNCH(true, true, true);
    }
#undef FP8LIN_BLOCK_LAUNCH
}

// ------------------------------------------- power-of-two block scaling

// Block scaling with power-of-two scales, in the granularity the tensor
// cores' block-scaled MMA applies them (one scale per 32 contraction
// elements): every block's scale is 2^e, e the largest integer with
// max(amax, 1e-12) * 2^e <= fmt_max (clamped to [-127, 127]); the codes are
// sat_RNE(fp32(x) * 2^e) (an exact product).  The GEMM reads the inverse
// scale 2^-e as the unsigned-exponent byte 127 - e; a block with a NaN or
// infinite amax gets 0xFF (NaN).  Exponent from the bit patterns: with
// a = ma 2^ea and fmt_max = mf 2^ef (ma, mf in [1, 2)), a 2^e <= fmt_max
// exactly when e <= ef - ea - (ma > mf).
__device__ __forceinline__ uint32_t pow2_scale_byte(uint32_t amax_bits, uint32_t fmax_bits) {
    if (amax_bits >= 0x7F800000u) return 0xFFu;
    const uint32_t a = amax_bits < 0x2B8CBCCCu ? 0x2B8CBCCCu : amax_bits;  // floor at 1e-12f
    int e = (int)(fmax_bits >> 23) - (int)(a >> 23) - ((a & 0x7FFFFFu) > (fmax_bits & 0x7FFFFFu) ? 1 : 0);
    e = e > 127 ? 127 : (e < -127 ? -127 : e);
    return (uint32_t)(127 - e);
}

// The OCP Microscaling rule: the byte of the shared scale
// X = 2^(floor(log2 amax) - emax) (emax 8 for e4m3, 15 for e5m2), by which the
// elements are divided; floor(log2 amax) is the exponent field minus 127 for
// a normal amax, so the byte is the exponent field minus emax (0 for a zero
// or subnormal amax), clamped to 0 .. 254; 0xFF for a NaN or infinite amax.
__device__ __forceinline__ uint32_t ocp_scale_byte(uint32_t amax_bits, int emax) {
    if (amax_bits >= 0x7F800000u) return 0xFFu;
    const int b = (int)(amax_bits >> 23) - emax;
    return (uint32_t)(b < 0 ? 0 : (b > 254 ? 254 : b));
}

// The block's scale byte under either rule (ocp_emax 0: the largest power of
// two not above fmt_max / amax).
__device__ __forceinline__ uint32_t mx_scale_byte(uint32_t amax_bits, uint32_t fmax_bits, int ocp_emax) {
    return ocp_emax ? ocp_scale_byte(amax_bits, ocp_emax) : pow2_scale_byte(amax_bits, fmax_bits);
}

// The bf16 bit pattern of 2^e from the byte 127 - e: exponent field 127 + e,
// no mantissa; 2^-127 is the subnormal 0x0040; NaN for the byte 0xFF.
__device__ __forceinline__ uint32_t pow2_bf16_from_byte(uint32_t b) {
    if (b == 0xFFu) return 0x7FC0u;
    return b == 254u ? 0x0040u : (254u - b) << 7;
}

// Four bf16 elements (x01, x23) times their power-of-two scales (bf16 pairs
// s01, s23, same order) to FP8: each product by one mixed-precision FMA
// (fp32 result = x * s + (-0), rounded once: exact, and equal to
// __fmul_rn(fp32(x), fp32(s)) bit for bit, the sign of a zero included),
// then cvt.rn.satfinite as in cvt4.
template <int FMT>
__device__ __forceinline__ uint32_t cast4_pow2(uint32_t x01, uint32_t x23, uint32_t s01, uint32_t s23) {
    uint32_t r;
#define FP8LIN_CAST4_POW2(CVT)                                                                        \
    asm("{\n\t.reg .b16 a0, a1, a2, a3, b0, b1, b2, b3, lo, hi;\n\t.reg .f32 p0, p1, p2, p3;\n\t"     \
        "mov.b32 {a0, a1}, %1;\n\t"                                                                   \
        "mov.b32 {a2, a3}, %2;\n\t"                                                                   \
        "mov.b32 {b0, b1}, %3;\n\t"                                                                   \
        "mov.b32 {b2, b3}, %4;\n\t"                                                                   \
        "fma.rn.f32.bf16 p0, a0, b0, 0f80000000;\n\t"                                                 \
        "fma.rn.f32.bf16 p1, a1, b1, 0f80000000;\n\t"                                                 \
        "fma.rn.f32.bf16 p2, a2, b2, 0f80000000;\n\t"                                                 \
        "fma.rn.f32.bf16 p3, a3, b3, 0f80000000;\n\t"                                                 \
        CVT " lo, p1, p0;\n\t"                                                                        \
        CVT " hi, p3, p2;\n\t"                                                                        \
        "mov.b32 %0, {lo, hi};\n\t}"                                                                  \
        : "=r"(r)                                                                                     \
        : "r"(x01), "r"(x23), "r"(s01), "r"(s23))
    if (FMT == FP8LIN_E4M3)
        FP8LIN_CAST4_POW2("cvt.rn.satfinite.e4m3x2.f32");
    else
        FP8LIN_CAST4_POW2("cvt.rn.satfinite.e5m2x2.f32");
#undef FP8LIN_CAST4_POW2
    return r;
}

// Eight elements, the scales of each pair packed as in v.
template <int FMT>
__device__ __forceinline__ uint2 cast8_pow2(uint4 v, uint4 s) {
    return make_uint2(cast4_pow2<FMT>(v.x, v.y, s.x, s.y), cast4_pow2<FMT>(v.z, v.w, s.z, s.w));
}

// A persistent kernel over 128 x 128 tiles of x, any of two copies (each
// row-major like x):
//   ROW: 1 x 32 blocks (runs of 32 columns), read by a GEMM whose contraction
//        runs along the columns, scales in atom (tc, tr);
//   COL: 32 x 1 blocks (runs of 32 rows), read with the contraction along
//        the rows, scales in atom (tr, tc).
// A scale atom holds the bytes of 128 operand rows x 4 contraction blocks
// (128 contraction elements) in the order the tensor cores' scale-factor
// copy takes them: operand row p and block j at 16 (p % 32) + 4 (p / 32) + j;
// atom (kb, pb) is 512 bytes at (kb * operand row blocks + pb) * 512.  A tile
// is exactly one atom of each copy, so each CTA writes whole atoms, with 127
// (scale 1) for rows or blocks past the matrix's edge.
// Row blocks: the thread's 8-column maximum, then the 4 lanes of a 32-column
// run (shuffles of two rows per word; each lane works out two rows' scale
// bytes and shares them).  Column blocks: the thread's rows i = 2b, 2b + 1 of run b,
// the lane 16 apart, then the 8 warps through shared memory.
// Loads come through the TileRing (the next two tiles in flight).  One tile
// per CTA with the loads held in registers had DRAM 52% busy and the SM
// issuing on 55% of its cycles.
template <int FMT, bool ROW, bool COL>
__global__ void __launch_bounds__(kThreads, kRingCtasPerSm)
cast_mx_kernel(const uint16_t *__restrict__ x, int rows, int cols, int tiles_r, int tiles_c, uint32_t fmax_bits,
               int ocp_emax, uint8_t *__restrict__ q_row, uint8_t *__restrict__ sf_row, uint8_t *__restrict__ q_col,
               uint8_t *__restrict__ sf_col) {
    extern __shared__ __align__(16) uint8_t ring_smem[];                  // [stages][8][kThreads][16 B]
    __shared__ __align__(16) uint32_t col_part[COL ? kThreads / 32 : 1][4][kTile / 2];  // packed column pairs
    __shared__ __align__(16) uint16_t col_scale[COL ? 4 : 1][kTile];   // bf16 2^e
    __shared__ __align__(16) uint32_t atom_row[ROW ? 128 : 4];
    __shared__ __align__(16) uint32_t atom_col[COL ? 128 : 4];

    const int t = threadIdx.x, lane = t % 32, warp = t / 32;
    const int ch = t % 16;        // 8-column chunk of the tile row
    const int row_base = t / 16;  // rows row_base + 16 i
    const TileRing ring(x, rows, cols, tiles_r, tiles_c, ring_smem);
    const int num_tiles = ring.num_tiles;
    const int step = (int)gridDim.x;
    const uint64_t pol = evict_first_policy();

    if (t < 128) {
        if (ROW) atom_row[t] = 0x7F7F7F7Fu;
        if (COL) atom_col[t] = 0x7F7F7F7Fu;
    }
#pragma unroll
    for (int s = 0; s < kRingStages - 1; ++s) ring.issue((int)blockIdx.x + s * step, s);

    int stage = 0;
    for (int tile = (int)blockIdx.x; tile < num_tiles; tile += step) {
        // the stage read in the previous tile takes the tile kRingStages - 1 ahead
        ring.issue(tile + (kRingStages - 1) * step, stage == 0 ? kRingStages - 1 : stage - 1);
        cp_async_wait<kRingStages - 1>();   // this tile's group has landed
        const int tr = tile / tiles_c, tc = tile % tiles_c;
        const int r0 = tr * kTile, c0 = tc * kTile;
        const bool col_in = (c0 + ch * 8) < cols;
        uint4 v[8];
        ring.read(r0, c0, stage, v);
        stage = stage + 1 == kRingStages ? 0 : stage + 1;
        // magnitudes as bf16 bit patterns without the sign (unsigned order = order of |x|)
        const uint32_t k = 0x7FFF7FFFu;
        uint32_t rowm[8];
        uint32_t colm[4][4];  // [run b][packed column pair j]
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int j = 0; j < 4; ++j) colm[b][j] = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t a = v[i].x & k, b = v[i].y & k, c = v[i].z & k, d = v[i].w & k;
            const uint32_t m = __vmaxu2(__vmaxu2(a, b), __vmaxu2(c, d));
            rowm[i] = max(m & 0xFFFFu, m >> 16);
            colm[i / 2][0] = __vmaxu2(colm[i / 2][0], a);
            colm[i / 2][1] = __vmaxu2(colm[i / 2][1], b);
            colm[i / 2][2] = __vmaxu2(colm[i / 2][2], c);
            colm[i / 2][3] = __vmaxu2(colm[i / 2][3], d);
        }
        uint32_t rbyte[8];
        if (ROW) {
            // the run's maxima over its 4 lanes, two rows per word (rows 2j,
            // 2j + 1 in the low and high halves)
            uint32_t pm[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pm[j] = rowm[2 * j] | (rowm[2 * j + 1] << 16);
                pm[j] = __vmaxu2(pm[j], __shfl_xor_sync(0xFFFFFFFFu, pm[j], 1));
                pm[j] = __vmaxu2(pm[j], __shfl_xor_sync(0xFFFFFFFFu, pm[j], 2));
            }
            // lane q of the run works out the scale bytes of rows 2q and 2q + 1;
            // two exchanges hand every lane all eight (row i: byte i % 4 of the
            // word of rows 0..3 or 4..7)
            const int q = lane & 3;
            const uint32_t mine = q == 0 ? pm[0] : (q == 1 ? pm[1] : (q == 2 ? pm[2] : pm[3]));
            const uint32_t two = mx_scale_byte(mine << 16, fmax_bits, ocp_emax) |
                                 (mx_scale_byte(mine & 0xFFFF0000u, fmax_bits, ocp_emax) << 8);
            uint32_t w = two << (16 * (q & 1));                 // rows 2q, 2q + 1 at bytes 2 (q % 2), + 1
            w |= __shfl_xor_sync(0xFFFFFFFFu, w, 1);            // rows 4 (q / 2) .. + 3
            const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, w, 2);
            const uint32_t lo = q < 2 ? w : other, hi = q < 2 ? other : w;
#pragma unroll
            for (int i = 0; i < 8; ++i) rbyte[i] = ((i < 4 ? lo : hi) >> (8 * (i % 4))) & 0xFFu;
        }
        if (COL) {
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t m = __vmaxu2(colm[b][j], __shfl_xor_sync(0xFFFFFFFFu, colm[b][j], 16));
                    if (lane < 16) col_part[warp][b][ch * 4 + j] = m;   // columns ch 8 + 2 j, + 1
                }
        }
        __syncthreads();
        if (COL) {
            // thread t: column t % 128, runs t / 128 and t / 128 + 2
            const int c = t % kTile;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int b = t / kTile + 2 * h;
                uint32_t m = 0;
#pragma unroll
                for (int w = 0; w < kThreads / 32; ++w) m = max(m, (col_part[w][b][c / 2] >> (16 * (c % 2))) & 0xFFFFu);
                const uint32_t byte = mx_scale_byte(m << 16, fmax_bits, ocp_emax);
                col_scale[b][c] = (uint16_t)pow2_bf16_from_byte(byte);
                if (c0 + c < cols && r0 + 32 * b < rows)
                    reinterpret_cast<uint8_t *>(atom_col)[16 * (c % 32) + 4 * (c / 32) + b] = (uint8_t)byte;
            }
        }
        if (ROW && (ch & 3) == 0 && col_in) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int rr = row_base + 16 * i;
                if (r0 + rr < rows)
                    reinterpret_cast<uint8_t *>(atom_row)[16 * (rr % 32) + 4 * (rr / 32) + ch / 4] = (uint8_t)rbyte[i];
            }
        }
        __syncthreads();
        // the atoms go out and are reset for the next tile (whose writers
        // start after the next tile's first barrier)
        if (ROW && t < 32) {
            uint4 *a = reinterpret_cast<uint4 *>(atom_row) + t;
            reinterpret_cast<uint4 *>(sf_row + ((int64_t)tc * tiles_r + tr) * 512)[t] = *a;
            *a = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        }
        if (COL && t >= 32 && t < 64) {
            uint4 *a = reinterpret_cast<uint4 *>(atom_col) + (t - 32);
            reinterpret_cast<uint4 *>(sf_col + ((int64_t)tr * tiles_c + tc) * 512)[t - 32] = *a;
            *a = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = r0 + row_base + 16 * i;
            const bool ok = col_in && r < rows;
            const int64_t off = (int64_t)r * cols + c0 + ch * 8;
            if (ROW && ok) {
                const uint32_t s2 = pow2_bf16_from_byte(rbyte[i]) * 0x10001u;
                st_stream8(q_row + off, cast8_pow2<FMT>(v[i], make_uint4(s2, s2, s2, s2)), pol);
            }
            if (COL && ok)
                st_stream8(q_col + off, cast8_pow2<FMT>(v[i], *reinterpret_cast<const uint4 *>(&col_scale[i / 2][ch * 8])),
                           pol);
        }
    }
    cp_async_wait<0>();   // no copy outlives the CTA (the tail's groups are empty)
}

template <int FMT, bool ROW, bool COL>
fp8lin_status launch_mx(int device, int sm_count, int num_tiles, cudaStream_t stream, const uint16_t *x, int rows,
                        int cols, int tiles_r, int tiles_c, uint32_t fmax_bits, int ocp_emax, uint8_t *q_row,
                        uint8_t *sf_row, uint8_t *q_col, uint8_t *sf_col) {
    static std::atomic<int> ctas_per_sm[64];
    int grid = 0;
    const fp8lin_status st = ring_grid(&cast_mx_kernel<FMT, ROW, COL>, ctas_per_sm, device, sm_count, num_tiles, &grid);
    if (st != FP8LIN_OK) return st;
    cast_mx_kernel<FMT, ROW, COL><<<grid, kThreads, kRingSmem, stream>>>(x, rows, cols, tiles_r, tiles_c, fmax_bits,
                                                                        ocp_emax, q_row, sf_row, q_col, sf_col);
    return FP8LIN_OK;
}

template <int FMT>
fp8lin_status launch_mx_any(int device, int sm_count, int num_tiles, cudaStream_t stream, const uint16_t *x, int rows, int cols,
                            int tiles_r, int tiles_c, uint32_t fmax_bits, int ocp_emax, uint8_t *qr, uint8_t *sr,
                            uint8_t *qc, uint8_t *sc) {
    if (qr != nullptr && qc != nullptr)
        return launch_mx<FMT, true, true>(device, sm_count, num_tiles, stream, x, rows, cols, tiles_r, tiles_c, fmax_bits, ocp_emax, qr, sr,
                                          qc, sc);
    if (qr != nullptr)
        return launch_mx<FMT, true, false>(device, sm_count, num_tiles, stream, x, rows, cols, tiles_r, tiles_c, fmax_bits, ocp_emax, qr, sr,
                                           qc, sc);
    return launch_mx<FMT, false, true>(device, sm_count, num_tiles, stream, x, rows, cols, tiles_r, tiles_c, fmax_bits, ocp_emax, qr, sr, qc,
                                       sc);
}

// Checks shared by the three scalings, then the launch.
fp8lin_status cast_common(int mode, const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt, float fmt_max,
                          const float *src, int hist_len, int slot, float *scale, float *inv_scale, uint8_t *q,
                          uint8_t *qT, float *amax_record, cudaStream_t stream, const float *col_src = nullptr,
                          float *col_inv = nullptr) {
    using namespace fp8lin;
    if (mode == kRowwise) {
        // q needs the row statistics and receives row inverse scales; qT the column ones
        if (q != nullptr && (src == nullptr || inv_scale == nullptr)) return FP8LIN_ERR_INVALID_ARG;
        if (qT != nullptr && (col_src == nullptr || col_inv == nullptr)) return FP8LIN_ERR_INVALID_ARG;
        if (!aligned(col_src, 4) || !aligned(col_inv, 4)) return FP8LIN_ERR_MISALIGNED;
    } else {
        if (src == nullptr || inv_scale == nullptr) return FP8LIN_ERR_INVALID_ARG;
        if (mode != kStatic && scale == nullptr) return FP8LIN_ERR_INVALID_ARG;
    }
    if (rows < 0 || cols < 0) return FP8LIN_ERR_INVALID_ARG;
    if (fmt != FP8LIN_E4M3 && fmt != FP8LIN_E5M2) return FP8LIN_ERR_INVALID_ARG;
    if (mode != kStatic && (!(fmt_max > 0.0f) || !(fmt_max <= 3.4e38f))) return FP8LIN_ERR_INVALID_ARG;
    if (mode == kRowwise && rows * cols == 0) return FP8LIN_OK;  // no rows or columns: nothing to scale
    const bool empty = rows == 0 || cols == 0;
    if (!empty && x == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (!aligned(src, 4) || !aligned(scale, 4) || !aligned(inv_scale, 4) || !aligned(amax_record, 4))
        return FP8LIN_ERR_MISALIGNED;
    if (!empty && (!aligned(x, 16) || !aligned(q, 16) || !aligned(qT, 16))) return FP8LIN_ERR_MISALIGNED;
    if (!dim_ok(rows) || !dim_ok(cols) || rows % 16 || cols % 16) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo dev;
    fp8lin_status st = current_device(&dev);
    if (st != FP8LIN_OK) return st;

    const int64_t tiles_r = (rows + kTile - 1) / kTile, tiles_c = (cols + kTile - 1) / kTile;
    const int64_t num_tiles = empty ? 0 : tiles_r * tiles_c;
    if (num_tiles > INT32_MAX) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    const int grid = num_tiles > 0 ? (int)num_tiles : 1;  // one CTA publishes the scale
    const int tc = tiles_c > 0 ? (int)tiles_c : 1;
    st = fmt == FP8LIN_E4M3 ? set_carveouts<FP8LIN_E4M3>(dev.device) : set_carveouts<FP8LIN_E5M2>(dev.device);
    if (st != FP8LIN_OK) return st;
    const bool record = amax_record != nullptr;
    if (record && cudaMemsetAsync(amax_record, 0, sizeof(float), stream) != cudaSuccess) return FP8LIN_ERR_CUDA;
    const uint16_t *xs = static_cast<const uint16_t *>(x);
    unsigned int *rec = reinterpret_cast<unsigned int *>(amax_record);
    if (fmt == FP8LIN_E4M3)
        launch_mode<FP8LIN_E4M3>(mode, record, grid, stream, xs, (int)rows, (int)cols, tc, (int)num_tiles, fmt_max,
                                 src, hist_len, slot, scale, inv_scale, q, qT, rec, col_src, col_inv);
    else
        launch_mode<FP8LIN_E5M2>(mode, record, grid, stream, xs, (int)rows, (int)cols, tc, (int)num_tiles, fmt_max,
                                 src, hist_len, slot, scale, inv_scale, q, qT, rec, col_src, col_inv);
    return check_launch();
}

}  // namespace

extern "C" fp8lin_status fp8lin_cast_transpose(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt,
                                               float fmt_max, const float *amax, float *scale,
                                               float *inv_scale, uint8_t *q, uint8_t *qT,
                                               cudaStream_t stream) {
    return cast_common(kDynamic, x, rows, cols, fmt, fmt_max, amax, 0, 0, scale, inv_scale, q, qT, nullptr,
                       stream);
}

extern "C" fp8lin_status fp8lin_quantize(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt, float fmt_max,
                                         float *amax, float *scale, float *inv_scale, uint8_t *q, uint8_t *qT,
                                         cudaStream_t stream) {
    using namespace fp8lin;
    if (amax == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (!aligned(amax, 4)) return FP8LIN_ERR_MISALIGNED;
    // the cast's checks first, so that nothing is launched for a bad argument
    if (rows < 0 || cols < 0 || scale == nullptr || inv_scale == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (fmt != FP8LIN_E4M3 && fmt != FP8LIN_E5M2) return FP8LIN_ERR_INVALID_ARG;
    if (!(fmt_max > 0.0f) || !(fmt_max <= 3.4e38f)) return FP8LIN_ERR_INVALID_ARG;
    const bool empty = rows == 0 || cols == 0;
    if (!empty && x == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (!aligned(scale, 4) || !aligned(inv_scale, 4)) return FP8LIN_ERR_MISALIGNED;
    if (!empty && (!aligned(x, 16) || !aligned(q, 16) || !aligned(qT, 16))) return FP8LIN_ERR_MISALIGNED;
    if (!dim_ok(rows) || !dim_ok(cols) || rows % 16 || cols % 16) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    if (q != nullptr && qT == nullptr && !empty) {
        bool launched = false;
        const QuantizeItem item{x, rows * cols, amax, scale, inv_scale, q};
        fp8lin_status st = launch_quantize_batch(&item, 1, fmt, fmt_max, stream, &launched);
        if (st != FP8LIN_OK || launched) return st;
    }
    fp8lin_status st = launch_amax(x, rows * cols, amax, stream, true);
    if (st != FP8LIN_OK) return st;
    return cast_common(kDynamic, x, rows, cols, fmt, fmt_max, amax, 0, 0, scale, inv_scale, q, qT, nullptr,
                       stream);
}

extern "C" fp8lin_status fp8lin_quantize_batch(const fp8lin_quantize_item *items, int count, fp8lin_fmt fmt,
                                               float fmt_max, cudaStream_t stream) {
    using namespace fp8lin;
    if (items == nullptr || count < 1 || count > FP8LIN_MAX_QUANTIZE_BATCH) return FP8LIN_ERR_INVALID_ARG;
    if (fmt != FP8LIN_E4M3 && fmt != FP8LIN_E5M2) return FP8LIN_ERR_INVALID_ARG;
    if (!(fmt_max > 0.0f) || !(fmt_max <= 3.4e38f)) return FP8LIN_ERR_INVALID_ARG;
    // every item's checks first, so that nothing is launched for a bad argument
    QuantizeItem qi[FP8LIN_MAX_QUANTIZE_BATCH];
    for (int k = 0; k < count; ++k) {
        const fp8lin_quantize_item &it = items[k];
        if (it.amax == nullptr || it.scale == nullptr || it.inv_scale == nullptr) return FP8LIN_ERR_INVALID_ARG;
        if (it.rows < 0 || it.cols < 0) return FP8LIN_ERR_INVALID_ARG;
        const bool empty = it.rows == 0 || it.cols == 0;
        if (!empty && (it.x == nullptr || it.q == nullptr)) return FP8LIN_ERR_INVALID_ARG;
        if (!aligned(it.amax, 4) || !aligned(it.scale, 4) || !aligned(it.inv_scale, 4)) return FP8LIN_ERR_MISALIGNED;
        if (!empty && (!aligned(it.x, 16) || !aligned(it.q, 16))) return FP8LIN_ERR_MISALIGNED;
        if (!dim_ok(it.rows) || !dim_ok(it.cols) || it.rows % 16 || it.cols % 16) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
        // each tensor needs slots of its own: the launch counts and waits on the first tensor's
        const float *mine[3] = {it.amax, it.scale, it.inv_scale};
        for (int a = 0; a < 3; ++a)
            for (int c = a + 1; c < 3; ++c)
                if (mine[a] == mine[c]) return FP8LIN_ERR_INVALID_ARG;
        for (int j = 0; j < k; ++j) {
            const float *theirs[3] = {items[j].amax, items[j].scale, items[j].inv_scale};
            for (int a = 0; a < 3; ++a)
                for (int c = 0; c < 3; ++c)
                    if (mine[a] == theirs[c]) return FP8LIN_ERR_INVALID_ARG;
        }
        qi[k] = QuantizeItem{it.x, it.rows * it.cols, it.amax, it.scale, it.inv_scale, it.q};
    }
    bool launched = false;
    fp8lin_status st = launch_quantize_batch(qi, count, fmt, fmt_max, stream, &launched);
    if (st != FP8LIN_OK || launched) return st;
    for (int k = 0; k < count; ++k) {   // one tensor at a time: amax, then cast
        const fp8lin_quantize_item &it = items[k];
        st = launch_amax(it.x, it.rows * it.cols, it.amax, stream, true);
        if (st == FP8LIN_OK)
            st = cast_common(kDynamic, it.x, it.rows, it.cols, fmt, fmt_max, it.amax, 0, 0, it.scale, it.inv_scale,
                             it.q, nullptr, nullptr, stream);
        if (st != FP8LIN_OK) return st;
    }
    return FP8LIN_OK;
}

extern "C" fp8lin_status fp8lin_cast_transpose_static(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt,
                                                      const float *scale, float *inv_scale, uint8_t *q,
                                                      uint8_t *qT, float *amax, cudaStream_t stream) {
    return cast_common(kStatic, x, rows, cols, fmt, 0.0f, scale, 0, 0, nullptr, inv_scale, q, qT, amax,
                       stream);
}

extern "C" fp8lin_status fp8lin_cast_transpose_delayed(const void *x, int64_t rows, int64_t cols,
                                                       fp8lin_fmt fmt, float fmt_max, float *amax_history,
                                                       int64_t history_len, int64_t slot, float *scale,
                                                       float *inv_scale, uint8_t *q, uint8_t *qT,
                                                       cudaStream_t stream) {
    if (amax_history == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (history_len < 2 || history_len > FP8LIN_MAX_HISTORY || slot < 0 || slot >= history_len)
        return FP8LIN_ERR_INVALID_ARG;
    return cast_common(kDelayed, x, rows, cols, fmt, fmt_max, amax_history, (int)history_len, (int)slot, scale,
                       inv_scale, q, qT, amax_history + slot, stream);
}

extern "C" fp8lin_status fp8lin_cast_blockwise(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt,
                                               float fmt_max, uint8_t *q_row, float *inv_row, uint8_t *q_col,
                                               float *inv_col, uint8_t *q_tile, float *inv_tile,
                                               cudaStream_t stream) {
    using namespace fp8lin;
    // each copy comes with its inverse scales, or neither is asked for
    if ((q_row == nullptr) != (inv_row == nullptr) || (q_col == nullptr) != (inv_col == nullptr) ||
        (q_tile == nullptr) != (inv_tile == nullptr))
        return FP8LIN_ERR_INVALID_ARG;
    const int which = (q_row ? 1 : 0) | (q_col ? 2 : 0) | (q_tile ? 4 : 0);
    if (which == 0) return FP8LIN_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return FP8LIN_ERR_INVALID_ARG;
    if (fmt != FP8LIN_E4M3 && fmt != FP8LIN_E5M2) return FP8LIN_ERR_INVALID_ARG;
    if (!(fmt_max > 0.0f) || !(fmt_max <= 3.4e38f)) return FP8LIN_ERR_INVALID_ARG;
    const bool empty = rows == 0 || cols == 0;
    if (!empty && x == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (!aligned(inv_row, 4) || !aligned(inv_col, 4) || !aligned(inv_tile, 4)) return FP8LIN_ERR_MISALIGNED;
    if (!empty && (!aligned(x, 16) || !aligned(q_row, 16) || !aligned(q_col, 16) || !aligned(q_tile, 16)))
        return FP8LIN_ERR_MISALIGNED;
    if (!dim_ok(rows) || !dim_ok(cols) || rows % 16 || cols % 16) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    const int64_t tiles_r = (rows + kTile - 1) / kTile, tiles_c = (cols + kTile - 1) / kTile;
    if (tiles_r * tiles_c > INT32_MAX - (1 << 20)) return FP8LIN_ERR_UNSUPPORTED_SHAPE;  // tile + ring lookahead fits an int
    DeviceInfo dev;
    fp8lin_status st = current_device(&dev);
    if (st != FP8LIN_OK) return st;
    if (empty) return FP8LIN_OK;
    const int num_tiles = (int)(tiles_r * tiles_c);
    const uint16_t *xs = static_cast<const uint16_t *>(x);
    st = fmt == FP8LIN_E4M3
             ? launch_block_any<FP8LIN_E4M3>(dev.device, dev.sm_count, which, num_tiles, stream, xs, (int)rows,
                                             (int)cols, (int)tiles_r, (int)tiles_c, fmt_max, q_row, inv_row, q_col,
                                             inv_col, q_tile, inv_tile)
             : launch_block_any<FP8LIN_E5M2>(dev.device, dev.sm_count, which, num_tiles, stream, xs, (int)rows,
                                             (int)cols, (int)tiles_r, (int)tiles_c, fmt_max, q_row, inv_row, q_col,
                                             inv_col, q_tile, inv_tile);
    if (st != FP8LIN_OK) return st;
    return check_launch();
}

extern "C" fp8lin_status fp8lin_cast_transpose_rowwise(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt,
                                                       float fmt_max, const float *row_amax, const float *col_amax,
                                                       float *row_inv_scale, float *col_inv_scale, uint8_t *q,
                                                       uint8_t *qT, cudaStream_t stream) {
    if (q == nullptr && qT == nullptr) return FP8LIN_ERR_INVALID_ARG;
    return cast_common(kRowwise, x, rows, cols, fmt, fmt_max, row_amax, 0, 0, nullptr, row_inv_scale, q, qT, nullptr,
                       stream, col_amax, col_inv_scale);
}

namespace {

// Checks and launch shared by the two power-of-two scale rules.
fp8lin_status cast_mx_common(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt, float fmt_max, int ocp_emax,
                             uint8_t *q_row, uint8_t *sf_row, uint8_t *q_col, uint8_t *sf_col, cudaStream_t stream) {
    using namespace fp8lin;
    if ((q_row == nullptr) != (sf_row == nullptr) || (q_col == nullptr) != (sf_col == nullptr))
        return FP8LIN_ERR_INVALID_ARG;
    if (q_row == nullptr && q_col == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return FP8LIN_ERR_INVALID_ARG;
    if (fmt != FP8LIN_E4M3 && fmt != FP8LIN_E5M2) return FP8LIN_ERR_INVALID_ARG;
    // a normal, finite fmt_max: the exponent rule reads its bit pattern
    if (!(fmt_max >= 1.17549435e-38f) || !(fmt_max <= 3.4e38f)) return FP8LIN_ERR_INVALID_ARG;
    const bool empty = rows == 0 || cols == 0;
    if (!empty && x == nullptr) return FP8LIN_ERR_INVALID_ARG;
    if (!empty && (!aligned(x, 16) || !aligned(q_row, 16) || !aligned(q_col, 16) || !aligned(sf_row, 16) ||
                   !aligned(sf_col, 16)))
        return FP8LIN_ERR_MISALIGNED;
    if (!dim_ok(rows) || !dim_ok(cols) || rows % 16 || cols % 16) return FP8LIN_ERR_UNSUPPORTED_SHAPE;
    const int64_t tiles_r = (rows + kTile - 1) / kTile, tiles_c = (cols + kTile - 1) / kTile;
    if (tiles_r * tiles_c > INT32_MAX - (1 << 20)) return FP8LIN_ERR_UNSUPPORTED_SHAPE;  // tile + ring lookahead fits an int
    DeviceInfo dev;
    fp8lin_status st = current_device(&dev);
    if (st != FP8LIN_OK) return st;
    if (empty) return FP8LIN_OK;
    const int num_tiles = (int)(tiles_r * tiles_c);
    uint32_t fmax_bits;
    memcpy(&fmax_bits, &fmt_max, 4);
    const uint16_t *xs = static_cast<const uint16_t *>(x);
    st = fmt == FP8LIN_E4M3 ? launch_mx_any<FP8LIN_E4M3>(dev.device, dev.sm_count, num_tiles, stream, xs, (int)rows, (int)cols,
                                                         (int)tiles_r, (int)tiles_c, fmax_bits, ocp_emax, q_row,
                                                         sf_row, q_col, sf_col)
                            : launch_mx_any<FP8LIN_E5M2>(dev.device, dev.sm_count, num_tiles, stream, xs, (int)rows, (int)cols,
                                                         (int)tiles_r, (int)tiles_c, fmax_bits, ocp_emax, q_row,
                                                         sf_row, q_col, sf_col);
    if (st != FP8LIN_OK) return st;
    return check_launch();
}

}  // namespace

extern "C" fp8lin_status fp8lin_cast_mx(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt, float fmt_max,
                                        uint8_t *q_row, uint8_t *sf_row, uint8_t *q_col, uint8_t *sf_col,
                                        cudaStream_t stream) {
    return cast_mx_common(x, rows, cols, fmt, fmt_max, 0, q_row, sf_row, q_col, sf_col, stream);
}

extern "C" fp8lin_status fp8lin_cast_mx_ocp(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt,
                                            uint8_t *q_row, uint8_t *sf_row, uint8_t *q_col, uint8_t *sf_col,
                                            cudaStream_t stream) {
    // the element format's own exponent range fixes the rule (fmt_max only passes the shared checks)
    const int emax = fmt == FP8LIN_E4M3 ? 8 : 15;
    return cast_mx_common(x, rows, cols, fmt, 448.0f, emax, q_row, sf_row, q_col, sf_col, stream);
}
