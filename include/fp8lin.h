/*
 * fp8lin.h -- C ABI of the Float8 linear layer hot path for one GB300 GPU
 * (sm_103a): dynamic per-tensor scaling and the three scaled FP8 GEMMs of a
 * linear layer's forward and backward pass, with the other scaling recipes
 * beside it: static and delayed per-tensor scaling, row-wise scales, fp32
 * block scales (1 x 128 / 128 x 128) and power-of-two block scales per 32
 * contraction elements applied by the tensor cores.
 *
 * Source of the method: "TorchTitan: a one-stop PyTorch-native solution for
 * production LLM pre-training" (zenmind.me paper analysis), section 3.3
 * "Memory and compute optimisations", bullet "Mixed precision and Float8":
 * Float8 is a derived dtype applied selectively to linear layers, with
 * dynamic / delayed / static per-tensor scaling, composable with autograd.
 * "Lecture 9 exercises" (juanwang-buaa tutorials), the answer on fp16 loss
 * scaling versus FP8 scaling: FP8 scaling is one factor per tensor, and FP8
 * saves only what is stored in FP8 (the FP8 copies are what the backward
 * pass keeps).  The pages fix neither the formats nor the arithmetic; this
 * library takes e4m3 for activations and weights, e5m2 for output
 * gradients, scale = fmt_max / amax (fmt_max = 448), a saturating
 * round-to-nearest-even cast, fp32 accumulation and the inverse scales
 * applied to the fp32 accumulator before the bf16 store.
 *
 * Conventions (nn.Linear):  X is [M x K] (tokens x in-features), W is
 * [N x K] (out-features x in-features), dY is [M x N]; every matrix is
 * row-major.  One linear's step is
 *     forward : fp8lin_amax(X), fp8lin_amax(W),
 *               fp8lin_cast_transpose(X -> Xq, XqT), (W -> Wq, WqT),
 *               fp8lin_fwd(Xq, Wq) -> Y
 *     backward: fp8lin_amax(dY), fp8lin_cast_transpose(dY -> dYq, dYqT),
 *               fp8lin_dgrad(dYq, WqT) -> dX, fp8lin_wgrad(dYqT, XqT) -> dW
 * or, with no transposed copies (qT = NULL in every cast):
 *               fp8lin_dgrad_mn(dYq, Wq) -> dX, fp8lin_wgrad_mn(dYq, Xq) -> dW
 *
 * Ownership: the caller allocates and owns every buffer (device memory),
 * including the one-float amax / scale / inverse-scale slots.  No entry
 * point allocates device memory; the GEMM kernels allocate and free tensor
 * memory (TMEM) on chip inside the kernel.
 *
 * Synchronisation: every call is asynchronous on `stream` (a CUDA stream of
 * the current device; 0 = legacy default stream).  Scales never leave the
 * device, so no call synchronises with the host.  Calls on one stream run in
 * order; the caller orders calls across streams.
 *
 * Errors: argument checks run on the host before anything is launched.  A
 * failed check returns its status and launches nothing.  A launch failure
 * returns FP8LIN_ERR_CUDA.  Faults inside a kernel surface, as usual with
 * CUDA, at the caller's next synchronisation.  Every wait inside the GEMM
 * kernels is bounded in time: a wait that runs out makes the kernel stop
 * cleanly and record FP8LIN_ERR_TIMEOUT in a device word that
 * fp8lin_device_error() reads back.
 */
#ifndef FP8LIN_H
#define FP8LIN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp8lin_status {
    FP8LIN_OK = 0,
    FP8LIN_ERR_INVALID_ARG = 1,        /* NULL pointer, negative size, bad format or fmt_max */
    FP8LIN_ERR_MISALIGNED = 2,         /* a pointer breaks the alignment stated on the call  */
    FP8LIN_ERR_UNSUPPORTED_SHAPE = 3,  /* a dimension is not a multiple of 16 or too large   */
    FP8LIN_ERR_CUDA = 4,               /* the CUDA runtime reported an error                 */
    FP8LIN_ERR_TIMEOUT = 5,            /* a bounded wait inside a kernel ran out             */
    FP8LIN_ERR_UNSUPPORTED_DEVICE = 6  /* the current device is not compute capability 10.3  */
} fp8lin_status;

typedef enum fp8lin_fmt {
    FP8LIN_E4M3 = 0,  /* 1-4-3, bias 7, no Inf, largest finite 448 (activations, weights) */
    FP8LIN_E5M2 = 1   /* 1-5-2, bias 15, largest finite 57344 (output gradients)          */
} fp8lin_fmt;

/* Largest dimension accepted by any call (rows, columns, M, N or K). */
#define FP8LIN_MAX_DIM ((int64_t)1 << 30)

/* Longest amax history accepted by fp8lin_cast_transpose_delayed. */
#define FP8LIN_MAX_HISTORY 1024

/*
 * amax of one bf16 tensor: *amax = max_i |x_i| (fp32, exact).
 * Dynamic per-tensor scaling takes this statistic of the tensor itself each
 * step (TorchTitan analysis page, section 3.3, "Mixed precision and Float8";
 * Lecture 9 exercises, FP8 scaling is one factor per tensor).
 *
 *   x      device, n bf16 values, contiguous, 16-byte aligned.
 *   n      element count, >= 0 (n == 0 gives amax = 0).
 *   amax   device, one float, 4-byte aligned.  Overwritten: the call clears
 *          it on `stream` before the reduction.
 * Magnitudes are ordered like the IEEE 754 totalOrder predicate: a NaN in x
 * gives a NaN amax, an infinity gives +Inf.
 */
fp8lin_status fp8lin_amax(const void *x, int64_t n, float *amax, cudaStream_t stream);

/*
 * Scale and cast one bf16 matrix to FP8, writing the row-major copy and/or
 * its transpose (the copy whose contiguous index is the row index), so that
 * each GEMM reads both operands with the contraction index contiguous.
 * Source: the Float8 derived dtype (TorchTitan analysis page, section 3.3).
 *
 *   x          device, bf16 [rows x cols] row-major, 16-byte aligned.
 *   rows, cols >= 0, multiples of 16, <= FP8LIN_MAX_DIM.
 *   fmt        FP8LIN_E4M3 (X, W) or FP8LIN_E5M2 (dY).
 *   fmt_max    finite, > 0: the scale's numerator (448 for all three tensors).
 *   amax       device, one float written by fp8lin_amax (read only).
 *   scale      device, one float: receives fmt_max / max(amax, 1e-12) (fp32,
 *              round to nearest even).
 *   inv_scale  device, one float: receives 1 / scale (fp32 RN), the factor
 *              the GEMM epilogues apply.
 *   q          device, u8 [rows x cols] or NULL; 16-byte aligned.
 *   qT         device, u8 [cols x rows] or NULL; 16-byte aligned.
 * Every code is sat_RNE(fp32(x) * scale): the binary32 product rounded to
 * nearest even, then rounded to nearest even into the format, saturating at
 * the format's largest finite value (Inf included); every NaN (either sign,
 * any payload) casts to the code 0x7F; the sign of zero is kept.  A NaN amax
 * gives a NaN scale (0x7FFFFFFF) and every code 0x7F.
 */
fp8lin_status fp8lin_cast_transpose(const void *x, int64_t rows, int64_t cols,
                                    fp8lin_fmt fmt, float fmt_max, const float *amax,
                                    float *scale, float *inv_scale,
                                    uint8_t *q, uint8_t *qT, cudaStream_t stream);

/*
 * Dynamic per-tensor scaling of one tensor in one call: fp8lin_amax followed
 * by fp8lin_cast_transpose on the same stream, with the same results bit for
 * bit (TorchTitan analysis page, section 3.3: dynamic scaling takes the
 * tensor's own statistic every step; Lecture 9 exercises: one factor per
 * tensor).  For a cast that runs with no GEMM beside it -- the cast a GEMM
 * waits for.  With q and no qT (and fmt_max <= 65504) it is one launch.  Up
 * to 786432 elements (1.5 MB of bf16) one cluster of 8 CTAs holds the whole
 * tensor in shared memory, exchanges the CTAs' maxima through distributed
 * shared memory at a cluster barrier, writes the three slots and casts;
 * nothing is cleared first.  Larger tensors take a cooperative launch with
 * one CTA on every SM: the grid reads x once for the amax, keeping part of
 * it in shared memory, meets at a grid barrier held in the amax / scale /
 * inverse-scale slots themselves (the call clears them first; no other
 * device memory is used), and casts.  Otherwise it is
 * fp8lin_amax (with the tensor's last 64 MB kept in L2 for the cast) and
 * fp8lin_cast_transpose.  Beside a running GEMM, or for two casts at once on
 * two streams (each grid wants every SM), call fp8lin_amax and
 * fp8lin_cast_transpose instead.  A grid barrier that does not complete
 * within 2 s records FP8LIN_ERR_TIMEOUT for fp8lin_device_error.
 *
 *   amax       device, one float: receives max |x|.
 *   x, rows, cols, fmt, fmt_max, scale, inv_scale, q, qT as for
 *   fp8lin_cast_transpose; arguments are checked before anything is launched.
 */
fp8lin_status fp8lin_quantize(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt, float fmt_max,
                              float *amax, float *scale, float *inv_scale, uint8_t *q, uint8_t *qT,
                              cudaStream_t stream);

/* Most tensors one fp8lin_quantize_batch call takes. */
#define FP8LIN_MAX_QUANTIZE_BATCH 4

/* One tensor of fp8lin_quantize_batch: the arguments of fp8lin_quantize
 * without the transposed copy. */
typedef struct fp8lin_quantize_item {
    const void *x;        /* device, bf16 [rows x cols] row-major, 16-byte aligned           */
    int64_t rows, cols;   /* >= 0, multiples of 16, <= FP8LIN_MAX_DIM                        */
    float *amax;          /* device, one float each, 4-byte aligned: receives max |x|,       */
    float *scale;         /*   fmt_max / max(amax, 1e-12) and 1 / scale; no two slots of a   */
    float *inv_scale;     /*   call (of this tensor or another) may coincide                 */
    uint8_t *q;           /* device, u8 [rows x cols], 16-byte aligned (NULL if empty)      */
} fp8lin_quantize_item;

/*
 * fp8lin_quantize for several tensors of one format, each with its own amax
 * and scale (TorchTitan analysis page, section 3.3: dynamic scaling takes
 * each tensor's own statistic every step; Lecture 9 exercises: one factor
 * per tensor), in one launch: the casts that gate the same GEMM, such as the
 * X and W of a forward pass, share one grid, one barrier and one clearing
 * memset instead of one each.  Every tensor's amax, scale, inverse scale and
 * FP8 bytes are bit for bit those of fp8lin_quantize on that tensor alone.
 * Up to 786432 elements in all the tensors take one cluster of 8 CTAs (no
 * memset); larger batches the whole-GPU cooperative grid.  With fmt_max
 * above 65504, or no cooperative launch on the device, the tensors are cast
 * one after another through fp8lin_amax and fp8lin_cast_transpose.  The same
 * conditions as fp8lin_quantize hold: nothing beside it, a grid barrier
 * bounded at 2 s (FP8LIN_ERR_TIMEOUT for fp8lin_device_error).
 *
 *   items   host array of `count` items, read during the call only.
 *   count   1 .. FP8LIN_MAX_QUANTIZE_BATCH.
 *   fmt, fmt_max  as for fp8lin_cast_transpose, shared by every item.
 * Every item is checked before anything is launched.
 */
fp8lin_status fp8lin_quantize_batch(const fp8lin_quantize_item *items, int count, fp8lin_fmt fmt,
                                    float fmt_max, cudaStream_t stream);

/*
 * Static scaling: cast with a scale the caller fixes (TorchTitan analysis
 * page, section 3.3: torchao offers dynamic, delayed and static per-tensor
 * scaling).  Same layouts, rounding and saturation as fp8lin_cast_transpose.
 *
 *   scale      device, one float, read only: the scale to apply.
 *   inv_scale  device, one float: receives 1 / scale (fp32 RN).
 *   amax       device, one float, or NULL: when given, receives max |x| of
 *              this tensor (cleared by the call first), e.g. to calibrate or
 *              to monitor the fixed scale.
 *   x, rows, cols, fmt, q, qT as for fp8lin_cast_transpose.
 */
fp8lin_status fp8lin_cast_transpose_static(const void *x, int64_t rows, int64_t cols,
                                           fp8lin_fmt fmt, const float *scale, float *inv_scale,
                                           uint8_t *q, uint8_t *qT, float *amax,
                                           cudaStream_t stream);

/*
 * Delayed scaling: the scale comes from the statistics of previous steps, so
 * no amax pass has to run before the cast (TorchTitan analysis page, section
 * 3.3, "delayed" per-tensor scaling; Lecture 9 exercises: delayed scaling
 * uses the previous step's statistics so the scaling work can hide in an
 * overlap window).  The pages give no history rule; this library keeps a
 * caller-owned ring of amax values:
 *
 *   scale          = fmt_max / max(max_{i != slot} amax_history[i], 1e-12)
 *   amax_history[slot] = max |x| of this tensor (cleared by the call first,
 *                        then recorded by the cast kernel itself)
 *
 * and the caller advances slot = (slot + 1) % history_len every step.  A
 * history whose other slots are all zero (the first step) gives the floor
 * scale, which saturates everything: seed slot (slot + 1) % history_len with
 * one fp8lin_amax of the tensor first.
 *
 *   amax_history  device, history_len floats (4-byte aligned), read and written.
 *   history_len   2 .. FP8LIN_MAX_HISTORY.
 *   slot          0 .. history_len - 1: the entry this step writes.
 *   fmt_max, scale, inv_scale, x, rows, cols, fmt, q, qT as for
 *   fp8lin_cast_transpose.  Values beyond the scaled range saturate.
 */
fp8lin_status fp8lin_cast_transpose_delayed(const void *x, int64_t rows, int64_t cols,
                                            fp8lin_fmt fmt, float fmt_max, float *amax_history,
                                            int64_t history_len, int64_t slot, float *scale,
                                            float *inv_scale, uint8_t *q, uint8_t *qT,
                                            cudaStream_t stream);

/*
 * Row-wise ("per block") scaling, statistics: row_amax[r] = max_c |x[r][c]|
 * and col_amax[c] = max_r |x[r][c]| of a bf16 [rows x cols] matrix.
 * "Lecture 9 exercises": FP8 scaling is one factor per tensor, or even per
 * block.  The block taken here is one row of each GEMM operand: the finest
 * block that is constant along the GEMM's contraction, so that its scale
 * factors out of the sum and is applied in the epilogue.
 *
 *   x          device, bf16 [rows x cols] row-major, 16-byte aligned.
 *   rows, cols >= 0, multiples of 16, <= FP8LIN_MAX_DIM.
 *   row_amax   device, rows floats, or NULL; cleared by the call first.
 *   col_amax   device, cols floats, or NULL (not both NULL); cleared first.
 */
fp8lin_status fp8lin_amax_rowcol(const void *x, int64_t rows, int64_t cols, float *row_amax,
                                 float *col_amax, cudaStream_t stream);

/*
 * Row-wise scaling, cast: q[r][c] = sat_RNE(fp32(x[r][c]) * s_row[r]) and
 * qT[c][r] = sat_RNE(fp32(x[r][c]) * s_col[c]) with
 * s_row[r] = fmt_max / max(row_amax[r], 1e-12), s_col[c] likewise from
 * col_amax; each copy is cast from the bf16 source with the scales of its
 * own rows, so qT is in general not the byte transpose of q.
 *
 *   row_amax, row_inv_scale   device, rows floats: read / receives 1 / s_row
 *                             (needed when q is not NULL).
 *   col_amax, col_inv_scale   device, cols floats: read / receives 1 / s_col
 *                             (needed when qT is not NULL).
 *   q, qT      device, as for fp8lin_cast_transpose (not both NULL).
 */
fp8lin_status fp8lin_cast_transpose_rowwise(const void *x, int64_t rows, int64_t cols,
                                            fp8lin_fmt fmt, float fmt_max, const float *row_amax,
                                            const float *col_amax, float *row_inv_scale,
                                            float *col_inv_scale, uint8_t *q, uint8_t *qT,
                                            cudaStream_t stream);

/*
 * Forward GEMM of the Float8 linear: Y = bf16_RN( (Xq . Wq^T)_fp32 * (inv_x * inv_w) ).
 * Source: Float8 applied to the linear layer's matmul (TorchTitan analysis
 * page, section 3.3).
 *
 *   xq     device, e4m3 [M x K] row-major (K contiguous), 16-byte aligned.
 *   inv_x  device, one float (inverse scale of X).
 *   wq     device, e4m3 [N x K] row-major, 16-byte aligned.
 *   inv_w  device, one float (inverse scale of W).
 *   y      device, bf16 [M x N] row-major, 16-byte aligned; fully overwritten.
 *   M, N, K  >= 0, multiples of 16, <= FP8LIN_MAX_DIM.  K == 0 writes zeros.
 */
fp8lin_status fp8lin_fwd(const uint8_t *xq, const float *inv_x, const uint8_t *wq,
                         const float *inv_w, void *y, int64_t M, int64_t N, int64_t K,
                         cudaStream_t stream);

/*
 * Input-gradient GEMM: dX = bf16_RN( (dYq . WqT^T)_fp32 * (inv_dy * inv_w) ),
 * i.e. dY . W.  Source: the backward pass of the Float8 linear through
 * autograd (TorchTitan analysis page, section 3.3).
 *
 *   dyq     device, e5m2 [M x N] row-major (N contiguous), 16-byte aligned.
 *   inv_dy  device, one float.
 *   wqT     device, e4m3 [K x N] (the transposed copy of Wq), 16-byte aligned.
 *   inv_w   device, one float.
 *   dx      device, bf16 [M x K] row-major, 16-byte aligned; fully overwritten.
 *   M, N, K  as for fp8lin_fwd.  N == 0 writes zeros.
 */
fp8lin_status fp8lin_dgrad(const uint8_t *dyq, const float *inv_dy, const uint8_t *wqT,
                           const float *inv_w, void *dx, int64_t M, int64_t N, int64_t K,
                           cudaStream_t stream);

/*
 * Weight-gradient GEMM: dW = bf16_RN( (dYqT . XqT^T)_fp32 * (inv_dy * inv_x) ),
 * i.e. dY^T . X.  Source: as for fp8lin_dgrad.
 *
 *   dyqT    device, e5m2 [N x M] (the transposed copy of dYq), 16-byte aligned.
 *   inv_dy  device, one float.
 *   xqT     device, e4m3 [K x M] (the transposed copy of Xq), 16-byte aligned.
 *   inv_x   device, one float.
 *   dw      device, bf16 [N x K] row-major, 16-byte aligned; fully overwritten.
 *   M, N, K  as for fp8lin_fwd.  M == 0 writes zeros.
 */
fp8lin_status fp8lin_wgrad(const uint8_t *dyqT, const float *inv_dy, const uint8_t *xqT,
                           const float *inv_x, void *dw, int64_t M, int64_t N, int64_t K,
                           cudaStream_t stream);

/*
 * The two backward GEMMs on the row-major FP8 copies (q of
 * fp8lin_cast_transpose), so a per-tensor-scaled linear needs no transposed
 * copy.  Same products, bit for bit, as fp8lin_dgrad / fp8lin_wgrad on the
 * transposed copies: the tensor cores read an 8-bit operand either
 * contraction-contiguous or row-index-contiguous, and these entry points
 * read Wq, dYq and Xq the second way.  With them each tensor of a
 * per-tensor-scaled step (TorchTitan analysis page, section 3.3: Float8
 * forward and backward through autograd) is cast once, to the one FP8 copy
 * that all three GEMMs read.  Row-wise scaling still needs the transposed
 * copies, whose scales run along the other axis.
 *
 * fp8lin_dgrad_mn: dX = bf16_RN( (dYq . Wq)_fp32 * (inv_dy * inv_w) ) = dY . W
 *   dyq     device, e5m2 [M x N] row-major, 16-byte aligned.
 *   wq      device, e4m3 [N x K] row-major (the copy fp8lin_fwd reads).
 *   dx      device, bf16 [M x K] row-major, 16-byte aligned; fully overwritten.
 * fp8lin_wgrad_mn: dW = bf16_RN( (dYq^T . Xq)_fp32 * (inv_dy * inv_x) ) = dY^T . X
 *   dyq     device, e5m2 [M x N] row-major, 16-byte aligned.
 *   xq      device, e4m3 [M x K] row-major (the copy fp8lin_fwd reads).
 *   dw      device, bf16 [N x K] row-major, 16-byte aligned; fully overwritten.
 * inv_*, M, N, K and the errors as for fp8lin_dgrad / fp8lin_wgrad.
 */
fp8lin_status fp8lin_dgrad_mn(const uint8_t *dyq, const float *inv_dy, const uint8_t *wq,
                              const float *inv_w, void *dx, int64_t M, int64_t N, int64_t K,
                              cudaStream_t stream);
fp8lin_status fp8lin_wgrad_mn(const uint8_t *dyq, const float *inv_dy, const uint8_t *xq,
                              const float *inv_x, void *dw, int64_t M, int64_t N, int64_t K,
                              cudaStream_t stream);

/*
 * Block scaling: every block of x is scaled like a tensor of its own
 * ("one factor per tensor, or even per block": Lecture 9 exercises, the
 * answer on fp16 loss scaling versus FP8 scaling) -- amax of the block,
 * scale = fmt_max / max(amax, 1e-12) (binary32, round to nearest even), a
 * saturating round-to-nearest-even cast -- in one pass over x, with no
 * separate amax call.  Any of three copies, each row-major [rows x cols]
 * like x, with its inverse scales (1 / scale, binary32):
 *   q_row,  inv_row  [ceil(cols/128) x rows]            1 x 128 blocks
 *   q_col,  inv_col  [ceil(rows/128) x cols]            128 x 1 blocks
 *   q_tile, inv_tile [ceil(rows/128) x ceil(cols/128)]  128 x 128 blocks
 * Blocks at the right and bottom edges are cut short.  Scales are stored
 * block-major (one block column's scales, or one block row's, contiguous),
 * so that the GEMM reads one contraction block's scales of consecutive rows
 * in one transaction.  A linear takes X as
 * q_row (forward) and q_col (weight gradient), W as q_tile, dY as q_row
 * (input gradient) and q_col (weight gradient); see fp8lin_fwd_block.
 *
 *   x        device, bf16 [rows x cols] row-major, 16-byte aligned.
 *   fmt      FP8LIN_E4M3 or FP8LIN_E5M2; fmt_max > 0 (448 by default).
 *   q_*      device, u8 [rows x cols], 16-byte aligned, or NULL.
 *   inv_*    device floats (sizes above), or NULL together with their q_*.
 *   rows, cols  >= 0, multiples of 16, <= FP8LIN_MAX_DIM.
 * Errors: a q_* without its inv_* (or the reverse), or no copy at all, is
 * FP8LIN_ERR_INVALID_ARG; alignment and shape as for fp8lin_cast_transpose,
 * and FP8LIN_ERR_UNSUPPORTED_SHAPE when the 128 x 128 tiles of x number more
 * than 2^31 - 2^20 - 1 (checked before the device is touched).
 */
fp8lin_status fp8lin_cast_blockwise(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt,
                                    float fmt_max, uint8_t *q_row, float *inv_row, uint8_t *q_col,
                                    float *inv_col, uint8_t *q_tile, float *inv_tile,
                                    cudaStream_t stream);

/*
 * The three GEMMs of a block-scaled linear (copies from
 * fp8lin_cast_blockwise).  The contraction is cut into blocks of 128; the
 * tensor cores sum each block in fp32, the partial sum is multiplied by the
 * two operands' inverse scales for that block (fp32) and added to an fp32
 * total, which is rounded to bf16 (round to nearest even) at the end:
 *   fwd  : Y [M x N]  = sum_j (Xq Wq^T)_j  * inv_x[j][m]  * inv_w[n/128][j]   contraction K
 *   dgrad: dX [M x K] = sum_j (dYq Wq)_j   * inv_dy[j][m] * inv_w[j][k/128]   contraction N
 *   wgrad: dW [N x K] = sum_j (dYq^T Xq)_j * inv_dy[j][n] * inv_x[j][k]       contraction M
 * (Lecture 9 exercises: FP8 scaling per tensor or per block; TorchTitan
 * analysis page, section 3.3: the Float8 linear's three GEMMs.)
 *
 * fp8lin_fwd_block:   xq = q_row of X [M x K] e4m3, inv_x [ceil(K/128) x M];
 *                     wq = q_tile of W [N x K] e4m3, inv_w [ceil(N/128) x ceil(K/128)].
 * fp8lin_dgrad_block: dyq = q_row of dY [M x N] e5m2, inv_dy [ceil(N/128) x M];
 *                     wq, inv_w as for the forward.
 * fp8lin_wgrad_block: dyq = q_col of dY [M x N] e5m2, inv_dy [ceil(M/128) x N];
 *                     xq = q_col of X [M x K] e4m3, inv_x [ceil(M/128) x K].
 * The scales of the row and column blocks (inv_x, inv_dy; for the weight
 * gradient both) are read four rows at a time and must be 16-byte aligned
 * (FP8LIN_ERR_MISALIGNED otherwise); inv_w needs 4 bytes.  Outputs bf16
 * row-major, 16-byte aligned, fully overwritten.  Pointers, shapes and
 * errors otherwise as for fp8lin_fwd.
 */
fp8lin_status fp8lin_fwd_block(const uint8_t *xq, const float *inv_x, const uint8_t *wq,
                               const float *inv_w, void *y, int64_t M, int64_t N, int64_t K,
                               cudaStream_t stream);
fp8lin_status fp8lin_dgrad_block(const uint8_t *dyq, const float *inv_dy, const uint8_t *wq,
                                 const float *inv_w, void *dx, int64_t M, int64_t N, int64_t K,
                                 cudaStream_t stream);
fp8lin_status fp8lin_wgrad_block(const uint8_t *dyq, const float *inv_dy, const uint8_t *xq,
                                 const float *inv_x, void *dw, int64_t M, int64_t N, int64_t K,
                                 cudaStream_t stream);

/*
 * The three GEMMs with row-wise scales: C[p][q] = bf16_RN(acc[p][q] *
 * (inv_a[p] * inv_b[q])), inv_a one float per row of A and inv_b one per row
 * of B (16-byte aligned device vectors).  Operands, shapes and outputs as for
 * fp8lin_fwd / fp8lin_dgrad / fp8lin_wgrad:
 *   fwd   inv_x_rows [M] (X's row scales),   inv_w_rows [N] (W's row scales)
 *   dgrad inv_dy_rows [M] (dY's row scales), inv_w_cols [K] (W's column scales)
 *   wgrad inv_dy_cols [N] (dY's column scales), inv_x_cols [K] (X's column scales)
 */
fp8lin_status fp8lin_fwd_rowwise(const uint8_t *xq, const float *inv_x_rows, const uint8_t *wq,
                                 const float *inv_w_rows, void *y, int64_t M, int64_t N, int64_t K,
                                 cudaStream_t stream);
fp8lin_status fp8lin_dgrad_rowwise(const uint8_t *dyq, const float *inv_dy_rows, const uint8_t *wqT,
                                   const float *inv_w_cols, void *dx, int64_t M, int64_t N, int64_t K,
                                   cudaStream_t stream);
fp8lin_status fp8lin_wgrad_rowwise(const uint8_t *dyqT, const float *inv_dy_cols, const uint8_t *xqT,
                                   const float *inv_x_cols, void *dw, int64_t M, int64_t N, int64_t K,
                                   cudaStream_t stream);

/*
 * Block scaling with power-of-two scales, applied by the tensor cores.  The
 * "per block" factor of the Lecture 9 exercises (the answer on fp16 loss
 * scaling versus FP8 scaling: one factor per tensor, or even per block),
 * restricted to powers of two in the granularity the sm_103a block-scaled
 * MMA (tcgen05.mma kind::mxf8f6f4.block_scale) applies: one scale per 32
 * contraction elements.  A block's scale is 2^e, e the largest integer with
 * max(amax, 1e-12) * 2^e <= fmt_max (clamped to -127 .. 127): the largest
 * power of two not above the per-tensor recipe's fmt_max / amax, so the
 * block's largest magnitude lands in [fmt_max / 2, fmt_max] and nothing
 * saturates.  Codes are sat_RNE(fp32(x) * 2^e) (the product is exact).
 *
 * Scales are stored as bytes 127 - e (the unsigned-exponent code of the
 * inverse scale 2^-e; 0xFF for a block whose amax is NaN or infinite), in
 * the order the tensor cores read them: "atoms" of 512 bytes, one per 128
 * operand rows x 128 contraction elements.  For a copy read by a GEMM with
 * operand rows p (P of them) and contraction index k (K of them), atom
 * (k / 128, p / 128) starts at byte ((k / 128) * ceil(P / 128) + p / 128) * 512,
 * and holds the scale of row p, block j = k / 32 at byte
 * 16 (p % 32) + 4 ((p % 128) / 32) + j % 4.  Entries past P or past the
 * last block hold 127 (scale 1).  Size: ceil(P/128) * ceil(K/128) * 512 bytes.
 */

/*
 * One pass over a bf16 [rows x cols] matrix x, writing either or both of
 *   q_row, sf_row: 1 x 32 blocks (runs of 32 columns); the copy is read with
 *                  its rows as operand rows and the contraction along the
 *                  columns (P = rows, K = cols);
 *   q_col, sf_col: 32 x 1 blocks (runs of 32 rows); read with its columns as
 *                  operand rows and the contraction along the rows
 *                  (P = cols, K = rows).
 * Both copies are row-major [rows x cols] like x.  A linear takes X as q_row
 * (forward) and q_col (weight gradient), W as q_row (forward) and q_col
 * (input gradient), dY as q_row (input gradient) and q_col (weight gradient).
 *
 *   x        device, bf16 [rows x cols] row-major, 16-byte aligned.
 *   rows, cols  >= 0, multiples of 16, <= FP8LIN_MAX_DIM.
 *   fmt      FP8LIN_E4M3 or FP8LIN_E5M2; fmt_max a normal finite float > 0
 *            (448 by default).
 *   q_*      device, u8 [rows x cols], 16-byte aligned, or NULL.
 *   sf_*     device, u8 scale atoms (sizes above), 16-byte aligned, or NULL
 *            together with their q_*.  Every byte is written.
 * Errors: a q_* without its sf_* (or the reverse), or no copy at all, is
 * FP8LIN_ERR_INVALID_ARG; alignment and shapes as for fp8lin_cast_transpose,
 * and FP8LIN_ERR_UNSUPPORTED_SHAPE when the 128 x 128 tiles of x number more
 * than 2^31 - 2^20 - 1 (checked before the device is touched).
 */
fp8lin_status fp8lin_cast_mx(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt, float fmt_max,
                             uint8_t *q_row, uint8_t *sf_row, uint8_t *q_col, uint8_t *sf_col,
                             cudaStream_t stream);

/*
 * fp8lin_cast_mx with the OCP Microscaling scale rule instead: the block's
 * shared scale is X = 2^(floor(log2 amax) - emax), emax the exponent of the
 * element format's largest normal (8 for e4m3, 15 for e5m2), and the codes
 * are sat_RNE(fp32(x) / X) -- the top binade's magnitudes above the format's
 * maximum saturate.  The scale byte is the code of X, 127 + log2 X (0 for an
 * all-zero block, 0xFF for a NaN or infinite amax, clamped to 0 .. 254), in
 * the same atoms, so the copies feed the same GEMMs.  For copies exchanged
 * with other producers of OCP MX data; the pages fix no rule (see
 * fp8lin_cast_mx for the one that never saturates).  Arguments and errors as
 * for fp8lin_cast_mx, with no fmt_max.
 */
fp8lin_status fp8lin_cast_mx_ocp(const void *x, int64_t rows, int64_t cols, fp8lin_fmt fmt, uint8_t *q_row,
                                 uint8_t *sf_row, uint8_t *q_col, uint8_t *sf_col, cudaStream_t stream);

/*
 * The three GEMMs of a linear on power-of-two block-scaled copies
 * (fp8lin_cast_mx).  The tensor cores apply the scales inside the MMA and
 * accumulate in fp32 across the whole contraction; the result is rounded to
 * bf16 (round to nearest even):
 *   fwd  : Y [M x N]  = sum_k (Xq[m][k] 2^-ex[m][k/32]) (Wq[n][k] 2^-ew[n][k/32])
 *   dgrad: dX [M x K] = sum_n (dYq[m][n] 2^-edy[m][n/32]) (Wq[n][k] 2^-ew'[n/32][k])
 *   wgrad: dW [N x K] = sum_m (dYq[m][n] 2^-edy'[m/32][n]) (Xq[m][k] 2^-ex'[m/32][k])
 * fp8lin_fwd_mx:   xq, sf_x = q_row, sf_row of X [M x K] (e4m3);
 *                  wq, sf_w = q_row, sf_row of W [N x K] (e4m3).
 * fp8lin_dgrad_mx: dyq, sf_dy = q_row, sf_row of dY [M x N] (e5m2);
 *                  wq, sf_w = q_col, sf_col of W [N x K] (e4m3).
 * fp8lin_wgrad_mx: dyq, sf_dy = q_col, sf_col of dY [M x N] (e5m2);
 *                  xq, sf_x = q_col, sf_col of X [M x K] (e4m3).
 * Pointers 16-byte aligned (the scale atoms too); outputs bf16 row-major,
 * fully overwritten.  M, N, K and the errors as for fp8lin_fwd.
 */
fp8lin_status fp8lin_fwd_mx(const uint8_t *xq, const uint8_t *sf_x, const uint8_t *wq, const uint8_t *sf_w,
                            void *y, int64_t M, int64_t N, int64_t K, cudaStream_t stream);
fp8lin_status fp8lin_dgrad_mx(const uint8_t *dyq, const uint8_t *sf_dy, const uint8_t *wq, const uint8_t *sf_w,
                              void *dx, int64_t M, int64_t N, int64_t K, cudaStream_t stream);
fp8lin_status fp8lin_wgrad_mx(const uint8_t *dyq, const uint8_t *sf_dy, const uint8_t *xq, const uint8_t *sf_x,
                              void *dw, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Static English description of a status code (never NULL). */
const char *fp8lin_status_str(fp8lin_status status);

/*
 * Read and clear the device words in which a GEMM kernel or the one-launch
 * cast of fp8lin_quantize records a bounded wait that ran out.  Synchronises `stream` first.  Returns FP8LIN_OK when
 * no kernel timed out since the last call, FP8LIN_ERR_TIMEOUT when one did
 * (and writes the raw word to *word when word is not NULL).
 */
fp8lin_status fp8lin_device_error(cudaStream_t stream, uint32_t *word);

/*
 * Self-test of the bounded waits: launches one CTA that waits on an mbarrier
 * nothing arrives on, for at most limit_ns nanoseconds (1 us .. 1 s), using
 * the same wait as the GEMM kernels.  The wait runs out and records
 * FP8LIN_ERR_TIMEOUT in the device word that fp8lin_device_error() reads;
 * the context stays usable.  Failure detection on this path is tested
 * without any GPU fault (bounded waits of the GEMM pipeline: the pipeline
 * has no counterpart on the pages; it follows from making every wait of an
 * asynchronous producer/consumer ring finite).
 */
fp8lin_status fp8lin_selftest_bounded_wait(uint64_t limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8LIN_H */
