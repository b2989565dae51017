/*
 * fp8bs.h -- fine-grained FP8 (E4M3) block-scaled quantisation and GEMMs for
 * B300 (sm_103a).  C ABI; no C++ or framework types cross it.
 *
 * The method (from the pages describing DeepSeek-V3's FP8 training):
 *   - activations are quantised in 1x128 tiles (per row, per 128 columns of
 *     K) and weights in 128x128 blocks, each group with its own scale;
 *     ["DeepSeek-V3 training walkthrough" (deepseek.csdn.net), section 二(四)
 *      "FP8 low-precision training", fine-grained quantisation item;
 *      "DeepSeek-V3 Technical Report digest" (sherconan.github.io), section 3
 *      "FP8 mixed-precision training"; qqstock.cn walkthrough, FP8 section,
 *      report figure 7a]
 *   - the GEMM multiplies FP8 operands and, every 128 accumulated K-elements,
 *     promotes the partial result into FP32 accumulators, applying the two
 *     groups' scales; forward, data-gradient and weight-gradient GEMMs all
 *     run in FP8.
 *     [Technical Report digest, section 3, precision-promotion and
 *      FP8-operations bullets; walkthrough 二(四), MMA-into-FP32 item;
 *      qqstock.cn walkthrough, report figure 7b]
 * The pages do not fix the FP8 format or the scale rule.  This library uses
 * E4M3 ("FN": bias 7, largest finite +-448, no infinities), scale =
 * fp32(amax / 448) (one IEEE binary32 division), and codes
 * q = E4M3_round_to_nearest_even_saturating(fp32(x / scale)).  A group whose
 * elements are all +-0 gets scale 0 and codes 0x00 / 0x80 by the sign of each
 * zero.  Inputs must be finite (NaN / Inf inputs give unspecified codes).
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers (global memory of the current device)
 *     unless stated.  The caller owns every buffer and stream; the library
 *     keeps no reference to them after the call returns.
 *   - Calls are asynchronous on `stream`: they validate their arguments on
 *     the host, enqueue kernels and return.  They never synchronise and never
 *     allocate device memory.
 *   - Argument errors are returned synchronously and enqueue nothing.
 *     Device-side errors (a pipeline wait that exceeded its time limit) are
 *     recorded in a per-device error word and reported by fp8bs_last_error().
 *   - Leading dimensions (ld*) are row strides in ELEMENTS of that array.
 *   - Rows of every FP8 and BF16 INPUT and of the quantisers' outputs must
 *     start on 16-byte boundaries: base pointers 16-byte aligned and
 *     ld * element_size a multiple of 16.  GEMM outputs need only element
 *     alignment.
 *   - The device must be compute capability 10.3 (B300); else FP8BS_ERR_DEVICE.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8BS_OK = 0,
    FP8BS_ERR_NULL = -1,        /* a required pointer is NULL                        */
    FP8BS_ERR_SHAPE = -2,       /* a size is negative, or K / C not a multiple of 128 */
    FP8BS_ERR_ALIGN = -3,       /* a pointer or row stride breaks the 16-byte rule    */
    FP8BS_ERR_ARG = -4,         /* an enum value is out of range, or bad offsets size */
    FP8BS_ERR_LAUNCH = -5,      /* the CUDA runtime refused a launch                  */
    FP8BS_ERR_DEVICE = -6,      /* the current device is not sm_103                   */
    FP8BS_ERR_TIMEOUT = -7,     /* (fp8bs_last_error only) a device-side wait timed out */
    FP8BS_ERR_INDEX = -8,       /* (fp8bs_last_error only) a device-side row index was out of range */
    FP8BS_ERR_SCRATCH = -9      /* the size needs more than the library's fixed scratch holds */
} fp8bs_status;

enum { FP8BS_OUT_BF16 = 0, FP8BS_OUT_FP32 = 1 };
enum { FP8BS_MAX_EXPERTS = 2048 };
enum { FP8BS_B_KMAJOR = 0, FP8BS_B_MNMAJOR = 1 };

/*
 * 1x128 activation quantisation.
 *   x_bf16 : [M][K] BF16, row stride ldx (elements).
 *   q_e4m3 : [M][K] E4M3 codes (1 byte each), row stride ldq (bytes).
 *   sA     : [K/128][M] FP32, M contiguous: sA[kb*M + m] is the scale of
 *            row m, columns [128*kb, 128*kb + 128).
 * M >= 0 arbitrary; K a multiple of 128 (else FP8BS_ERR_SHAPE).
 * M == 0 or K == 0 is a no-op.
 */
int fp8_quant_act_1x128(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                        void *q_e4m3, int64_t ldq, float *sA, cudaStream_t stream);

/*
 * 128x128 block quantisation of a weight stored as [R][C].
 *   w_bf16 : [R][C] BF16, row stride ldw (elements).
 *   q_e4m3 : [R][C] E4M3 codes, row stride ldq (bytes).
 *   sW     : [ceil(R/128)][C/128] FP32 row-major; sW[rb*(C/128) + cb] is the
 *            scale of rows [128*rb, 128*rb+128) x columns [128*cb, 128*cb+128).
 * R >= 0 arbitrary (a last, shorter row block takes its amax over the rows
 * that exist); C a multiple of 128.
 * For a K-major GEMM weight W[N][K] call it with (R, C) = (N, K).  For a weight
 * stored [K][N] (the MN-major B operand) call it with (R, C) = (K, N).
 */
int fp8_quant_w_128x128(const void *w_bf16, int64_t R, int64_t C, int64_t ldw,
                        void *q_e4m3, int64_t ldq, float *sW, cudaStream_t stream);

/*
 * Both operands of one GEMM quantised in a single launch: the activation x
 * with the 1x128 rule and the weight w with the 128x128 rule.  The pages
 * quantise both inputs of every FP8 GEMM this way before the GEMM runs
 * ("DeepSeek-V3 Technical Report digest", section 3, fine-grained
 * quantisation: 1x128 tiles for activations, 128x128 blocks for weights).
 * The outputs are exactly those of fp8_quant_act_1x128(x, M, K, ...) and
 * fp8_quant_w_128x128(w, R, C, ...), bit for bit, and every argument has the
 * same meaning, layout, checks and error codes as in those two calls.  One
 * kernel walks both operands' 32 KiB units through one TMA ring, which keeps
 * the small activation pass from running as a second kernel beside the
 * weight pass.  Either operand may be empty (M == 0 or K == 0; R == 0 or
 * C == 0).  Nothing is launched when an argument is rejected.
 */
int fp8_quant_act_w(const void *x_bf16, int64_t M, int64_t K, int64_t ldx, void *qa_e4m3, int64_t ldqa, float *sA,
                    const void *w_bf16, int64_t R, int64_t C, int64_t ldw, void *qw_e4m3, int64_t ldqw, float *sW,
                    cudaStream_t stream);

/*
 * Block-scaled FP8 GEMM:  C[m][n] = sum_kb  sA[kb][m] * sB(n, kb) *
 *                                   sum_{k in kb} qA[m][k] * qB(n, k)
 * with each 128-wide K slice's FP8 product formed on the tensor cores in FP32
 * and promoted into an FP32 accumulator with its two scales applied.
 *   qA, sA : as written by fp8_quant_act_1x128 ([M][K], ld = K; [K/128][M]).
 *   b_major == FP8BS_B_KMAJOR : qB is [N][K] (ld = K), sB [ceil(N/128)][K/128]
 *                               (fp8_quant_w_128x128 with R = N, C = K).
 *   b_major == FP8BS_B_MNMAJOR: qB is stored [K][N] (ld = N), sB [K/128][N/128]
 *                               (fp8_quant_w_128x128 with R = K, C = N);
 *                               this is the data-gradient form dX = dY . W for
 *                               a weight kept as [K][N].  N % 128 == 0 required
 *                               (the weight quantiser's column rule).
 *   C      : [M][N], row stride ldc >= N (elements), BF16 (round to nearest
 *            even) or FP32 by c_dtype.  C needs only element alignment; a
 *            16-byte aligned base and row stride enable vector stores.
 * M, N >= 0 arbitrary (partial tiles are masked); K a multiple of 128.
 * K == 0 writes zeros.  M, N < 2^31.
 */
int fp8_gemm_blockscaled(const void *qA, const float *sA, const void *qB, const float *sB,
                         int64_t M, int64_t N, int64_t K, int b_major,
                         void *C, int c_dtype, int64_t ldc, cudaStream_t stream);

/*
 * Block-scaled GEMM with a quantised output: the same C = A . B^T (same
 * arguments, same arithmetic, same BF16 rounding of each output element), but
 * the epilogue quantises every 1x128 tile of each output row with the
 * activation rule of fp8_quant_act_1x128 -- amax over the tile's BF16 values,
 * scale = fp32(amax / 448), code = E4M3_RNE_sat(fp32(c / scale)) -- and
 * writes codes and scales instead of BF16.  The pages store activations and
 * pass them between devices in low-precision formats ("DeepSeek-V3 training
 * walkthrough", section 二(四), last item; qqstock.cn walkthrough, FP8
 * section, low-precision storage and communication, report figure 10); this
 * call produces that FP8 form without a BF16 round trip through HBM.  The
 * result is bit-identical to
 * fp8_gemm_blockscaled (BF16 out) followed by fp8_quant_act_1x128.
 *   qC : [M][N] E4M3 codes, row stride ldqc BYTES (>= N, multiple of 16;
 *        base 16-byte aligned).
 *   sC : [N/128][M] FP32: sC[nb*M + m] is the scale of row m, columns
 *        [128*nb, 128*nb + 128) -- the layout fp8_quant_act_1x128 gives sA.
 * N must be a multiple of 128 (else FP8BS_ERR_SHAPE).  K == 0 writes zero
 * codes and zero scales.  Other rules and errors as fp8_gemm_blockscaled.
 */
int fp8_gemm_blockscaled_e4m3_out(const void *qA, const float *sA, const void *qB, const float *sB,
                                  int64_t M, int64_t N, int64_t K, int b_major, void *qC, int64_t ldqc,
                                  float *sC, cudaStream_t stream);

/*
 * Gather + 1x128 activation quantisation, for routed-expert dispatch: output
 * row i is the 1x128 quantisation of input row rows[i].  The pages dispatch
 * activations to experts in FP8 ("DeepSeek-V3 training walkthrough", section
 * 二(四), last item; qqstock.cn walkthrough, FP8 section, report figure 10);
 * since quantising then gathering rows equals gathering then quantising, the
 * result is bit-identical to fp8_quant_act_1x128 of the gathered BF16 matrix
 * x[rows], which is never materialised.
 *   x_bf16 : [T][K] BF16 token rows, row stride ldx (elements).
 *   rows   : [M] int32 on the device, each in [0, T).
 *   q_e4m3 : [M][K] E4M3, row stride ldq (bytes); sA : [K/128][M] FP32.
 * K a multiple of 128.  An index outside [0, T) produces zero codes and zero
 * scales for that row and makes the next fp8bs_last_error report
 * FP8BS_ERR_INDEX.  Alignment rules as fp8_quant_act_1x128 (rows 4-byte
 * aligned).
 */
int fp8_quant_act_1x128_gather(const void *x_bf16, int64_t T, int64_t K, int64_t ldx, const int32_t *rows,
                               int64_t M, void *q_e4m3, int64_t ldq, float *sA, cudaStream_t stream);

/*
 * Scatter + 1x128 activation quantisation: the expert dispatch written from
 * the token side.  Token row t is quantised ONCE and its codes and scales are
 * written to each of its topk destination rows: output row dest[t*topk + j]
 * (j < topk) is the 1x128 quantisation of x row t.  The pages quantise
 * activations to FP8 before dispatching them to the routed experts
 * ("DeepSeek-V3 training walkthrough", section 二(四), last item; qqstock.cn
 * walkthrough, FP8 section, report figure 10), so every routed copy of a
 * token carries the same bytes; this call produces them with one read and
 * one encoding per token instead of one per copy, and its output equals
 * fp8_quant_act_1x128_gather with rows[dest[t*topk + j]] = t, bit for bit.
 *   x_bf16 : [T][K] BF16 token rows, row stride ldx (elements).
 *   dest   : [T][topk] int32 on the device; 1 <= topk <= 32.
 *   q_e4m3 : [M][K] E4M3, row stride ldq (bytes); sA : [K/128][M] FP32.
 * Output rows that no dest entry names are not written.  A destination
 * outside [0, M) is skipped and makes the next fp8bs_last_error report
 * FP8BS_ERR_INDEX; a row named by two entries receives one of the two tokens.
 * Alignment rules as fp8_quant_act_1x128 (dest 4-byte aligned).
 */
int fp8_quant_act_1x128_scatter(const void *x_bf16, int64_t T, int64_t K, int64_t ldx, const int32_t *dest, int topk,
                                int64_t M, void *q_e4m3, int64_t ldq, float *sA, cudaStream_t stream);

/*
 * Expert-parallel dispatch, sending side: the routed copies of token rows,
 * gathered and quantised per 1x128 tile exactly as
 * fp8_quant_act_1x128_gather does, but each output row PACKED with its own
 * scales so that one all-to-all moves a routed row in FP8 together with the
 * FP32 scales it needs.  The pages dispatch activations to the experts on
 * other devices in FP8 over an all-to-all ("DeepSeek-V3 training
 * walkthrough", section 二, cross-node all-to-all / expert parallelism, and
 * section 二(四), last item: activations cached and dispatched in FP8;
 * qqstock.cn walkthrough, FP8 section, report figure 10).
 *   x_bf16 : [T][K] BF16 token rows, row stride ldx (elements).
 *   rows   : [M] int32 on the device: the token row of each routed copy, in
 *            send order.
 *   packed : [M] rows of ld_packed bytes: bytes [0, K) are row i's E4M3
 *            codes, bytes [K, K + 4*K/128) its K/128 FP32 scales (tile kb's
 *            scale at float index kb).  ld_packed >= K + 4*K/128 and a
 *            multiple of 16.
 * Codes and scales equal fp8_quant_act_1x128 of the gathered rows, bit for
 * bit.  Index errors and alignment rules as fp8_quant_act_1x128_gather.
 */
int fp8_ep_dispatch_pack(const void *x_bf16, int64_t T, int64_t K, int64_t ldx, const int32_t *rows, int64_t M,
                         void *packed, int64_t ld_packed, cudaStream_t stream);

/*
 * The sending side of the expert-parallel dispatch in scatter form: token row
 * t is quantised once (1x128 tiles) and its codes and scales are packed into
 * each of its topk send rows dest[t*topk + j], in the fp8_ep_dispatch_pack
 * layout.  Equal, bit for bit, to fp8_ep_dispatch_pack with rows[dest[t*topk
 * + j]] = t, with one read and one encoding per token instead of one per
 * routed copy (fp8_quant_act_1x128_scatter's rules for dest and its errors).
 */
int fp8_ep_dispatch_pack_scatter(const void *x_bf16, int64_t T, int64_t K, int64_t ldx, const int32_t *dest, int topk,
                                 int64_t M, void *packed, int64_t ld_packed, cudaStream_t stream);

/*
 * Expert-parallel dispatch, receiving side: packed rows (fp8_ep_dispatch_pack
 * layout) as they arrive from the all-to-all, grouped by source rank, are
 * reordered into expert-major order for the grouped GEMM: output row i is
 * packed row perm[i]; its codes go to q_e4m3[i] and its scales to
 * sA[kb][i] (the [K/128][M] layout the GEMMs read).
 *   packed : [n_src] rows, row stride ld_packed bytes.
 *   perm   : [M] int32 on the device, each in [0, n_src).
 *   q_e4m3 : [M][K] E4M3, row stride ldq bytes; sA : [K/128][M] FP32.
 * An index outside [0, n_src) gives a zero row and zero scales and makes the
 * next fp8bs_last_error report FP8BS_ERR_INDEX.  Pure data movement: the
 * output is bit-identical to the packed input.
 */
int fp8_ep_unpack(const void *packed, int64_t n_src, int64_t ld_packed, int64_t K, const int32_t *perm, int64_t M,
                  void *q_e4m3, int64_t ldq, float *sA, cudaStream_t stream);

/*
 * Row gather of byte rows, the data movement of the expert-parallel return
 * path (expert outputs back to their source rank, then into token/slot
 * order): dst row i = src row rows[i], row_bytes bytes each.
 *   src : [n_src] rows, row stride ld_src bytes;  dst : [M] rows, ld_dst.
 *   rows: [M] int32 on the device.
 * row_bytes, ld_src, ld_dst multiples of 16; src and dst 16-byte aligned.
 * An index outside [0, n_src) gives a zero row and FP8BS_ERR_INDEX at the
 * next fp8bs_last_error.
 */
int fp8bs_gather_rows(const void *src, int64_t n_src, int64_t ld_src, const int32_t *rows, int64_t M,
                      int64_t row_bytes, void *dst, int64_t ld_dst, cudaStream_t stream);

/*
 * Token-dimension 1x128 quantisation, for the operands of the weight-gradient
 * GEMM dW = dY^T . X, whose contraction runs over tokens.  The pages run all
 * three GEMM kinds (forward, data gradient, weight gradient) in FP8 with
 * 1x128 tiles for activation-like operands ("DeepSeek-V3 Technical Report
 * digest", section 3, "FP8 operations" and fine-grained quantisation
 * bullets); the tiles of the weight-gradient operands lie along the tokens,
 * so each feature column of the [tokens][features] matrix is cut into runs of
 * 128 tokens, each with its own scale (same amax/448 rule and encoder as
 * fp8_quant_act_1x128), and the codes are written transposed so that the GEMM
 * reads them token-contiguous.
 *   x_bf16 : [T][F] BF16, row stride ldx (elements).
 *   qT     : [F][T] E4M3 codes, row stride ldq (bytes, >= T).
 *   s      : [T/128][F] FP32: s[tb*F + f] is the scale of feature f over
 *            tokens [128*tb, 128*tb + 128).
 * T a multiple of 128 (else FP8BS_ERR_SHAPE); F >= 0 arbitrary.  Alignment
 * rules as fp8_quant_act_1x128.  Equals fp8_quant_act_1x128 of the
 * transposed matrix, bit for bit.
 */
int fp8_quant_tokens_1x128(const void *x_bf16, int64_t T, int64_t F, int64_t ldx, void *qT, int64_t ldq,
                           float *s, cudaStream_t stream);

/*
 * Weight-gradient GEMM: C[M][N] = sum_k A^[m][k] * B^[n][k] where BOTH
 * operands carry one FP32 scale per row and 128-wide K-slice (both produced
 * by fp8_quant_tokens_1x128, K = tokens): each slice's FP32 partial is
 * promoted with sA[kb][m] * sB[kb][n].
 *   qA : [M][K] E4M3 (K contiguous), sA : [K/128][M].
 *   qB : [N][K] E4M3 (K contiguous), sB : [K/128][N].
 *   C  : [M][N] BF16 or FP32 (c_dtype), row stride ldc.
 * For dW = dY^T . X: A = dY quantised along tokens (M = output features),
 * B = X quantised along tokens (N = input features), K = tokens.  Shape,
 * alignment and error rules as fp8_gemm_blockscaled.
 */
int fp8_gemm_wgrad(const void *qA, const float *sA, const void *qB, const float *sB, int64_t M, int64_t N,
                   int64_t K, void *C, int c_dtype, int64_t ldc, cudaStream_t stream);

/*
 * Grouped block-scaled FP8 GEMM for routed experts (one expert per segment of
 * rows).  The pages' MoE layer routes every token to 8 of 256 routed experts,
 * each a separate FFN with its own weights ("DeepSeek-V3 training
 * walkthrough", section 一, DeepSeekMoE item), and runs its GEMMs in FP8 with
 * the same fine-grained tiles; the rows routed to one expert are one segment
 * here.  Rows [seg_offsets[e], seg_offsets[e+1]) of qA belong to expert e:
 *   C[m][n] = sum_kb sA[kb][m] * sB[e][n/128][kb] * sum_{k in kb} qA[m][k] * qB[e][n][k]
 *   qA          : [M_total][K] E4M3, sA [K/128][M_total] (quantise the
 *                 gathered rows, or gather rows and scale columns of a
 *                 quantised token matrix: the two are identical).
 *   qB          : [E][N][K] E4M3 (K contiguous), sB [E][ceil(N/128)][K/128].
 *   seg_offsets : DEVICE int32[E+1], nondecreasing, [0] == 0, [E] == M_total.
 *                 Read on the device only: no host synchronisation.  Offsets
 *                 that break these rules give unspecified output rows (never
 *                 an out-of-bounds access: rows are clamped to [0, M_total)).
 *   C           : [M_total][N], row stride ldc, BF16 or FP32.
 * Segments may be empty.  1 <= E <= FP8BS_MAX_EXPERTS (2048: the per-expert
 * tile table lives in shared memory); any other E returns FP8BS_ERR_ARG.
 */
int fp8_grouped_gemm_blockscaled(const void *qA, const float *sA,
                                 const void *qB, const float *sB,
                                 const int32_t *seg_offsets, int E, int64_t M_total,
                                 int64_t N, int64_t K,
                                 void *C, int c_dtype, int64_t ldc, cudaStream_t stream);

/*
 * Per-tensor FP8 quantisation, the contrast variant: ONE scale for the whole
 * tensor instead of one per 1x128 tile or 128x128 block.  The pages present
 * their fine-grained groups as the alternative to this, because a single
 * outlier sets the scale of every element of the tensor ("qqstock.cn
 * walkthrough", FP8 section: fine-grained rather than per-tensor
 * quantisation; "DeepSeek-V3 Technical Report digest", section 3,
 * fine-grained quantisation bullet).  The rules are the library's rules with
 * the group being the tensor: scale = fp32(amax / 448) over all R x C
 * elements, q = E4M3_RNE_sat(fp32(x / scale)); an all-zero tensor has scale 0
 * and codes 0x00 / 0x80.
 *   x_bf16 : [R][C] BF16, row stride ldx (elements); C a multiple of 128.
 *   q_e4m3 : [R][C] E4M3 codes, row stride ldq (bytes).
 *   scale  : one FP32 on the device.
 *   workspace : device scratch of at least the size that
 *            fp8_quant_per_tensor_workspace_size(R, C) reports (4 bytes per
 *            128x128 unit, plus 4), 4-byte aligned, owned by the caller; its
 *            contents on entry do not matter and on return are unspecified.
 *            Calls that share one workspace must not overlap on the GPU.
 * Three kernels on `stream`: the amax of every 128x128 unit into the
 * workspace, one CTA that reduces them to the tensor's amax and scale, and
 * the encoding pass (which reads the tensor a second time).  R == 0 or
 * C == 0 is a no-op.  A workspace smaller than required: FP8BS_ERR_ARG.
 * Other rules and errors as fp8_quant_w_128x128.
 */
int fp8_quant_per_tensor_workspace_size(int64_t R, int64_t C, int64_t *bytes);
int fp8_quant_per_tensor(const void *x_bf16, int64_t R, int64_t C, int64_t ldx, void *q_e4m3, int64_t ldq,
                         float *scale, void *workspace, int64_t workspace_bytes, cudaStream_t stream);

/*
 * Per-tensor FP8 quantisation with DELAYED scaling: the scale comes from an
 * amax the caller supplies (the usual choice is the largest amax recorded
 * over earlier steps), so the tensor is encoded in one pass while its own
 * amax is recorded for later steps.
 *   amax_in  : one FP32 on the device, finite and >= 0; scale =
 *              fp32(amax_in / 448) is stored in *scale.  Elements with
 *              |x| / scale >= 464 saturate to +-448; amax_in == 0 gives scale 0
 *              and codes E4M3(x).
 *   amax_out : one FP32 on the device (not the same word as amax_in): set to
 *              max |x| over this tensor (the call first zeroes it, on
 *              `stream`).
 * Other arguments, rules and errors as fp8_quant_per_tensor (no workspace).
 */
int fp8_quant_per_tensor_delayed(const void *x_bf16, int64_t R, int64_t C, int64_t ldx, const float *amax_in,
                                 void *q_e4m3, int64_t ldq, float *scale, float *amax_out, cudaStream_t stream);

/*
 * GEMM over per-tensor quantised operands:
 *   C[m][n] = sA * sB * sum_k qA[m][k] * qB(n, k)
 * with the WHOLE K sum accumulated by the tensor cores in their FP32
 * accumulator (no per-128 promotion: with one scale per tensor there is
 * nothing to apply per slice), then multiplied by fp32(sA * sB) and rounded
 * to the output type.  This is the scheme the fine-grained GEMM is compared
 * with.
 *   sA, sB : one FP32 each, on the device (from fp8_quant_per_tensor or
 *            fp8_quant_per_tensor_delayed).
 *   qB     : [N][K] (b_major == FP8BS_B_KMAJOR) or stored [K][N]
 *            (FP8BS_B_MNMAJOR, N a multiple of 16).
 * Other arguments, rules and errors as fp8_gemm_blockscaled.
 */
int fp8_gemm_per_tensor(const void *qA, const float *sA, const void *qB, const float *sB, int64_t M, int64_t N,
                        int64_t K, int b_major, void *C, int c_dtype, int64_t ldc, cudaStream_t stream);

/*
 * fp8_quant_per_tensor without a workspace argument: the same result, bit
 * for bit (same scale, same codes), from the same kernels, with the scratch
 * held by the library itself.  The pages have no counterpart to this call;
 * it exists for callers that cannot allocate device memory around a call --
 * for example code embedded in a host application that owns every device
 * buffer and grants none for scratch, or a serving loop that forbids any
 * allocation once it has started -- and so cannot provide the workspace
 * that fp8_quant_per_tensor needs.  The call itself allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *   Scratch: a fixed array of FP8BS_NOALLOC_MAX_UNITS + 1 32-bit words
 *   (64 KiB) that every GPU which loads the library holds until the process
 *   exits.  A tensor of more than FP8BS_NOALLOC_MAX_UNITS 128x128 units
 *   (ceil(R/128) * C/128) is refused with FP8BS_ERR_SCRATCH before anything
 *   is enqueued.
 *   Set-up: the first call on a device, with that device current, looks up
 *   the array's device address (cudaGetSymbolAddress) and keeps it; make that
 *   first call before any stream capture.
 *   Sharing: every call on a device uses the same array and leaves its
 *   contents there; nothing in it needs to start at zero, because each call
 *   writes every word it later reads.  Calls whose kernels overlap on the GPU
 *   (e.g. on two streams) race on the array and must be serialised by the
 *   caller.
 * Arguments, other rules and errors as fp8_quant_per_tensor.
 */
enum { FP8BS_NOALLOC_MAX_UNITS = 16384 };
int fp8_quant_per_tensor_noalloc(const void *x_bf16, int64_t R, int64_t C, int64_t ldx, void *q_e4m3, int64_t ldq,
                                 float *scale, cudaStream_t stream);

/*
 * Synchronises `stream`, then reports and clears one condition of the current
 * device's error word: FP8BS_OK (no condition), FP8BS_ERR_TIMEOUT (a kernel's
 * pipeline wait exceeded its time limit; that kernel's outputs are
 * incomplete), FP8BS_ERR_INDEX (a gather index was out of range), or
 * FP8BS_ERR_LAUNCH (the CUDA runtime reported an error for the stream).
 * When both device conditions are set, the time-out is reported and cleared
 * first and the index error stays set for the next call.
 * The error word is ONE word per device, shared by every stream and every
 * caller in the process: a condition raised by a kernel on another stream is
 * reported (and cleared) by whichever call reads it first.  Only `stream` is
 * synchronised, so kernels still running on other streams may set a bit
 * after this call returns.
 */
int fp8bs_last_error(cudaStream_t stream);

/*
 * Self-test of the failure detection (no counterpart in the pages: it checks
 * the library's own device-side time-out machinery).  Enqueues on `stream`
 * one single-CTA kernel that waits, through the same bounded mbarrier wait
 * that every pipeline of the library uses, on a barrier that nothing ever
 * signals, with a limit of `limit_us` microseconds.  The wait runs out, the
 * kernel records the time-out in the device error word and returns; the
 * next fp8bs_last_error(stream) reports FP8BS_ERR_TIMEOUT and clears it, and
 * the CUDA context stays usable.  No memory is read or written besides the
 * error word.
 * Returns FP8BS_OK (enqueued), FP8BS_ERR_ARG (limit_us outside
 * [1, 1000000]), FP8BS_ERR_DEVICE or FP8BS_ERR_LAUNCH.
 */
int fp8bs_selftest_wait_timeout(int64_t limit_us, cudaStream_t stream);

/*
 * Test hook for the abort paths of the real kernels (no counterpart in the
 * pages).  Sets the time limit, in nanoseconds, of every pipeline wait of the
 * kernels launched AFTER this call by the quantisers (fp8_quant_act_1x128,
 * fp8_quant_w_128x128, fp8_quant_act_w, fp8_quant_tokens_1x128) and by the
 * single-CTA GEMMs (fp8_gemm_blockscaled / _e4m3_out / fp8_gemm_wgrad with
 * M <= 128, and fp8_grouped_gemm_blockscaled).  CTA-pair GEMMs (M > 128)
 * always keep the default limit.  limit_ns == 0 restores the default (2 s).
 * With a limit of a few microseconds a wait that has to wait for memory runs
 * out: the kernel records FP8BS_ERR_TIMEOUT, drains its own copies and
 * MMAs, frees its tensor memory and returns; its outputs are incomplete but
 * nothing outside them is written.  The setting is process-wide and not
 * meant for concurrent use.  Returns FP8BS_OK, or FP8BS_ERR_ARG for a limit
 * outside [0, 2e9].
 */
int fp8bs_selftest_set_wait_limit(int64_t limit_ns);

/*
 * Test hook for the E4M3 encoder (the pages fix no FP8 format; the reading
 * taken is OCP E4M3 "FN", round to nearest even, saturating to +-448).
 * q[i] = the code of the fp32 value whose bit pattern is first_bits + i,
 * for i in [0, n), formed by the same conversion instruction every quantiser
 * of the library encodes with (cvt.rn.satfinite.e4m3x2.f32), so that a test
 * can compare it with an independent encoder over every fp32 pattern.
 *   q : [n] bytes on the device.
 * n >= 0 and first_bits + n <= 2^32 (else FP8BS_ERR_ARG); non-finite
 * patterns are converted too (their codes are the hardware's, not part of
 * the library's contract).  Asynchronous on `stream`; returns FP8BS_OK,
 * FP8BS_ERR_NULL, FP8BS_ERR_DEVICE or FP8BS_ERR_LAUNCH.
 */
int fp8bs_selftest_encode_e4m3(uint32_t first_bits, int64_t n, uint8_t *q, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
