/*
 * fp8bs.h -- C ABI of the GB300 (sm_103a) FP8 linear-layer library.
 *
 * The method: the FP8 linear layer of block-scaled FP8 training.  Linear
 * layers run their products in FP8 while attention, normalisation and
 * non-linear layers stay in bf16; weights are block-quantized to E4M3 with
 * 128x128 tiles and activations with 1x128 tiles ("NVIDIA NeMo RL logra una
 * aceleracion del 48%...", hotbookzone.com, section "El avance tecnico").
 * E4M3 (up to +-448) carries forward activations and weights and E5M2 the
 * gradients; per-tensor delayed scaling takes the scale from the amax history
 * of earlier iterations ("Infraestructura de Entrenamiento FP8", introl.com,
 * sections "El panorama de la precision numerica" and "Transformer Engine: la
 * base de software").
 *
 * Conventions (all entry points):
 *   - Every pointer is a DEVICE pointer unless stated otherwise.  The caller
 *     allocates and owns every buffer; the library never allocates device
 *     memory, frees it or keeps a pointer after the call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  A return value other than FP8BS_OK means nothing was
 *     launched; fp8bs_last_error() then describes the problem.
 *   - bf16 inputs are raw bf16 bit patterns (2 bytes per element).
 *   - FP8 data are raw 8-bit codes.  E4M3 is the "FN" variant (no infinities,
 *     max 448, NaN = S.1111.111); E5M2 has IEEE infinities, max 57344.
 *   - Scales are DEQUANTIZATION multipliers: value = decode(code) * scale.
 *   - Encoding rounds to nearest, ties to even, and saturates finite overflow
 *     and infinities to +-max; the element computed is fp32(x * fp32(1/s)).
 *   - Alignment: data pointers 16-byte aligned, leading dimensions (in
 *     bytes) multiples of 16; otherwise FP8BS_ERR_MISALIGNED.
 *   - Contraction lengths (columns of a quantized matrix, K of a product) must
 *     be multiples of 128; otherwise FP8BS_ERR_UNSUPPORTED.  Empty inputs
 *     (a zero dimension) are valid and launch nothing, except a product with
 *     K == 0, which writes zeros to Y.
 *   - Device-side waits are bounded; a kernel that gives up records it in a
 *     status word (one per process and device, shared by all streams) read
 *     by fp8bs_device_status().
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fp8bs_stream_t;   /* same type as cudaStream_t */

enum fp8bs_status {
    FP8BS_OK = 0,
    FP8BS_ERR_INVALID_ARG = -1,     /* null pointer, bad enum, bad size */
    FP8BS_ERR_UNSUPPORTED = -2,     /* valid request this library does not run */
    FP8BS_ERR_MISALIGNED = -3,      /* pointer or leading dimension alignment */
    FP8BS_ERR_CUDA = -4,            /* CUDA runtime/driver error (message kept) */
    FP8BS_ERR_DEVICE_TIMEOUT = -5   /* a bounded device-side wait expired */
};

enum fp8bs_format { FP8BS_E4M3 = 0, FP8BS_E5M2 = 1 };
enum fp8bs_scale_mode { FP8BS_SCALE_FP32 = 0, FP8BS_SCALE_POW2 = 1 };
enum fp8bs_out_dtype { FP8BS_OUT_F32 = 0, FP8BS_OUT_BF16 = 1 };
enum fp8bs_granularity { FP8BS_GRAN_1x128 = 0, FP8BS_GRAN_128x128 = 1, FP8BS_GRAN_TENSOR = 2,
                         FP8BS_GRAN_1x32 = 3 /* MXFP8 */ };
enum fp8bs_epilogue { FP8BS_EPI_NONE = 0, FP8BS_EPI_SWIGLU = 1 };

/* ------------------------------------------------------------ quantizers */

/*
 * Activation quantizer, one scale per 1x128 tile ("1x128" granularity for
 * activations, hotbookzone.com "El avance tecnico").
 *   x      [rows][ld_x] bf16, the 128-element tiles run along each row.
 *   q      [rows][ld_q] 8-bit codes (output).
 *   scales [cols/128][rows] fp32, rows contiguous (output).
 * Per tile: amax = max|x|; s = amax/fmax in fp32 (mode FP32; amax == 0 gives
 * 1, floor 2^-126) or the smallest power of two 2^e, e in [-126, 127], with
 * amax <= fmax * 2^e (mode POW2; the power-of-two option of hotbookzone.com
 * "Por que esto es importante..."); q = enc(x * (1/s)).
 * fmt selects E4M3 (fmax 448) or E5M2 (fmax 57344).
 * Errors: INVALID_ARG (nulls, rows/cols < 0, ld < cols, bad enum),
 * UNSUPPORTED (cols % 128), MISALIGNED (x, q not 16-byte aligned, ld_x*2 or
 * ld_q not a multiple of 16, scales not 4-byte aligned).
 */
int fp8_quantize_1x128(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                       int32_t fmt, int32_t mode,
                       uint8_t* q, int64_t ld_q, float* scales, fp8bs_stream_t stream);

/*
 * Weight quantizer, one scale per 128x128 tile ("128x128" granularity for
 * weights, hotbookzone.com "El avance tecnico").  Weights are re-quantized
 * after every optimizer step ("Ganancias de rendimiento en el mundo real").
 *   w      [rows][ld_w] bf16;  q [rows][ld_q] codes (output);
 *   scales [ceil(rows/128)][cols/128] fp32 (output).
 * A last row-tile with fewer than 128 rows covers only the rows that exist.
 * Scale and element rules as fp8_quantize_1x128, over the whole tile.
 * Errors as fp8_quantize_1x128.
 */
int fp8_quantize_128x128(const void* w, int64_t rows, int64_t cols, int64_t ld_w,
                         int32_t fmt, int32_t mode,
                         uint8_t* q, int64_t ld_q, float* scales, fp8bs_stream_t stream);

/*
 * Both FP8 operands of one linear layer in one call: X [m][k] quantized
 * exactly as fp8_quantize_1x128 does (codes qx [m][ld_qx], scales sx
 * [k/128][m]) and W [n][k] exactly as fp8_quantize_128x128 does (codes qw
 * [n][ld_qw], scales sw [ceil(n/128)][k/128]), with the same fmt and mode.
 * The results equal the two separate calls bit for bit.  The weight half is
 * launched as a programmatic dependent of the activation half, so it runs
 * alongside that grid's last wave instead of after it (part of the
 * quantization overhead the NeMo RL page counts against the FP8 linear
 * layer, hotbookzone.com "Ganancias de rendimiento en el mundo real"); work
 * queued after this call on the stream still starts only once both are done.
 * The outputs must not overlap the inputs.  Either operand may be empty (m
 * or n == 0: its pointers are not read).
 * Errors: those of fp8_quantize_1x128 for X and of fp8_quantize_128x128 for W.
 */
int fp8_quantize_linear(const void* x, int64_t m, int64_t ld_x, uint8_t* qx, int64_t ld_qx, float* sx,
                        const void* w, int64_t n, int64_t ld_w, uint8_t* qw, int64_t ld_qw, float* sw,
                        int64_t k, int32_t fmt, int32_t mode, fp8bs_stream_t stream);

/*
 * MXFP8 (microscaling FP8) quantizer: one power-of-two scale per 32
 * consecutive elements of a row.  The introl page names MXFP8 as Blackwell's
 * hardware block scaling ("Requisitos de hardware para entrenamiento FP8";
 * "Escalado por bloque (MXFP8)" in "Estrategias de escalado y estabilidad";
 * "Blackwell MXFP8 y NVFP4") without the block size or the scale rule; this
 * follows the open microscaling format the name refers to:
 *   per 32-element block: e = floor(log2(amax)) - Emax (Emax = 8 for E4M3,
 *   15 for E5M2), clamped to [-127, 127] (amax == 0 or subnormal: -127);
 *   code = e + 127 (E8M0); elements q = enc(x * 2^-e), rounded to nearest
 *   even and saturated (the block maximum lies in [2^Emax, 2^(Emax+1)) and
 *   may saturate); a non-finite amax gives code 255 (NaN) and NaN elements.
 *   x      [rows][ld_x] bf16;  q [rows][ld_q] codes (output);
 *   scales [cols/128][rows][4] uint8 codes (output): byte j of entry
 *          (kb, r) is the scale of columns 128 kb + 32 j .. 128 kb + 32 j + 31
 *          -- one 32-bit word per (128-column block, row), the rows of a
 *          block contiguous, as the block-scaled product reads them.
 * Errors as fp8_quantize_1x128 (scales 4-byte aligned).
 */
int fp8_quantize_mx(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int32_t fmt,
                    uint8_t* q, int64_t ld_q, uint8_t* scales, fp8bs_stream_t stream);

/*
 * Column-wise 1x128 quantizer for the backward products.  The block recipe
 * ("El avance tecnico": 1x128 activation tiles) applied to products that
 * contract over the token dimension (wgrad dW = dY^T X) needs tiles of 128
 * consecutive ROWS of one column of dY and of X.  This call quantizes x with
 * such 128x1 tiles and writes the result transposed, so the product reads a
 * K-major operand with the ordinary 1x128 layout; from the same read of x it
 * can also write the row-wise 1x128 copy (dY's dgrad operand, or X's
 * forward operand).
 *   x        [rows][ld_x] bf16.
 *   qt       [cols][ld_qt] codes: qt[c][r] = enc(x[r][c] * (1/st)), st the
 *            scale of tile (r/128, c) -- the fp8_quantize_1x128 rules
 *            applied to x^T.
 *   scales_t [rows/128][cols] fp32 (the 1x128 table of the [cols][rows]
 *            operand qt).
 *   q, scales: the row-wise copy exactly as fp8_quantize_1x128 writes it
 *            (ld_q), or both NULL to skip it.
 * Errors: INVALID_ARG (nulls, one of q/scales null, ld too small, bad enum),
 * UNSUPPORTED (rows % 128 or cols % 128), MISALIGNED (x, qt, q 16-byte
 * aligned with 16-byte row pitches, scale tables 4-byte aligned).
 */
int fp8_quantize_1x128_colwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                               int32_t fmt, int32_t mode,
                               uint8_t* qt, int64_t ld_qt, float* scales_t,
                               uint8_t* q, int64_t ld_q, float* scales, fp8bs_stream_t stream);

/*
 * Per-tensor delayed-scaling quantizer ("Escalado diferido", introl.com
 * "Estrategias de escalado y estabilidad"; recipe of "Transformer Engine: la
 * base de software").  Quantizes with the scale already in use, built from
 * earlier steps only, and measures this step's amax for the history:
 *   q[i] = enc(x[i] * fp32(1 / *scale));  *amax_out = max_i |x[i]|.
 *   x        [numel] bf16, contiguous;  q [numel] codes (output);
 *   scale    device scalar, the dequantization scale in use (read);
 *   amax_out device scalar (written, not accumulated).
 * The hybrid recipe uses fmt E5M2 for gradients and E4M3 for activations
 * and weights.  Errors: INVALID_ARG, MISALIGNED (x, q 16-byte aligned).
 */
int fp8_quantize_tensor_delayed(const void* x, int64_t numel, int32_t fmt,
                                const float* scale, uint8_t* q, float* amax_out,
                                fp8bs_stream_t stream);

/*
 * Delayed-scaling state update (fields margin, amax_history_len and
 * amax_compute_algo = "max" of the recipe on introl.com "Transformer Engine:
 * la base de software"):
 *   history[*head] = *amax; *head = (*head + 1) % history_len;
 *   amax_h = max(history[0..history_len));
 *   t = fp32(fp32(amax_h / fmax) * 2^margin);
 *   if amax_h > 0 and t is finite: *scale = max(t, 2^-126), else unchanged.
 *   history [history_len] fp32, head int32 scalar, scale fp32 scalar: all
 *   device memory, read and written in place; amax: device scalar (read).
 * A fresh state is history = 0, head = 0, scale = 1.
 * Errors: INVALID_ARG (nulls, history_len < 1, margin outside [-126, 126]).
 */
int fp8_amax_history_update(float* history, int32_t* head, int32_t history_len,
                            const float* amax, int32_t fmt, int32_t margin,
                            float* scale, fp8bs_stream_t stream);

/* ---------------------------------------------------------------- GEMM */

/*
 * One FP8 operand of Y = deq(A) . deq(B)^T.  Logical shape [rows][K]
 * (rows = M for A, N for B).
 *   transposed = 0: stored [rows][ld], K contiguous ("K-major").
 *   transposed = 1: stored [K][ld], rows contiguous ("MN-major"), as in the
 *                   backward products (dgrad reads W and wgrad reads dY and X
 *                   across their stored rows).
 * Scale tables (fp32), in the orientation of the stored matrix:
 *   GRAN_1x128   (transposed = 0 only): [K/128][rows].  On B (one scale per
 *                128 K-elements of each column of the product) it is the
 *                wgrad operand of the block recipe's backward pass (see
 *                fp8_quantize_1x128_colwise); not in grouped products, only
 *                with a non-transposed A and a float output (fp8_block_gemm),
 *                with 16-byte aligned scale tables, and, for a 1x128 A, rows
 *                of A a multiple of 4.
 *   GRAN_128x128, transposed = 0: [ceil(rows/128)][K/128]
 *   GRAN_128x128, transposed = 1: [K/128][ceil(rows/128)]
 *   GRAN_TENSOR: one value.
 */
/*   GRAN_1x32 (MXFP8; transposed = 0, both operands, not grouped): the
 *                uint8 table of fp8_quantize_mx, [K/128][rows][4] codes,
 *                passed through the `scales` pointer (cast); the tensor core
 *                applies each 32-element block's scale.  A's table needs
 *                rows % 4 == 0 and 16-byte alignment. */
typedef struct {
    const uint8_t* data;
    int64_t ld;            /* elements (= bytes) between stored rows */
    int32_t transposed;
    int32_t fmt;           /* fp8bs_format */
    int32_t gran;          /* fp8bs_granularity */
    int32_t reserved;      /* must be 0 */
    const float* scales;
} fp8bs_operand;

/*
 * Block-scaled FP8 product with fp32 accumulation (the FP8 linear layer's
 * product, hotbookzone.com "El avance tecnico"):
 *   Y[m][n] = sum_k decode(A[m][k]) sA(m,k) * decode(B[n][k]) sB(n,k)
 * fprop: A = Xq (1x128), B = Wq (128x128).  dgrad: A = dYq, B = Wq stored
 * transposed.  wgrad: A = dYq^T, B = Xq^T, both stored transposed.
 * A and B may use different formats (E5M2 gradients x E4M3 weights).
 * Partial products of each 128-long K block are accumulated in fp32 and
 * promoted with that block's two scales into an fp32 accumulator.
 *   mode = POW2 declares that every BLOCK scale (GRAN_1x128, GRAN_128x128)
 *   is an exact power of two in [2^-126, 2^127] (from the POW2 quantizers);
 *   the result is the same sum.  The library cannot check this on the host;
 *   other block scales under POW2 give a wrong result.  A per-tensor scale
 *   (GRAN_TENSOR, e.g. a delayed-scaling scale) may be any fp32 value in
 *   either mode.
 *   Y [M][ld_y], fp32 or bf16 (round to nearest even), written, not
 *   accumulated.
 * Errors: INVALID_ARG, UNSUPPORTED (K % 128, N % 8, GRAN_1x128 on a
 * transposed operand, GRAN_1x128 B with a transposed A), MISALIGNED (data 16-byte aligned, ld % 16, Y 16-byte
 * aligned with ld_y * element size a multiple of 16).
 */
int fp8_block_gemm(int64_t M, int64_t N, int64_t K,
                   const fp8bs_operand* A, const fp8bs_operand* B,
                   int32_t mode, void* Y, int64_t ld_y, int32_t out_dtype,
                   fp8bs_stream_t stream);

/*
 * Grouped product for mixture-of-experts expert GEMMs (the FP8 recipe on a
 * mixture-of-experts model, hotbookzone.com "Ganancias de rendimiento en el
 * mundo real"): for each group g the rows [row_offsets[g], row_offsets[g+1])
 * of A are multiplied by expert g's weights.
 *   row_offsets     device int32 [num_groups + 1], non-decreasing,
 *                   row_offsets[0] = 0, row_offsets[G] <= a_rows.  Entries
 *                   are clamped into [0, a_rows], so no tile writes outside
 *                   Y; a table that decreases (after clamping) makes the
 *                   kernel write nothing and record FP8BS_ERR_INVALID_ARG for
 *                   fp8bs_device_status() -- it lives in device memory, so
 *                   the host cannot check it before the launch.
 *   a_rows          rows of A as stored (its 1x128 scale table is
 *                   [K/128][a_rows]); sizes the launch on the host.
 *   A               [a_rows][K], transposed = 0, GRAN_1x128 or GRAN_TENSOR.
 *   B               [G][N][K] stored as one [G*N][ld] matrix, transposed = 0,
 *                   GRAN_128x128 (scales [G][ceil(N/128)][K/128]) or
 *                   GRAN_TENSOR (one value for all groups).
 *   Y               [a_rows][ld_y]; rows outside every group are not written
 *                   (K == 0: every row of Y is zeroed).
 * Errors as fp8_block_gemm; num_groups in [1, 1024].
 */
int fp8_grouped_block_gemm(int32_t num_groups, const int32_t* row_offsets, int64_t a_rows,
                           int64_t N, int64_t K,
                           const fp8bs_operand* A, const fp8bs_operand* B,
                           int32_t mode, void* Y, int64_t ld_y, int32_t out_dtype,
                           fp8bs_stream_t stream);

/*
 * Product with a quantized output: the GEMM epilogue emits the next linear
 * layer's FP8 activation operand directly, with no float round trip through
 * memory and no separate quantization pass (the quantization-kernel overhead
 * that hotbookzone.com "Ganancias de rendimiento en el mundo real" names as
 * part of the gap between the theoretical 2x and the 15-25 % measured on
 * linear layers).
 *   epilogue = FP8BS_EPI_NONE:   Z = Y (as fp8_block_gemm computes it, fp32).
 *   epilogue = FP8BS_EPI_SWIGLU: B's rows [0, N/2) are gate rows and
 *     [N/2, N) the matching up rows; Z[m][j] = silu(Y[m][j]) * Y[m][N/2 + j]
 *     with silu(g) = g / (1 + e^-g), evaluated in fp32 (the non-linear
 *     function stays out of FP8 math, as "El avance tecnico" keeps
 *     non-linear layers in higher precision); Z has N/2 columns.
 * Z is then quantized exactly as fp8_quantize_1x128 quantizes its input,
 * with the fp32 values of Z in place of bf16 ones:
 *   Q        [M][ld_q] codes of Z (format q_fmt), Z's columns;
 *   q_scales [cols(Z)/128][M] fp32 (scale mode q_mode): the 1x128 operand
 *            layout, ready to be the A operand of the next product.
 * The fp32 values of Z are those of the float-output product (same
 * accumulation), so they match the exact sum within fp8_block_gemm's
 * tolerance; codes and scales follow from those values.
 * K == 0: Q = 0 and every scale 1.
 * Errors as fp8_block_gemm, plus UNSUPPORTED (N % 128, or N % 256 with
 * SwiGLU; SwiGLU with a transposed operand), INVALID_ARG (bad epilogue,
 * q_fmt or q_mode, null Q or q_scales), MISALIGNED (Q 16-byte aligned,
 * ld_q % 16, q_scales 4-byte aligned).
 */
int fp8_block_gemm_quant(int64_t M, int64_t N, int64_t K,
                         const fp8bs_operand* A, const fp8bs_operand* B, int32_t mode,
                         int32_t epilogue, int32_t q_fmt, int32_t q_mode,
                         uint8_t* Q, int64_t ld_q, float* q_scales, fp8bs_stream_t stream);

/*
 * Grouped form of fp8_block_gemm_quant (mixture-of-experts expert layers:
 * the gate/up product with SwiGLU feeds the down product's FP8 operand).
 * Operands, groups and offsets as fp8_grouped_block_gemm; with SwiGLU each
 * expert's B block [N][K] holds its N/2 gate rows then its N/2 up rows.
 *   Q [a_rows][ld_q], q_scales [cols(Z)/128][a_rows]; rows outside every
 *   group are not written (K == 0: every row is written, Q = 0, scales 1).
 * Errors as fp8_block_gemm_quant and fp8_grouped_block_gemm.
 */
int fp8_grouped_block_gemm_quant(int32_t num_groups, const int32_t* row_offsets, int64_t a_rows,
                                 int64_t N, int64_t K,
                                 const fp8bs_operand* A, const fp8bs_operand* B, int32_t mode,
                                 int32_t epilogue, int32_t q_fmt, int32_t q_mode,
                                 uint8_t* Q, int64_t ld_q, float* q_scales, fp8bs_stream_t stream);

/* ----------------------------------------------------------- attention */

/* One FP8 input of the attention: codes [rows][ld], head h (of its heads) at
 * columns 128 h .. 128 h + 127, with its scale table. */
typedef struct {
    const uint8_t* data;
    int64_t ld;            /* bytes between rows (tokens) */
    int32_t fmt;           /* fp8bs_format */
    int32_t reserved;      /* must be 0 */
    const float* scales;
} fp8bs_attn_input;

/*
 * FP8 attention over an FP8 KV cache, forward, one sequence ("NVIDIA NeMo RL
 * logra una aceleracion del 48%...", hotbookzone.com, "Ganancias de
 * rendimiento en el mundo real": FP8 extended to the KV cache and the
 * attention operations).  Both products run on the FP8 tensor cores:
 *   S = scale * deq(Q_h) deq(K_g)^T, masked (causal: key j visible to query
 *       i iff j <= i + seq_k - seq_q), g = h / (heads_q / heads_kv);
 *   P = exp(S - running row max) in fp32; P times (its key tile's V scale /
 *       the largest V tile scale of head g), at most 1, quantized to E4M3
 *       with the scale 1/448; row sums l from the unrounded, unscaled values;
 *   O = (P deq(V_g)) / l, accumulated in fp32 in the unit of that largest V
 *       scale, stored as bf16.
 * Scales (readings; the pages give none): Q one per token and head, as the
 * 1x128 activation tiles -- fp8_quantize_1x128 of the [seq_q][heads_q * 128]
 * matrix, table [heads_q][seq_q]; K and V (the KV cache) one per 128 tokens
 * and head, as the 128x128 tiles -- fp8_quantize_128x128 of the
 * [seq_k][heads_kv * 128] matrices, tables [ceil(seq_k/128)][heads_kv].
 *   O: bf16 [seq_q][ld_o], head h at columns 128 h.  Rows that see no key
 *   are 0.  softmax_scale > 0 (typically 1/sqrt(128)).
 * Errors: INVALID_ARG (sizes, heads_q % heads_kv, nulls, bad format),
 * UNSUPPORTED (head_dim != 128), MISALIGNED (data and O 16-byte aligned,
 * ld % 16 bytes, scales 4-byte aligned).
 */
int fp8_attention_fwd(int64_t seq_q, int64_t seq_k, int32_t heads_q, int32_t heads_kv, int32_t head_dim,
                      int32_t causal, float softmax_scale, const fp8bs_attn_input* Q,
                      const fp8bs_attn_input* K, const fp8bs_attn_input* V, void* O, int64_t ld_o,
                      fp8bs_stream_t stream);

/* ------------------------------------------------------------ diagnostics */

/* Message for the last non-OK status returned on the calling host thread. */
const char* fp8bs_last_error(void);

/* Synchronizes `stream`, then reads and clears the library's device status
 * word: FP8BS_ERR_INVALID_ARG if a grouped product found its row_offsets
 * decreasing (it then wrote nothing), FP8BS_ERR_DEVICE_TIMEOUT if a kernel
 * gave up on a bounded wait, FP8BS_ERR_CUDA on a CUDA error, else FP8BS_OK.
 * The status word is one per process and device, shared by every stream:
 * it covers the kernels of all streams since the previous call, and it is
 * only complete once every stream that ran this library's kernels has been
 * synchronized (this call synchronizes `stream` alone). */
int fp8bs_device_status(fp8bs_stream_t stream);

/* Self-test of the device-side failure detection: launches one thread that
 * waits, with the same bounded mbarrier wait the GEMM roles use, on a barrier
 * nothing arrives at, giving up after `limit_ms` (1..10000).  It then records
 * FP8BS_ERR_DEVICE_TIMEOUT exactly as a stalled GEMM would, writes 0 to the
 * device int *waited_ok (1 if the wait had completed) and returns; the CUDA
 * context stays usable.  fp8bs_device_status() afterwards reports the timeout.
 * Errors: INVALID_ARG (null output, limit out of range). */
int fp8bs_selftest_wait_timeout(int32_t limit_ms, int32_t* waited_ok, fp8bs_stream_t stream);

/* Library version, for the binding's load check. */
int fp8bs_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FP8BS_H */
