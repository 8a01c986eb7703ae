/*
 * fp8_oracle.c -- plain, slow CPU oracle for the FP8 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path (the CUDA library
 * and its Python binding) may include, link or call this file; only the
 * test-suite, the smoke check and the CPU-baseline leg of the benchmark do.
 * It shares no code, header, table or constant generator with the CUDA path.
 *
 * What it follows (the method is described in three web pages on FP8
 * training; the pages give the formats and the recipe, not the arithmetic):
 *   - "Infraestructura de Entrenamiento FP8" (introl.com), section
 *     "El panorama de la precision numerica": E4M3 for activations and
 *     weights with values up to +-448, E5M2 for gradients.
 *   - same page, "Transformer Engine: la base de software": the delayed
 *     scaling recipe (margin, amax history length, "max" over the history,
 *     HYBRID = E4M3 forward / E5M2 backward) and the statement that the
 *     scale comes from the maximum absolute values of earlier iterations.
 *   - same page, "Estrategias de escalado y estabilidad": per-tensor versus
 *     block scaling; delayed scaling avoids a same-step reduction.
 *   - "NVIDIA NeMo RL logra una aceleracion del 48%..." (hotbookzone.com),
 *     "El avance tecnico": block-quantized E4M3 with 128x128 tiles for
 *     weights and 1x128 tiles for activations; linear layers run FP8 math.
 *   - same page, "Por que esto es importante...": power-of-two scales.
 * Where the pages are silent (rounding, ties, saturation, the scale formula,
 * the tolerance of the product) this file takes the readings stated beside
 * each function.  Every choice is deliberately the plainest one.
 *
 * Floating point: compile with -O2 -ffp-contract=off and without any
 * fast-math flag, so that float expressions are evaluated as written, each
 * operation rounded once to nearest-even.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>

#define ORC_E4M3 0
#define ORC_E5M2 1
#define ORC_SCALE_FP32 0
#define ORC_SCALE_POW2 1
#define ORC_GRAN_1x128 0
#define ORC_GRAN_128x128 1
#define ORC_GRAN_TENSOR 2
#define ORC_GRAN_1x32 3

/* ---------------------------------------------------------------- formats */

/* Format parameters.  E4M3 here is the "FN" variant: no infinities, the
 * only NaN codes are S.1111.111, so the largest finite magnitude is
 * 1.75 * 2^8 = 448, matching the +-448 the introl page gives for E4M3.
 * E5M2 follows IEEE conventions (infinities at exponent 31, mantissa 0),
 * largest finite 1.75 * 2^15 = 57344. */
typedef struct {
    int mbits;      /* stored mantissa bits */
    int bias;
    int emin;       /* exponent of the smallest normal binade */
    int maxcode;    /* code (sign bit clear) of the largest finite value */
    double fmax;
} orc_fmt;

static orc_fmt fmt_params(int fmt) {
    orc_fmt f;
    if (fmt == ORC_E4M3) {
        f.mbits = 3; f.bias = 7; f.emin = 1 - 7; f.maxcode = 0x7E; f.fmax = 448.0;
    } else {
        f.mbits = 2; f.bias = 15; f.emin = 1 - 15; f.maxcode = 0x7B; f.fmax = 57344.0;
    }
    return f;
}

/* Exact decode of one 8-bit code to fp64 (closed form of the format). */
double fp8o_decode(uint32_t code, int fmt) {
    int s = (code >> 7) & 1;
    double sign = s ? -1.0 : 1.0;
    if (fmt == ORC_E4M3) {
        int e = (code >> 3) & 0xF, m = code & 0x7;
        if (e == 15 && m == 7) return NAN;
        if (e == 0) return sign * ldexp((double)m, -9);          /* m/8 * 2^(1-7) */
        return sign * ldexp(8.0 + m, e - 7 - 3);                 /* (1+m/8) 2^(e-7) */
    } else {
        int e = (code >> 2) & 0x1F, m = code & 0x3;
        if (e == 31) return m == 0 ? sign * INFINITY : NAN;
        if (e == 0) return sign * ldexp((double)m, -16);         /* m/4 * 2^(1-15) */
        return sign * ldexp(4.0 + m, e - 15 - 2);                /* (1+m/4) 2^(e-15) */
    }
}

double fp8o_fmax(int fmt) { return fmt_params(fmt).fmax; }

static uint32_t f32_bits(float v) { uint32_t b; memcpy(&b, &v, 4); return b; }
static float bits_f32(uint32_t b) { float v; memcpy(&v, &b, 4); return v; }

/* bf16 -> fp32 is exact: the bf16 pattern is the top half of the fp32 one. */
float fp8o_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Encode an fp32 value: round to nearest, ties to the even code, saturate
 * finite overflow and infinities to +-max ("satfinite").  The sign survives
 * rounding to zero (-0 and tiny negatives give 0x80).  NaN gives 0x7F.
 *
 * Reading: the pages give neither the rounding nor the overflow rule; the
 * method's statement fixes round-to-nearest-even and saturation at 448.
 *
 * Method: with |v| = sig * 2^(E-23) (sig the 24-bit significand), the
 * target grid inside binade E is 2^(max(E,emin) - mbits).  Rounding |v| to
 * that grid is an integer rounding of sig at bit position `shift`; the
 * rounded integer n, offset by the binade, is directly the code magnitude
 * (a carry out of the mantissa moves to the next exponent by itself). */
uint32_t fp8o_encode(float v, int fmt) {
    orc_fmt f = fmt_params(fmt);
    uint32_t b = f32_bits(v);
    uint32_t sign = (b >> 31) << 7;
    uint32_t a = b & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return 0x7F;                 /* NaN */
    if (a == 0x7F800000u) return sign | (uint32_t)f.maxcode;   /* inf saturates */
    if (a < 0x00800000u) return sign;                 /* fp32 zero/subnormal: far below half the smallest subnormal */
    int E = (int)(a >> 23) - 127;
    uint32_t sig = (a & 0x7FFFFFu) | 0x800000u;
    int e_eff = E > f.emin ? E : f.emin;
    int shift = 23 - f.mbits + (e_eff - E);
    uint64_t n;
    if (shift > 40) {
        n = 0;                                        /* < quarter of the grid step */
    } else {
        uint64_t s64 = sig;
        n = s64 >> shift;
        uint64_t rem = s64 & ((1ull << shift) - 1);
        uint64_t half = 1ull << (shift - 1);
        if (rem > half || (rem == half && (n & 1))) n += 1;
    }
    int64_t mag = ((int64_t)(e_eff - f.emin) << f.mbits) + (int64_t)n;
    if (mag > f.maxcode) mag = f.maxcode;
    return sign | (uint32_t)mag;
}

/* -------------------------------------------------------------- scales */

/* Dequantization scale of one block from its amax (reading: the pages give
 * no formula; the method's statement gives amax/448, stored as fp32 or
 * rounded to a power of two).
 *   fp32: s = fl32(amax / fmax), with amax == 0 -> 1 and a floor at 2^-126
 *         so that 1/s stays finite for bf16-subnormal blocks.
 *   pow2: s = 2^e with e the smallest integer in [-126, 127] such that
 *         amax <= fmax * 2^e, so no element of the block saturates; the
 *         search runs upward from -126 and stops at 127; amax == 0 -> 1.
 * The power-of-two rounding direction is a reading: rounding up is the
 * only one under which the block's own maximum never overflows. */
float fp8o_block_scale(float amax, int fmt, int mode) {
    orc_fmt f = fmt_params(fmt);
    if (!(amax > 0.0f)) return 1.0f;                  /* zero (or NaN) block */
    if (mode == ORC_SCALE_FP32) {
        float s = amax / (float)f.fmax;
        if (s < 0x1p-126f) s = 0x1p-126f;
        return s;
    }
    int e;
    for (e = -126; e < 127; e++)
        if ((double)amax <= ldexp(f.fmax, e)) break;
    return (float)ldexp(1.0, e);
}

/* One element: q = enc(fl32(x * fl32(1/s))).  Reading: multiplying by the
 * rounded reciprocal (one rounding) rather than dividing by s. */
static uint8_t quant_elem(float x, float s, int fmt) {
    float r = 1.0f / s;
    float v = x * r;
    return (uint8_t)fp8o_encode(v, fmt);
}

/* Activation tiles: one scale per 128 consecutive elements of a row, along
 * the contraction (column) dimension ("1x128" on the NeMo RL page).
 * x: [rows][ldx] bf16 bits, q: [rows][ldq] codes,
 * scales: [ceil(cols/128)][rows], rows contiguous. */
void fp8o_quantize_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                         int fmt, int mode, uint8_t* q, int64_t ldq, float* scales) {
    int64_t nkb = (cols + 127) / 128;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t kb = 0; kb < nkb; kb++) {
            int64_t c0 = kb * 128, c1 = c0 + 128 < cols ? c0 + 128 : cols;
            float amax = 0.0f;
            for (int64_t c = c0; c < c1; c++) {
                float a = fabsf(fp8o_bf16_to_f32(x[r * ldx + c]));
                if (a > amax) amax = a;
            }
            float s = fp8o_block_scale(amax, fmt, mode);
            scales[kb * rows + r] = s;
            for (int64_t c = c0; c < c1; c++)
                q[r * ldq + c] = quant_elem(fp8o_bf16_to_f32(x[r * ldx + c]), s, fmt);
        }
    }
}

/* The same 1x128 rule on fp32 input: the quantization a product's epilogue
 * applies to its own fp32 result so that it can feed the next FP8 linear
 * layer directly (the quantization step the NeMo RL page counts among the
 * overheads of "Ganancias de rendimiento en el mundo real", done on the
 * product's output).  Reading: the same scale and element rules as for a
 * bf16 input, with the fp32 value in place of the widened bf16 one.
 * y: [rows][ldy] fp32; q, scales as fp8o_quantize_1x128. */
void fp8o_quantize_1x128_f32(const float* y, int64_t rows, int64_t cols, int64_t ldy,
                             int fmt, int mode, uint8_t* q, int64_t ldq, float* scales) {
    int64_t nkb = (cols + 127) / 128;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t kb = 0; kb < nkb; kb++) {
            int64_t c0 = kb * 128, c1 = c0 + 128 < cols ? c0 + 128 : cols;
            float amax = 0.0f;
            for (int64_t c = c0; c < c1; c++) {
                float a = fabsf(y[r * ldy + c]);
                if (a > amax) amax = a;
            }
            float s = fp8o_block_scale(amax, fmt, mode);
            scales[kb * rows + r] = s;
            for (int64_t c = c0; c < c1; c++)
                q[r * ldq + c] = quant_elem(y[r * ldy + c], s, fmt);
        }
    }
}

/* MXFP8 (microscaling FP8): one shared power-of-two scale per 32 consecutive
 * elements of a row.  The introl page names MXFP8 as Blackwell's block
 * scaling -- a separate scale factor for each block of a tensor, applied by
 * the hardware ("Requisitos de hardware para entrenamiento FP8",
 * "Estrategias de escalado y estabilidad", "Blackwell MXFP8 y NVFP4") --
 * without giving the block size or the scale rule.  Reading: the open
 * microscaling format the name refers to --
 *   32-element blocks; an 8-bit power-of-two scale X = 2^e stored as the
 *   code e + 127 (E8M0, 255 = NaN);
 *   e = floor(log2(amax)) - emax, emax the exponent of the element format's
 *   largest binade (8 for E4M3, 15 for E5M2), clamped to [-127, 127];
 *   elements enc(x * 2^-e) with the usual rounding and saturation (the
 *   block maximum lies in [2^emax, 2^(emax+1)) and may saturate);
 *   amax == 0 -> e = -127 (code 0); a non-finite amax -> code 255 and NaN
 *   elements.
 * floor(log2(amax)) is exact from frexp (amax = m 2^ex, m in [0.5, 1)). */
uint8_t fp8o_mx_scale_code(float amax, int fmt) {
    if (!isfinite(amax)) return 255;
    if (amax == 0.0f) return 0;
    int ex;
    frexp((double)amax, &ex);
    int e = (ex - 1) - (fmt == ORC_E4M3 ? 8 : 15);
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint8_t)(e + 127);
}

/* x: [rows][ldx] bf16 bits; q: [rows][ldq] codes;
 * scales: [ceil(cols/128)][rows][4] codes -- byte j of entry (kb, r) is
 * the scale of columns 128 kb + 32 j .. 128 kb + 32 j + 31 of row r. */
void fp8o_quantize_mx(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                      uint8_t* q, int64_t ldq, uint8_t* scales) {
    int64_t nkb = (cols + 127) / 128;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < nkb * 4; b++) {
            int64_t c0 = b * 32, c1 = c0 + 32 < cols ? c0 + 32 : cols;
            uint8_t code = 0;
            if (c0 < cols) {
                float amax = 0.0f;
                for (int64_t c = c0; c < c1; c++) {
                    float a = fabsf(fp8o_bf16_to_f32(x[r * ldx + c]));
                    if (a > amax) amax = a;   /* as in the other quantizers: NaN does not enter */
                }
                code = fp8o_mx_scale_code(amax, fmt);
                float mult = code == 255 ? NAN : (float)ldexp(1.0, 127 - (int)code);
                for (int64_t c = c0; c < c1; c++)
                    q[r * ldq + c] = (uint8_t)fp8o_encode(fp8o_bf16_to_f32(x[r * ldx + c]) * mult, fmt);
            }
            scales[((b / 4) * rows + r) * 4 + (b % 4)] = code;
        }
    }
}

/* Weight tiles: one scale per 128x128 tile ("128x128" on the NeMo RL page).
 * A partial last tile covers only the rows/columns that exist.
 * scales: [ceil(rows/128)][ceil(cols/128)]. */
void fp8o_quantize_128x128(const uint16_t* w, int64_t rows, int64_t cols, int64_t ldw,
                           int fmt, int mode, uint8_t* q, int64_t ldq, float* scales) {
    int64_t nrb = (rows + 127) / 128, nkb = (cols + 127) / 128;
    for (int64_t rb = 0; rb < nrb; rb++) {
        int64_t r0 = rb * 128, r1 = r0 + 128 < rows ? r0 + 128 : rows;
        for (int64_t kb = 0; kb < nkb; kb++) {
            int64_t c0 = kb * 128, c1 = c0 + 128 < cols ? c0 + 128 : cols;
            float amax = 0.0f;
            for (int64_t r = r0; r < r1; r++)
                for (int64_t c = c0; c < c1; c++) {
                    float a = fabsf(fp8o_bf16_to_f32(w[r * ldw + c]));
                    if (a > amax) amax = a;
                }
            float s = fp8o_block_scale(amax, fmt, mode);
            scales[rb * nkb + kb] = s;
            for (int64_t r = r0; r < r1; r++)
                for (int64_t c = c0; c < c1; c++)
                    q[r * ldq + c] = quant_elem(fp8o_bf16_to_f32(w[r * ldw + c]), s, fmt);
        }
    }
}

/* Per-tensor delayed scaling, quantization half: quantize with the scale
 * already in use (built from earlier steps only) and report this tensor's
 * amax for the history.  The amax covers every element, exactly. */
void fp8o_quantize_tensor(const uint16_t* x, int64_t n, int fmt, float scale,
                          uint8_t* q, float* amax_out) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; i++) {
        float v = fp8o_bf16_to_f32(x[i]);
        float a = fabsf(v);
        if (a > amax) amax = a;
        q[i] = quant_elem(v, scale, fmt);
    }
    *amax_out = amax;
}

/* Per-tensor delayed scaling, state half (recipe fields margin,
 * amax_history_len and amax_compute_algo="max" as on the introl page):
 *   history[head] = amax; head = (head + 1) mod L;
 *   amax_h = max over the whole history;
 *   if amax_h > 0 and t = fl32(fl32(amax_h / fmax) * 2^margin) is finite
 *   and > 0: scale = max(t, 2^-126); otherwise the scale is kept.
 * Reading: margin is an integer power-of-two exponent, as in the recipe's
 * margin=0 example; the stored scale is a dequantization multiplier. */
void fp8o_amax_history_update(float* history, int32_t* head, int32_t L, float amax,
                              int fmt, int32_t margin, float* scale) {
    orc_fmt f = fmt_params(fmt);
    history[*head] = amax;
    *head = (*head + 1) % L;
    float amax_h = 0.0f;
    for (int32_t i = 0; i < L; i++)
        if (history[i] > amax_h) amax_h = history[i];
    if (amax_h > 0.0f) {
        float t = amax_h / (float)f.fmax;
        t = t * (float)ldexp(1.0, margin);
        if (isfinite(t) && t > 0.0f) *scale = t < 0x1p-126f ? 0x1p-126f : t;
    }
}

/* ---------------------------------------------------------------- GEMM */

/* One FP8 operand of the product, as the library sees it.
 * Logical shape [rows][K] (rows = M for A, N for B).
 *   transposed == 0: stored [rows][ld], K contiguous.
 *   transposed == 1: stored [K][ld], rows contiguous.
 * Scale tables, in the orientation of the stored matrix:
 *   GRAN_1x128   (transposed == 0 only): [ceil(K/128)][rows]
 *   GRAN_128x128, transposed == 0: [ceil(rows/128)][ceil(K/128)]
 *   GRAN_128x128, transposed == 1: [ceil(K/128)][ceil(rows/128)]
 *   GRAN_TENSOR: one value.
 *   GRAN_1x32    (transposed == 0 only): MXFP8 codes, [ceil(K/128)][rows][4]
 *                bytes (see fp8o_quantize_mx), the pointer cast to float*. */
typedef struct {
    const uint8_t* data;
    int64_t ld;
    int32_t transposed;
    int32_t fmt;
    int32_t gran;
    int32_t pad_;
    const float* scales;
} fp8o_operand;

static double deq(const fp8o_operand* o, const double* lut, int64_t rows, int64_t K,
                  int64_t r, int64_t k) {
    uint8_t c = o->transposed ? o->data[k * o->ld + r] : o->data[r * o->ld + k];
    double s;
    int64_t nkb = (K + 127) / 128, nrb = (rows + 127) / 128;
    if (o->gran == ORC_GRAN_1x32) {   /* MXFP8: code of the 32-element block, 2^(code - 127) */
        uint8_t code = ((const uint8_t*)o->scales)[((k / 128) * rows + r) * 4 + (k % 128) / 32];
        s = code == 255 ? NAN : ldexp(1.0, (int)code - 127);
    } else if (o->gran == ORC_GRAN_1x128) s = o->scales[(k / 128) * rows + r];
    else if (o->gran == ORC_GRAN_128x128)
        s = o->transposed ? o->scales[(k / 128) * nrb + r / 128]
                          : o->scales[(r / 128) * nkb + k / 128];
    else s = o->scales[0];
    return lut[c] * s;
}

static void make_lut(int fmt, double* lut) {
    for (int c = 0; c < 256; c++) lut[c] = fp8o_decode((uint32_t)c, fmt);
}

/* Y = deq(A) . deq(B)^T on a selection of outputs, in fp64:
 *   y[i][j]    = sum_k deqA[row_i][k] * deqB[col_j][k]
 *   yabs[i][j] = sum_k |deqA[row_i][k] * deqB[col_j][k]|
 * (the GEMM of the NeMo RL page's linear layers; fp64 so that the result is
 * the exact sum up to fp64 rounding, far below any fp32 tolerance).
 * row_sel / col_sel may be NULL for "all rows" / "all columns". */
int fp8o_gemm(int64_t M, int64_t N, int64_t K,
              const fp8o_operand* A, const fp8o_operand* B,
              int64_t nr, const int64_t* row_sel, int64_t nc, const int64_t* col_sel,
              double* y, double* yabs) {
    double lutA[256], lutB[256];
    make_lut(A->fmt, lutA);
    make_lut(B->fmt, lutB);
    if (A->transposed && (A->gran == ORC_GRAN_1x128 || A->gran == ORC_GRAN_1x32)) return -1;
    if (B->transposed && (B->gran == ORC_GRAN_1x128 || B->gran == ORC_GRAN_1x32)) return -1;
    for (int64_t i = 0; i < nr; i++) {
        int64_t m = row_sel ? row_sel[i] : i;
        if (m < 0 || m >= M) return -1;
        for (int64_t j = 0; j < nc; j++) {
            int64_t n = col_sel ? col_sel[j] : j;
            if (n < 0 || n >= N) return -1;
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = deq(A, lutA, M, K, m, k) * deq(B, lutB, N, K, n, k);
                acc += p;
                aacc += fabs(p);
            }
            y[i * nc + j] = acc;
            yabs[i * nc + j] = aacc;
        }
    }
    return 0;
}

/* Grouped product (mixture-of-experts expert GEMMs): rows
 * [off[g], off[g+1]) of A are multiplied by expert g's weights, which sit
 * at B.data + g * N * B.ld with scales at B.scales + g * (scale table size).
 * A has a_rows rows as stored (its 1x128 scale table is [ceil(K/128)][a_rows]);
 * off[G] <= a_rows.  B must be non-transposed here (weights stored [G][N][K]).
 * A selected row outside every group yields NaN. */
int fp8o_grouped_gemm(int32_t G, const int32_t* off, int64_t a_rows, int64_t N, int64_t K,
                      const fp8o_operand* A, const fp8o_operand* B,
                      int64_t nr, const int64_t* row_sel, int64_t nc, const int64_t* col_sel,
                      double* y, double* yabs) {
    if (off[G] > a_rows) return -1;
    int64_t nkb = (K + 127) / 128, nrb = (N + 127) / 128;
    int64_t sc_per_group = B->gran == ORC_GRAN_128x128 ? nrb * nkb
                         : B->gran == ORC_GRAN_1x128 ? nkb * N : 1;
    if (B->transposed) return -1;
    for (int64_t i = 0; i < nr; i++) {
        int64_t m = row_sel ? row_sel[i] : i;
        int32_t g = -1;
        for (int32_t t = 0; t < G; t++)
            if (m >= off[t] && m < off[t + 1]) { g = t; break; }
        if (g < 0) {
            for (int64_t j = 0; j < nc; j++) { y[i * nc + j] = NAN; yabs[i * nc + j] = NAN; }
            continue;
        }
        fp8o_operand Bg = *B;
        Bg.data = B->data + (int64_t)g * N * B->ld;
        Bg.scales = B->scales + (int64_t)g * sc_per_group;
        int64_t one = m;
        int rc = fp8o_gemm(a_rows, N, K, A, &Bg, 1, &one, nc, col_sel, y + i * nc, yabs + i * nc);
        if (rc) return rc;
    }
    return 0;
}

/* ------------------------------------------------------------ attention */

/* FP8 attention with an FP8 KV cache (hotbookzone.com, "Ganancias de
 * rendimiento en el mundo real": extending FP8 to the KV cache and the
 * attention operations takes the speedup from +15-25 % to ~48 %; "El avance
 * tecnico": attention otherwise stays in BF16).  The pages give no recipe;
 * the readings: Q is quantized like an activation (1x128 tiles = one scale per
 * token and head, head_dim 128), K and V like the 128x128 weight tiles (one
 * scale per 128 tokens per head) -- the cache layout [tokens][heads * 128]
 * makes both the library's existing quantizers.
 * What is computed (the definition; the kernel's P rounding is judged by the
 * tolerance, see fp8o_attention's outputs): for query row i of head h, kv
 * head g = h / (hq / hkv),
 *   S_ij = scale * sum_d deqQ[i][h][d] deqK[j][g][d]   (j visible: j <= i +
 *          seq_k - seq_q when causal)
 *   P_ij = exp(S_ij - max_j S_ij), l_i = sum_j P_ij
 *   O[i][h][d] = sum_j P_ij deqV[j][g][d] / l_i
 * and, for the tolerance, oap[i][h][d] = sum_j P_ij |deqV| / l_i and
 * oav[i][h][d] = sum_j |deqV| (svm_g / sv_t(j)) / l_i = sum_j |V code| svm_g
 * / l_i, all in fp64, where sv_t(j) is key j's V tile scale and svm_g the
 * largest V tile scale of kv head g (the kernel quantizes P times sv_t / svm_g,
 * so the absolute error of a subnormal P code, read back in P units, grows by
 * svm_g / sv_t).
 * q: [seq_q][hq][128] codes, sq: [hq][seq_q] (1x128 table of the [seq_q][hq*128]
 * matrix); k, v: [seq_k][hkv][128] codes, sk, sv: [ceil(seq_k/128)][hkv].
 * Selected (row, head) pairs: rows[n], heads[n].  Output [n][128]. */
int fp8o_attention(int64_t seq_q, int64_t seq_k, int32_t hq, int32_t hkv, int causal, double scale,
                   const uint8_t* q, const float* sq, int fmt_q, const uint8_t* k, const float* sk,
                   int fmt_k, const uint8_t* v, const float* sv, int fmt_v,
                   int64_t n, const int64_t* rows, const int32_t* heads,
                   double* o, double* oap, double* oav) {
    const int D = 128;
    if (hq <= 0 || hkv <= 0 || hq % hkv) return -1;
    double lq[256], lk[256], lv[256];
    make_lut(fmt_q, lq);
    make_lut(fmt_k, lk);
    make_lut(fmt_v, lv);
    double* sc = (double*)malloc(sizeof(double) * (size_t)(seq_k > 0 ? seq_k : 1));
    if (!sc) return -2;
    for (int64_t t = 0; t < n; t++) {
        int64_t i = rows[t];
        int32_t h = heads[t];
        if (i < 0 || i >= seq_q || h < 0 || h >= hq) { free(sc); return -1; }
        int32_t g = h / (hq / hkv);
        double qs = sq[(int64_t)h * seq_q + i];
        double svm = 0.0;
        for (int64_t tt = 0; tt < (seq_k + 127) / 128; tt++)
            if (sv[tt * hkv + g] > svm) svm = sv[tt * hkv + g];
        int64_t jend = causal ? i + (seq_k - seq_q) + 1 : seq_k;
        if (jend > seq_k) jend = seq_k;
        double m = -INFINITY;
        for (int64_t j = 0; j < jend; j++) {
            double ks = sk[(j / 128) * hkv + g], acc = 0.0;
            for (int d = 0; d < D; d++)
                acc += lq[q[(i * hq + h) * D + d]] * qs * lk[k[(j * hkv + g) * D + d]] * ks;
            sc[j] = acc * scale;
            if (sc[j] > m) m = sc[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < jend; j++) { sc[j] = exp(sc[j] - m); l += sc[j]; }
        for (int d = 0; d < D; d++) {
            double a = 0.0, ap = 0.0, av = 0.0;
            for (int64_t j = 0; j < jend; j++) {
                double vv = lv[v[(j * hkv + g) * D + d]] * sv[(j / 128) * hkv + g];
                a += sc[j] * vv;
                ap += sc[j] * fabs(vv);
                av += fabs(lv[v[(j * hkv + g) * D + d]]) * svm;
            }
            o[t * D + d] = jend > 0 ? a / l : 0.0;
            oap[t * D + d] = jend > 0 ? ap / l : 0.0;
            oav[t * D + d] = jend > 0 ? av / l : 0.0;
        }
    }
    free(sc);
    return 0;
}

/* Element-wise encoder over an array (the same fp8o_encode, looped), so the
 * tests can sweep many fp32 patterns without a Python-level loop. */
void fp8o_encode_array(const float* v, int64_t n, int fmt, uint8_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)fp8o_encode(v[i], fmt);
}
