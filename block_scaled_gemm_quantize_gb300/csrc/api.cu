// api.cu -- the C ABI (include/fp8bs.h): argument validation, TMA tensor-map
// construction and kernel launches.  No device memory is allocated here.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "fp8bs.h"
#include "attn_kernels.h"
#include "gemm_kernels.h"
#include "quant_kernels.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* where) {
    return fail(FP8BS_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool valid_fmt(int32_t f) { return f == FP8BS_E4M3 || f == FP8BS_E5M2; }
bool valid_mode(int32_t m) { return m == FP8BS_SCALE_FP32 || m == FP8BS_SCALE_POW2; }

// Shared checks of the two block quantizers.
int check_block_quant(const char* fn, const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                      int32_t fmt, int32_t mode, const uint8_t* q, int64_t ld_q,
                      const float* scales) {
    if (rows < 0 || cols < 0) return fail(FP8BS_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!valid_fmt(fmt) || !valid_mode(mode))
        return fail(FP8BS_ERR_INVALID_ARG, "%s: bad format %d or scale mode %d", fn, fmt, mode);
    if (rows == 0 || cols == 0) return FP8BS_OK;
    if (!x || !q || !scales) return fail(FP8BS_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (ld_x < cols || ld_q < cols)
        return fail(FP8BS_ERR_INVALID_ARG, "%s: leading dimension smaller than cols", fn);
    if (cols % 128) return fail(FP8BS_ERR_UNSUPPORTED, "%s: cols %% 128 != 0 (cols=%lld)", fn, (long long)cols);
    if (!aligned16(x) || !aligned16(q) || (ld_x * 2) % 16 || ld_q % 16 || !aligned4(scales))
        return fail(FP8BS_ERR_MISALIGNED, "%s: x/q must be 16-byte aligned with 16-byte row pitch", fn);
    return 1;  // proceed
}

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

int get_encoder() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return fail(FP8BS_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)",
                               cudaGetErrorString(g_encode_err));
    return FP8BS_OK;
}

// 2-D uint8 tensor [outer][inner] with row pitch `pitch` bytes; box
// {128, box_outer}, 128-byte swizzle, out-of-bounds elements read as zero.
int make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch,
             uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {128, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FP8BS_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return FP8BS_OK;
}

// Output tensor [rows][N] of fp32, bf16 or 8-bit codes (esz 4, 2, 1) with
// row pitch `pitch` bytes; box 32 rows x 64 bytes, 64-byte swizzle (matches
// the epilogue's staging slabs).
int make_out_map(CUtensorMap* m, void* base, int esz, uint64_t N, uint64_t rows, uint64_t pitch) {
    cuuint64_t dims[2] = {N, rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {64u / static_cast<cuuint32_t>(esz), 32u};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = esz == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = g_encode(m, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FP8BS_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (CUresult %d)", (int)r);
    return FP8BS_OK;
}

// fp32 scale table [nkb][rows] (rows contiguous); box 128 rows x 1 K block.
int make_scale_map(CUtensorMap* m, const float* base, uint64_t rows, uint64_t nkb) {
    cuuint64_t dims[2] = {rows, nkb};
    cuuint64_t strides[1] = {rows * 4};
    cuuint32_t box[2] = {128, 1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FP8BS_ERR_CUDA, "cuTensorMapEncodeTiled (scales) failed (CUresult %d)", (int)r);
    return FP8BS_OK;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

int check_operand(const char* fn, const char* name, const fp8bs_operand* o, int64_t rows,
                  int64_t K, bool is_b, bool grouped) {
    if (!o) return fail(FP8BS_ERR_INVALID_ARG, "%s: %s is null", fn, name);
    if (!o->data || !o->scales) return fail(FP8BS_ERR_INVALID_ARG, "%s: %s data/scales null", fn, name);
    if (!valid_fmt(o->fmt)) return fail(FP8BS_ERR_INVALID_ARG, "%s: %s bad format", fn, name);
    if (o->gran < 0 || o->gran > 3 || o->reserved != 0)
        return fail(FP8BS_ERR_INVALID_ARG, "%s: %s bad granularity", fn, name);
    if (o->gran == FP8BS_GRAN_1x32 && (o->transposed || grouped))
        return fail(FP8BS_ERR_UNSUPPORTED, "%s: %s MXFP8 (1x32) operands must be non-transposed, not grouped",
                    fn, name);
    if (o->transposed != 0 && o->transposed != 1)
        return fail(FP8BS_ERR_INVALID_ARG, "%s: %s bad transposed flag", fn, name);
    if (o->gran == FP8BS_GRAN_1x128 && o->transposed)
        return fail(FP8BS_ERR_UNSUPPORTED, "%s: %s 1x128 scales only on a non-transposed operand", fn, name);
    if (o->gran == FP8BS_GRAN_1x128 && is_b && grouped)
        return fail(FP8BS_ERR_UNSUPPORTED, "%s: 1x128 B scales not supported in a grouped product", fn);
    if (grouped && o->transposed)
        return fail(FP8BS_ERR_UNSUPPORTED, "%s: %s must be non-transposed in a grouped product", fn, name);
    if (grouped && !is_b && o->gran == FP8BS_GRAN_128x128)
        return fail(FP8BS_ERR_UNSUPPORTED, "%s: grouped A takes 1x128 or per-tensor scales", fn);
    const int64_t inner = o->transposed ? rows : K;
    if (o->ld < inner) return fail(FP8BS_ERR_INVALID_ARG, "%s: %s ld too small", fn, name);
    if (!aligned16(o->data) || o->ld % 16)
        return fail(FP8BS_ERR_MISALIGNED, "%s: %s data must be 16-byte aligned, ld %% 16 == 0", fn, name);
    if (!aligned4(o->scales)) return fail(FP8BS_ERR_MISALIGNED, "%s: %s scales not 4-byte aligned", fn, name);
    return FP8BS_OK;
}

// Where and how a product writes its result.
struct OutSpec {
    void* y;              // Y (float output) or Q (8-bit codes)
    int64_t ld;           // elements between rows
    int32_t dtype;        // FP8BS_OUT_F32 / FP8BS_OUT_BF16 (float output)
    bool quant;           // quantized output: codes + 1x128 scales
    int32_t epilogue;     // FP8BS_EPI_NONE / FP8BS_EPI_SWIGLU (quantized output)
    int32_t q_fmt, q_mode;
    float* q_scales;      // [n_out/128][a_rows]
};

int run_gemm(const char* fn, int32_t G, const int32_t* offsets, int64_t a_rows, int64_t M,
             int64_t N, int64_t K, const fp8bs_operand* A, const fp8bs_operand* B, int32_t mode,
             const OutSpec& o, cudaStream_t stream) {
    const bool grouped = offsets != nullptr;
    if (M < 0 || N < 0 || K < 0 || a_rows < 0) return fail(FP8BS_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!valid_mode(mode)) return fail(FP8BS_ERR_INVALID_ARG, "%s: bad scale mode", fn);
    if (!o.quant && o.dtype != FP8BS_OUT_F32 && o.dtype != FP8BS_OUT_BF16)
        return fail(FP8BS_ERR_INVALID_ARG, "%s: bad output dtype", fn);
    if (o.quant && (o.epilogue != FP8BS_EPI_NONE && o.epilogue != FP8BS_EPI_SWIGLU))
        return fail(FP8BS_ERR_INVALID_ARG, "%s: bad epilogue", fn);
    if (o.quant && (!valid_fmt(o.q_fmt) || !valid_mode(o.q_mode)))
        return fail(FP8BS_ERR_INVALID_ARG, "%s: bad output format or scale mode", fn);
    if (grouped && (G < 1 || G > fp8bs::kMaxGroups))
        return fail(FP8BS_ERR_INVALID_ARG, "%s: num_groups must be in [1, %d]", fn, fp8bs::kMaxGroups);
    const bool swiglu = o.quant && o.epilogue == FP8BS_EPI_SWIGLU;
    if (swiglu && N % 256) return fail(FP8BS_ERR_UNSUPPORTED, "%s: SwiGLU needs N %% 256 == 0", fn);
    if (o.quant && N % 128) return fail(FP8BS_ERR_UNSUPPORTED, "%s: quantized output needs N %% 128 == 0", fn);
    if (M == 0 || N == 0) return FP8BS_OK;
    const int64_t n_out = swiglu ? N / 2 : N;
    const int64_t esz = o.quant ? 1 : (o.dtype == FP8BS_OUT_BF16 ? 2 : 4);
    if (!o.y) return fail(FP8BS_ERR_INVALID_ARG, "%s: output is null", fn);
    if (o.quant && !o.q_scales) return fail(FP8BS_ERR_INVALID_ARG, "%s: output scales are null", fn);
    if (o.ld < n_out) return fail(FP8BS_ERR_INVALID_ARG, "%s: output leading dimension too small", fn);
    if (!aligned16(o.y) || (o.ld * esz) % 16 || (o.quant && !aligned4(o.q_scales)))
        return fail(FP8BS_ERR_MISALIGNED, "%s: output must be 16-byte aligned with 16-byte row pitch", fn);
    if (K == 0) {  // empty contraction: Y = 0 (quantized: codes 0, scales 1)
        cudaError_t e = cudaMemset2DAsync(o.y, o.ld * esz, 0, n_out * esz, M, stream);
        if (e == cudaSuccess && o.quant) e = fp8bs::launch_fill_f32(o.q_scales, (n_out / 128) * M, 1.0f, stream);
        return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, fn);
    }
    if (K % 128) return fail(FP8BS_ERR_UNSUPPORTED, "%s: K %% 128 != 0 (K=%lld)", fn, (long long)K);
    if (N % 8) return fail(FP8BS_ERR_UNSUPPORTED, "%s: N %% 8 != 0", fn);
    int rc;
    if ((rc = check_operand(fn, "A", A, M, K, false, grouped)) != FP8BS_OK) return rc;
    if ((rc = check_operand(fn, "B", B, N, K, true, grouped)) != FP8BS_OK) return rc;
    if (swiglu && (A->transposed || B->transposed))
        return fail(FP8BS_ERR_UNSUPPORTED, "%s: SwiGLU needs non-transposed operands", fn);
    if (B->gran == FP8BS_GRAN_1x128) {
        // the kernel bulk-copies B's (and a 1x128 A's) scale rows per K block
        if (o.quant || A->transposed)
            return fail(FP8BS_ERR_UNSUPPORTED, "%s: 1x128 B scales need a non-transposed A and a float output", fn);
        if (A->gran == FP8BS_GRAN_1x128 && a_rows % 4)
            return fail(FP8BS_ERR_UNSUPPORTED, "%s: 1x128 B scales with a 1x128 A need rows of A %% 4 == 0", fn);
        if (!aligned16(B->scales) || (A->gran == FP8BS_GRAN_1x128 && !aligned16(A->scales)))
            return fail(FP8BS_ERR_MISALIGNED, "%s: 1x128 B scales need 16-byte aligned scale tables", fn);
    }
    const bool mx32 = A->gran == FP8BS_GRAN_1x32 || B->gran == FP8BS_GRAN_1x32;
    if (mx32 && (A->gran != B->gran || swiglu))
        return fail(FP8BS_ERR_UNSUPPORTED, "%s: MXFP8 (1x32) needs both operands 1x32 and no SwiGLU", fn);
    if (mx32 && (a_rows % 4 || !aligned16(A->scales)))
        return fail(a_rows % 4 ? FP8BS_ERR_UNSUPPORTED : FP8BS_ERR_MISALIGNED,
                    "%s: MXFP8 A scales need rows %% 4 == 0 and a 16-byte aligned table", fn);
    if (a_rows > (int64_t)INT32_MAX - 256 || N * (grouped ? G : 1) > (int64_t)INT32_MAX - 256 ||
        K > (int64_t)INT32_MAX)
        return fail(FP8BS_ERR_UNSUPPORTED, "%s: dimension beyond 2^31", fn);
    if ((rc = get_encoder()) != FP8BS_OK) return rc;

    const int BN = fp8bs::gemm_tile_n(), BM = fp8bs::gemm_tile_m();
    const bool a_mn = A->transposed, b_mn = B->transposed;
    CUtensorMap tmA, tmB;
    if (a_mn) rc = make_map(&tmA, A->data, M, K, A->ld, 128);
    else rc = make_map(&tmA, A->data, K, a_rows, A->ld, 128);
    if (rc) return rc;
    const int64_t b_rows_total = grouped ? (int64_t)G * N : N;
    if (b_mn) rc = make_map(&tmB, B->data, N, K, B->ld, 128);
    else rc = make_map(&tmB, B->data, K, b_rows_total, B->ld, swiglu ? 64 : BN);
    if (rc) return rc;

    CUtensorMap tmY;
    if ((rc = make_out_map(&tmY, o.y, static_cast<int>(esz), n_out, a_rows, o.ld * esz)) != FP8BS_OK)
        return rc;

    fp8bs::GemmParams p;
    memset(&p, 0, sizeof(p));
    p.tma_store = 1;
    p.M = M;
    p.N = N;
    p.K = K;
    p.a_rows = a_rows;
    p.a_rblocks = (M + 127) / 128;
    p.b_rblocks = (N + 127) / 128;
    p.b_scale_group_stride = B->gran == FP8BS_GRAN_128x128 ? ((N + 127) / 128) * (K / 128) : 0;
    p.sa = A->scales;
    p.sb = B->scales;
    p.offsets = offsets;
    p.y = o.y;
    p.ldy = o.ld;
    p.num_groups = grouped ? G : 1;
    p.b_rows_per_group = grouped ? static_cast<int32_t>(N) : 0;
    p.a_gran = A->gran;
    p.b_gran = B->gran;
    p.sa_bulk = A->gran == FP8BS_GRAN_1x128 && a_rows % 4 == 0 && aligned16(A->scales);
    p.tiles_n = static_cast<int32_t>(swiglu ? n_out / 128 : (N + BN - 1) / BN);
    p.promote = (A->gran == FP8BS_GRAN_TENSOR && B->gran == FP8BS_GRAN_TENSOR) ? 0 : 1;
    p.out_bf16 = !o.quant && o.dtype == FP8BS_OUT_BF16;
    p.out_q = o.quant;
    p.q_fmt = o.q_fmt;
    p.q_mode = o.q_mode;
    p.sq = o.q_scales;
    p.n_out = n_out;
    p.swiglu = swiglu;
    p.swiglu_i = swiglu ? N / 2 : 0;
    p.mx32 = mx32;
    p.idesc = fp8bs::make_idesc_f8f6f4(A->fmt, B->fmt, a_mn, b_mn,
                                       b_mn ? 128 : fp8bs::gemm_mma_n(B->gran == FP8BS_GRAN_1x128));

    // upper bound on tiles (the grouped count is only known on the device)
    const int64_t slots = grouped ? (a_rows + BM - 1) / BM + G : (M + BM - 1) / BM;
    const int64_t tiles = slots * p.tiles_n;
    if (tiles > (int64_t)INT32_MAX) return fail(FP8BS_ERR_UNSUPPORTED, "%s: too many tiles", fn);
    const int sms = sm_count();
    if (sms <= 0) return fail(FP8BS_ERR_CUDA, "%s: cannot query the device", fn);
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    if (grid <= 0) return FP8BS_OK;
    // (1x128 A scales reach the MX kernel by TMA: a row pitch of 16 bytes
    // needed.)  Only block-scaled operands go there: a per-tensor scale
    // (delayed scaling) is in general not a power of two, so those products
    // keep the promotion kernel.
    const bool sa_tma_ok = A->gran != FP8BS_GRAN_1x128 || (a_rows % 4 == 0 && aligned16(A->scales));
    const bool blocks_only = A->gran != FP8BS_GRAN_TENSOR && B->gran != FP8BS_GRAN_TENSOR;
#ifndef FP8BS_NO_MX
    const bool use_mx = mx32 || (mode == FP8BS_SCALE_POW2 && !a_mn && !b_mn && !grouped && sa_tma_ok &&
                                 blocks_only && B->gran != FP8BS_GRAN_1x128);
#else
    const bool use_mx = mx32;
#endif
    // Power-of-two scales on K-major operands go to the block-scaled (MX)
    // kernel: the tensor core applies the UE8M0 scales, no promotion.
    cudaError_t e;
    if (mx32) {   // MXFP8: the block-scaled kernel reads the E8M0 words directly
        CUtensorMap tmSA;
        if ((rc = make_scale_map(&tmSA, A->scales, a_rows, K / 128)) != FP8BS_OK) return rc;
        p.idesc = fp8bs::make_idesc_mx(A->fmt, B->fmt, BN);
        e = fp8bs::launch_fp8_gemm_mx(tmA, tmB, tmY, tmSA, p, grid, stream);
        return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, fn);
    }
    if (use_mx) {
        CUtensorMap tmSA;
        memset(&tmSA, 0, sizeof(tmSA));
        if (A->gran == FP8BS_GRAN_1x128 && (rc = make_scale_map(&tmSA, A->scales, a_rows, K / 128)) != FP8BS_OK)
            return rc;
        p.idesc = fp8bs::make_idesc_mx(A->fmt, B->fmt, BN);
        e = fp8bs::launch_fp8_gemm_mx(tmA, tmB, tmY, tmSA, p, grid, stream);
    } else {
        e = fp8bs::launch_fp8_gemm(tmA, tmB, tmY, p, a_mn, b_mn, grid, stream);
    }
    return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, fn);
}

OutSpec float_out(void* Y, int64_t ld_y, int32_t out_dtype) {
    OutSpec o;
    memset(&o, 0, sizeof(o));
    o.y = Y;
    o.ld = ld_y;
    o.dtype = out_dtype;
    return o;
}

OutSpec quant_out(uint8_t* Q, int64_t ld_q, int32_t epilogue, int32_t q_fmt, int32_t q_mode, float* q_scales) {
    OutSpec o;
    memset(&o, 0, sizeof(o));
    o.y = Q;
    o.ld = ld_q;
    o.quant = true;
    o.epilogue = epilogue;
    o.q_fmt = q_fmt;
    o.q_mode = q_mode;
    o.q_scales = q_scales;
    return o;
}

}  // namespace

extern "C" {

int fp8bs_version(void) { return 1; }

const char* fp8bs_last_error(void) { return g_err; }

int fp8_quantize_1x128(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int32_t fmt,
                       int32_t mode, uint8_t* q, int64_t ld_q, float* scales,
                       fp8bs_stream_t stream) {
    int rc = check_block_quant("fp8_quantize_1x128", x, rows, cols, ld_x, fmt, mode, q, ld_q, scales);
    if (rc <= 0) return rc;
    cudaError_t e = fp8bs::launch_quant_1x128(static_cast<const uint16_t*>(x), rows, cols, ld_x, fmt,
                                              mode, q, ld_q, scales, (cudaStream_t)stream);
    return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, "fp8_quantize_1x128");
}

int fp8_quantize_128x128(const void* w, int64_t rows, int64_t cols, int64_t ld_w, int32_t fmt,
                         int32_t mode, uint8_t* q, int64_t ld_q, float* scales,
                         fp8bs_stream_t stream) {
    int rc = check_block_quant("fp8_quantize_128x128", w, rows, cols, ld_w, fmt, mode, q, ld_q, scales);
    if (rc <= 0) return rc;
    cudaError_t e = fp8bs::launch_quant_128x128(static_cast<const uint16_t*>(w), rows, cols, ld_w,
                                                fmt, mode, q, ld_q, scales, (cudaStream_t)stream);
    return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, "fp8_quantize_128x128");
}

int fp8_quantize_linear(const void* x, int64_t m, int64_t ld_x, uint8_t* qx, int64_t ld_qx, float* sx,
                        const void* w, int64_t n, int64_t ld_w, uint8_t* qw, int64_t ld_qw, float* sw,
                        int64_t k, int32_t fmt, int32_t mode, fp8bs_stream_t stream) {
    const char* fn = "fp8_quantize_linear";
    if (m < 0 || n < 0 || k < 0) return fail(FP8BS_ERR_INVALID_ARG, "%s: negative size", fn);
    // each operand is checked exactly as its own quantizer checks it
    int rx = check_block_quant(fn, x, m, k, ld_x, fmt, mode, qx, ld_qx, sx);
    if (rx < 0) return rx;
    int rw = check_block_quant(fn, w, n, k, ld_w, fmt, mode, qw, ld_qw, sw);
    if (rw < 0) return rw;
    if (rx == 0 && rw == 0) return FP8BS_OK;
    cudaError_t e = fp8bs::launch_quant_linear(
        static_cast<const uint16_t*>(x), rx ? m : 0, ld_x, qx, ld_qx, sx, static_cast<const uint16_t*>(w),
        rw ? n : 0, ld_w, qw, ld_qw, sw, k, fmt, mode, (cudaStream_t)stream);
    return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, fn);
}

int fp8_quantize_mx(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int32_t fmt, uint8_t* q,
                    int64_t ld_q, uint8_t* scales, fp8bs_stream_t stream) {
    const char* fn = "fp8_quantize_mx";
    int rc = check_block_quant(fn, x, rows, cols, ld_x, fmt, FP8BS_SCALE_POW2, q, ld_q,
                               reinterpret_cast<const float*>(scales));
    if (rc <= 0) return rc;
    cudaError_t e = fp8bs::launch_quant_mx(static_cast<const uint16_t*>(x), rows, cols, ld_x, fmt, q, ld_q,
                                           reinterpret_cast<uint32_t*>(scales), (cudaStream_t)stream);
    return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, fn);
}

int fp8_quantize_1x128_colwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int32_t fmt,
                               int32_t mode, uint8_t* qt, int64_t ld_qt, float* scales_t, uint8_t* q,
                               int64_t ld_q, float* scales, fp8bs_stream_t stream) {
    const char* fn = "fp8_quantize_1x128_colwise";
    if (rows < 0 || cols < 0) return fail(FP8BS_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!valid_fmt(fmt) || !valid_mode(mode))
        return fail(FP8BS_ERR_INVALID_ARG, "%s: bad format %d or scale mode %d", fn, fmt, mode);
    if ((q == nullptr) != (scales == nullptr))
        return fail(FP8BS_ERR_INVALID_ARG, "%s: row-wise q and scales must both be given or both be null", fn);
    if (rows == 0 || cols == 0) return FP8BS_OK;
    if (!x || !qt || !scales_t) return fail(FP8BS_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (ld_x < cols || ld_qt < rows || (q && ld_q < cols))
        return fail(FP8BS_ERR_INVALID_ARG, "%s: leading dimension too small", fn);
    if (rows % 128 || cols % 128)
        return fail(FP8BS_ERR_UNSUPPORTED, "%s: rows and cols must be multiples of 128", fn);
    if (!aligned16(x) || (ld_x * 2) % 16 || !aligned16(qt) || ld_qt % 16 || !aligned4(scales_t) ||
        (q && (!aligned16(q) || ld_q % 16 || !aligned4(scales))))
        return fail(FP8BS_ERR_MISALIGNED, "%s: x/q/qt must be 16-byte aligned with 16-byte row pitch", fn);
    cudaError_t e = fp8bs::launch_quant_colwise(static_cast<const uint16_t*>(x), rows, cols, ld_x, fmt, mode,
                                                qt, ld_qt, scales_t, q, ld_q, scales, (cudaStream_t)stream);
    return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, fn);
}

int fp8_quantize_tensor_delayed(const void* x, int64_t numel, int32_t fmt, const float* scale,
                                uint8_t* q, float* amax_out, fp8bs_stream_t stream) {
    const char* fn = "fp8_quantize_tensor_delayed";
    if (numel < 0) return fail(FP8BS_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!valid_fmt(fmt)) return fail(FP8BS_ERR_INVALID_ARG, "%s: bad format", fn);
    if (!scale || !amax_out) return fail(FP8BS_ERR_INVALID_ARG, "%s: null scale/amax", fn);
    if (numel > 0 && (!x || !q)) return fail(FP8BS_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned4(scale) || !aligned4(amax_out) || (numel > 0 && (!aligned16(x) || !aligned16(q))))
        return fail(FP8BS_ERR_MISALIGNED, "%s: x/q must be 16-byte aligned", fn);
    cudaError_t e = fp8bs::launch_quant_tensor(static_cast<const uint16_t*>(x), numel, fmt, scale, q,
                                               amax_out, (cudaStream_t)stream);
    return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, fn);
}

int fp8_amax_history_update(float* history, int32_t* head, int32_t history_len, const float* amax,
                            int32_t fmt, int32_t margin, float* scale, fp8bs_stream_t stream) {
    const char* fn = "fp8_amax_history_update";
    if (!history || !head || !amax || !scale) return fail(FP8BS_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (history_len < 1) return fail(FP8BS_ERR_INVALID_ARG, "%s: history_len < 1", fn);
    if (!valid_fmt(fmt)) return fail(FP8BS_ERR_INVALID_ARG, "%s: bad format", fn);
    if (margin < -126 || margin > 126) return fail(FP8BS_ERR_INVALID_ARG, "%s: margin outside [-126, 126]", fn);
    if (!aligned4(history) || !aligned4(head) || !aligned4(amax) || !aligned4(scale))
        return fail(FP8BS_ERR_MISALIGNED, "%s: scalars must be 4-byte aligned", fn);
    cudaError_t e = fp8bs::launch_amax_history(history, head, history_len, amax, fmt, margin, scale,
                                               (cudaStream_t)stream);
    return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, fn);
}

int fp8_block_gemm(int64_t M, int64_t N, int64_t K, const fp8bs_operand* A,
                   const fp8bs_operand* B, int32_t mode, void* Y, int64_t ld_y, int32_t out_dtype,
                   fp8bs_stream_t stream) {
    return run_gemm("fp8_block_gemm", 1, nullptr, M, M, N, K, A, B, mode, float_out(Y, ld_y, out_dtype),
                    (cudaStream_t)stream);
}

int fp8_block_gemm_quant(int64_t M, int64_t N, int64_t K, const fp8bs_operand* A,
                         const fp8bs_operand* B, int32_t mode, int32_t epilogue, int32_t q_fmt,
                         int32_t q_mode, uint8_t* Q, int64_t ld_q, float* q_scales,
                         fp8bs_stream_t stream) {
    return run_gemm("fp8_block_gemm_quant", 1, nullptr, M, M, N, K, A, B, mode,
                    quant_out(Q, ld_q, epilogue, q_fmt, q_mode, q_scales), (cudaStream_t)stream);
}

int fp8_grouped_block_gemm(int32_t num_groups, const int32_t* row_offsets, int64_t a_rows,
                           int64_t N, int64_t K, const fp8bs_operand* A, const fp8bs_operand* B,
                           int32_t mode, void* Y, int64_t ld_y, int32_t out_dtype,
                           fp8bs_stream_t stream) {
    if (!row_offsets) return fail(FP8BS_ERR_INVALID_ARG, "fp8_grouped_block_gemm: null row_offsets");
    if (!aligned4(row_offsets)) return fail(FP8BS_ERR_MISALIGNED, "fp8_grouped_block_gemm: offsets");
    return run_gemm("fp8_grouped_block_gemm", num_groups, row_offsets, a_rows, a_rows, N, K, A, B,
                    mode, float_out(Y, ld_y, out_dtype), (cudaStream_t)stream);
}

int fp8_grouped_block_gemm_quant(int32_t num_groups, const int32_t* row_offsets, int64_t a_rows,
                                 int64_t N, int64_t K, const fp8bs_operand* A, const fp8bs_operand* B,
                                 int32_t mode, int32_t epilogue, int32_t q_fmt, int32_t q_mode,
                                 uint8_t* Q, int64_t ld_q, float* q_scales, fp8bs_stream_t stream) {
    if (!row_offsets) return fail(FP8BS_ERR_INVALID_ARG, "fp8_grouped_block_gemm_quant: null row_offsets");
    if (!aligned4(row_offsets)) return fail(FP8BS_ERR_MISALIGNED, "fp8_grouped_block_gemm_quant: offsets");
    return run_gemm("fp8_grouped_block_gemm_quant", num_groups, row_offsets, a_rows, a_rows, N, K, A, B,
                    mode, quant_out(Q, ld_q, epilogue, q_fmt, q_mode, q_scales), (cudaStream_t)stream);
}

int fp8_attention_fwd(int64_t seq_q, int64_t seq_k, int32_t heads_q, int32_t heads_kv, int32_t head_dim,
                      int32_t causal, float softmax_scale, const fp8bs_attn_input* Q, const fp8bs_attn_input* K,
                      const fp8bs_attn_input* V, void* O, int64_t ld_o, fp8bs_stream_t stream) {
    const char* fn = "fp8_attention_fwd";
    if (seq_q < 0 || seq_k < 0) return fail(FP8BS_ERR_INVALID_ARG, "%s: negative size", fn);
    if (heads_q < 1 || heads_kv < 1 || heads_q % heads_kv)
        return fail(FP8BS_ERR_INVALID_ARG, "%s: heads_q must be a positive multiple of heads_kv", fn);
    if (head_dim != 128) return fail(FP8BS_ERR_UNSUPPORTED, "%s: head_dim must be 128", fn);
    if (causal != 0 && causal != 1) return fail(FP8BS_ERR_INVALID_ARG, "%s: causal must be 0 or 1", fn);
    if (!(softmax_scale > 0.0f) || !(softmax_scale < 1e30f))
        return fail(FP8BS_ERR_INVALID_ARG, "%s: softmax_scale must be positive and finite", fn);
    if (!Q || !K || !V) return fail(FP8BS_ERR_INVALID_ARG, "%s: null input descriptor", fn);
    if (seq_q == 0) return FP8BS_OK;
    if (!O) return fail(FP8BS_ERR_INVALID_ARG, "%s: O is null", fn);
    const int64_t wq = (int64_t)heads_q * 128, wkv = (int64_t)heads_kv * 128;
    if (ld_o < wq) return fail(FP8BS_ERR_INVALID_ARG, "%s: ld_o < heads_q * 128", fn);
    if (!aligned16(O) || (ld_o * 2) % 16) return fail(FP8BS_ERR_MISALIGNED, "%s: O alignment", fn);
    const fp8bs_attn_input* in[3] = {Q, K, V};
    const int64_t width[3] = {wq, wkv, wkv};
    const int64_t rows[3] = {seq_q, seq_k, seq_k};
    for (int i = 0; i < 3; i++) {
        if (!valid_fmt(in[i]->fmt) || in[i]->reserved != 0)
            return fail(FP8BS_ERR_INVALID_ARG, "%s: bad format of input %d", fn, i);
        if (rows[i] == 0) continue;
        if (!in[i]->data || !in[i]->scales) return fail(FP8BS_ERR_INVALID_ARG, "%s: null data/scales (%d)", fn, i);
        if (in[i]->ld < width[i]) return fail(FP8BS_ERR_INVALID_ARG, "%s: ld too small (%d)", fn, i);
        if (!aligned16(in[i]->data) || in[i]->ld % 16 || !aligned4(in[i]->scales))
            return fail(FP8BS_ERR_MISALIGNED, "%s: input %d alignment", fn, i);
    }
    if (seq_q > (int64_t)INT32_MAX - 256 || seq_k > (int64_t)INT32_MAX - 256 || heads_q > 65535)
        return fail(FP8BS_ERR_UNSUPPORTED, "%s: dimension too large", fn);
    int rc;
    if ((rc = get_encoder()) != FP8BS_OK) return rc;
    CUtensorMap tmQ, tmK, tmV;
    if ((rc = make_map(&tmQ, Q->data, wq, seq_q, Q->ld, 128)) != FP8BS_OK) return rc;
    if (seq_k > 0) {
        if ((rc = make_map(&tmK, K->data, wkv, seq_k, K->ld, 128)) != FP8BS_OK) return rc;
        if ((rc = make_map(&tmV, V->data, wkv, seq_k, V->ld, 128)) != FP8BS_OK) return rc;
    } else {
        tmK = tmQ;   // never read: no key tile exists
        tmV = tmQ;
    }
    fp8bs::AttnParams p;
    memset(&p, 0, sizeof(p));
    p.seq_q = seq_q;
    p.seq_k = seq_k;
    p.hq = heads_q;
    p.hkv = heads_kv;
    p.causal = causal;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.sq = Q->scales;
    p.sk = K->scales;
    p.sv = V->scales;
    p.o = O;
    p.ldo = ld_o;
    p.idesc_s = fp8bs::make_idesc_f8f6f4(Q->fmt, K->fmt, false, false, 128);
    p.idesc_o = fp8bs::make_idesc_f8f6f4(FP8BS_E4M3, V->fmt, false, true, 128);
    cudaError_t e = fp8bs::launch_fp8_attn_fwd(tmQ, tmK, tmV, p, (cudaStream_t)stream);
    return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, fn);
}

int fp8bs_selftest_wait_timeout(int32_t limit_ms, int32_t* waited_ok, fp8bs_stream_t stream) {
    const char* fn = "fp8bs_selftest_wait_timeout";
    if (!waited_ok) return fail(FP8BS_ERR_INVALID_ARG, "%s: null output", fn);
    if (limit_ms < 1 || limit_ms > 10000) return fail(FP8BS_ERR_INVALID_ARG, "%s: limit_ms in [1, 10000]", fn);
    cudaError_t e = fp8bs::launch_wait_selftest(static_cast<uint64_t>(limit_ms) * 1000000ull, waited_ok,
                                                (cudaStream_t)stream);
    return e == cudaSuccess ? FP8BS_OK : cuda_fail(e, fn);
}

int fp8bs_device_status(fp8bs_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "fp8bs_device_status");
    int st = 0, sta = 0;
    e = fp8bs::read_and_clear_status(&st);
    if (e == cudaSuccess) e = fp8bs::read_and_clear_attn_status(&sta);
    if (e != cudaSuccess) return cuda_fail(e, "fp8bs_device_status");
    if (st == fp8bs::kStatusBadOffsets)
        return fail(FP8BS_ERR_INVALID_ARG, "a grouped product found decreasing row_offsets and wrote nothing");
    if (sta != 0) st = sta;
    if (st != 0) return fail(FP8BS_ERR_DEVICE_TIMEOUT, "a kernel gave up on a bounded device wait");
    return FP8BS_OK;
}

}  // extern "C"
