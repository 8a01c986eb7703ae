// gemm_kernels.h -- launch interface of the tcgen05 FP8 GEMM (gemm.cu),
// called by the C ABI layer after argument validation.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fp8bs {

constexpr int kMaxGroups = 1024;
constexpr int kStatusDeviceTimeout = -5;   // FP8BS_ERR_DEVICE_TIMEOUT
constexpr int kStatusBadOffsets = -1;      // FP8BS_ERR_INVALID_ARG: decreasing group offsets

struct GemmParams {
    int64_t M, N, K;          // logical product size (M = rows of A as stored)
    int64_t a_rows;           // rows of A as stored: 1x128 scale table stride
    int64_t a_rblocks;        // ceil(M / 128): transposed 128x128 A scale stride
    int64_t b_rblocks;        // ceil(N / 128): transposed 128x128 B scale stride
    int64_t b_scale_group_stride;  // floats between groups' B scale tables
    const float* sa;
    const float* sb;
    const int32_t* offsets;   // device [num_groups + 1] or null (one group [0, M))
    void* y;
    int64_t ldy;
    int32_t num_groups;
    int32_t b_rows_per_group; // rows of the B tensor map per group (grouped: N)
    int32_t a_gran, b_gran;   // fp8bs_granularity
    int32_t tiles_n;
    int32_t promote;          // 1: scale per 128-K block; 0: one scale per tensor pair
    int32_t out_bf16;
    int32_t tma_store;        // 1: tmY describes Y (box 32 rows x 64 B, 64-B swizzle)
    int32_t sa_bulk;          // 1: 1x128 A scale table 16-byte aligned with a_rows % 4 == 0
                              //    (copied by bulk copies, a K block's rows at once)
    uint32_t idesc;
    // Quantized output: Y holds 8-bit codes [rows][n_out] and sq its 1x128
    // scales [n_out/128][a_rows] (the next linear's activation operand).
    int32_t out_q, q_fmt, q_mode;
    float* sq;
    int64_t n_out;            // columns of Y (N, or N/2 with SwiGLU)
    // SwiGLU: B's rows [0, swiglu_i) are gate rows and [swiglu_i, 2 swiglu_i)
    // the matching up rows (per group); Y = silu(gate) * up.
    int32_t swiglu;
    int64_t swiglu_i;
    // MXFP8 operands (both): scale tables of 32-bit E8M0 words [K/128][rows],
    // byte j = scale of the K elements 32 j .. 32 j + 31 of the block
    int32_t mx32;
};

uint32_t make_idesc_f8f6f4(int a_fmt, int b_fmt, bool a_mn, bool b_mn, int n);
int gemm_tile_n();
int gemm_mma_n(bool b_col);   // N of one tcgen05.mma (K-major B; b_col: per-column B scales);
                              // an MN-major B always uses 128
int gemm_tile_m();
cudaError_t launch_fp8_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmY,
                            const GemmParams& p, bool a_mn, bool b_mn, int grid, cudaStream_t st);
uint32_t make_idesc_mx(int a_fmt, int b_fmt, int n);
cudaError_t launch_fp8_gemm_mx(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmY,
                               const CUtensorMap& tmSA, const GemmParams& p, int grid, cudaStream_t st);
cudaError_t read_and_clear_status(int* status);
cudaError_t launch_wait_selftest(uint64_t limit_ns, int* out, cudaStream_t st);
cudaError_t launch_fill_f32(float* p, int64_t n, float v, cudaStream_t st);

}  // namespace fp8bs
