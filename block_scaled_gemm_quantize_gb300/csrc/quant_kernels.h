// quant_kernels.h -- launchers of the quantizer kernels (quant.cu), called
// by the C ABI layer after argument validation.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

namespace fp8bs {
cudaError_t launch_quant_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                               int fmt, int mode, uint8_t* q, int64_t ldq, float* scales,
                               cudaStream_t st);
cudaError_t launch_quant_128x128(const uint16_t* w, int64_t rows, int64_t cols, int64_t ldw,
                                 int fmt, int mode, uint8_t* q, int64_t ldq, float* scales,
                                 cudaStream_t st);
// X [m][k] per 1x128 tile and W [n][k] per 128x128 tile in one launch
cudaError_t launch_quant_linear(const uint16_t* x, int64_t m, int64_t ldx, uint8_t* qx, int64_t ldqx, float* sx,
                                const uint16_t* w, int64_t n, int64_t ldw, uint8_t* qw, int64_t ldqw, float* sw,
                                int64_t k, int fmt, int mode, cudaStream_t st);
cudaError_t launch_quant_mx(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, int fmt,
                            uint8_t* q, int64_t ldq, uint32_t* scales, cudaStream_t st);
cudaError_t launch_quant_colwise(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                                int fmt, int mode, uint8_t* qt, int64_t ldqt, float* sqt,
                                uint8_t* q, int64_t ldq, float* sq, cudaStream_t st);
cudaError_t launch_quant_tensor(const uint16_t* x, int64_t n, int fmt, const float* scale,
                                uint8_t* q, float* amax_out, cudaStream_t st);
cudaError_t launch_amax_history(float* history, int32_t* head, int32_t L, const float* amax,
                                int fmt, int32_t margin, float* scale, cudaStream_t st);
}  // namespace fp8bs
