// quant.cu -- memory-bound FP8 quantizers for sm_103a.
//
//   k_quant_1x128     activations, one scale per 1x128 row tile
//   k_quant_128x128   weights, one scale per 128x128 tile
//   k_quant_tensor    per-tensor delayed scaling (scale in use + amax)
//   k_amax_history    delayed-scaling state update
//
// Block granularities from "NVIDIA NeMo RL logra una aceleracion del 48%..."
// (hotbookzone.com), "El avance tecnico"; formats and the delayed-scaling
// recipe from "Infraestructura de Entrenamiento FP8" (introl.com), "El
// panorama de la precision numerica" and "Transformer Engine: la base de
// software".
//
// Bit-exactness: each element is fp32(x * rcp_rn(s)) rounded once
// (__fmul_rn, no contraction), then cvt.rn.satfinite to the 8-bit format;
// the fp32 scale is the correctly rounded quotient __fdiv_rn(amax, fmax).
// This TU must not be built with fast-math or flush-to-zero.
#include <cuda_runtime.h>
#include <cstdint>
#include <cstring>

#include "quant_kernels.h"

namespace fp8bs {

template <int FMT>
struct Fmt;
template <>
struct Fmt<0> {  // E4M3 (FN)
    static constexpr float kMax = 448.0f;
    static constexpr int kEmax = 8;  // 448 = 1.75 * 2^8
};
template <>
struct Fmt<1> {  // E5M2
    static constexpr float kMax = 57344.0f;
    static constexpr int kEmax = 15;  // 57344 = 1.75 * 2^15
};

// Dequantization scale of a block (mode 0: fp32 amax/fmax, mode 1: power of
// two rounded up so the block maximum never saturates).
template <int FMT, int MODE>
__device__ __forceinline__ float block_scale(float amax) {
    if (!(amax > 0.0f)) return 1.0f;
    if (MODE == 0) {
        float s = __fdiv_rn(amax, Fmt<FMT>::kMax);
        return fmaxf(s, 0x1p-126f);
    }
    // amax = (1 + f) 2^E.  With fmax = 1.75 * 2^Emax the smallest e with
    // amax <= fmax 2^e is E - Emax, plus one when 1 + f > 1.75 (fraction
    // field above 0x600000).  Subnormal amax -> -126; infinity -> 127.
    const uint32_t b = __float_as_uint(amax);
    const int ef = static_cast<int>(b >> 23);
    int e;
    if (ef == 0) {
        e = -126;
    } else if (ef == 255) {
        e = 127;
    } else {
        e = (ef - 127) - Fmt<FMT>::kEmax + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
        e = max(-126, min(127, e));
    }
    return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// Two fp32 values -> two 8-bit codes (lo in bits 0-7, hi in bits 8-15).
template <int FMT>
__device__ __forceinline__ uint32_t cvt2(float lo, float hi) {
    uint16_t r;
    if (FMT == 0)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v2(void* p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ float amax8(const float (&f)[8]) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) m = fmaxf(m, fabsf(f[i]));
    return m;
}

template <int FMT>
__device__ __forceinline__ void quant8(const float (&f)[8], float r, uint32_t& lo, uint32_t& hi) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = __fmul_rn(f[i], r);
    lo = cvt2<FMT>(v[0], v[1]) | (cvt2<FMT>(v[2], v[3]) << 16);
    hi = cvt2<FMT>(v[4], v[5]) | (cvt2<FMT>(v[6], v[7]) << 16);
}

// ---------------------------------------------------------------- 1x128
// A half-warp owns one 1x128 tile: 16 lanes x 8 bf16 (one 16-byte load per
// lane), a 4-step shuffle-xor amax inside the half-warp, one 8-byte store per
// lane (128 contiguous code bytes per tile) and one scale store.  Grid: y =
// K block, x = group of 16*U rows; the 16 half-warps of a CTA take 16
// consecutive rows, so each of the U rounds writes 16 consecutive scales, and
// each thread keeps U loads in flight.
template <int FMT, int MODE, int U>
__global__ void __launch_bounds__(256) k_quant_1x128(const uint16_t* __restrict__ x, int64_t rows,
                                                    int64_t ldx, uint8_t* __restrict__ q, int64_t ldq,
                                                    float* __restrict__ scales) {
    const int l16 = threadIdx.x & 15;
    const int hw = threadIdx.x >> 4;
    const int64_t kb = blockIdx.y;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * (16 * U) + hw;
    const uint16_t* xk = x + kb * 128 + l16 * 8;
    uint4 v[U];
#pragma unroll
    for (int i = 0; i < U; i++) {
        const int64_t r = r0 + 16 * i;
        v[i] = make_uint4(0, 0, 0, 0);
        if (r < rows) v[i] = ld_stream_v4(xk + r * ldx);
    }
#pragma unroll
    for (int i = 0; i < U; i++) {
        const int64_t r = r0 + 16 * i;
        float f[8];
        unpack8(v[i], f);
        float m = amax8(f);
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (r < rows) {
            const float s = block_scale<FMT, MODE>(m);
            const float rc = __frcp_rn(s);
            uint32_t lo, hi;
            quant8<FMT>(f, rc, lo, hi);
            st_v2(q + r * ldq + kb * 128 + l16 * 8, lo, hi);
            if (l16 == 0) scales[kb * rows + r] = s;
        }
    }
}

// -------------------------------------------------------------- 128x128
// One CTA (256 threads) per 128x128 tile, held in registers: thread t reads
// the 16-byte chunk (t % 16) of rows t/16 + 16 i, i < 8 (a half-warp covers
// one 256-byte row segment).  CTA amax (shuffles + shared memory), one
// scale, then convert and store -- a single pass over the tile.
#ifndef FP8BS_Q128_MINB
#define FP8BS_Q128_MINB 3
#endif
template <int FMT, int MODE>
__global__ void __launch_bounds__(256, FP8BS_Q128_MINB) k_quant_128x128(const uint16_t* __restrict__ w, int64_t rows,
                                                      int64_t ldw, int64_t nkb,
                                                      uint8_t* __restrict__ q, int64_t ldq,
                                                      float* __restrict__ scales) {
    __shared__ float red[8];
    const int64_t rb = blockIdx.x / nkb;
    const int64_t kb = blockIdx.x - rb * nkb;
    const int c = threadIdx.x & 15;
    const int r0 = threadIdx.x >> 4;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int64_t row = rb * 128 + r0 + 16 * i;
        v[i] = make_uint4(0, 0, 0, 0);
        if (row < rows) v[i] = ld_stream_v4(w + row * ldw + kb * 128 + c * 8);
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        float f[8];
        unpack8(v[i], f);
        m = fmaxf(m, amax8(f));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int i = 1; i < 8; i++) m = fmaxf(m, red[i]);
    const float s = block_scale<FMT, MODE>(m);
    const float r = __frcp_rn(s);
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int64_t row = rb * 128 + r0 + 16 * i;
        if (row < rows) {
            float f[8];
            unpack8(v[i], f);
            uint32_t lo, hi;
            quant8<FMT>(f, r, lo, hi);
            st_v2(q + row * ldq + kb * 128 + c * 8, lo, hi);
        }
    }
    if (threadIdx.x == 0) scales[rb * nkb + kb] = s;
}

// ------------------------------------------------------- per-tensor delayed
// Quantize with the scale in use and reduce this tensor's amax: each thread
// handles U 16-byte vectors (grid-contiguous per iteration), CTA reduction,
// one atomicMax on the float bits (amax >= 0, so unsigned order is float
// order).  amax_out is zeroed on the stream before the launch.
template <int FMT, int U>
__global__ void __launch_bounds__(256) k_quant_tensor(const uint16_t* __restrict__ x, int64_t n,
                                                     const float* __restrict__ scale,
                                                     uint8_t* __restrict__ q,
                                                     float* __restrict__ amax_out) {
    __shared__ float red[8];
    const float r = __frcp_rn(*scale);
    const int64_t nvec = n >> 3;
    const int64_t base = static_cast<int64_t>(blockIdx.x) * (256 * U) + threadIdx.x;
    uint4 v[U];
#pragma unroll
    for (int i = 0; i < U; i++) {
        const int64_t idx = base + 256 * i;
        v[i] = make_uint4(0, 0, 0, 0);
        if (idx < nvec) v[i] = ld_stream_v4(x + idx * 8);
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < U; i++) {
        const int64_t idx = base + 256 * i;
        if (idx < nvec) {
            float f[8];
            unpack8(v[i], f);
            m = fmaxf(m, amax8(f));
            uint32_t lo, hi;
            quant8<FMT>(f, r, lo, hi);
            st_v2(q + idx * 8, lo, hi);
        }
    }
    if (blockIdx.x == 0) {  // ragged tail (numel % 8)
        for (int64_t i = nvec * 8 + threadIdx.x; i < n; i += blockDim.x) {
            const float f = __uint_as_float(static_cast<uint32_t>(x[i]) << 16);
            m = fmaxf(m, fabsf(f));
            q[i] = static_cast<uint8_t>(cvt2<FMT>(__fmul_rn(f, r), 0.0f));
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = red[0];
#pragma unroll
        for (int i = 1; i < 8; i++) b = fmaxf(b, red[i]);
        atomicMax(reinterpret_cast<unsigned int*>(amax_out), __float_as_uint(b));
    }
}

// ------------------------------------------------------ history update
template <int FMT>
__global__ void __launch_bounds__(256) k_amax_history(float* __restrict__ history,
                                                     int32_t* __restrict__ head, int32_t L,
                                                     const float* __restrict__ amax,
                                                     float margin_mult,
                                                     float* __restrict__ scale) {
    __shared__ float red[8];
    __shared__ int32_t h;
    if (threadIdx.x == 0) {
        h = *head;
        history[h] = *amax;
    }
    __syncthreads();
    float m = 0.0f;
    for (int32_t i = threadIdx.x; i < L; i += blockDim.x) m = fmaxf(m, history[i]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = red[0];
        for (int i = 1; i < 8; i++) a = fmaxf(a, red[i]);
        *head = (h + 1) % L;
        if (a > 0.0f) {
            float t = __fmul_rn(__fdiv_rn(a, Fmt<FMT>::kMax), margin_mult);
            if (isfinite(t) && t > 0.0f) *scale = fmaxf(t, 0x1p-126f);
        }
    }
}

// ------------------------------------------------------------ launchers
namespace {
#ifndef FP8BS_U1
#define FP8BS_U1 4
#endif
constexpr int kU1 = FP8BS_U1;   // tiles in flight per half-warp (1x128)
#ifndef FP8BS_UT
#define FP8BS_UT 8
#endif
constexpr int kUT = FP8BS_UT;   // vectors in flight per thread (per-tensor)
}  // namespace

cudaError_t launch_quant_1x128(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                               int fmt, int mode, uint8_t* q, int64_t ldq, float* scales,
                               cudaStream_t st) {
    const int64_t gx = (rows + 16 * kU1 - 1) / (16 * kU1), gy = cols / 128;
    if (gx > 0x7FFFFFFF || gy > 65535) return cudaErrorInvalidValue;
    auto k = fmt == 0 ? (mode == 0 ? k_quant_1x128<0, 0, kU1> : k_quant_1x128<0, 1, kU1>)
                      : (mode == 0 ? k_quant_1x128<1, 0, kU1> : k_quant_1x128<1, 1, kU1>);
    k<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), 256, 0, st>>>(x, rows, ldx, q, ldq,
                                                                                 scales);
    return cudaGetLastError();
}

cudaError_t launch_quant_128x128(const uint16_t* w, int64_t rows, int64_t cols, int64_t ldw,
                                 int fmt, int mode, uint8_t* q, int64_t ldq, float* scales,
                                 cudaStream_t st) {
    const int64_t nkb = cols / 128, nrb = (rows + 127) / 128;
    const int64_t grid = nkb * nrb;
    if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
    auto k = fmt == 0 ? (mode == 0 ? k_quant_128x128<0, 0> : k_quant_128x128<0, 1>)
                      : (mode == 0 ? k_quant_128x128<1, 0> : k_quant_128x128<1, 1>);
    k<<<static_cast<unsigned>(grid), 256, 0, st>>>(w, rows, ldw, nkb, q, ldq, scales);
    return cudaGetLastError();
}

cudaError_t launch_quant_tensor(const uint16_t* x, int64_t n, int fmt, const float* scale,
                                uint8_t* q, float* amax_out, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), st);
    if (e != cudaSuccess) return e;
    const int64_t nvec = n >> 3;
    int64_t grid = (nvec + 256 * kUT - 1) / (256 * kUT);
    if (grid < 1) grid = 1;  // the tail and the amax write still need a CTA
    if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
    auto k = fmt == 0 ? k_quant_tensor<0, kUT> : k_quant_tensor<1, kUT>;
    k<<<static_cast<unsigned>(grid), 256, 0, st>>>(x, n, scale, q, amax_out);
    return cudaGetLastError();
}

cudaError_t launch_amax_history(float* history, int32_t* head, int32_t L, const float* amax,
                                int fmt, int32_t margin, float* scale, cudaStream_t st) {
    const uint32_t bits = static_cast<uint32_t>(margin + 127) << 23;  // 2^margin, |margin| <= 126
    float mult;
    memcpy(&mult, &bits, sizeof(mult));
    auto k = fmt == 0 ? k_amax_history<0> : k_amax_history<1>;
    k<<<1, 256, 0, st>>>(history, head, L, amax, mult, scale);
    return cudaGetLastError();
}

}  // namespace fp8bs
