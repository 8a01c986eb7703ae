// fp8_math.cuh -- the FP8 element and block-scale rules shared by the
// quantizer kernels (quant.cu) and the GEMM epilogue that quantizes its own
// output (gemm.cu).
//
// Formats: E4M3 (the "FN" variant, max 448) for activations and weights, E5M2
// (max 57344) for gradients ("Infraestructura de Entrenamiento FP8",
// introl.com, "El panorama de la precision numerica").  Block scales are
// dequantization multipliers built from the block's amax; the power-of-two
// option follows "NVIDIA NeMo RL logra una aceleracion del 48%..."
// (hotbookzone.com), "Por que esto es importante...".
//
// Elements are fp32(x * rcp_rn(s)) rounded once (__fmul_rn, no contraction),
// then cvt.rn.satfinite to the 8-bit format.  Units including this header
// must not be built with fast-math or flush-to-zero.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

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

// Runtime-format form for kernels that take fmt and mode as parameters.
__device__ __forceinline__ float block_scale_rt(float amax, int fmt, int mode) {
    if (fmt == 0) return mode == 0 ? block_scale<0, 0>(amax) : block_scale<0, 1>(amax);
    return mode == 0 ? block_scale<1, 0>(amax) : block_scale<1, 1>(amax);
}

// MXFP8 block scale (32-element blocks, E8M0 code = e + 127): e =
// floor(log2(amax)) - Emax of the element format, clamped to [-127, 127]
// (zero and subnormal amax give -127); a non-finite amax gives code 255 (NaN)
// and a NaN multiplier.  `mult` = 2^-e, exact.
template <int FMT>
__device__ __forceinline__ void mx_scale(float amax, uint32_t& code, float& mult) {
    const int ef = static_cast<int>(__float_as_uint(amax) >> 23);   // amax >= 0
    if (ef >= 255) {
        code = 255u;
        mult = __uint_as_float(0x7FC00000u);
        return;
    }
    const int e = ef == 0 ? -127 : max(-127, ef - 127 - Fmt<FMT>::kEmax);
    code = static_cast<uint32_t>(e + 127);
    mult = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
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

// Four fp32 values -> four E4M3 codes in one word (element 0 in the low byte),
// the two halves packed by a register-pair move.
__device__ __forceinline__ uint32_t cvt4_e4m3(float a, float b, float c, float d) {
    uint32_t w;
    asm("{\n.reg .b16 lo, hi;\n"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
        "mov.b32 %0, {lo, hi};\n}"
        : "=r"(w)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return w;
}

__device__ __forceinline__ uint32_t cvt2_rt(float lo, float hi, int fmt) {
    return fmt == 0 ? cvt2<0>(lo, hi) : cvt2<1>(lo, hi);
}

// Four fp32 values (two packed pairs) times r -> four codes in one word,
// element 0 in the low byte.
__device__ __forceinline__ uint32_t quant4_rt(float a, float b, float c, float d, float r, int fmt) {
    return cvt2_rt(__fmul_rn(a, r), __fmul_rn(b, r), fmt) |
           (cvt2_rt(__fmul_rn(c, r), __fmul_rn(d, r), fmt) << 16);
}

}  // namespace fp8bs
