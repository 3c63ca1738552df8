// mxq_quant_math.cuh -- device-side MXFP8 quantization arithmetic shared by the
// quantizer kernels and the GEMM's quantizing epilogue: the rceil exponent from
// BF16 bits, exact power-of-two scaling, packed maxima and FP8 conversions.
// One E8M0 scale per 32 elements with the exponent rounded up (torchtitan-npu
// low-precision tutorial, "MXFP8 与 HiF8 架构原理速览" and its "mxfp8_rceil" log
// keyword); payload E4M3 or E5M2 (MindSpeed RFC section 3.5.2.3).
#pragma once

#include <cstdint>

#include "mxq_device.cuh"

namespace mxq {

// E8M0 exponent of a finite, non-negative amax given as BF16 bits
// (sign cleared): e = ceil(log2(amax/448)), clamped below at -127.
// With amax = 1.m * 2^(E-127): amax/448 = (1.m/1.75) * 2^(E-135), and the
// ceiling steps up exactly when the 7-bit mantissa exceeds 1.75 (m > 96).
// Subnormal and zero amax (E == 0) fall below -127 and are clamped.
//
// Payload formats: kFmt 0 = E4M3 (max 448), 1 = E5M2 (max 57344 = 1.75 * 2^15,
// so the same mantissa test with the exponent offset 142 instead of 135).
template <int kFmt = 0>
__device__ __forceinline__ int rceil_exponent(uint32_t amax_bits) {
    const int E = static_cast<int>(amax_bits >> 7);
    const int m = static_cast<int>(amax_bits & 0x7Fu);
    const int e = E - (kFmt == 0 ? 135 : 142) + (m > 96 ? 1 : 0);
    return e < -127 ? -127 : e;
}

template <int kFmt>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
    return kFmt == 0 ? cvt_e4m3x2(lo, hi) : cvt_e5m2x2(lo, hi);
}

// 2^-e as a float for e in [-127, 120] (always a normal number).
__device__ __forceinline__ float pow2_neg(int e) { return __int_as_float((127 - e) << 23); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Per-half unsigned maximum of two packed 16-bit pairs (one instruction).
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Per-half max(|a|, |b|) of two BF16 pairs, NaN if either is NaN (the sign bit
// of the result is the XOR of the signs: mask it off).  One instruction.
__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Per-half BF16 product, round to nearest even.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// BF16 bits of 2^-e for e in [-127, 126] (a normal number).
__device__ __forceinline__ uint32_t pow2_neg_bf16(int e) { return static_cast<uint32_t>(127 - e) << 7; }

// Largest |x| (as BF16 bits, sign cleared) of 8 BF16 values; a group holding a
// NaN gives a NaN pattern, one holding an Inf (and no NaN) 0x7F80: both >= 0x7F80.
__device__ __forceinline__ uint32_t amax8_bits(const uint4 v) {
    const uint32_t m = max_abs_bf16x2(max_abs_bf16x2(v.x, v.y), max_abs_bf16x2(v.z, v.w)) & 0x7FFF7FFFu;
    return max(m & 0xFFFFu, m >> 16);
}

// Payload of a group holding NaN or Inf: every byte 0x7F | sign.
__device__ __forceinline__ uint32_t nan_bytes4(uint32_t w0, uint32_t w1) {
    return 0x7F7F7F7Fu | ((w0 >> 8) & 0x80u) | ((w0 >> 16) & 0x8000u) | ((w1 << 8) & 0x800000u) |
           (w1 & 0x80000000u);
}


}  // namespace mxq
