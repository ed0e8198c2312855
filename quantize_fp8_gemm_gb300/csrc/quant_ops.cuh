// quant_ops.cuh -- per-element arithmetic of the fused quantize, shared by
// the stand-alone quantize kernels (quant.cu) and the fused quantize + GEMM
// kernel (gemm.cu).
//
// "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records" (second
// paragraph): the activation is applied in registers, the BF16 copy kept for
// backward is written, and the FP8 copy is emitted under the delayed scale.
// Per element:  a = act(h);  abf = BF16(a);  v = abf * s (float32);
//               q = FP8(v) (round to nearest even, saturate);  amax = max |abf|.
#pragma once

#include "common.cuh"

#include <cfloat>

namespace fp8q {

template <int ACT>
__device__ __forceinline__ float act_f32(float h) {
    if constexpr (ACT == FP8Q_ACT_IDENTITY) {
        return h;
    } else {
        float r = h > 0.0f ? h : 0.0f;  // ReLU: +0 for h <= 0, -0 and NaN
        if constexpr (ACT == FP8Q_ACT_RELU) return r;
        return __fmul_rn(r, r);         // exact: a BF16 square fits in float32
    }
}

// ReLU^2 of two packed BF16 values, rounded to BF16: max(h, 0) (a NaN gives
// 0) squared by one BF16 multiply, which rounds the exact square once.  That
// equals BF16(float32(max(h, 0)^2)): a BF16 value has 8 significant bits, so
// its square has at most 16, whose lowest lies at or above 2^-148 whenever the
// square reaches 2^-134 -- there float32 holds it exactly -- and a square below
// 2^-134 (under half the smallest BF16 subnormal) gives 0 by either route.
__device__ __forceinline__ uint32_t relu2_bf16x2(uint32_t h2) {
    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&h2);
    const __nv_bfloat162 r = __hmax2(h, __float2bfloat162_rn(0.0f));  // a NaN lane gives the 0
    const __nv_bfloat162 q = __hmul2(r, r);
    return *reinterpret_cast<const uint32_t*>(&q);
}

// act + BF16 rounding of 8 packed BF16 inputs; returns the packed BF16 results
// and folds their magnitudes into `amax2` (two 16-bit lanes).  PACKED takes
// ReLU^2 through relu2_bf16x2 (the same results in fewer instructions: the
// fused kernel, whose quantize warps share issue slots with the GEMM); the
// stand-alone kernels, bound by HBM, keep the float32 route, with which they
// need no spills.
template <int ACT, bool PACKED = false>
__device__ __forceinline__ uint4 act8(uint4 x, uint32_t& amax2) {
    uint32_t in[4] = {x.x, x.y, x.z, x.w};
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (ACT == FP8Q_ACT_IDENTITY) {
            out[j] = in[j];
            amax2 = __vmaxu2(amax2, out[j] & 0x7FFF7FFFu);
        } else if constexpr (ACT == FP8Q_ACT_RELU2 && PACKED) {
            out[j] = relu2_bf16x2(in[j]);
            amax2 = __vmaxu2(amax2, out[j]);  // a square carries no sign
        } else {
            out[j] = cvt_bf16x2(act_f32<ACT>(bf16lo_to_f32(in[j])), act_f32<ACT>(bf16hi_to_f32(in[j])));
            amax2 = __vmaxu2(amax2, out[j] & 0x7FFF7FFFu);
        }
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// scale + FP8 cast of 8 packed BF16 values; counts |v| > max into `nsat`.
template <int FMT>
__device__ __forceinline__ uint2 cast8(uint4 a, float s, uint32_t& nsat) {
    constexpr float fmax = fp8_max_value(FMT);
    uint32_t in[4] = {a.x, a.y, a.z, a.w};
    uint32_t q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float v0 = __fmul_rn(bf16lo_to_f32(in[j]), s);
        float v1 = __fmul_rn(bf16hi_to_f32(in[j]), s);
        nsat += (fabsf(v0) > fmax) + (fabsf(v1) > fmax);
        q[j] = cvt_fp8x2<FMT>(v0, v1);
    }
    return make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

__device__ __forceinline__ uint32_t max16x2(uint32_t a2) { return max(a2 & 0xFFFFu, a2 >> 16); }

// The FP8 codes of 8 packed BF16 values scaled by s, as cast8 but without the
// saturation count: the two products of a pair are one packed float32
// multiply (mul.rn.f32x2: each lane one IEEE multiply, rounded once).
template <int FMT>
__device__ __forceinline__ uint2 cast8_codes(uint4 a, float s) {
    uint32_t in[4] = {a.x, a.y, a.z, a.w};
    uint32_t q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float v0, v1;
        asm("{\n\t.reg .b64 a, g;\n\t"
            "mov.b64 a, {%2, %3};\n\t"
            "mov.b64 g, {%4, %4};\n\t"
            "mul.rn.f32x2 a, a, g;\n\t"
            "mov.b64 {%0, %1}, a;\n\t}"
            : "=f"(v0), "=f"(v1)
            : "r"(in[j] << 16), "r"(in[j] & 0xFFFF0000u), "f"(s));
        q[j] = cvt_fp8x2<FMT>(v0, v1);
    }
    return make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

// #{ |float32(a_k * s)| > max } over 8 packed BF16 values.
template <int FMT>
__device__ __forceinline__ uint32_t sat_count8(uint4 a, float s) {
    constexpr float fmax = fp8_max_value(FMT);
    uint32_t in[4] = {a.x, a.y, a.z, a.w};
    uint32_t n = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        n += (fabsf(__fmul_rn(bf16lo_to_f32(in[j]), s)) > fmax) + (fabsf(__fmul_rn(bf16hi_to_f32(in[j]), s)) > fmax);
    return n;
}

// Whether any value of a batch whose magnitudes folded into m2 (act8's
// amax2) can saturate under s: the float32 product is monotonic in |a|, so
// the batch's largest |v| is float32(max |a| * s).
template <int FMT>
__device__ __forceinline__ bool may_saturate(uint32_t m2, float s) {
    return __fmul_rn(__uint_as_float(max16x2(m2) << 16), s) > fp8_max_value(FMT);
}

// Online group scale: max / amax_g (IEEE division), 1 for an all-zero group,
// clamped to FLT_MAX when the quotient overflows.
template <int FMT>
__device__ __forceinline__ float group_scale(uint32_t amax_bf16_bits) {
    if (amax_bf16_bits == 0) return 1.0f;
    float s = __fdiv_rn(fp8_max_value(FMT), __uint_as_float(amax_bf16_bits << 16));
    return s > FLT_MAX ? FLT_MAX : s;
}


}  // namespace fp8q
