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

// act + BF16 rounding of 8 packed BF16 inputs; returns the packed BF16 results
// and folds their magnitudes into `amax2` (two 16-bit lanes).
template <int ACT>
__device__ __forceinline__ uint4 act8(uint4 x, uint32_t& amax2) {
    uint32_t in[4] = {x.x, x.y, x.z, x.w};
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (ACT == FP8Q_ACT_IDENTITY) {
            out[j] = in[j];
        } else {
            out[j] = cvt_bf16x2(act_f32<ACT>(bf16lo_to_f32(in[j])), act_f32<ACT>(bf16hi_to_f32(in[j])));
        }
        amax2 = __vmaxu2(amax2, out[j] & 0x7FFF7FFFu);
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

// Online group scale: max / amax_g (IEEE division), 1 for an all-zero group,
// clamped to FLT_MAX when the quotient overflows.
template <int FMT>
__device__ __forceinline__ float group_scale(uint32_t amax_bf16_bits) {
    if (amax_bf16_bits == 0) return 1.0f;
    float s = __fdiv_rn(fp8_max_value(FMT), __uint_as_float(amax_bf16_bits << 16));
    return s > FLT_MAX ? FLT_MAX : s;
}


}  // namespace fp8q
