// naive.cu -- the unfused three-pass quantize (measured comparator only).
// Built into its own library, libfp8q_naive.so, not into libfp8q.so: it is
// not part of the down-projection path.
//
// "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records", second
// paragraph: write the intermediate tensor, scan it for its maximum, read it
// again to convert it.  Each pass is its own grid-stride kernel with 16-byte
// accesses, so the comparison with the fused kernel is about passes over HBM,
// not about code quality.
#include "../common.cuh"
#include "../../../include/fp8q_naive.h"

#include <algorithm>

namespace fp8q {
namespace {

constexpr int kT = 256;

int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
        (void)cudaGetLastError();
        return 1;
    }
    return sms;
}

unsigned grid_for(int64_t nchunks) {
    const int64_t want = (nchunks + kT - 1) / kT;
    const int64_t cap = static_cast<int64_t>(device_sms()) * (2048 / kT);
    return static_cast<unsigned>(std::max<int64_t>(1, std::min(want, cap)));
}

template <int ACT>
__global__ void __launch_bounds__(kT) naive_act_kernel(const uint4* __restrict__ h, int64_t n8, uint4* __restrict__ out) {
    for (int64_t i = blockIdx.x * int64_t(kT) + threadIdx.x; i < n8; i += int64_t(gridDim.x) * kT) {
        uint4 x = ld_stream_v4(h + i);
        uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (ACT != FP8Q_ACT_IDENTITY) {
                float lo = bf16lo_to_f32(w[j]), hi = bf16hi_to_f32(w[j]);
                lo = lo > 0.0f ? lo : 0.0f;
                hi = hi > 0.0f ? hi : 0.0f;
                if (ACT == FP8Q_ACT_RELU2) { lo = __fmul_rn(lo, lo); hi = __fmul_rn(hi, hi); }
                w[j] = cvt_bf16x2(lo, hi);
            }
        }
        st_v4(out + i, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

__global__ void __launch_bounds__(kT) naive_amax_kernel(const uint4* __restrict__ x, int64_t n8, float* amax_out) {
    uint32_t m2 = 0;
    for (int64_t i = blockIdx.x * int64_t(kT) + threadIdx.x; i < n8; i += int64_t(gridDim.x) * kT) {
        uint4 v = ld_stream_v4(x + i);
        m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __shared__ uint32_t s[kT / 32];
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kT / 32; ++w) m = max(m, s[w]);
        m = max(m, s[0]);
        if (m) atomicMax(reinterpret_cast<unsigned int*>(amax_out), m << 16);
    }
}

template <int FMT>
__global__ void __launch_bounds__(kT) naive_cast_kernel(const uint4* __restrict__ x, int64_t n8, const float* amax,
                                                        float margin, float* scale_out, uint2* __restrict__ q) {
    const float a = *amax;
    const float s = a > 0.0f ? __fdiv_rn(fp8_max_value(FMT), __fmul_rn(margin, a)) : 1.0f;
    if (scale_out && blockIdx.x == 0 && threadIdx.x == 0) *scale_out = s;
    for (int64_t i = blockIdx.x * int64_t(kT) + threadIdx.x; i < n8; i += int64_t(gridDim.x) * kT) {
        uint4 v = ld_stream_v4(x + i);
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            c[j] = cvt_fp8x2<FMT>(__fmul_rn(bf16lo_to_f32(w[j]), s), __fmul_rn(bf16hi_to_f32(w[j]), s));
        st_v2(q + i, make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16)));
    }
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" int fp8q_naive_act(const void* h, int64_t M, int64_t K, int act, void* act_out, cudaStream_t stream) {
    if (!h || !act_out) return FP8Q_ERR_NULL;
    if (M < 0 || K < 16 || K % 16) return FP8Q_ERR_SHAPE;
    if (act < 0 || act > 2) return FP8Q_ERR_UNSUPPORTED;
    if (!aligned16(h) || !aligned16(act_out)) return FP8Q_ERR_ALIGN;
    const int64_t n8 = M * K / 8;
    if (n8 == 0) return FP8Q_OK;
    const unsigned g = grid_for(n8);
    if (act == FP8Q_ACT_IDENTITY) naive_act_kernel<FP8Q_ACT_IDENTITY><<<g, kT, 0, stream>>>((const uint4*)h, n8, (uint4*)act_out);
    else if (act == FP8Q_ACT_RELU) naive_act_kernel<FP8Q_ACT_RELU><<<g, kT, 0, stream>>>((const uint4*)h, n8, (uint4*)act_out);
    else naive_act_kernel<FP8Q_ACT_RELU2><<<g, kT, 0, stream>>>((const uint4*)h, n8, (uint4*)act_out);
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}

extern "C" int fp8q_naive_amax(const void* x, int64_t n, float* amax_out, cudaStream_t stream) {
    if (!x || !amax_out) return FP8Q_ERR_NULL;
    if (n < 0 || n % 8) return FP8Q_ERR_SHAPE;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(amax_out) & 3u)) return FP8Q_ERR_ALIGN;
    if (cudaMemsetAsync(amax_out, 0, sizeof(float), stream) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (n == 0) return FP8Q_OK;
    naive_amax_kernel<<<grid_for(n / 8), kT, 0, stream>>>((const uint4*)x, n / 8, amax_out);
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}

extern "C" int fp8q_naive_cast(const void* x, int64_t n, int fmt, const float* amax, float margin,
                               float* scale_out, void* q_out, cudaStream_t stream) {
    if (!x || !amax || !q_out) return FP8Q_ERR_NULL;
    if (n < 0 || n % 8) return FP8Q_ERR_SHAPE;
    if (fmt != FP8Q_E4M3 && fmt != FP8Q_E5M2) return FP8Q_ERR_UNSUPPORTED;
    if (!(margin > 0.0f)) return FP8Q_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q_out)) return FP8Q_ERR_ALIGN;
    if (n == 0) return FP8Q_OK;
    const unsigned g = grid_for(n / 8);
    if (fmt == FP8Q_E5M2) naive_cast_kernel<FP8Q_E5M2><<<g, kT, 0, stream>>>((const uint4*)x, n / 8, amax, margin, scale_out, (uint2*)q_out);
    else naive_cast_kernel<FP8Q_E4M3><<<g, kT, 0, stream>>>((const uint4*)x, n / 8, amax, margin, scale_out, (uint2*)q_out);
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}
