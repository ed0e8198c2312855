/*
 * fp8q_naive.h -- the unfused three-pass quantize, kept as a measured
 * comparator for fp8_quant_fused.  Not part of the down-projection path.
 *
 * "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records", second
 * paragraph: done naively, quantization writes out the whole intermediate
 * tensor, scans it once to find the maximum, and reads it again to convert
 * it; those extra passes erase most of the FP8 speed-up.  These three calls
 * are those passes (9 bytes of HBM traffic per element against the fused
 * kernel's 5), with a just-in-time scale from the tensor's own amax
 * ("FP8 Training & Inference", Delayed Scaling: the problem with just-in-time
 * scaling).
 *
 * Same conventions as fp8q.h: device pointers, caller-owned memory, 16-byte
 * aligned tensors, stream-ordered, fp8q_status return codes.
 */
#ifndef FP8Q_NAIVE_H
#define FP8Q_NAIVE_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Pass 1: act_out[M,K] = BF16(act(h)).  K % 16 == 0, M >= 0. */
int fp8q_naive_act(const void* h, int64_t M, int64_t K, int act, void* act_out, cudaStream_t stream);

/* Pass 2: *amax_out = max |x| over n BF16 values (n % 8 == 0); zeroed first. */
int fp8q_naive_amax(const void* x, int64_t n, float* amax_out, cudaStream_t stream);

/* Pass 3: s = float32(fmt_max / float32(margin * *amax)) (1 when *amax is 0),
 * q_out[i] = FP8(float32(x[i] * s)); s is also stored to *scale_out
 * (device float, may be NULL).  n % 8 == 0. */
int fp8q_naive_cast(const void* x, int64_t n, int fmt, const float* amax, float margin,
                    float* scale_out, void* q_out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_NAIVE_H */
