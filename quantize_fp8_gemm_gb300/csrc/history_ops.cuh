// history_ops.cuh -- one delayed-scaling update, done by one warp: used by the
// history kernel (history.cu) and by the last CTA of the fused step kernel
// (gemm.cu).
//
// "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records" (second
// paragraph): the scale uses the previous step's maximum multiplied by a
// safety margin.  "FP8 training: what it is and how it works", Step 2 (scale
// = format max / amax) and Trade-offs (a stored history of amax values).
//
//   *head = (*head + 1) % L;  history[*head] = amax_new;
//   amax_ref = max(history);  s = float32(fmt_max / float32(margin * amax_ref));
//   *scale_out = s if amax_ref and s are positive and finite, else the
//   previous scale (*scale_prev when given, or left alone) and FP8Q_DEV_BAD_AMAX
//   into *status;  then *amax_clear = 0, *sat_clear = 0 when given.
#pragma once

#include "common.cuh"

namespace fp8q {

struct HistoryArgs {
    float* history;
    int L;
    int* head;
    float margin;
    float fmt_max;
    const float* scale_prev;        // or nullptr
    float* scale_out;
    int* status;                    // or nullptr
    float* amax_clear;              // or nullptr
    unsigned long long* sat_clear;  // or nullptr
};

// Called by all 32 lanes of one warp.
__device__ __forceinline__ void history_update_warp(const HistoryArgs& a, const float* amax_new) {
    const int lane = threadIdx.x & 31;
    // the loads are independent: issue them together
    const int h0 = *a.head;
    const float a_new = __ldcg(amax_new);  // final in L2 (atomics), never from L1
    const float prev = a.scale_prev ? *a.scale_prev : 0.0f;
    const float first = lane < a.L ? a.history[lane] : 0.0f;
    const int slot = (h0 + 1) % a.L;
    // |x| as an ordered key: bit patterns of non-negative floats sort like the
    // floats, and a NaN magnitude sorts above infinity
    uint32_t key = 0;
    for (int i = lane; i < a.L; i += 32) {
        const float v = (i == slot) ? a_new : (i == lane ? first : a.history[i]);
        key = max(key, __float_as_uint(v) & 0x7FFFFFFFu);
    }
    key = __reduce_max_sync(0xFFFFFFFFu, key);
    __syncwarp();
    if (lane == 0) {
        a.history[slot] = a_new;
        *a.head = slot;
        const float ref = __uint_as_float(key);
        bool ok = ref > 0.0f && ref <= 3.402823466e38f;
        float s = 0.0f;
        if (ok) {
            const float d = __fmul_rn(a.margin, ref);
            s = __fdiv_rn(a.fmt_max, d);
            ok = s > 0.0f && s <= 3.402823466e38f;
        }
        if (ok) {
            *a.scale_out = s;
        } else {
            if (a.scale_prev) *a.scale_out = prev;
            if (a.status) atomicOr(a.status, FP8Q_DEV_BAD_AMAX);
        }
        if (a.amax_clear) *a.amax_clear = 0.0f;
        if (a.sat_clear) *a.sat_clear = 0ull;
    }
}

// Host check of one fp8q_history_args (the rules of amax_history_update_ex)
// and its device form.
inline int check_history(const fp8q_history_args* h, const float* amax_new, HistoryArgs* out) {
    if (!h->history || !h->head || !h->scale_out || !amax_new) return FP8Q_ERR_NULL;
    if (h->L < 1 || h->L > 4096) return FP8Q_ERR_SHAPE;
    if (h->fmt != FP8Q_E4M3 && h->fmt != FP8Q_E5M2) return FP8Q_ERR_UNSUPPORTED;
    if (!(h->margin > 0.0f) || h->margin > 3.402823466e38f) return FP8Q_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(h->history) | reinterpret_cast<uintptr_t>(h->head) |
         reinterpret_cast<uintptr_t>(h->scale_out) | reinterpret_cast<uintptr_t>(h->scale_prev) |
         reinterpret_cast<uintptr_t>(h->status) | reinterpret_cast<uintptr_t>(h->amax_clear)) & 3u)
        return FP8Q_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(h->sat_clear) & 7u) return FP8Q_ERR_ALIGN;
    if (h->amax_clear && h->amax_clear == amax_new) return FP8Q_ERR_SHAPE;
    out->history = h->history;
    out->L = h->L;
    out->head = h->head;
    out->margin = h->margin;
    out->fmt_max = fp8_max_value(h->fmt);
    out->scale_prev = h->scale_prev;
    out->scale_out = h->scale_out;
    out->status = h->status;
    out->amax_clear = h->amax_clear;
    out->sat_clear = h->sat_clear;
    return FP8Q_OK;
}

}  // namespace fp8q
