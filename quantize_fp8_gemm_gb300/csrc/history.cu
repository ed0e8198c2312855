// history.cu -- delayed per-tensor scaling: the amax history ring and the
// scale for the next step, plus the library's small host utilities.
//
// "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records" (second
// paragraph): the scale uses the previous step's maximum multiplied by a
// safety margin, so no step waits on its own maximum.  "FP8 training: what it
// is and how it works", Step 2 (scale = format max / amax) and Trade-offs
// (delayed scaling keeps a stored history of amax values).  "FP8 Training &
// Inference", Delayed Scaling.
//
// One warp: the newest amax goes into the next ring slot, the window maximum
// is a warp reduction over the L entries, and the scale is
//     s = float32( fmt_max / float32(margin * amax_ref) ),
// written only when amax_ref and s are positive and finite (else the previous
// scale is kept, copied from scale_prev when one is given).  The same launch
// can zero the accumulators the next step's cast folds into.
#include "common.cuh"
#include "history_ops.cuh"

#include <mutex>

namespace fp8q {

namespace {

constexpr int kMaxDevices = 64;

__global__ void __launch_bounds__(32)
amax_history_kernel(float* __restrict__ history, int L, int* __restrict__ head,
                    const float* __restrict__ amax_new, float margin, float fmt_max,
                    float* __restrict__ scale_out, int* __restrict__ status, const float* scale_prev,
                    float* amax_clear, unsigned long long* sat_clear) {
    pdl_launch_dependents();
    pdl_wait();
    HistoryArgs a;
    a.history = history;
    a.L = L;
    a.head = head;
    a.margin = margin;
    a.fmt_max = fmt_max;
    a.scale_prev = scale_prev;
    a.scale_out = scale_out;
    a.status = status;
    a.amax_clear = amax_clear;
    a.sat_clear = sat_clear;
    history_update_warp(a, amax_new);
}

struct DeviceInfo {
    int sms = 0;
    int major = 0;
    int minor = 0;
};

DeviceInfo g_info[kMaxDevices];
std::once_flag g_once[kMaxDevices];

const DeviceInfo* current_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::call_once(g_once[dev], [dev] {
        cudaDeviceGetAttribute(&g_info[dev].sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&g_info[dev].major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&g_info[dev].minor, cudaDevAttrComputeCapabilityMinor, dev);
    });
    return &g_info[dev];
}

}  // namespace

int sm_count() {
    const DeviceInfo* d = current_info();
    return (d && d->sms > 0) ? d->sms : 1;
}

bool device_is_sm103() {
    const DeviceInfo* d = current_info();
    return d && d->major == 10 && d->minor == 3;
}

}  // namespace fp8q

using namespace fp8q;

extern "C" int amax_history_update(float* history, int L, int* head, const float* amax_new,
                                   float margin, int fmt, float* scale_out, int* status,
                                   cudaStream_t stream) {
    return amax_history_update_ex(history, L, head, amax_new, margin, fmt, nullptr, scale_out, status, nullptr,
                                  nullptr, stream);
}

extern "C" int amax_history_update_ex(float* history, int L, int* head, const float* amax_new, float margin,
                                      int fmt, const float* scale_prev, float* scale_out, int* status,
                                      float* amax_clear, unsigned long long* sat_clear, cudaStream_t stream) {
    if (!history || !head || !amax_new || !scale_out) return FP8Q_ERR_NULL;
    if (L < 1 || L > 4096) return FP8Q_ERR_SHAPE;
    if (fmt != FP8Q_E4M3 && fmt != FP8Q_E5M2) return FP8Q_ERR_UNSUPPORTED;
    if (!(margin > 0.0f) || margin > 3.402823466e38f) return FP8Q_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(history) | reinterpret_cast<uintptr_t>(head) |
         reinterpret_cast<uintptr_t>(amax_new) | reinterpret_cast<uintptr_t>(scale_out) |
         reinterpret_cast<uintptr_t>(status) | reinterpret_cast<uintptr_t>(scale_prev) |
         reinterpret_cast<uintptr_t>(amax_clear)) & 3u)
        return FP8Q_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(sat_clear) & 7u) return FP8Q_ERR_ALIGN;
    if (amax_clear && amax_clear == amax_new) return FP8Q_ERR_SHAPE;  // it is read, not cleared
    if (!device_is_sm103()) return FP8Q_ERR_UNSUPPORTED;
    if (launch_pdl(amax_history_kernel, dim3(1), dim3(32), 0, stream, history, L, head, amax_new, margin,
                   fp8_max_value(fmt), scale_out, status, scale_prev, amax_clear, sat_clear) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8Q_ERR_CUDA;
    }
    return FP8Q_OK;
}

extern "C" const char* fp8q_status_string(int status) {
    switch (status) {
        case FP8Q_OK: return "ok";
        case FP8Q_ERR_NULL: return "a required pointer is NULL";
        case FP8Q_ERR_ALIGN: return "a tensor pointer is not suitably aligned";
        case FP8Q_ERR_SHAPE: return "a size is out of range or breaks a multiple-of rule";
        case FP8Q_ERR_UNSUPPORTED: return "unsupported enum value or device (needs sm_103)";
        case FP8Q_ERR_CUDA: return "a CUDA call or kernel launch failed";
        default: return "unknown status";
    }
}

extern "C" int fp8q_version(void) { return 100; }
