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
// written only when amax_ref and s are positive and finite.
#include "common.cuh"

#include <mutex>

namespace fp8q {

namespace {

constexpr int kMaxDevices = 64;

__global__ void __launch_bounds__(32)
amax_history_kernel(float* __restrict__ history, int L, int* __restrict__ head,
                    const float* __restrict__ amax_new, float margin, float fmt_max,
                    float* __restrict__ scale_out, int* __restrict__ status) {
    const int lane = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait();
    // the three loads are independent: issue them together
    const int h0 = *head;
    const float a_new = *amax_new;
    float first = lane < L ? history[lane] : 0.0f;
    const int slot = (h0 + 1) % L;
    // |x| as an ordered key: bit patterns of non-negative floats sort like the
    // floats, and a NaN magnitude sorts above infinity
    uint32_t key = 0;
    for (int i = lane; i < L; i += 32) {
        const float v = (i == slot) ? a_new : (i == lane ? first : history[i]);
        key = max(key, __float_as_uint(v) & 0x7FFFFFFFu);
    }
    key = __reduce_max_sync(0xFFFFFFFFu, key);
    __syncwarp();
    if (lane == 0) {
        history[slot] = a_new;
        *head = slot;
        const float ref = __uint_as_float(key);
        bool ok = ref > 0.0f && ref <= 3.402823466e38f;
        float s = 0.0f;
        if (ok) {
            const float d = __fmul_rn(margin, ref);
            s = __fdiv_rn(fmt_max, d);
            ok = s > 0.0f && s <= 3.402823466e38f;
        }
        if (ok) *scale_out = s;
        else if (status) atomicOr(status, FP8Q_DEV_BAD_AMAX);
    }
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
    if (!history || !head || !amax_new || !scale_out) return FP8Q_ERR_NULL;
    if (L < 1 || L > 4096) return FP8Q_ERR_SHAPE;
    if (fmt != FP8Q_E4M3 && fmt != FP8Q_E5M2) return FP8Q_ERR_UNSUPPORTED;
    if (!(margin > 0.0f) || margin > 3.402823466e38f) return FP8Q_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(history) | reinterpret_cast<uintptr_t>(head) |
         reinterpret_cast<uintptr_t>(amax_new) | reinterpret_cast<uintptr_t>(scale_out) |
         reinterpret_cast<uintptr_t>(status)) & 3u)
        return FP8Q_ERR_ALIGN;
    if (!device_is_sm103()) return FP8Q_ERR_UNSUPPORTED;
    if (launch_pdl(amax_history_kernel, dim3(1), dim3(32), 0, stream, history, L, head, amax_new, margin,
                   fp8_max_value(fmt), scale_out, status) != cudaSuccess) {
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
