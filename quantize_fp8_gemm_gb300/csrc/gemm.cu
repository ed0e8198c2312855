// gemm.cu -- FP8 x FP8 -> FP32-accumulated, dequantised BF16 GEMM on the
// fifth-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// "FP8 Training & Inference", FP8 Training Recipe: the forward Y = X x W with
// both operands E4M3, and the activation gradient dX = dY x W^T with dY in
// E5M2 and W in E4M3; Per-Tensor Scaling for FP8: the scales are factored out
// of the matmul and the output is rescaled.  "FP8 training: what it is and how
// it works", Step 3: FP8 inputs, a wider running sum (here FP32 in TMEM), and
// the 1x128 / 128x128 scale groups of Trade-offs and edge cases, whose partial
// sums are promoted into FP32 registers once per 128-long slice.
//
// Both GEMMs are D[M,N] = A[M,K] . B[N,K]^T with A and B K-major:
//   forward: A = X_q [M,K],   B = W_q^T [N,K]
//   dgrad:   A = dY_q [M,N],  B = W_q [K,N]   (the contraction runs over N)
//
// CTA = 6 warps, persistent over 128 x BN output tiles (static round robin):
//   warp 0     TMA producer: one elected lane streams A/B k-blocks (128 B of
//              K per row, 128-byte swizzle) into a STAGES-deep ring.
//   warp 1     MMA issuer: allocates TMEM; one lane issues 4 x
//              tcgen05.mma.kind::f8f6f4 (M=128, N=BN, K=32) per k-block and
//              commits each stage back to the producer.
//   warps 2-5  epilogue: tcgen05.ld the FP32 accumulator (each warp its 32
//              TMEM lanes), scale by 1/(s_a s_b), round to BF16, store.
// Two TMEM accumulators let the epilogue of tile i overlap the main loop of
// tile i+1.  Every mbarrier wait is bounded; on time-out the CTA sets
// FP8Q_DEV_TIMEOUT, drains its in-flight copies and MMAs and exits.
#include "common.cuh"

#include <algorithm>
#include <cudaTypedefs.h>
#include <mutex>

namespace fp8q {

namespace {

constexpr int BM = 128;            // tile rows (MMA M, TMEM lanes)
constexpr int BK = 128;            // K bytes per stage = one 128-byte swizzle row
constexpr int UMMA_K = 32;         // K per tcgen05.mma for 8-bit operands
constexpr int kThreadsGemm = 192;  // 6 warps
constexpr int kEpiWarps = 4;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait: far above any real wait

template <int BN>
struct Cfg {
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (220 * 1024) / STAGE_BYTES < 8 ? (220 * 1024) / STAGE_BYTES : 8;
    static constexpr int TMEM_COLS = (2 * BN <= 256) ? 256 : 512;  // two accumulators, power of 2
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;  // + alignment slack
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN: multiple of 32 in [64, 256]");
    static_assert(STAGES >= 2, "at least a double-buffered ring");
    static_assert((2 * STAGES + 5) * 8 + 16 <= BAR_BYTES, "barrier area");
};

struct SharedCtl {
    // lives at the end of the dynamic shared memory, after the stage ring
    uint64_t* full;
    uint64_t* empty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint64_t* drain;
    uint32_t* tmem_holder;
    int* abort_flag;
};

// Bounded wait on an mbarrier phase.  Returns false when this thread gave up
// or another role of the CTA already aborted.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           int* status) {
    const uint32_t b = smem_u32(bar);
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(b, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kTimeoutNs) {
            *abort_flag = 1;
            if (status) atomicOr(status, FP8Q_DEV_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait used while draining after an abort (no abort check).
__device__ __forceinline__ void wait_phase_drain(uint64_t* bar, uint32_t parity) {
    const uint32_t b = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(b, parity)) {
        if (globaltimer_ns() - t0 > kTimeoutNs) return;
    }
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* __restrict__ D, int64_t row, int64_t col0,
                                              int64_t M, int64_t N, const float (&v)[32]) {
    if (row >= M) return;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t col = col0 + 8 * j;
        if (col < N) {
            uint4 p;
            p.x = cvt_bf16x2(v[8 * j + 0], v[8 * j + 1]);
            p.y = cvt_bf16x2(v[8 * j + 2], v[8 * j + 3]);
            p.z = cvt_bf16x2(v[8 * j + 4], v[8 * j + 5]);
            p.w = cvt_bf16x2(v[8 * j + 6], v[8 * j + 7]);
            st_v4(D + row * N + col, p);
        }
    }
}

// GROUP = false: per-tensor scales, one accumulation per tile.
// GROUP = true : BN must be 128; each 128-long K slice is accumulated into a
//                fresh TMEM buffer and promoted into FP32 registers with its
//                own 1/(s_a[row, kb] * s_b[kb, n_blk]).
template <int BN, bool GROUP>
__global__ void __launch_bounds__(kThreadsGemm, 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const float* __restrict__ scale_a, const float* __restrict__ scale_b,
                __nv_bfloat16* __restrict__ D, int64_t M, int64_t N, int64_t K, uint32_t idesc,
                int* __restrict__ status) {
    using C = Cfg<BN>;
    static_assert(!GROUP || BN == 128, "group mode uses 128-wide tiles");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    SharedCtl ctl;
    ctl.full = bars;
    ctl.empty = bars + C::STAGES;
    ctl.tfull = bars + 2 * C::STAGES;
    ctl.tempty = bars + 2 * C::STAGES + 2;
    ctl.drain = bars + 2 * C::STAGES + 4;
    ctl.tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 5);
    ctl.abort_flag = reinterpret_cast<int*>(bars + 2 * C::STAGES + 5) + 1;
    volatile int* abort_flag = ctl.abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t num_m = (M + BM - 1) / BM;
    const int64_t num_n = (N + BN - 1) / BN;
    const int64_t num_tiles = num_m * num_n;
    const int num_kb = static_cast<int>((K + BK - 1) / BK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&ctl.full[s]), 1);
            mbar_init(smem_u32(&ctl.empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&ctl.tfull[a]), 1);
            mbar_init(smem_u32(&ctl.tempty[a]), kEpiWarps);
        }
        mbar_init(smem_u32(ctl.drain), 1);
        *ctl.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(ctl.tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *ctl.tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                const int32_t m0 = static_cast<int32_t>((tile / num_n) * BM);
                const int32_t n0 = static_cast<int32_t>((tile % num_n) * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!wait_phase(&ctl.empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
                    const uint32_t fb = smem_u32(&ctl.full[stage]);
                    uint8_t* sa = smem + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                    tma_load_2d(smem_u32(sa), &tmA, fb, kb * BK, m0);
                    tma_load_2d(smem_u32(sa + C::A_BYTES), &tmB, fb, kb * BK, n0);
                    ++issued;
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Make sure no copy is still landing in shared memory when the CTA
            // exits: wait for the last (up to STAGES) loads to complete.
            const int64_t tail = issued < C::STAGES ? issued : C::STAGES;
            for (int64_t j = 1; j <= tail; ++j) {
                int s = stage - static_cast<int>(j);
                uint32_t ph = phase;
                if (s < 0) { s += C::STAGES; ph ^= 1u; }
                wait_phase_drain(&ctl.full[s], ph);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                if (!GROUP) {
                    if (!wait_phase(&ctl.tempty[acc], acc_phase ^ 1u, abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                }
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (GROUP) {
                        if (!wait_phase(&ctl.tempty[acc], acc_phase ^ 1u, abort_flag, status)) { ok = false; break; }
                        tc_fence_after();
                    }
                    if (!wait_phase(&ctl.full[stage], phase, abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                    const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        const uint32_t accumulate = GROUP ? (k > 0) : (kb > 0 || k > 0);
                        mma_f8f6f4(d_tmem, smem_desc_k_sw128(a_addr + k * UMMA_K),
                                   smem_desc_k_sw128(b_addr + k * UMMA_K), idesc, accumulate);
                    }
                    mma_commit(smem_u32(&ctl.empty[stage]));  // stage free once these MMAs finish
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                    if (GROUP) {
                        mma_commit(smem_u32(&ctl.tfull[acc]));
                        acc ^= 1;
                        if (acc == 0) acc_phase ^= 1u;
                    }
                }
                if (!GROUP && ok) {
                    mma_commit(smem_u32(&ctl.tfull[acc]));  // accumulator ready for the epilogue
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                }
            }
            // all MMAs of this thread complete before TMEM is released
            mma_commit(smem_u32(ctl.drain));
            wait_phase_drain(ctl.drain, 0);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        float inv = 1.0f;
        if (!GROUP) inv = 1.0f / (__ldg(scale_a) * __ldg(scale_b));
        const int64_t kg = K / BK;                    // group mode: K % 128 == 0
        const int64_t ng = (N + 127) / 128;
        for (int64_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const int64_t m_blk = tile / num_n, n_blk = tile % num_n;
            const int64_t row = m_blk * BM + q * 32 + lane;
            if (!GROUP) {
                ok = wait_phase(&ctl.tfull[acc], acc_phase, abort_flag, status);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_x32(tmem_base + lane_base + static_cast<uint32_t>(acc * BN + c * 32), r);
                    tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * inv;
                    store_bf16x32(D, row, n_blk * BN + c * 32, M, N, v);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctl.tempty[acc]));
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            } else {
                float sum[BN];
#pragma unroll
                for (int j = 0; j < BN; ++j) sum[j] = 0.0f;
                const int64_t srow = row < M ? row : M - 1;
                for (int kb = 0; kb < num_kb; ++kb) {
                    const float sa = __ldg(scale_a + srow * kg + kb);
                    const float sb = __ldg(scale_b + kb * ng + n_blk);
                    const float ginv = 1.0f / (sa * sb);
                    ok = wait_phase(&ctl.tfull[acc], acc_phase, abort_flag, status);
                    ok = __all_sync(0xFFFFFFFFu, ok);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld_x32(tmem_base + lane_base + static_cast<uint32_t>(acc * BN + c * 32), r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) sum[c * 32 + j] = fmaf(__uint_as_float(r[j]), ginv, sum[c * 32 + j]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ctl.tempty[acc]));
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                }
                if (!ok) break;
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = sum[c * 32 + j];
                    store_bf16x32(D, row, n_blk * BN + c * 32, M, N, v);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------- host --
using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// K-major 8-bit operand [rows, K]: box = 128 bytes of K x box_rows rows, 128-byte swizzle.
bool make_kmajor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN, bool GROUP>
int launch_gemm(const void* a, const void* b, const float* sa, const float* sb, void* d, int64_t M,
                int64_t N, int64_t K, uint32_t afmt, uint32_t bfmt, int* status, cudaStream_t stream) {
    using C = Cfg<BN>;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(fp8_gemm_kernel<BN, GROUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return FP8Q_ERR_CUDA;
    alignas(64) CUtensorMap mapA, mapB;
    if (!make_kmajor_map(&mapA, a, M, K, BM) || !make_kmajor_map(&mapB, b, N, K, BN)) return FP8Q_ERR_CUDA;
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int grid = static_cast<int>(std::min<int64_t>(tiles, sm_count()));
    const uint32_t idesc = idesc_f8(afmt, bfmt, BM, BN);
    fp8_gemm_kernel<BN, GROUP><<<grid, kThreadsGemm, C::SMEM_BYTES, stream>>>(
        mapA, mapB, sa, sb, static_cast<__nv_bfloat16*>(d), M, N, K, idesc, status);
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}

// Tile width: the candidate with the least work on the busiest SM
// (ceil(tiles / SMs) * BN); ties go to the wider tile.
int pick_bn(int64_t M, int64_t N) {
    const int cands[] = {256, 192, 160, 128};
    const int64_t sms = sm_count();
    int best = 128;
    int64_t best_cost = -1;
    for (int bn : cands) {
        const int64_t tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
        const int64_t cost = ((tiles + sms - 1) / sms) * bn;
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = bn; }
    }
    return best;
}

int gemm_dispatch(const void* a, const void* b, const float* sa, const float* sb, int group, void* d,
                  int64_t M, int64_t N, int64_t K, uint32_t afmt, uint32_t bfmt, int* status,
                  cudaStream_t stream) {
    if (group) return launch_gemm<128, true>(a, b, sa, sb, d, M, N, K, afmt, bfmt, status, stream);
    switch (pick_bn(M, N)) {
        case 256: return launch_gemm<256, false>(a, b, sa, sb, d, M, N, K, afmt, bfmt, status, stream);
        case 192: return launch_gemm<192, false>(a, b, sa, sb, d, M, N, K, afmt, bfmt, status, stream);
        case 160: return launch_gemm<160, false>(a, b, sa, sb, d, M, N, K, afmt, bfmt, status, stream);
        default: return launch_gemm<128, false>(a, b, sa, sb, d, M, N, K, afmt, bfmt, status, stream);
    }
}

int check_gemm_args(const void* a, const void* b, const float* sa, const float* sb, const void* d,
                    int64_t M, int64_t N, int64_t K, const int* status) {
    if (!b || !sa || !sb) return FP8Q_ERR_NULL;
    if ((!a || !d) && M != 0) return FP8Q_ERR_NULL;  // an empty A / D may have no storage
    if (M < 0 || N < 16 || K < 16 || N % 16 != 0 || K % 16 != 0) return FP8Q_ERR_SHAPE;
    if (M > (int64_t(1) << 31) - BM || N > (int64_t(1) << 31) - 256 || K > (int64_t(1) << 31) - BK)
        return FP8Q_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return FP8Q_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(sa) | reinterpret_cast<uintptr_t>(sb) |
         reinterpret_cast<uintptr_t>(status)) & 3u)
        return FP8Q_ERR_ALIGN;
    if (!device_is_sm103()) return FP8Q_ERR_UNSUPPORTED;
    return FP8Q_OK;
}

}  // namespace

}  // namespace fp8q

using namespace fp8q;

extern "C" int fp8_gemm_fwd(const void* x_q, const void* wt_q, const float* scale_x, const float* scale_w,
                            int group_mode, void* y, int64_t M, int64_t N, int64_t K, int* status,
                            cudaStream_t stream) {
    int st = check_gemm_args(x_q, wt_q, scale_x, scale_w, y, M, N, K, status);
    if (st != FP8Q_OK) return st;
    if (group_mode != 0 && group_mode != 1) return FP8Q_ERR_UNSUPPORTED;
    if (group_mode && K % FP8Q_GROUP != 0) return FP8Q_ERR_SHAPE;
    if (M == 0) return FP8Q_OK;
    return gemm_dispatch(x_q, wt_q, scale_x, scale_w, group_mode, y, M, N, K, FP8Q_E4M3, FP8Q_E4M3, status,
                         stream);
}

extern "C" int fp8_gemm_dgrad(const void* dy_q, const void* w_q, const float* scale_dy, const float* scale_w,
                              void* dx, int64_t M, int64_t N, int64_t K, int* status, cudaStream_t stream) {
    // D = dX [M,K], A = dY [M,N] (contraction N), B = W [K,N]
    int st = check_gemm_args(dy_q, w_q, scale_dy, scale_w, dx, M, K, N, status);
    if (st != FP8Q_OK) return st;
    if (M == 0) return FP8Q_OK;
    return gemm_dispatch(dy_q, w_q, scale_dy, scale_w, 0, dx, M, K, N, FP8Q_E5M2, FP8Q_E4M3, status, stream);
}
