// gemm_parts.cuh -- pieces shared by the tcgen05 GEMM kernels (gemm.cu: the
// per-tensor, group-scaled and fused GEMMs; mx.cu: the block-scaled MX GEMM):
// tile constants, bounded mbarrier waits, the BF16 epilogue store through a
// swizzled shared-memory block and TMA, and the host-side tensor maps.
#pragma once

#include "common.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace fp8q {

namespace {

constexpr int BM = 128;            // rows per CTA (MMA rows per SM, TMEM lanes)
constexpr int BK = 128;            // K bytes per stage = one 128-byte swizzle row
constexpr int UMMA_K = 32;         // K per tcgen05.mma for 8-bit operands
constexpr int kEpiChunkBytes = 32 * 32 * 2;  // one warp's 32 rows x 32 BF16 columns
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait: far above any real wait

// Next accumulator (of ACCS) and the phase its barriers are in.
template <int ACCS>
__device__ __forceinline__ void next_acc(int& acc, uint32_t& acc_phase) {
    if (++acc == ACCS) {
        acc = 0;
        acc_phase ^= 1u;
    }
}

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

// One warp's 32 rows x 32 columns of output: round to BF16, stage in shared
// memory with the 64-byte swizzle (row r's 16-byte piece j sits at piece
// j ^ ((r >> 1) & 3), so the warp's writes spread over all banks) and write
// it with one TMA store; the box is clipped at the edges of D.  Two staging
// buffers per warp alternate; a buffer is reused once the store issued from
// it two chunks earlier has finished reading it.
template <int NBUF = 2>
__device__ __forceinline__ void epi_store_chunk(const CUtensorMap* tmD, uint8_t* warp_stage, int& nchunk,
                                                int lane, const float (&v)[32], int32_t col0, int32_t row0,
                                                int64_t M, int64_t N) {
    static_assert(NBUF == 1 || NBUF == 2, "one or two staging blocks per warp");
    // A box wholly outside D is skipped outright: nchunk counts committed
    // store groups, so the wait below covers the store that last read `buf`.
    if (row0 >= M || col0 >= N) return;
    uint8_t* buf = warp_stage + (NBUF == 2 ? (nchunk & 1) * kEpiChunkBytes : 0);
    if (nchunk >= NBUF) {
        if (lane == 0) bulk_wait_group_read<NBUF - 1>();
        __syncwarp();
    }
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 p;
        p.x = cvt_bf16x2(v[8 * j + 0], v[8 * j + 1]);
        p.y = cvt_bf16x2(v[8 * j + 2], v[8 * j + 3]);
        p.z = cvt_bf16x2(v[8 * j + 4], v[8 * j + 5]);
        p.w = cvt_bf16x2(v[8 * j + 6], v[8 * j + 7]);
        *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ sw) << 4)) = p;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmD, smem_u32(buf), col0, row0);
        bulk_commit_group();
    }
    ++nchunk;
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

// BF16 output D [rows, cols]: box = 32 columns x 32 rows, 64-byte swizzle (stores).
bool make_out_map(CUtensorMap* map, void* base, int64_t rows, int64_t cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

}  // namespace fp8q
