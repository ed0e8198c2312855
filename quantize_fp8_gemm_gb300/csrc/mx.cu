// mx.cu -- MXFP8: FP8 codes with one power-of-two scale per block of 32
// adjacent values along the contraction ("FP8 training: what it is and how
// it works", Trade-offs and edge cases: the microscaling format Blackwell
// supports natively, 32-value blocks with power-of-two scales), and the GEMM
// that consumes them on the block-scaled tensor-core path
// (tcgen05.mma.kind::mxf8f6f4.block_scale: the scales ride in tensor memory
// beside the accumulator and are applied inside the MMA, so the epilogue is a
// plain BF16 store).
//
// The block scale (Step 2's scale = format max / amax, rounded down to a
// power of two so that no value of the block saturates):
//   s_b = 2^e,  e = the largest integer with amax_b * 2^e <= fmt_max,
//   clamped to [-127, 127]; an all-zero block gets e = 0.
// The byte kept per block is the 8-bit biased exponent of the dequantisation
// factor 1/s_b: 127 - e (the E8M0 scale format of the block-scaled MMA).
//
// Kernels:
//   quant_mx_rows_kernel   H [M,K] -> act(H) BF16 copy, E4M3/E5M2 codes, one
//                          scale byte per 32 values of a row; four lanes per
//                          block, two shuffles for its amax.
//   quant_mx_cols_kernel   W [R,C] -> W^T codes [C,R] with one scale byte per
//                          32 values of a column of W (a row of W^T, the GEMM's
//                          K-major operand); a thread per two columns x 32 rows.
//   mx_gemm_kernel         Y = sum_k (x_q 2^-e_x)(w_q 2^-e_w) -> BF16, 1-CTA
//                          128 x BN tiles (BN 128, 192 or 256).
#include "common.cuh"
#include "gemm_parts.cuh"
#include "quant_ops.cuh"

#include <algorithm>
#include <atomic>
#include <mutex>

namespace fp8q {

namespace {

constexpr int kMxBlock = 32;
constexpr int kMxThreads = 256;

// ---------------------------------------------------------------- scales --
// e of the block scale for a block whose largest magnitude is the
// non-negative BF16 value amax16 (bit pattern).  The format maximum is
// 1.75 * 2^P (448 = 1.75 * 2^8, 57344 = 1.75 * 2^15); with amax = (1 + f) 2^E,
// amax * 2^e <= 1.75 * 2^P holds for e = P - E when f <= 0.75 and for
// e = P - E - 1 otherwise.  Exact: integer arithmetic on the bit pattern.  An
// infinite or NaN maximum (outside the inputs this path is defined on) gets
// e = 0 like an all-zero block.
template <int FMT>
__device__ __forceinline__ int mx_exponent(uint32_t amax16) {
    constexpr int P = FMT == FP8Q_E5M2 ? 15 : 8;
    if (amax16 == 0 || amax16 >= 0x7F80u) return 0;
    const uint32_t ex = amax16 >> 7, mn = amax16 & 0x7Fu;
    int E;
    bool big;
    if (ex != 0) {
        E = static_cast<int>(ex) - 127;
        big = mn > 96u;  // f = mn / 128 > 0.75
    } else {             // subnormal: mn * 2^-133, mn in 1 .. 127
        const int b = 31 - __clz(mn);
        E = b - 133;
        big = 4u * mn > (7u << b);  // mn / 2^b > 1.75
    }
    int e = P - E - (big ? 1 : 0);
    return e > 127 ? 127 : (e < -127 ? -127 : e);
}

// 2^e as a float32, e in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int e) {
    return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// CTA-wide (amax bits, saturation count) -> one atomic each.
__device__ __forceinline__ void mx_publish(uint32_t amax16, uint32_t nsat, float* amax_out,
                                           unsigned long long* sat_out) {
    __shared__ uint32_t s_amax[kMxThreads / 32], s_sat[kMxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    amax16 = __reduce_max_sync(0xFFFFFFFFu, amax16);
    nsat = __reduce_add_sync(0xFFFFFFFFu, nsat);
    if (lane == 0) { s_amax[warp] = amax16; s_sat[warp] = nsat; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kMxThreads / 32; ++w) { amax16 = max(amax16, s_amax[w]); nsat += s_sat[w]; }
        if (amax_out && amax16) atomicMax(reinterpret_cast<unsigned int*>(amax_out), amax16 << 16);
        if (sat_out && nsat) atomicAdd(sat_out, static_cast<unsigned long long>(nsat));
    }
}

// ------------------------------------------------------ quantize: row blocks --
// Chunk c (8 values, 16 bytes of H) lies in block c / 4 of the flattened
// [M, K/32] block grid (K % 32 == 0): the four lanes 4j .. 4j + 3 of a warp
// hold one block, so its maximum is two xor-shuffles away.  A warp takes 32 x
// U consecutive chunks per trip (U loads in flight per lane).
template <int ACT, int FMT>
__global__ void __launch_bounds__(kMxThreads)
quant_mx_rows_kernel(const uint4* __restrict__ h, int64_t nchunks, uint4* __restrict__ act_out,
                     uint2* __restrict__ q_out, uint8_t* __restrict__ sf_out, float* __restrict__ amax_out,
                     unsigned long long* __restrict__ sat_out) {
    constexpr int U = 4;
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    uint32_t amax2 = 0, nsat = 0;
    pdl_wait();
    for (int64_t w0 = warp_id * (32 * U); w0 < nchunks; w0 += nwarps * (32 * U)) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = w0 + u * 32 + lane;
            x[u] = c < nchunks ? ld_stream_v4(h + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = w0 + u * 32 + lane;
            uint32_t m2 = 0;
            const uint4 a = act8<ACT, true>(x[u], m2);
            uint32_t m = max16x2(m2);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            const int e = mx_exponent<FMT>(m);
            if (c < nchunks) {  // nchunks % 4 == 0: a block is wholly inside or outside
                amax2 = max(amax2, m);
                if (act_out) st_stream_v4(act_out + c, a);
                const float sc = pow2f(e);
                st_v2(q_out + c, cast8_codes<FMT>(a, sc));
                // a finite block saturates nothing: e is the largest exponent with
                // amax 2^e <= max, and its clamp at -127 would need amax above
                // max 2^127 > FLT_MAX; only a block holding an inf or a NaN (e = 0)
                // is counted, value by value
                if (m >= 0x7F80u) nsat += sat_count8<FMT>(a, sc);
                if ((lane & 3) == 0) sf_out[c >> 2] = static_cast<uint8_t>(127 - e);
            }
        }
    }
    pdl_launch_dependents();
    mx_publish(amax2, nsat, amax_out, sat_out);
}

// --------------------------------------------------- quantize: column blocks --
// The transposed copy with blocks along the rows of the input: h [R,C] ->
// q_t [C,R], block (c, rb) = h[32 rb .. 32 rb + 31, c], its scale byte at
// sf_t[c * (R / 32) + rb].  A CTA takes a tile of 128 rows (four blocks) x 64
// columns through shared memory: 16-byte loads of whole 128-byte row pieces
// (the activation applied on the way in), then thread (column c, block b)
// reads its 32 values down the column, takes the block maximum, the
// exponent and the 32 codes, and the codes go out as whole 128-byte runs of
// q_t rows and the scale bytes four to a word.  (A thread per two columns x 32
// rows writing its own two 32-byte runs and two single scale bytes filled the
// store queue with partial sectors: 15.7 us for W [6400,1600], 0.27 of the
// copy rate.)
constexpr int kMxColTileR = 128;  // rows of W per CTA (four blocks)
constexpr int kMxColTileC = 64;   // columns of W per CTA

template <int ACT, int FMT>
__global__ void __launch_bounds__(kMxThreads)
quant_mx_cols_kernel(const uint4* __restrict__ h, int64_t R, int64_t C, uint8_t* __restrict__ q_t,
                     uint8_t* __restrict__ sf_t, float* __restrict__ amax_out,
                     unsigned long long* __restrict__ sat_out) {
    static_assert(kMxThreads == 256 && kMxColTileC * kMxColTileR / kMxBlock == kMxThreads, "one block per thread");
    constexpr int TR = kMxColTileR, TC = kMxColTileC;
    __shared__ __align__(16) uint16_t s_in[TR][TC];         // the tile after the activation (BF16 bits)
    __shared__ __align__(16) uint8_t s_q[TC][TR + 16];      // codes by column (+16 B: fewer bank conflicts)
    __shared__ __align__(16) uint8_t s_sf[TC][TR / kMxBlock];
    const int t = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * TR, c0 = static_cast<int64_t>(blockIdx.y) * TC;
    uint32_t m2 = 0, nsat = 0;
    pdl_wait();
#pragma unroll
    for (int i = 0; i < TR * TC / 8 / kMxThreads; ++i) {
        const int idx = t + kMxThreads * i, row = idx / (TC / 8), col = (idx % (TC / 8)) * 8;
        uint4 x = make_uint4(0, 0, 0, 0);
        if (r0 + row < R && c0 + col < C) x = ld_stream_v4(h + ((r0 + row) * C + c0 + col) / 8);
        *reinterpret_cast<uint4*>(&s_in[row][col]) = act8<ACT>(x, m2);  // act(0) = 0 past the edges
    }
    __syncthreads();
    // a warp: 32 consecutive columns of one block (conflict-free column reads)
    const int c = ((t >> 5) % (TC / 32)) * 32 + (t & 31), b = t / TC;
    uint32_t m = 0;
#pragma unroll
    for (int r = 0; r < kMxBlock; ++r) m = max(m, static_cast<uint32_t>(s_in[kMxBlock * b + r][c] & 0x7FFFu));
    const int e = mx_exponent<FMT>(m);
    const float sc = pow2f(e);
    constexpr float fmax = fp8_max_value(FMT);
    uint32_t q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t w = 0;
#pragma unroll
        for (int k = 0; k < 4; k += 2) {
            const float v0 = __fmul_rn(__uint_as_float(static_cast<uint32_t>(s_in[kMxBlock * b + 4 * j + k][c]) << 16), sc);
            const float v1 = __fmul_rn(__uint_as_float(static_cast<uint32_t>(s_in[kMxBlock * b + 4 * j + k + 1][c]) << 16), sc);
            nsat += (fabsf(v0) > fmax) + (fabsf(v1) > fmax);
            w |= static_cast<uint32_t>(cvt_fp8x2<FMT>(v0, v1)) << (8 * k);
        }
        q[j] = w;
    }
    *reinterpret_cast<uint4*>(&s_q[c][kMxBlock * b]) = make_uint4(q[0], q[1], q[2], q[3]);
    *reinterpret_cast<uint4*>(&s_q[c][kMxBlock * b + 16]) = make_uint4(q[4], q[5], q[6], q[7]);
    s_sf[c][b] = static_cast<uint8_t>(127 - e);
    __syncthreads();
    // R % 32 == 0 and C % 16 == 0: a 16-byte piece, a block, lies wholly inside or outside
#pragma unroll
    for (int i = 0; i < TC * TR / 16 / kMxThreads; ++i) {
        const int idx = t + kMxThreads * i, row = idx / (TR / 16), seg = (idx % (TR / 16)) * 16;
        if (c0 + row < C && r0 + seg < R)
            st_v4(q_t + (c0 + row) * R + r0 + seg, *reinterpret_cast<const uint4*>(&s_q[row][seg]));
    }
    if (t < TC && c0 + t < C) {
        const int64_t nb = R / kMxBlock;
        uint8_t* dst = sf_t + (c0 + t) * nb + r0 / kMxBlock;
        if (r0 + TR <= R && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
            *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(&s_sf[t][0]);
        } else {
            for (int k = 0; k < TR / kMxBlock && r0 + kMxBlock * k < R; ++k) dst[k] = s_sf[t][k];
        }
    }
    pdl_launch_dependents();
    mx_publish(max16x2(m2), nsat, amax_out, sat_out);
}

// ------------------------------------------------------------------- GEMM --
// D[M,N] = A[M,K] . B[N,K]^T with per-block scales: A and B K-major E4M3 /
// E5M2 codes, sf_a [M, K/32] and sf_b [N, K/32] bytes (2^(byte - 127) is the
// block's dequantisation factor).
//
// CTA = 6 warps, persistent over 128 x BN tiles (static round robin):
//   warp 0     producer.  Lane 0 streams the A and B k-blocks (128 bytes of K,
//              128-byte swizzle) by TMA into a STAGES-deep ring.  All 32 lanes
//              fill the stage's scale block in shared memory in the layout the
//              tensor-memory copy takes (32 rows of 16 bytes: row l holds the
//              4 scale bytes of the stage's four 32-value blocks for the tile
//              rows l, l + 32, l + 64, l + 96 -- one 32-bit column of tensor
//              memory per 32 tile rows); the words of the next stage are
//              loaded while this one is written, so their latency is hidden.
//   warp 1     MMA issuer.  Per stage: tcgen05.cp of the scale blocks into a
//              tensor-memory slot (32x128b.warpx4: the 32 rows land in all four
//              lane quarters), then 4 block-scaled MMAs (K = 32 each), the
//              k-th selecting byte k of every scale column.
//   warps 2-5  epilogue: tcgen05.ld of the FP32 accumulator, BF16, TMA store.
// Tensor memory: ACCS accumulators of BN columns, then STAGES scale slots of
// 4 (A) + 4 * ceil(BN / 128) (B) columns.
constexpr int kMxGemmThreads = 192;
constexpr int kMxEpiWarps = 4;

template <int BN>
struct MxCfg {
    static constexpr int BNC = (BN + 127) / 128;               // 128-row scale blocks of B per tile
    static constexpr int ACCS = BN == 256 ? 1 : 2;             // TMEM holds 512 columns
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SF_BYTES = 512 * (1 + BNC);           // A's and B's scale blocks of a stage
    static constexpr int SF_COLS = 4 * (1 + BNC);
    static constexpr int EPI_BYTES = kMxEpiWarps * 2 * kEpiChunkBytes;
    static constexpr int BUDGET = 220 * 1024 - EPI_BYTES;
    static constexpr int STAGES = BUDGET / (STAGE_BYTES + SF_BYTES) < 8 ? BUDGET / (STAGE_BYTES + SF_BYTES) : 8;
    static constexpr int TMEM_COLS = 512;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = STAGES * (STAGE_BYTES + SF_BYTES) + EPI_BYTES + BAR_BYTES + 1024;
    static_assert(BN == 128 || BN == 192 || BN == 256, "MX tiles: 128, 192 or 256 wide");
    static_assert(STAGES >= 2, "at least a double-buffered ring");
    static_assert(ACCS * BN + STAGES * SF_COLS <= TMEM_COLS, "accumulators and scale slots fit TMEM");
    static_assert((2 * STAGES + 2 * ACCS + 1) * 8 + 16 <= BAR_BYTES, "barrier area");
    static_assert(SMEM_BYTES <= 232448, "dynamic shared memory per CTA");
};

// The block-scaled MMA: D[tmem] (+)= (A * 2^(sfa - 127)) (B * 2^(sfb - 127))^T,
// the scale bytes read from tensor memory at sfa_tmem / sfb_tmem (the byte of
// each 32-bit column that the instruction descriptor's scale ids select).
__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copy a 32-row x 16-byte block of shared memory into 4 tensor-memory columns
// of lanes 0-31, repeated in each of the four lane quarters.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}

// Shared-memory descriptor of a 32-row x 16-byte block, no swizzle: 8-row
// core matrices of 128 contiguous bytes, stacked 128 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sf(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address   [0,14)
    d |= static_cast<uint64_t>(128 >> 4) << 16;           // leading offset  [16,30)
    d |= static_cast<uint64_t>(128 >> 4) << 32;           // stride offset   [32,46)
    d |= static_cast<uint64_t>(1) << 46;                  // descriptor version [46,48)
    return d;                                             // no swizzle       [61,64) = 0
}

// Instruction descriptor of the block-scaled kind::mxf8f6f4 MMA: A/B formats
// (0 = E4M3, 1 = E5M2), both K-major, E8M0 scales, shape M x N; sf_id picks the
// byte of the A and B scale columns (the MMA's 32-value block in the stage).
__host__ __device__ constexpr uint32_t idesc_mx(uint32_t afmt, uint32_t bfmt, uint32_t m, uint32_t n,
                                                uint32_t sf_id) {
    return (sf_id << 4) | (afmt << 7) | (bfmt << 10) | ((n >> 3) << 17) | (1u << 23) | ((m >> 4) << 24) |
           (sf_id << 29);
}

// Four scale bytes (blocks 4g .. 4g + 3) of row `row` of a [rows, KB] byte
// array as one 32-bit word; rows and blocks past the end read 127 (factor 1).
__device__ __forceinline__ uint32_t sf_word(const uint8_t* __restrict__ sf, int64_t row, int64_t rows, int64_t KB,
                                            int64_t g, bool words) {
    if (row >= rows) return 0x7F7F7F7Fu;
    const uint8_t* p = sf + row * KB + 4 * g;
    if (words) return __ldg(reinterpret_cast<const uint32_t*>(p));  // (unused by the cp.async route)
    uint32_t w = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) w |= static_cast<uint32_t>(4 * g + b < KB ? __ldg(p + b) : 0x7Fu) << (8 * b);
    return w;
}

// 4-byte asynchronous copy global -> shared (no register holds it in flight);
// src_bytes = 0 writes zeros instead of reading.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// Arrive on the mbarrier once every cp.async this thread issued so far has
// landed (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}

template <int BN>
__global__ void __launch_bounds__(kMxGemmThreads, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmD, const uint8_t* __restrict__ sf_a,
               const uint8_t* __restrict__ sf_b, int64_t M, int64_t N, int64_t K, uint32_t idesc0,
               int* __restrict__ status) {
    using C = MxCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sf_smem = smem + C::STAGES * C::STAGE_BYTES;
    uint8_t* epi_stage = sf_smem + C::STAGES * C::SF_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi_stage + C::EPI_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* tfull = bars + 2 * C::STAGES;
    uint64_t* tempty = tfull + C::ACCS;
    uint64_t* drain = tempty + C::ACCS;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<int*>(tmem_holder) + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t num_m = (M + BM - 1) / BM;
    const int64_t num_n = (N + BN - 1) / BN;
    const int64_t num_tiles = num_m * num_n;
    const int num_kb = static_cast<int>((K + BK - 1) / BK);
    const int64_t KB = K / kMxBlock;  // scale bytes per row
    // Whole 32-bit words of scale bytes per row and stage (K % 128 == 0, aligned
    // arrays): the producer's lanes copy them into place with cp.async and the
    // stage's barrier counts each lane's completion; otherwise they are read
    // into registers a stage ahead and stored (bytes past K read as 127).
    const bool words = (KB % 4 == 0) &&
                       ((reinterpret_cast<uintptr_t>(sf_a) | reinterpret_cast<uintptr_t>(sf_b)) & 3u) == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            // the TMA bytes' arrival + the scale block's arrival(s)
            mbar_init(smem_u32(&full[s]), words ? 1 + 32 : 2);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < C::ACCS; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), kMxEpiWarps);
        }
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmD);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------ producer (whole warp)
        uint32_t wa[4], wb[4 * C::BNC];
        auto load_sf = [&](int64_t tile, int kb) {
            const int64_t m0 = (tile / num_n) * BM, n0 = (tile % num_n) * BN;
#pragma unroll
            for (int c = 0; c < 4; ++c) wa[c] = sf_word(sf_a, m0 + 32 * c + lane, M, KB, kb, false);
#pragma unroll
            for (int j = 0; j < 4 * C::BNC; ++j)
                wb[j] = 32 * j < BN ? sf_word(sf_b, n0 + 32 * j + lane, N, KB, kb, false) : 0x7F7F7F7Fu;
        };
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        int64_t tile = blockIdx.x;
        int kb = 0;
        if (tile < num_tiles && !words) load_sf(tile, kb);
        while (tile < num_tiles) {
            int64_t ntile = tile;
            int nkb = kb + 1;
            if (nkb == num_kb) { nkb = 0; ntile += gridDim.x; }
            int ok = 1;
            if (lane == 0) ok = wait_phase(&empty[stage], phase ^ 1u, abort_flag, status);
            if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
            const int32_t m0 = static_cast<int32_t>((tile / num_n) * BM);
            const int32_t n0 = static_cast<int32_t>((tile % num_n) * BN);
            uint8_t* sa = smem + stage * C::STAGE_BYTES;
            if (lane == 0) {
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                tma_load_2d(smem_u32(sa), &tmA, fb, kb * BK, m0);
                tma_load_2d(smem_u32(sa + C::A_BYTES), &tmB, fb, kb * BK, n0);
            }
            uint8_t* sf = sf_smem + stage * C::SF_BYTES;
            if (words) {
                // word c of lane l: rows 32 c + l of the tile; rows past the
                // matrix are zero-filled (their codes are zero-filled too)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int64_t row = m0 + 32 * c + lane;
                    const bool in = row < M;
                    cp_async4(smem_u32(sf + lane * 16 + 4 * c), sf_a + (in ? row * KB + 4 * kb : 0), in ? 4u : 0u);
                }
#pragma unroll
                for (int j = 0; j < 4 * C::BNC; ++j) {
                    const int64_t row = n0 + 32 * j + lane;
                    const bool in = 32 * j < BN && row < N;
                    cp_async4(smem_u32(sf + 512 + 512 * (j / 4) + lane * 16 + 4 * (j % 4)),
                              sf_b + (in ? row * KB + 4 * kb : 0), in ? 4u : 0u);
                }
                cp_async_arrive_noinc(smem_u32(&full[stage]));
            } else {
                *reinterpret_cast<uint4*>(sf + lane * 16) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
#pragma unroll
                for (int j = 0; j < C::BNC; ++j)
                    *reinterpret_cast<uint4*>(sf + 512 * (j + 1) + lane * 16) =
                        make_uint4(wb[4 * j], wb[4 * j + 1], wb[4 * j + 2], wb[4 * j + 3]);
                if (ntile < num_tiles) load_sf(ntile, nkb);  // in flight while the next stage is awaited
                fence_proxy_async_smem();  // the scale block is read by tcgen05.cp (async proxy)
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&full[stage]));
            }
            ++issued;
            if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
            tile = ntile;
            kb = nkb;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");  // this lane's scale copies have landed
        if (lane == 0) {
            // no copy may still be landing in shared memory when the CTA exits
            const int64_t tail = issued < C::STAGES ? issued : C::STAGES;
            for (int64_t j = 1; j <= tail; ++j) {
                int s = stage - static_cast<int>(j);
                uint32_t ph = phase;
                if (s < 0) { s += C::STAGES; ph ^= 1u; }
                wait_phase_drain(&full[s], ph);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                if (!wait_phase(&tempty[acc], acc_phase ^ 1u, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!wait_phase(&full[stage], phase, abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    // the scale block was written through the generic proxy (st.shared or
                    // cp.async); tcgen05.cp reads it through the async proxy
                    fence_proxy_async_smem();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                    const uint32_t sf_t = tmem_base + static_cast<uint32_t>(C::ACCS * BN + stage * C::SF_COLS);
                    const uint32_t sf_s = smem_u32(sf_smem + stage * C::SF_BYTES);
#pragma unroll
                    for (int j = 0; j <= C::BNC; ++j)
                        tmem_cp_32x128b_x4(sf_t + 4 * j, smem_desc_sf(sf_s + 512 * j));
                    const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(k) << 4) |
                                               (static_cast<uint32_t>(k) << 29);
                        mma_mxf8(d_tmem, smem_desc_k_sw128(a_addr + k * UMMA_K),
                                 smem_desc_k_sw128(b_addr + k * UMMA_K), idesc, sf_t, sf_t + 4,
                                 (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&empty[stage]));  // the stage and its scale slot are free
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (ok) {
                    mma_commit(smem_u32(&tfull[acc]));
                    next_acc<C::ACCS>(acc, acc_phase);
                }
            }
            mma_commit(smem_u32(drain));  // every MMA completes before TMEM is released
            wait_phase_drain(drain, 0);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int q = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        uint8_t* warp_stage = epi_stage + (warp - 2) * 2 * kEpiChunkBytes;
        int nchunk = 0, acc = 0;
        uint32_t acc_phase = 0;
        for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int64_t m_blk = tile / num_n, n_blk = tile % num_n;
            const int64_t row0 = m_blk * BM + q * 32;
            bool ok = wait_phase(&tfull[acc], acc_phase, abort_flag, status);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_x32_sync(tmem_base + lane_base + static_cast<uint32_t>(acc * BN + c * 32), r);
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                epi_store_chunk(&tmD, warp_stage, nchunk, lane, v, static_cast<int32_t>(n_blk * BN + c * 32),
                                static_cast<int32_t>(row0), M, N);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
            next_acc<C::ACCS>(acc, acc_phase);
        }
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------- host --
template <int BN>
int launch_mx_gemm(const void* a, const uint8_t* sfa, const void* b, const uint8_t* sfb, void* d, int64_t M,
                   int64_t N, int64_t K, int fa, int fb, int* status, cudaStream_t stream) {
    using C = MxCfg<BN>;
    static cudaError_t attr = cudaFuncSetAttribute(mx_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   C::SMEM_BYTES);
    if (attr != cudaSuccess) return FP8Q_ERR_CUDA;
    alignas(64) CUtensorMap mapA, mapB, mapD;
    if (!make_kmajor_map(&mapA, a, M, K, BM) || !make_kmajor_map(&mapB, b, N, K, BN) || !make_out_map(&mapD, d, M, N))
        return FP8Q_ERR_CUDA;
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int grid = static_cast<int>(std::min<int64_t>(tiles, sm_count()));
    const uint32_t idesc0 = idesc_mx(static_cast<uint32_t>(fa), static_cast<uint32_t>(fb), BM, BN, 0);
    if (launch_pdl(mx_gemm_kernel<BN>, dim3(grid), dim3(kMxGemmThreads), C::SMEM_BYTES, stream, mapA, mapB, mapD,
                   sfa, sfb, M, N, K, idesc0, status) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8Q_ERR_CUDA;
    }
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}

std::atomic<int> g_mx_bn{0};  // fp8q_mx_set_tile: 0 = automatic

// Tile width: whole waves of 1-CTA tiles, each width scored by its time per
// tile relative to the 128-wide tile (the per-tensor GEMM's measured 1-CTA
// ratios: 192 wide 1.06x, 256 wide 1.31x with one accumulator).
int pick_mx_bn(int64_t M, int64_t N) {
    const int ov = g_mx_bn.load(std::memory_order_relaxed);
    if (ov) return ov;
    struct Cand { int bn; double t; };
    static constexpr Cand kCands[] = {{128, 1.000}, {192, 1.064}, {256, 1.307}};
    const int64_t sms = sm_count();
    int best = 128;
    double best_cost = -1.0;
    for (const Cand& c : kCands) {
        const int64_t tiles = ((M + BM - 1) / BM) * ((N + c.bn - 1) / c.bn);
        const double cost = static_cast<double>((tiles + sms - 1) / sms) * c.t;
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = c.bn; }
    }
    return best;
}

template <int ACT>
int launch_quant_mx(int fmt, const void* h, int64_t M, int64_t K, void* act_out, void* q_out, uint8_t* sf_out,
                    void* q_t_out, uint8_t* sf_t_out, float* amax_out, unsigned long long* sat, cudaStream_t stream) {
    cudaError_t e;
    if (q_out) {
        const int64_t nchunks = M * K / 8;
        const int64_t per_cta = int64_t(kMxThreads) * 4;
        const unsigned grid = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>((nchunks + per_cta - 1) / per_cta, int64_t(1) << 30)));
        auto kern = fmt == FP8Q_E5M2 ? quant_mx_rows_kernel<ACT, FP8Q_E5M2> : quant_mx_rows_kernel<ACT, FP8Q_E4M3>;
        e = launch_pdl(kern, dim3(grid), dim3(kMxThreads), 0, stream, static_cast<const uint4*>(h), nchunks,
                       static_cast<uint4*>(act_out), static_cast<uint2*>(q_out), sf_out, amax_out, sat);
    } else {
        const dim3 grid(static_cast<unsigned>((M + kMxColTileR - 1) / kMxColTileR),
                        static_cast<unsigned>((K + kMxColTileC - 1) / kMxColTileC));
        auto kern = fmt == FP8Q_E5M2 ? quant_mx_cols_kernel<ACT, FP8Q_E5M2> : quant_mx_cols_kernel<ACT, FP8Q_E4M3>;
        e = launch_pdl(kern, grid, dim3(kMxThreads), 0, stream, static_cast<const uint4*>(h), M, K,
                       static_cast<uint8_t*>(q_t_out), sf_t_out, amax_out, sat);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8Q_ERR_CUDA;
    }
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}

}  // namespace

}  // namespace fp8q

using namespace fp8q;

extern "C" int fp8_quant_mx(const void* h, int64_t M, int64_t K, int act, int fmt, void* act_out, void* q_out,
                            uint8_t* sf_out, void* q_t_out, uint8_t* sf_t_out, float* amax_out,
                            unsigned long long* sat_count, cudaStream_t stream) {
    if (act < FP8Q_ACT_IDENTITY || act > FP8Q_ACT_RELU2 || (fmt != FP8Q_E4M3 && fmt != FP8Q_E5M2))
        return FP8Q_ERR_UNSUPPORTED;
    const bool rows = q_out != nullptr || sf_out != nullptr;
    const bool cols = q_t_out != nullptr || sf_t_out != nullptr;
    if (rows == cols) return FP8Q_ERR_UNSUPPORTED;  // exactly one of the two modes per call
    if (cols && act_out) return FP8Q_ERR_UNSUPPORTED;
    if (rows ? (!q_out || !sf_out) : (!q_t_out || !sf_t_out)) return FP8Q_ERR_NULL;
    if (!h && M != 0) return FP8Q_ERR_NULL;
    // rows: blocks along K; columns: blocks along M, tiles of 128 rows x 64 columns (at most 65535
    // tiles across K, the grid's second dimension)
    if (M < 0 || (rows ? (K < 32 || K % 32 != 0)
                       : (K < 16 || K % 16 != 0 || M % 32 != 0 || (K + kMxColTileC - 1) / kMxColTileC > 65535)))
        return FP8Q_ERR_SHAPE;
    if (!aligned16(h) || !aligned16(act_out) || !aligned16(q_out) || !aligned16(q_t_out) ||
        (reinterpret_cast<uintptr_t>(amax_out) & 3u) || (reinterpret_cast<uintptr_t>(sat_count) & 7u))
        return FP8Q_ERR_ALIGN;
    if (!device_is_sm103()) return FP8Q_ERR_UNSUPPORTED;
    if (amax_out && cudaMemsetAsync(amax_out, 0, sizeof(float), stream) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (sat_count && cudaMemsetAsync(sat_count, 0, sizeof(unsigned long long), stream) != cudaSuccess)
        return FP8Q_ERR_CUDA;
    if (M == 0) return FP8Q_OK;
    switch (act) {
        case FP8Q_ACT_IDENTITY:
            return launch_quant_mx<FP8Q_ACT_IDENTITY>(fmt, h, M, K, act_out, q_out, sf_out, q_t_out, sf_t_out,
                                                      amax_out, sat_count, stream);
        case FP8Q_ACT_RELU:
            return launch_quant_mx<FP8Q_ACT_RELU>(fmt, h, M, K, act_out, q_out, sf_out, q_t_out, sf_t_out,
                                                  amax_out, sat_count, stream);
        default:
            return launch_quant_mx<FP8Q_ACT_RELU2>(fmt, h, M, K, act_out, q_out, sf_out, q_t_out, sf_t_out,
                                                   amax_out, sat_count, stream);
    }
}

extern "C" int fp8_gemm_mx(const void* x_q, const uint8_t* sf_x, const void* wt_q, const uint8_t* sf_w, void* y,
                           int64_t M, int64_t N, int64_t K, int fmt_x, int fmt_w, int* status,
                           cudaStream_t stream) {
    if ((fmt_x != FP8Q_E4M3 && fmt_x != FP8Q_E5M2) || (fmt_w != FP8Q_E4M3 && fmt_w != FP8Q_E5M2))
        return FP8Q_ERR_UNSUPPORTED;
    if (!wt_q || !sf_w) return FP8Q_ERR_NULL;
    if ((!x_q || !sf_x || !y) && M != 0) return FP8Q_ERR_NULL;
    if (M < 0 || N < 16 || N % 16 != 0 || K < 32 || K % 32 != 0) return FP8Q_ERR_SHAPE;
    if (M > (int64_t(1) << 31) - BM || N > (int64_t(1) << 31) - 256 || K > (int64_t(1) << 31) - BK)
        return FP8Q_ERR_SHAPE;
    if (!aligned16(x_q) || !aligned16(wt_q) || !aligned16(y) || (reinterpret_cast<uintptr_t>(status) & 3u))
        return FP8Q_ERR_ALIGN;
    if (!device_is_sm103()) return FP8Q_ERR_UNSUPPORTED;
    if (M == 0) return FP8Q_OK;
    const int bn = pick_mx_bn(M, N);
    if (bn == 256) return launch_mx_gemm<256>(x_q, sf_x, wt_q, sf_w, y, M, N, K, fmt_x, fmt_w, status, stream);
    if (bn == 192) return launch_mx_gemm<192>(x_q, sf_x, wt_q, sf_w, y, M, N, K, fmt_x, fmt_w, status, stream);
    return launch_mx_gemm<128>(x_q, sf_x, wt_q, sf_w, y, M, N, K, fmt_x, fmt_w, status, stream);
}

extern "C" int fp8q_mx_set_tile(int bn) {
    if (bn != 0 && bn != 128 && bn != 192 && bn != 256) return FP8Q_ERR_UNSUPPORTED;
    g_mx_bn.store(bn);
    return FP8Q_OK;
}
