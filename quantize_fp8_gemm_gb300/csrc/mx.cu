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
//                          K-major operand); a 128 x 64 tile per CTA through
//                          shared memory.
//   mx_gemm_kernel         Y = sum_k (x_q 2^-e_x)(w_q 2^-e_w) -> BF16, 1-CTA
//                          128 x BN tiles or 2-SM 256 x BN tiles (BN 128, 192
//                          or 256).
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

// ------------------------------------------------- the tiled scale layout --
// The scale bytes of a [rows, KB] block grid (KB blocks of 32 values per row)
// are stored in atoms of 128 rows x 4 blocks, 512 bytes each: the layout the
// block-scaled MMA's tensor-memory copy takes, so that a GEMM stage (128
// values of K) fetches the scales of 128 rows with one TMA copy.  Atom (rows
// 128 i .. 128 i + 127, blocks 4 g .. 4 g + 3) starts at byte 512 (i G + g),
// G = ceil(KB / 4); in it, row 32 j + l (l < 32, j < 4) and block 4 g + k sit
// at byte 16 l + 4 j + k.  Blocks KB .. 4 G - 1 of a row are padding and hold
// 127 (factor 1); bytes of rows past the grid in the last atom row are not
// written.
constexpr int kMxAtomBytes = 512;

__host__ __device__ __forceinline__ int64_t mx_sf_offset(int64_t row, int64_t blk, int64_t G) {
    return ((row >> 7) * G + (blk >> 2)) * kMxAtomBytes + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (blk & 3);
}

// n / d for 32-bit n and a divisor fixed per launch, by a multiply with a
// precomputed reciprocal (Granlund and Montgomery, "Division by Invariant
// Integers using Multiplication", 1994, the unsigned case: l = ceil(log2 d),
// m = floor(2^32 (2^l - d) / d) + 1, t = mulhi(m, n),
// q = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0); exact for n < 2^32).
struct DivU32 {
    uint32_t m, sh1, sh2;
};
inline DivU32 make_divu32(uint32_t d) {
    uint32_t l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
    return DivU32{static_cast<uint32_t>(m), l < 1 ? l : 1u, l > 1 ? l - 1 : 0u};
}
__device__ __forceinline__ uint32_t divu32(uint32_t n, DivU32 d) {
    const uint32_t t = __umulhi(d.m, n);
    return (t + ((n - t) >> d.sh1)) >> d.sh2;
}

// ------------------------------------------------------ quantize: row blocks --
// Chunk c (8 values, 16 bytes of H) lies in block c / 4 of the flattened
// [M, K/32] block grid (K % 32 == 0): the four lanes 4j .. 4j + 3 of a warp
// hold one block, so its maximum is two xor-shuffles away.  A warp takes 32 x
// U consecutive chunks per trip (U loads in flight per lane).  The block's row
// and column come from its flat index by the invariant division (fewer than
// 2^32 blocks); the scale byte goes to its place in the tiled layout.
template <int ACT, int FMT>
__global__ void __launch_bounds__(kMxThreads, 4)
quant_mx_rows_kernel(const uint4* __restrict__ h, int64_t nchunks, uint32_t KB, DivU32 div_kb, int64_t G,
                     uint4* __restrict__ act_out, uint2* __restrict__ q_out, uint8_t* __restrict__ sf_out,
                     float* __restrict__ amax_out, unsigned long long* __restrict__ sat_out) {
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
                if ((lane & 3) == 0) {
                    const uint32_t fb = static_cast<uint32_t>(c >> 2);
                    const uint32_t row = divu32(fb, div_kb), blk = fb - row * KB;
                    sf_out[mx_sf_offset(row, blk, G)] = static_cast<uint8_t>(127 - e);
                    if (blk == KB - 1)  // the row's padding blocks, up to the atom's edge
                        for (int64_t p = KB; p < 4 * G; ++p) sf_out[mx_sf_offset(row, p, G)] = 127;
                }
            }
        }
    }
    pdl_launch_dependents();
    mx_publish(amax2, nsat, amax_out, sat_out);
}

// --------------------------------------------------- quantize: column blocks --
// The transposed copy with blocks along the rows of the input: h [R,C] ->
// q_t [C,R], block (c, rb) = h[32 rb .. 32 rb + 31, c], its scale byte at
// (row c, block rb) of the tiled layout of the [C, R/32] grid.  A CTA takes a
// tile of 128 rows (four blocks, one atom column) x 64
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
        // the column's four scale bytes are one aligned word of its atom; blocks
        // past R (zero rows, e = 0) hold 127, the layout's padding
        const int64_t G = (R / kMxBlock + 3) / 4;
        *reinterpret_cast<uint32_t*>(sf_t + mx_sf_offset(c0 + t, r0 / kMxBlock, G)) =
            *reinterpret_cast<const uint32_t*>(&s_sf[t][0]);
    }
    pdl_launch_dependents();
    mx_publish(max16x2(m2), nsat, amax_out, sat_out);
}

// ------------------------------------------------------------------- GEMM --
// D[M,N] = A[M,K] . B[N,K]^T with per-block scales: A and B K-major E4M3 /
// E5M2 codes, sf_a and sf_b the scale bytes of their [M, K/32] and [N, K/32]
// block grids in the tiled layout above (2^(byte - 127) is the block's
// dequantisation factor).
//
// CTA = 6 warps, persistent over 128 x BN tiles (PAIR = false) or, with
// PAIR = true, a cluster of two CTAs on two SMs per 256 x BN tile (static
// round robin):
//   warp 0     producer.  Lane 0 streams, per stage of 128 K values, the A and
//              B k-blocks (128-byte swizzle) and the scale atoms of the stage
//              (one for the CTA's 128 rows of A, BN / 128 for the tile's rows
//              of B: exactly the bytes the tensor-memory copy reads) by TMA
//              into a STAGES-deep ring.  In a pair each CTA loads its own 128
//              rows of A and half of B's rows, the scale atoms of its own A
//              rows and of all the tile's B rows, and both CTAs' copies
//              complete on the leader's barrier.
//   warp 1     MMA issuer (the leader's, in a pair).  Per stage: tcgen05.cp of
//              the scale atoms into a tensor-memory slot (32x128b.warpx4: the
//              atom's 32 rows of 16 bytes land in all four lane quarters; in a
//              pair the copy runs in both CTAs, each from its own shared memory
//              into its own tensor memory), then 4 block-scaled MMAs (K = 32
//              each), the k-th selecting byte k of every scale column.
//   warps 2-5  epilogue: tcgen05.ld of the FP32 accumulator, BF16, TMA store.
// Tensor memory: ACCS accumulators of BN columns, then STAGES scale slots of
// 4 (A) + 4 * BN / 128 (B) columns.
constexpr int kMxGemmThreads = 192;
constexpr int kMxEpiWarps = 4;

template <int BN, bool PAIR>
struct MxCfg {
    static constexpr int BNC = BN / 128;                       // scale atoms of B per tile and stage
    static constexpr int ACCS = BN == 256 ? 1 : 2;             // TMEM holds 512 columns
    static constexpr int TILE_M = PAIR ? 2 * BM : BM;
    static constexpr int MMA_M = TILE_M;
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;          // rows of B this CTA loads
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = B_ROWS * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SF_BYTES = kMxAtomBytes * (1 + BNC);  // A's and B's scale atoms of a stage
    static constexpr int SF_COLS = 4 * (1 + BNC);
    static constexpr int TX_BYTES = (STAGE_BYTES + SF_BYTES) * (PAIR ? 2 : 1);  // bytes one stage's barrier awaits
    static constexpr int EPI_BYTES = kMxEpiWarps * 2 * kEpiChunkBytes;
    static constexpr int BUDGET = 220 * 1024 - EPI_BYTES;
    static constexpr int STAGES = BUDGET / (STAGE_BYTES + SF_BYTES) < 8 ? BUDGET / (STAGE_BYTES + SF_BYTES) : 8;
    static constexpr int TMEM_COLS = 512;
    static constexpr int BAR_BYTES = 256;
    static constexpr int EPI_ARRIVALS = kMxEpiWarps * (PAIR ? 2 : 1);  // per accumulator drain
    static constexpr int SMEM_BYTES = STAGES * (STAGE_BYTES + SF_BYTES) + EPI_BYTES + BAR_BYTES + 1024;
    static_assert(BN == 128 || BN == 256, "MX tiles: 128 or 256 wide (whole scale atoms of B)");
    static_assert(B_BYTES % 1024 == 0, "each stage's B box starts on a 1 KB swizzle atom");
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
// The same issued by the leader of a CTA pair: A rows 0-127 and half of B from
// its own shared memory, the rest from the peer's (same offsets); each CTA's
// tensor memory holds its D rows and the scales at the same addresses.
__device__ __forceinline__ void mma_mxf8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copy a 32-row x 16-byte block of shared memory into 4 tensor-memory columns
// of lanes 0-31, repeated in each of the four lane quarters.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}
// The same in both CTAs of a pair, each from its own shared memory at the
// descriptor's offset into its own tensor memory at taddr.
__device__ __forceinline__ void tmem_cp_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}

// 3-D tiled loads (x innermost); completion bytes on `bar`, which for the
// pair form may be the leader CTA's barrier (a shared::cluster address).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                            int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z) : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                                 int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5}], [%2];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z) : "memory");
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

template <int BN, bool PAIR>
__global__ void __launch_bounds__(kMxGemmThreads, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmSA,
               const __grid_constant__ CUtensorMap tmSB, int64_t M, int64_t N, int64_t K, uint32_t idesc0,
               int* __restrict__ status) {
    using C = MxCfg<BN, PAIR>;
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
    const uint32_t rank = PAIR ? cluster_ctarank() : 0;  // 0 = leader of the pair
    const bool leader = rank == 0;
    const int64_t num_m = (M + C::TILE_M - 1) / C::TILE_M;
    const int64_t num_n = (N + BN - 1) / BN;
    const int64_t num_tiles = num_m * num_n;
    const int64_t first_tile = PAIR ? blockIdx.x / 2 : blockIdx.x;
    const int64_t tile_stride = PAIR ? gridDim.x / 2 : gridDim.x;
    const int num_kb = static_cast<int>((K + BK - 1) / BK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);  // the leader's expect-tx arrival; the rest is bytes
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < C::ACCS; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), C::EPI_ARRIVALS);
        }
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmD);
        tma_prefetch_desc(&tmSA);
        tma_prefetch_desc(&tmSB);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_holder), C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();  // the peer's barriers exist before any copy signals them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0) {
        // -------------------------------------------------------- producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t tile = first_tile; tile < num_tiles && ok; tile += tile_stride) {
                // this CTA's A rows and the tile's first B row (both multiples of 128)
                const int32_t m0 = static_cast<int32_t>((tile / num_n) * C::TILE_M + rank * BM);
                const int32_t n0 = static_cast<int32_t>((tile % num_n) * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!wait_phase(&empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
                    uint8_t* sa = smem + stage * C::STAGE_BYTES;
                    const uint32_t sf = smem_u32(sf_smem + stage * C::SF_BYTES);
                    if constexpr (PAIR) {
                        // both CTAs' copies complete on the leader's barrier
                        const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
                        if (leader) mbar_arrive_expect_tx(smem_u32(&full[stage]), C::TX_BYTES);
                        tma_load_2d_pair(smem_u32(sa), &tmA, fb, kb * BK, m0);
                        tma_load_2d_pair(smem_u32(sa + C::A_BYTES), &tmB, fb, kb * BK,
                                         n0 + static_cast<int32_t>(rank) * C::B_ROWS);
                        tma_load_3d_pair(sf, &tmSA, fb, 0, kb, m0 / BM);
                        tma_load_3d_pair(sf + kMxAtomBytes, &tmSB, fb, 0, kb, n0 / BM);
                    } else {
                        const uint32_t fb = smem_u32(&full[stage]);
                        mbar_arrive_expect_tx(fb, C::TX_BYTES);
                        tma_load_2d(smem_u32(sa), &tmA, fb, kb * BK, m0);
                        tma_load_2d(smem_u32(sa + C::A_BYTES), &tmB, fb, kb * BK, n0);
                        tma_load_3d(sf, &tmSA, fb, 0, kb, m0 / BM);
                        tma_load_3d(sf + kMxAtomBytes, &tmSB, fb, 0, kb, n0 / BM);
                    }
                    ++issued;
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // No copy may still be landing in shared memory when the CTA exits:
            // wait for the last (up to STAGES) loads.  In a pair the leader's
            // barriers also count the peer's bytes.
            if (leader) {
                const int64_t tail = issued < C::STAGES ? issued : C::STAGES;
                for (int64_t j = 1; j <= tail; ++j) {
                    int s = stage - static_cast<int>(j);
                    uint32_t ph = phase;
                    if (s < 0) { s += C::STAGES; ph ^= 1u; }
                    wait_phase_drain(&full[s], ph);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t tile = first_tile; tile < num_tiles && ok; tile += tile_stride) {
                if (!wait_phase(&tempty[acc], acc_phase ^ 1u, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!wait_phase(&full[stage], phase, abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                    const uint32_t sf_t = tmem_base + static_cast<uint32_t>(C::ACCS * BN + stage * C::SF_COLS);
                    const uint32_t sf_s = smem_u32(sf_smem + stage * C::SF_BYTES);
#pragma unroll
                    for (int j = 0; j <= C::BNC; ++j) {
                        if constexpr (PAIR) tmem_cp_32x128b_x4_pair(sf_t + 4 * j, smem_desc_sf(sf_s + kMxAtomBytes * j));
                        else tmem_cp_32x128b_x4(sf_t + 4 * j, smem_desc_sf(sf_s + kMxAtomBytes * j));
                    }
                    const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(k) << 4) |
                                               (static_cast<uint32_t>(k) << 29);
                        const uint64_t ad = smem_desc_k_sw128(a_addr + k * UMMA_K);
                        const uint64_t bd = smem_desc_k_sw128(b_addr + k * UMMA_K);
                        const uint32_t accumulate = (kb > 0 || k > 0) ? 1u : 0u;
                        if constexpr (PAIR) mma_mxf8_pair(d_tmem, ad, bd, idesc, sf_t, sf_t + 4, accumulate);
                        else mma_mxf8(d_tmem, ad, bd, idesc, sf_t, sf_t + 4, accumulate);
                    }
                    // the stage and its scale slot are free (in both CTAs of a pair)
                    if constexpr (PAIR) mma_commit_pair_mc(smem_u32(&empty[stage]), 0x3);
                    else mma_commit(smem_u32(&empty[stage]));
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (ok) {
                    if constexpr (PAIR) mma_commit_pair_mc(smem_u32(&tfull[acc]), 0x3);
                    else mma_commit(smem_u32(&tfull[acc]));
                    next_acc<C::ACCS>(acc, acc_phase);
                }
            }
            // every MMA completes before TMEM is released
            if constexpr (PAIR) mma_commit_pair(smem_u32(drain));
            else mma_commit(smem_u32(drain));
            wait_phase_drain(drain, 0);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int q = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        uint8_t* warp_stage = epi_stage + (warp - 2) * 2 * kEpiChunkBytes;
        // drained accumulators are reported to the leader's barrier
        const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(&tempty[0]), 0) : smem_u32(&tempty[0]);
        int nchunk = 0, acc = 0;
        uint32_t acc_phase = 0;
        for (int64_t tile = first_tile; tile < num_tiles; tile += tile_stride) {
            const int64_t m_blk = tile / num_n, n_blk = tile % num_n;
            const int64_t row0 = m_blk * C::TILE_M + rank * BM + q * 32;
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
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_cluster(tempty0 + 8u * static_cast<uint32_t>(acc));
                else mbar_arrive(smem_u32(&tempty[acc]));
            }
            next_acc<C::ACCS>(acc, acc_phase);
        }
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // a pair frees TMEM only after the leader's MMAs into both CTAs drained and
    // no arrival to the leader's barriers is still in flight
    if constexpr (PAIR) cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------- host --
// The scale atoms of a [rows, KB] block grid as a 3-D tensor of 32-bit words:
// x = the 128 words of an atom, y = atom column (G of them), z = atom row; a
// box of one atom column and `atoms` atom rows.  Atoms past the grid read as
// zeros (bytes 0, factor 2^-127) on rows whose codes are zero-filled too.
bool make_sf_map(CUtensorMap* map, const void* base, int64_t rows, int64_t KB, int atoms) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int64_t G = (KB + 3) / 4, RB = (rows + 127) / 128;
    cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(RB)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kMxAtomBytes), static_cast<cuuint64_t>(G * kMxAtomBytes)};
    cuuint32_t box[3] = {128, 1, static_cast<cuuint32_t>(atoms)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN, bool PAIR>
struct MxLaunchInfo {
    cudaError_t attr_err = cudaSuccess;
    int max_clusters = 0;  // co-resident 2-CTA clusters (PAIR only)
};

template <int BN, bool PAIR>
const MxLaunchInfo<BN, PAIR>& mx_launch_info() {
    using C = MxCfg<BN, PAIR>;
    static MxLaunchInfo<BN, PAIR> info;
    static std::once_flag once;
    std::call_once(once, [] {
        auto kern = mx_gemm_kernel<BN, PAIR>;
        info.attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (PAIR && info.attr_err == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * sm_count());
            cfg.blockDim = dim3(kMxGemmThreads);
            cfg.dynamicSmemBytes = C::SMEM_BYTES;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
                (void)cudaGetLastError();
                n = 0;
            }
            info.max_clusters = n;
        }
    });
    return info;
}

template <int BN, bool PAIR>
int launch_mx_gemm(const void* a, const uint8_t* sfa, const void* b, const uint8_t* sfb, void* d, int64_t M,
                   int64_t N, int64_t K, int fa, int fb, int* status, cudaStream_t stream) {
    using C = MxCfg<BN, PAIR>;
    const MxLaunchInfo<BN, PAIR>& info = mx_launch_info<BN, PAIR>();
    if (info.attr_err != cudaSuccess) return FP8Q_ERR_CUDA;
    alignas(64) CUtensorMap mapA, mapB, mapD, mapSA, mapSB;
    const int64_t KB = K / kMxBlock;
    if (!make_kmajor_map(&mapA, a, M, K, BM) || !make_kmajor_map(&mapB, b, N, K, C::B_ROWS) ||
        !make_out_map(&mapD, d, M, N) || !make_sf_map(&mapSA, sfa, M, KB, 1) ||
        !make_sf_map(&mapSB, sfb, N, KB, C::BNC))
        return FP8Q_ERR_CUDA;
    const int64_t tiles = ((M + C::TILE_M - 1) / C::TILE_M) * ((N + BN - 1) / BN);
    const uint32_t idesc0 = idesc_mx(static_cast<uint32_t>(fa), static_cast<uint32_t>(fb), C::MMA_M, BN, 0);
    auto kern = mx_gemm_kernel<BN, PAIR>;
    if constexpr (PAIR) {
        if (info.max_clusters < 1) return FP8Q_ERR_CUDA;
        const int clusters = static_cast<int>(std::min<int64_t>(tiles, info.max_clusters));
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(2 * clusters);
        cfg.blockDim = dim3(kMxGemmThreads);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        if (cudaLaunchKernelEx(&cfg, kern, mapA, mapB, mapD, mapSA, mapSB, M, N, K, idesc0, status) != cudaSuccess) {
            (void)cudaGetLastError();
            return FP8Q_ERR_CUDA;
        }
    } else {
        const int grid = static_cast<int>(std::min<int64_t>(tiles, sm_count()));
        if (launch_pdl(kern, dim3(grid), dim3(kMxGemmThreads), C::SMEM_BYTES, stream, mapA, mapB, mapD, mapSA,
                       mapSB, M, N, K, idesc0, status) != cudaSuccess) {
            (void)cudaGetLastError();
            return FP8Q_ERR_CUDA;
        }
    }
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}

struct MxShape {
    bool pair;
    int bn;
};

std::atomic<int> g_mx_tile{-1};  // fp8q_mx_set_tile: -1 = automatic, else (pair << 16) | bn

// Tile shape: whole waves of tiles (1-CTA tiles on the SMs, 256-row pair tiles
// on the SM pairs), each shape scored by its time per wave relative to the
// 1-CTA 128-wide tile (measured on GB300 at 16384 x 4096 -> 1024, 8192^3 and
// 131072 x 6400 -> 1600: 256 wide 1.24-1.31, pair 128 1.02, pair 256
// 1.23-1.35, i.e. pair and 1-CTA tiles level within a few per cent; ties go to
// the earlier candidate).  A pair needs M > 128; otherwise the 1-CTA tile of
// the same width runs.
MxShape pick_mx_shape(int64_t M, int64_t N) {
    const int ov = g_mx_tile.load(std::memory_order_relaxed);
    if (ov >= 0) return MxShape{(ov >> 16) != 0 && M > BM, ov & 0xFFFF};
    struct Cand { bool pair; int bn; double t; };
    static constexpr Cand kCands[] = {
        {false, 128, 1.00}, {false, 256, 1.28}, {true, 128, 1.02}, {true, 256, 1.29},
    };
    const int64_t sms = sm_count();
    MxShape best{false, 128};
    double best_cost = -1.0;
    for (const Cand& c : kCands) {
        if (c.pair && M <= BM) continue;
        const int64_t tile_m = c.pair ? 2 * BM : BM;
        const int64_t units = c.pair ? sms / 2 : sms;
        const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + c.bn - 1) / c.bn);
        const double cost = static_cast<double>((tiles + units - 1) / units) * c.t;
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = MxShape{c.pair, c.bn}; }
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
        const uint32_t KB = static_cast<uint32_t>(K / kMxBlock);
        auto kern = fmt == FP8Q_E5M2 ? quant_mx_rows_kernel<ACT, FP8Q_E5M2> : quant_mx_rows_kernel<ACT, FP8Q_E4M3>;
        e = launch_pdl(kern, dim3(grid), dim3(kMxThreads), 0, stream, static_cast<const uint4*>(h), nchunks, KB,
                       make_divu32(KB), static_cast<int64_t>((KB + 3) / 4), static_cast<uint4*>(act_out),
                       static_cast<uint2*>(q_out), sf_out, amax_out, sat);
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
    // (rows: fewer than 2^32 blocks, the kernel's 32-bit block index)
    if (M < 0 || (rows ? (K < 32 || K % 32 != 0 || M * (K / 32) > int64_t(0xFFFFFFFF))
                       : (K < 16 || K % 16 != 0 || M % 32 != 0 || (K + kMxColTileC - 1) / kMxColTileC > 65535)))
        return FP8Q_ERR_SHAPE;
    if (!aligned16(h) || !aligned16(act_out) || !aligned16(q_out) || !aligned16(q_t_out) || !aligned16(sf_out) ||
        !aligned16(sf_t_out) || (reinterpret_cast<uintptr_t>(amax_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(sat_count) & 7u))
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
    // TMA coordinates are 32-bit: the second CTA of the last pair tile starts at
    // row ceil(M / 256) * 256 - 128
    if (M > (int64_t(1) << 31) - 2 * BM || N > (int64_t(1) << 31) - 256 || K > (int64_t(1) << 31) - BK)
        return FP8Q_ERR_SHAPE;
    if (!aligned16(x_q) || !aligned16(wt_q) || !aligned16(y) || !aligned16(sf_x) || !aligned16(sf_w) ||
        (reinterpret_cast<uintptr_t>(status) & 3u))
        return FP8Q_ERR_ALIGN;
    if (!device_is_sm103()) return FP8Q_ERR_UNSUPPORTED;
    if (M == 0) return FP8Q_OK;
    const MxShape sh = pick_mx_shape(M, N);
    if (sh.pair) {
        if (sh.bn == 256) return launch_mx_gemm<256, true>(x_q, sf_x, wt_q, sf_w, y, M, N, K, fmt_x, fmt_w, status, stream);
        return launch_mx_gemm<128, true>(x_q, sf_x, wt_q, sf_w, y, M, N, K, fmt_x, fmt_w, status, stream);
    }
    if (sh.bn == 256) return launch_mx_gemm<256, false>(x_q, sf_x, wt_q, sf_w, y, M, N, K, fmt_x, fmt_w, status, stream);
    return launch_mx_gemm<128, false>(x_q, sf_x, wt_q, sf_w, y, M, N, K, fmt_x, fmt_w, status, stream);
}

extern "C" int64_t fp8_mx_scale_bytes(int64_t rows, int64_t K) {
    if (rows < 0 || K < 0 || K % 32 != 0) return -1;
    return ((rows + 127) / 128) * ((K / 32 + 3) / 4) * kMxAtomBytes;
}

extern "C" int fp8q_mx_set_tile(int pair, int bn) {
    if (pair == 0 && bn == 0) {
        g_mx_tile.store(-1);
        return FP8Q_OK;
    }
    if ((pair != 0 && pair != 1) || (bn != 128 && bn != 256)) return FP8Q_ERR_UNSUPPORTED;
    g_mx_tile.store((pair << 16) | bn);
    return FP8Q_OK;
}
