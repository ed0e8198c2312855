// quant.cu -- the fused activation + quantize step and its C entry point.
//
// "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records" (second
// paragraph): one kernel applies the activation while the values sit in
// registers, writes the BF16 copy kept for the backward pass, emits the FP8
// copy under a scale taken from the previous step's amax times a margin, and
// keeps small running maxima, so the large tensor is never read twice.
// "FP8 training: what it is and how it works", Step 2 (scale = max / amax) and
// Trade-offs (online amax per 1x128 activation tile / 128x128 weight block).
//
// Per element:  a = act(h);  abf = BF16(a);  v = abf * s (float32);
//               q = FP8(v) (round to nearest even, saturate);  amax = max |abf|.
//
// Kernels:
//   quant_stream_kernel  per-tensor scale, or 1x128 groups; row-major outputs.
//                        HBM-bound: 16-byte loads/stores, four loads in
//                        flight per thread, one pass over the tensor,
//                        amax by warp reduce -> shared memory -> 1 atomic/CTA.
//   quant_tile_kernel    128x128 tiles through shared memory: the transposed
//                        FP8 copy (the weight's K-major GEMM operand) and the
//                        128x128 block scales; the BF16 tile lands in shared
//                        memory by cp.async (large grids).
//   quant_tile_regs_kernel  the same with the loads landing in registers
//                        (grids of up to two rounds).
#include "common.cuh"
#include "quant_ops.cuh"

#include <algorithm>
#include <cfloat>

namespace fp8q {

namespace {

constexpr int kThreads = 256;

// CTA-wide reduction of (amax bits, saturation count), then one atomic each.
__device__ __forceinline__ void block_reduce_publish(uint32_t amax16, uint32_t nsat,
                                                     float* amax_out, unsigned long long* sat_out) {
    __shared__ uint32_t s_amax[kThreads / 32], s_sat[kThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    amax16 = __reduce_max_sync(0xFFFFFFFFu, amax16);
    nsat = __reduce_add_sync(0xFFFFFFFFu, nsat);
    if (lane == 0) { s_amax[warp] = amax16; s_sat[warp] = nsat; }
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        uint32_t a = lane < nw ? s_amax[lane] : 0u;
        uint32_t c = lane < nw ? s_sat[lane] : 0u;
        a = __reduce_max_sync(0xFFFFFFFFu, a);
        c = __reduce_add_sync(0xFFFFFFFFu, c);
        if (lane == 0) {
            // a non-negative float orders like its bit pattern
            if (amax_out && a) atomicMax(reinterpret_cast<unsigned int*>(amax_out), a << 16);
            if (sat_out && c) atomicAdd(sat_out, static_cast<unsigned long long>(c));
        }
    }
}

// The optional FP8 cache of the pre-activation itself ("FP8 training: what
// it is and how it works", Trade-offs and edge cases: the activations kept for
// the backward pass are stored in FP8): h_q = E4M3(float32(h * s_h)) of the
// BF16 input h, with its own delayed scale, maximum and saturation count, so a
// backward that needs act'(H) reads 1 byte per element instead of 2.
struct HCache {
    uint2* hq;           // [M,K] E4M3, or nullptr
    float s;             // s_h
    uint32_t amax2 = 0;  // max |h| (two 16-bit lanes)
    uint32_t nsat = 0;   // #{|h s_h| > 448}
};

__device__ __forceinline__ void h_cache8(HCache& c, uint4 x, uint2* dst) {
    c.amax2 = __vmaxu2(c.amax2, x.x & 0x7FFF7FFFu);
    c.amax2 = __vmaxu2(c.amax2, x.y & 0x7FFF7FFFu);
    c.amax2 = __vmaxu2(c.amax2, x.z & 0x7FFF7FFFu);
    c.amax2 = __vmaxu2(c.amax2, x.w & 0x7FFF7FFFu);
    st_v2(dst, cast8<FP8Q_E4M3>(x, c.s, c.nsat));
}

// Per-tensor streaming pass of CTA `cta` out of `ncta`: each thread owns
// 8-element chunks, U loads in flight, grid-stride over the tensor.  HQ: the
// chunk is also cast into the pre-activation cache.
template <int ACT, int FMT, int U = 4, bool HQ = false>
__device__ __forceinline__ void stream_body(const uint4* __restrict__ h, int64_t nchunks, float s,
                                            uint4* __restrict__ act_out, uint2* __restrict__ q_out,
                                            int64_t cta, int64_t ncta, uint32_t& amax2, uint32_t& nsat,
                                            HCache* hc = nullptr) {
    const int64_t tid = cta * blockDim.x + threadIdx.x;
    const int64_t nthreads = ncta * blockDim.x;
    int64_t i = tid;
    for (; i + (U - 1) * nthreads < nchunks; i += U * nthreads) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = ld_stream_v4(h + i + u * nthreads);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if constexpr (HQ) h_cache8(*hc, x[u], hc->hq + i + u * nthreads);
            uint4 a = act8<ACT>(x[u], amax2);
            if (act_out) st_stream_v4(act_out + i + u * nthreads, a);
            uint2 q = cast8<FMT>(a, s, nsat);
            if (q_out) st_v2(q_out + i + u * nthreads, q);
        }
    }
    for (; i < nchunks; i += nthreads) {
        const uint4 x = ld_stream_v4(h + i);
        if constexpr (HQ) h_cache8(*hc, x, hc->hq + i);
        uint4 a = act8<ACT>(x, amax2);
        if (act_out) st_stream_v4(act_out + i, a);
        uint2 q = cast8<FMT>(a, s, nsat);
        if (q_out) st_v2(q_out + i, q);
    }
}

// ---------------------------------------------------------------------------
// Streaming kernel.  GROUP = false: per-tensor scale, each thread owns 8-element
// chunks (16 B in), four loads in flight (a grid-stride loop covers grids
// smaller than the tensor).  GROUP = true:
// 1x128 groups, a half-warp owns one group (16 lanes x 8 elements), the group
// amax is a 16-lane shuffle reduction, two groups in flight per half-warp.
// ---------------------------------------------------------------------------
template <int ACT, int FMT, bool GROUP>
__global__ void __launch_bounds__(kThreads)
quant_stream_kernel(const uint4* __restrict__ h, int64_t nchunks, const float* __restrict__ scale,
                    uint4* __restrict__ act_out, uint2* __restrict__ q_out,
                    float* __restrict__ gscale, float* __restrict__ amax_out,
                    unsigned long long* __restrict__ sat_out) {
    uint32_t amax2 = 0, nsat = 0;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    pdl_wait();

    if constexpr (!GROUP) {
        stream_body<ACT, FMT>(h, nchunks, *scale, act_out, q_out, blockIdx.x, gridDim.x, amax2, nsat);
    } else {
        // chunk index = group * 16 + l16.  The loop is warp-uniform so all 32
        // lanes take part in the shuffles; a warp handles 2*U consecutive
        // groups per trip (half-warp `half` takes every other one).
        const int l16 = threadIdx.x & 15, half = (threadIdx.x >> 4) & 1;
        const int64_t ngroups = nchunks >> 4;
        const int64_t warp_id = tid >> 5, nwarps = nthreads >> 5;
        constexpr int U = 2;
        for (int64_t wg = warp_id; wg * (2 * U) < ngroups; wg += nwarps) {
            uint4 x[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t g = wg * (2 * U) + u * 2 + half;
                x[u] = g < ngroups ? ld_stream_v4(h + g * 16 + l16) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t g = wg * (2 * U) + u * 2 + half;
                uint32_t m2 = 0;
                uint4 a = act8<ACT>(x[u], m2);
                uint32_t m = max16x2(m2);
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                const float s = group_scale<FMT>(m);
                if (g < ngroups) {
                    amax2 = __vmaxu2(amax2, m);
                    if (act_out) st_stream_v4(act_out + g * 16 + l16, a);
                    uint2 q = cast8<FMT>(a, s, nsat);
                    if (q_out) st_v2(q_out + g * 16 + l16, q);
                    if (l16 == 0 && gscale) gscale[g] = s;
                }
            }
        }
    }
    pdl_launch_dependents();  // late: the next kernel's CTAs fill SMs as this grid drains
    block_reduce_publish(max16x2(amax2), nsat, amax_out, sat_out);
}

// ---------------------------------------------------------------------------
// Tiled kernel: one CTA per 128x128 tile of h [M,K].  Chunk c = it*256 + tid
// (it = 0..7) is row c/16, columns (c%16)*8..+7 of the tile, so a half-warp
// holds one 128-wide row segment (a 1x128 group when the tile is aligned).
// ---------------------------------------------------------------------------
constexpr int kTile = 128;
constexpr int kTqPitch = kTile;  // bytes per row of the FP8 tile in shared memory
constexpr int kTileCtasPerSm = 6;  // quant_tile_kernel: 32 KB of shared memory and <= 42 registers each

// Byte offset of the 8-byte piece j (columns 8j..8j+7) of tile row r in the
// shared-memory FP8 tile: the 4-byte words of row r are permuted by
// XOR-ing their index with 4 * ((r / 16) % 8), so that the column-wise reads
// of store_transposed hit every bank once; an 8-byte piece stays whole.
__device__ __forceinline__ int tq_offset(int r, int j) {
    return r * kTqPitch + ((j * 8) ^ (((r >> 4) & 7) << 4));
}

// Write the tile's FP8 codes (tq: complete, laid out by tq_offset) transposed
// into q_t [K,M]: output row k = col0 + j holds tile column j.  Thread t takes
// the 16 tile rows 16p..16p+15 (p = t % 8) of the four tile columns
// 4q..4q+3 (q = t / 8): sixteen 32-bit reads (one per row; a warp's 32 reads
// of a row fall in 32 different banks), a 4x4 byte transpose in registers
// (byte_perm), and four 16-byte stores, one per output row.  The eight threads
// with the same q write the 128 contiguous bytes m = row0 .. row0 + 127 of
// each of their output rows, so a warp's store covers four whole lines.
// M % 16 == 0, so a piece is inside q_t whenever its first row is.
__device__ __forceinline__ void store_transposed(const uint8_t* tq, uint8_t* __restrict__ q_t_out, int64_t M,
                                                 int64_t K, int64_t row0, int64_t col0) {
    static_assert(kThreads == 256 && kTile == 128, "256 threads: 8 row groups x 32 column groups");
    const int p = threadIdx.x & 7, q = threadIdx.x >> 3;
    uint32_t x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = p * 16 + i;
        x[i] = *reinterpret_cast<const uint32_t*>(tq + r * kTqPitch + ((q ^ (p << 2)) << 2));
    }
    const int64_t mcol = row0 + p * 16;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        // byte c of the first word -> byte 0, byte c of the second -> byte 1
        const uint32_t sel = static_cast<uint32_t>(c) | (static_cast<uint32_t>(4 + c) << 4);
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = __byte_perm(x[4 * j], x[4 * j + 1], sel);
            const uint32_t hi = __byte_perm(x[4 * j + 2], x[4 * j + 3], sel);
            o[j] = __byte_perm(lo, hi, 0x5410);  // lo bytes 0,1 then hi bytes 0,1
        }
        const int64_t krow = col0 + q * 4 + c;
        if (krow < K && mcol < M) st_v4(q_t_out + krow * M + mcol, make_uint4(o[0], o[1], o[2], o[3]));
    }
}

// One 128x128 tile (bx, by) of h [M,K]; per-tensor scale, or the tile's
// 128x128 block scale, or 1x128 row-group scales (gscale, group_rows).
// The BF16 tile lands in shared memory by cp.async (tbuf, 32 KB: no registers
// hold the loads in flight, so six CTAs fit an SM) as two groups, one per
// 64-row half, and each half is processed as soon as it has landed.  The FP8 tile of the transposed copy reuses tbuf's first
// 16 KB: its rows 0-63 are written after every thread has read the first
// half (one barrier), its rows 64-127 fall on input rows 32-63, read by then.
// Chunk c = it * 256 + tid (it = 0..7) is tile row c / 16, columns
// (c % 16) * 8 .. + 7, at tbuf + 16 c, so a half-warp holds one 128-wide row
// segment (a 1x128 group when the tile is aligned).  s_blk: one word per warp.
template <int ACT, int FMT>
__device__ __forceinline__ void tile_body(const uint16_t* __restrict__ h, int64_t M, int64_t K,
                                          const float* __restrict__ scale, uint16_t* __restrict__ act_out,
                                          uint8_t* __restrict__ q_out, uint8_t* __restrict__ q_t_out,
                                          float* __restrict__ gscale, int group_rows, int64_t bx, int64_t by,
                                          uint8_t* tbuf, uint32_t* s_blk, uint32_t& amax2, uint32_t& nsat) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, l16 = tid & 15;
    const int64_t row0 = by * kTile;
    const int64_t col0 = bx * kTile;
    const int64_t kgroups = K / kTile;

#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int c = it * kThreads + tid;
        const int64_t row = row0 + (c >> 4), col = col0 + (c & 15) * 8;
        uint8_t* dst = tbuf + c * 16;
        if (row < M && col < K) cp_async16(smem_u32(dst), h + row * K + col);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        if (it == 3 || it == 7) cp_async_commit();  // group 0: rows 0-63, group 1: rows 64-127
    }
    const bool block_scale = gscale != nullptr && group_rows == kTile;
    if (block_scale) cp_async_wait<0>();  // the block scale needs the whole tile first
    else cp_async_wait<1>();
    __syncthreads();

    float s_tensor = 1.0f;
    if (gscale == nullptr) {
        s_tensor = *scale;
    } else if (group_rows == kTile) {
        // the block scale needs the whole tile's maximum before any cast
        uint32_t m2 = 0;
#pragma unroll
        for (int it = 0; it < 8; ++it)
            (void)act8<ACT>(*reinterpret_cast<const uint4*>(tbuf + (it * kThreads + tid) * 16), m2);
        uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max16x2(m2));
        if (lane == 0) s_blk[warp] = m;
        __syncthreads();
        m = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) m = max(m, s_blk[w]);
        s_tensor = group_scale<FMT>(m);
        if (tid == 0) gscale[by * kgroups + bx] = s_tensor;
    }

    uint8_t* tq = tbuf;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        if (half == 1 && !block_scale) {
            cp_async_wait<0>();
            __syncthreads();
        }
        uint4 a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const uint4*>(tbuf + ((half * 4 + i) * kThreads + tid) * 16);
        if (half == 0 && q_t_out) __syncthreads();  // rows 0-63 read by all before tq overwrites them
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = (half * 4 + i) * kThreads + tid;
            const int r = c >> 4;
            const int64_t row = row0 + r, col = col0 + (c & 15) * 8;
            const bool ok = row < M && col < K;
            uint32_t m2 = 0;
            a[i] = act8<ACT>(a[i], m2);
            amax2 = __vmaxu2(amax2, m2);
            if (ok && act_out) st_stream_v4(act_out + row * K + col, a[i]);
            float s = s_tensor;
            if (gscale != nullptr && group_rows == 1) {
                uint32_t m = max16x2(m2);
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                s = group_scale<FMT>(m);
                if (ok && l16 == 0) gscale[row * kgroups + bx] = s;
            }
            uint32_t ns = 0;
            const uint2 q = cast8<FMT>(a[i], s, ns);
            if (ok) {
                nsat += ns;
                if (q_out) st_v2(q_out + row * K + col, q);
            }
            if (q_t_out) *reinterpret_cast<uint2*>(tq + tq_offset(r, c & 15)) = q;
        }
    }

    if (q_t_out) {
        __syncthreads();
        store_transposed(tq, q_t_out, M, K, row0, col0);
    }
}

template <int ACT, int FMT>
__global__ void __launch_bounds__(kThreads, kTileCtasPerSm)
quant_tile_kernel(const uint16_t* __restrict__ h, int64_t M, int64_t K, const float* __restrict__ scale,
                  uint16_t* __restrict__ act_out, uint8_t* __restrict__ q_out,
                  uint8_t* __restrict__ q_t_out, float* __restrict__ gscale, int group_rows,
                  float* __restrict__ amax_out, unsigned long long* __restrict__ sat_out) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ __align__(128) uint8_t tbuf[kTile * kTile * 2];
    __shared__ uint32_t s_blk[kThreads / 32];
    uint32_t amax2 = 0, nsat = 0;
    tile_body<ACT, FMT>(h, M, K, scale, act_out, q_out, q_t_out, gscale, group_rows, blockIdx.x, blockIdx.y, tbuf,
                        s_blk, amax2, nsat);
    block_reduce_publish(max16x2(amax2), nsat, amax_out, sat_out);
}

// tile_body with the tile's loads landing in registers (all eight of a thread
// issued before any store): shorter per CTA than the shared-memory landing, so
// it wins on grids the GPU holds in one or two rounds.
// tq: kTile x kTqPitch bytes of shared memory (16-byte aligned); s_blk: one
// word per warp.
template <int ACT, int FMT>
__device__ __forceinline__ void tile_body_regs(const uint16_t* __restrict__ h, int64_t M, int64_t K,
                                          const float* __restrict__ scale, uint16_t* __restrict__ act_out,
                                          uint8_t* __restrict__ q_out, uint8_t* __restrict__ q_t_out,
                                          float* __restrict__ gscale, int group_rows, int64_t bx, int64_t by,
                                          uint8_t* tq, uint32_t* s_blk, uint32_t& amax2, uint32_t& nsat) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, l16 = tid & 15;
    const int64_t row0 = by * kTile;
    const int64_t col0 = bx * kTile;
    const int64_t kgroups = K / kTile;

    uint4 a[8];
    uint32_t m16[8];
    // all eight loads are issued before any store, so they overlap in flight
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int c = it * kThreads + tid;
        const int64_t row = row0 + (c >> 4), col = col0 + (c & 15) * 8;
        a[it] = (row < M && col < K) ? ld_stream_v4(h + row * K + col) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int c = it * kThreads + tid;
        const int64_t row = row0 + (c >> 4), col = col0 + (c & 15) * 8;
        const bool ok = row < M && col < K;
        uint32_t m2 = 0;
        a[it] = act8<ACT>(a[it], m2);
        m16[it] = max16x2(m2);
        amax2 = __vmaxu2(amax2, m2);
        if (ok && act_out) st_stream_v4(act_out + row * K + col, a[it]);
    }

    float s_tensor = 1.0f;
    if (gscale == nullptr) {
        s_tensor = *scale;
    } else if (group_rows == kTile) {
        uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max16x2(amax2));
        if (lane == 0) s_blk[warp] = m;
        __syncthreads();
        m = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) m = max(m, s_blk[w]);
        s_tensor = group_scale<FMT>(m);
        if (tid == 0) gscale[by * kgroups + bx] = s_tensor;
    }

#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int c = it * kThreads + tid;
        const int r = c >> 4;
        const int64_t row = row0 + r, col = col0 + (c & 15) * 8;
        const bool ok = row < M && col < K;
        float s = s_tensor;
        if (gscale != nullptr && group_rows == 1) {
            uint32_t m = m16[it];
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            s = group_scale<FMT>(m);
            if (ok && l16 == 0) gscale[row * kgroups + bx] = s;
        }
        uint32_t ns = 0;
        uint2 q = cast8<FMT>(a[it], s, ns);
        if (ok) {
            nsat += ns;
            if (q_out) st_v2(q_out + row * K + col, q);
        }
        if (q_t_out) *reinterpret_cast<uint2*>(tq + tq_offset(r, c & 15)) = q;
    }

    if (q_t_out) {
        __syncthreads();
        store_transposed(tq, q_t_out, M, K, row0, col0);
    }
}

template <int ACT, int FMT>
__global__ void __launch_bounds__(kThreads)
quant_tile_regs_kernel(const uint16_t* __restrict__ h, int64_t M, int64_t K, const float* __restrict__ scale,
                  uint16_t* __restrict__ act_out, uint8_t* __restrict__ q_out,
                  uint8_t* __restrict__ q_t_out, float* __restrict__ gscale, int group_rows,
                  float* __restrict__ amax_out, unsigned long long* __restrict__ sat_out) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ __align__(16) uint8_t tq[kTile * kTqPitch];
    __shared__ uint32_t s_blk[kThreads / 32];
    uint32_t amax2 = 0, nsat = 0;
    tile_body_regs<ACT, FMT>(h, M, K, scale, act_out, q_out, q_t_out, gscale, group_rows, blockIdx.x, blockIdx.y, tq,
                        s_blk, amax2, nsat);
    block_reduce_publish(max16x2(amax2), nsat, amax_out, sat_out);
}

// ---------------------------------------------------------------------------
// Batched kernel: several per-tensor quantize calls in one grid.  CTA b runs
// entry i when block0[i] <= b < block0[i + 1]: the tile pass (transposed
// copy) for entries with q_t_out, the streaming pass otherwise.  Activation
// and format are per entry (uniform within a CTA).
// ---------------------------------------------------------------------------
struct BatchEntry {
    const uint16_t* h;
    int64_t M, K;
    const float* scale;
    uint16_t* act_out;
    uint8_t* q_out;
    uint8_t* q_t_out;
    float* amax_out;
    unsigned long long* sat_out;
    uint8_t* hq_out;                // the pre-activation's E4M3 cache, or nullptr
    const float* scale_h;
    float* amax_h;
    unsigned long long* sat_h;
    int64_t block0, nblocks;  // this entry's CTAs
    int64_t tiles_x;          // tile pass: tiles along K
    int act, fmt;
};

struct BatchParams {
    BatchEntry e[FP8Q_BATCH_MAX];
    int n;
};

constexpr int kBatchU = 8;           // streaming pass: loads in flight per thread
constexpr int kBatchCtasPerSm = 4;   // 64 registers per thread: no spills in either pass

// Per-tensor tile pass of the batched kernel: the same outputs as tile_body
// with a per-tensor scale, but the tile is taken in two 64-row halves of four
// loads per thread, which keeps the batched kernel's registers (and so its
// occupancy) set by the streaming pass.  Measured back to back on GB300 at
// 8192 x 3072 (+ the 3072 x 768 weight): 21.8 us for both tensors in one
// launch, against 19.5 + 12.0 us as two launches.
template <int ACT, int FMT, bool HQ = false>
__device__ __forceinline__ void tile_pt_body(const uint16_t* __restrict__ h, int64_t M, int64_t K, float s,
                                             uint16_t* __restrict__ act_out, uint8_t* __restrict__ q_out,
                                             uint8_t* __restrict__ q_t_out, int64_t bx, int64_t by, uint8_t* tq,
                                             uint32_t& amax2, uint32_t& nsat, HCache* hc = nullptr) {
    const int tid = threadIdx.x;
    const int64_t row0 = by * kTile;
    const int64_t col0 = bx * kTile;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        uint4 a[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int c = (half * 4 + it) * kThreads + tid;
            const int64_t row = row0 + (c >> 4), col = col0 + (c & 15) * 8;
            a[it] = (row < M && col < K) ? ld_stream_v4(h + row * K + col) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int c = (half * 4 + it) * kThreads + tid;
            const int r = c >> 4;
            const int64_t row = row0 + r, col = col0 + (c & 15) * 8;
            const bool ok = row < M && col < K;
            if constexpr (HQ) {
                if (ok) h_cache8(*hc, a[it], reinterpret_cast<uint2*>(hc->hq) + (row * K + col) / 8);
            }
            uint32_t m2 = 0;
            a[it] = act8<ACT>(a[it], m2);
            amax2 = __vmaxu2(amax2, m2);
            uint32_t ns = 0;
            const uint2 q = cast8<FMT>(a[it], s, ns);
            if (ok) {
                nsat += ns;
                if (act_out) st_stream_v4(act_out + row * K + col, a[it]);
                if (q_out) st_v2(q_out + row * K + col, q);
            }
            if (q_t_out) *reinterpret_cast<uint2*>(tq + tq_offset(r, c & 15)) = q;
        }
    }
    if (q_t_out) {
        __syncthreads();
        store_transposed(tq, q_t_out, M, K, row0, col0);
    }
}

template <int ACT, int FMT, bool HQ>
__device__ __forceinline__ void batch_entry_body_t(const BatchEntry& e, int64_t cta, uint8_t* tq,
                                                   uint32_t& amax2, uint32_t& nsat, HCache* hc) {
    if (e.q_t_out) {
        tile_pt_body<ACT, FMT, HQ>(e.h, e.M, e.K, *e.scale, e.act_out, e.q_out, e.q_t_out, cta % e.tiles_x,
                                   cta / e.tiles_x, tq, amax2, nsat, hc);
    } else {
        // with the cache a thread holds four loads in flight, not eight: the
        // extra cast keeps the 64-register budget without spills
        stream_body<ACT, FMT, HQ ? 4 : kBatchU, HQ>(reinterpret_cast<const uint4*>(e.h), e.M * e.K / 8, *e.scale,
                                           reinterpret_cast<uint4*>(e.act_out), reinterpret_cast<uint2*>(e.q_out),
                                           cta, e.nblocks, amax2, nsat, hc);
    }
}

template <int ACT, int FMT, bool HQ>
__device__ __forceinline__ void batch_entry_body(const BatchEntry& e, int64_t cta, uint8_t* tq, uint32_t* s_blk,
                                                 uint32_t& amax2, uint32_t& nsat, HCache* hc) {
    if (HQ && e.hq_out) batch_entry_body_t<ACT, FMT, HQ>(e, cta, tq, amax2, nsat, hc);
    else batch_entry_body_t<ACT, FMT, false>(e, cta, tq, amax2, nsat, hc);
}

// HQ: some entry writes the pre-activation's E4M3 cache (a kernel of its own,
// so the plain batch keeps its registers).
template <bool HQ>
__global__ void __launch_bounds__(kThreads, kBatchCtasPerSm)
quant_batch_kernel(const __grid_constant__ BatchParams p) {
    __shared__ __align__(16) uint8_t tq[kTile * kTqPitch];
    __shared__ uint32_t s_blk[kThreads / 32];
    int i = 0;
    while (i + 1 < p.n && static_cast<int64_t>(blockIdx.x) >= p.e[i + 1].block0) ++i;
    const BatchEntry& e = p.e[i];
    const int64_t cta = static_cast<int64_t>(blockIdx.x) - e.block0;
    uint32_t amax2 = 0, nsat = 0;
    HCache hc;
    hc.hq = reinterpret_cast<uint2*>(e.hq_out);
    pdl_wait();
    hc.s = e.hq_out ? *e.scale_h : 1.0f;
    const int key = e.act * 2 + e.fmt;
    switch (key) {
        case FP8Q_ACT_IDENTITY * 2 + FP8Q_E4M3:
            batch_entry_body<FP8Q_ACT_IDENTITY, FP8Q_E4M3, HQ>(e, cta, tq, s_blk, amax2, nsat, &hc);
            break;
        case FP8Q_ACT_IDENTITY * 2 + FP8Q_E5M2:
            batch_entry_body<FP8Q_ACT_IDENTITY, FP8Q_E5M2, HQ>(e, cta, tq, s_blk, amax2, nsat, &hc);
            break;
        case FP8Q_ACT_RELU * 2 + FP8Q_E4M3:
            batch_entry_body<FP8Q_ACT_RELU, FP8Q_E4M3, HQ>(e, cta, tq, s_blk, amax2, nsat, &hc);
            break;
        case FP8Q_ACT_RELU * 2 + FP8Q_E5M2:
            batch_entry_body<FP8Q_ACT_RELU, FP8Q_E5M2, HQ>(e, cta, tq, s_blk, amax2, nsat, &hc);
            break;
        case FP8Q_ACT_RELU2 * 2 + FP8Q_E4M3:
            batch_entry_body<FP8Q_ACT_RELU2, FP8Q_E4M3, HQ>(e, cta, tq, s_blk, amax2, nsat, &hc);
            break;
        default:
            batch_entry_body<FP8Q_ACT_RELU2, FP8Q_E5M2, HQ>(e, cta, tq, s_blk, amax2, nsat, &hc);
            break;
    }
    pdl_launch_dependents();  // late: the next kernel's CTAs fill SMs as this grid drains
    block_reduce_publish(max16x2(amax2), nsat, e.amax_out, e.sat_out);
    if (HQ && e.hq_out) {
        __syncthreads();  // the reduction's shared words are reused
        block_reduce_publish(max16x2(hc.amax2), hc.nsat, e.amax_h, e.sat_h);
    }
}

// CTAs of the streaming pass over nchunks 16-byte chunks: each thread takes
// one batch of loads (the hardware refills SMs as CTAs retire).
int64_t stream_blocks(int64_t nchunks, int chunks_per_thread) {
    const int64_t per_cta = int64_t(kThreads) * chunks_per_thread;
    const int64_t want = (nchunks + per_cta - 1) / per_cta;
    return std::max<int64_t>(1, std::min<int64_t>(want, int64_t(1) << 30));
}

template <int ACT, int FMT>
int launch_quant(const void* h, int64_t M, int64_t K, const float* scale, void* act_out,
                 void* q_out, void* q_t_out, float* amax_out, unsigned long long* sat_count,
                 float* gscale, int group_rows, cudaStream_t stream) {
    const bool tiled = (q_t_out != nullptr) || (gscale != nullptr && group_rows == kTile);
    if (tiled) {
        dim3 grid(static_cast<unsigned>((K + kTile - 1) / kTile), static_cast<unsigned>((M + kTile - 1) / kTile));
        const int64_t tiles = int64_t(grid.x) * grid.y;
        // Up to two rounds of the register-landing kernel (64 registers: four
        // CTAs per SM) its shorter per-CTA path wins; beyond, the shared-memory
        // landing holds more bytes in flight per SM (measured on GB300: W
        // 6400 x 1600, 650 tiles: 9.9 against 10.8 us; 8192 x 8192: 53.5
        // against 41.8 us; dY 131072 x 1600 transposed: 115.2 against 107.6 us).
        const bool regs = tiles <= int64_t(2) * 4 * sm_count();
        cudaError_t e;
        if (regs) {
            e = launch_pdl(quant_tile_regs_kernel<ACT, FMT>, grid, dim3(kThreads), 0, stream,
                           static_cast<const uint16_t*>(h), M, K, scale, static_cast<uint16_t*>(act_out),
                           static_cast<uint8_t*>(q_out), static_cast<uint8_t*>(q_t_out), gscale, group_rows,
                           amax_out, sat_count);
        } else {
            // six 32 KB CTAs per SM need most of the unified L1 / shared memory as shared
            static const cudaError_t carve =
                cudaFuncSetAttribute(quant_tile_kernel<ACT, FMT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
            e = carve != cudaSuccess ? carve
                                     : launch_pdl(quant_tile_kernel<ACT, FMT>, grid, dim3(kThreads), 0, stream,
                                                  static_cast<const uint16_t*>(h), M, K, scale,
                                                  static_cast<uint16_t*>(act_out), static_cast<uint8_t*>(q_out),
                                                  static_cast<uint8_t*>(q_t_out), gscale, group_rows, amax_out,
                                                  sat_count);
        }
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return FP8Q_ERR_CUDA;
        }
    } else {
        // One pass: enough CTAs that each thread handles one batch of loads
        // (4 chunks per tensor pass, 2 groups per half-warp); the hardware
        // refills SMs as CTAs retire.  Measured faster than a persistent
        // grid-stride grid on GB300 (0.99 vs 0.89 of the copy rate at 4 GB).
        const int64_t nchunks = M * K / 8;
        const unsigned grid = static_cast<unsigned>(stream_blocks(nchunks, gscale ? 2 : 4));
        cudaError_t e;
        if (gscale)
            e = launch_pdl(quant_stream_kernel<ACT, FMT, true>, dim3(grid), dim3(kThreads), 0, stream,
                           static_cast<const uint4*>(h), nchunks, scale, static_cast<uint4*>(act_out),
                           static_cast<uint2*>(q_out), gscale, amax_out, sat_count);
        else
            e = launch_pdl(quant_stream_kernel<ACT, FMT, false>, dim3(grid), dim3(kThreads), 0, stream,
                           static_cast<const uint4*>(h), nchunks, scale, static_cast<uint4*>(act_out),
                           static_cast<uint2*>(q_out), static_cast<float*>(nullptr), amax_out, sat_count);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return FP8Q_ERR_CUDA;
        }
    }
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}

template <int ACT>
int launch_quant_fmt(int fmt, const void* h, int64_t M, int64_t K, const float* scale, void* act_out,
                     void* q_out, void* q_t_out, float* amax_out, unsigned long long* sat_count,
                     float* gscale, int group_rows, cudaStream_t stream) {
    if (fmt == FP8Q_E5M2)
        return launch_quant<ACT, FP8Q_E5M2>(h, M, K, scale, act_out, q_out, q_t_out, amax_out,
                                            sat_count, gscale, group_rows, stream);
    return launch_quant<ACT, FP8Q_E4M3>(h, M, K, scale, act_out, q_out, q_t_out, amax_out,
                                        sat_count, gscale, group_rows, stream);
}

// FP32 -> FP8 elementwise (fp8_cast_f32): the conversion the quantize
// kernels apply to v = BF16(act(h)) * s, four values per thread and step; the
// thread with i == n4 converts the last n % 4 values one by one.
template <int FMT>
__global__ void __launch_bounds__(kThreads)
cast_f32_kernel(const float4* __restrict__ x, uint32_t* __restrict__ q, int64_t n4, int64_t n) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i <= n4; i += stride) {
        if (i < n4) {
            const float4 v = x[i];
            q[i] = static_cast<uint32_t>(cvt_fp8x2<FMT>(v.x, v.y)) |
                   (static_cast<uint32_t>(cvt_fp8x2<FMT>(v.z, v.w)) << 16);
        } else {
            const float* xs = reinterpret_cast<const float*>(x);
            uint8_t* qs = reinterpret_cast<uint8_t*>(q);
            for (int64_t j = 4 * n4; j < n; ++j) qs[j] = static_cast<uint8_t>(cvt_fp8x2<FMT>(xs[j], 0.0f) & 0xFFu);
        }
    }
}

}  // namespace

}  // namespace fp8q

using namespace fp8q;

extern "C" int fp8_cast_f32(const float* x, void* q, int64_t n, int fmt, cudaStream_t stream) {
    if (n < 0) return FP8Q_ERR_SHAPE;
    if (fmt != FP8Q_E4M3 && fmt != FP8Q_E5M2) return FP8Q_ERR_UNSUPPORTED;
    if (n == 0) return FP8Q_OK;
    if (x == nullptr || q == nullptr) return FP8Q_ERR_NULL;
    if (!aligned16(x) || !aligned16(q)) return FP8Q_ERR_ALIGN;
    if (!device_is_sm103()) return FP8Q_ERR_UNSUPPORTED;
    const int64_t n4 = n / 4;
    const int64_t want = (n4 + kThreads) / kThreads;  // threads for i = 0 .. n4
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(want, int64_t(sm_count()) * 16));
    const float4* xv = reinterpret_cast<const float4*>(x);
    uint32_t* qv = static_cast<uint32_t*>(q);
    const cudaError_t e = fmt == FP8Q_E5M2
        ? launch_pdl(cast_f32_kernel<FP8Q_E5M2>, dim3(grid), dim3(kThreads), 0, stream, xv, qv, n4, n)
        : launch_pdl(cast_f32_kernel<FP8Q_E4M3>, dim3(grid), dim3(kThreads), 0, stream, xv, qv, n4, n);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8Q_ERR_CUDA;
    }
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}

// Argument checks of one quantize call (fp8_quant_fused_ex); the device check is the caller's.
static int check_quant_args(const void* h, int64_t M, int64_t K, int act, int fmt, const float* scale,
                            const void* act_out, const void* q_out, const void* q_t_out, const float* amax_out,
                            const unsigned long long* sat_count, const float* group_scales_out, int group_rows,
                            unsigned flags) {
    if (flags & ~static_cast<unsigned>(FP8Q_ACCUMULATE)) return FP8Q_ERR_UNSUPPORTED;
    if (h == nullptr && M != 0) return FP8Q_ERR_NULL;  // an empty tensor may have no storage
    if (act < FP8Q_ACT_IDENTITY || act > FP8Q_ACT_RELU2) return FP8Q_ERR_UNSUPPORTED;
    if (fmt != FP8Q_E4M3 && fmt != FP8Q_E5M2) return FP8Q_ERR_UNSUPPORTED;
    const bool group = group_scales_out != nullptr;
    if (group) {
        if (group_rows != 1 && group_rows != FP8Q_GROUP) return FP8Q_ERR_UNSUPPORTED;
        if (K % FP8Q_GROUP != 0) return FP8Q_ERR_SHAPE;
    } else if (scale == nullptr) {
        return FP8Q_ERR_NULL;
    }
    if (M < 0 || K < 16 || K % 16 != 0) return FP8Q_ERR_SHAPE;
    if (q_t_out != nullptr && M % 16 != 0) return FP8Q_ERR_SHAPE;
    if ((M + 127) / 128 > 65535 && (q_t_out != nullptr || (group && group_rows == FP8Q_GROUP)))
        return FP8Q_ERR_SHAPE;
    if (!aligned16(h) || !aligned16(act_out) || !aligned16(q_out) || !aligned16(q_t_out))
        return FP8Q_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(amax_out) & 3u) || (reinterpret_cast<uintptr_t>(group_scales_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(sat_count) & 7u))
        return FP8Q_ERR_ALIGN;
    return FP8Q_OK;
}

extern "C" int fp8_quant_fused(const void* h, int64_t M, int64_t K, int act, int fmt,
                               const float* scale, void* act_out, void* q_out, void* q_t_out,
                               float* amax_out, unsigned long long* sat_count,
                               float* group_scales_out, int group_rows, cudaStream_t stream) {
    return fp8_quant_fused_ex(h, M, K, act, fmt, scale, act_out, q_out, q_t_out, amax_out, sat_count,
                              group_scales_out, group_rows, 0u, stream);
}

extern "C" int fp8_quant_fused_ex(const void* h, int64_t M, int64_t K, int act, int fmt,
                                  const float* scale, void* act_out, void* q_out, void* q_t_out,
                                  float* amax_out, unsigned long long* sat_count,
                                  float* group_scales_out, int group_rows, unsigned flags,
                                  cudaStream_t stream) {
    const int st = check_quant_args(h, M, K, act, fmt, scale, act_out, q_out, q_t_out, amax_out, sat_count,
                                    group_scales_out, group_rows, flags);
    if (st != FP8Q_OK) return st;
    if (!device_is_sm103()) return FP8Q_ERR_UNSUPPORTED;

    const bool zero = !(flags & FP8Q_ACCUMULATE);
    if (zero && amax_out && cudaMemsetAsync(amax_out, 0, sizeof(float), stream) != cudaSuccess)
        return FP8Q_ERR_CUDA;
    if (zero && sat_count && cudaMemsetAsync(sat_count, 0, sizeof(unsigned long long), stream) != cudaSuccess)
        return FP8Q_ERR_CUDA;
    if (M == 0) return FP8Q_OK;

    switch (act) {
        case FP8Q_ACT_IDENTITY:
            return launch_quant_fmt<FP8Q_ACT_IDENTITY>(fmt, h, M, K, scale, act_out, q_out, q_t_out, amax_out,
                                                       sat_count, group_scales_out, group_rows, stream);
        case FP8Q_ACT_RELU:
            return launch_quant_fmt<FP8Q_ACT_RELU>(fmt, h, M, K, scale, act_out, q_out, q_t_out, amax_out,
                                                   sat_count, group_scales_out, group_rows, stream);
        default:
            return launch_quant_fmt<FP8Q_ACT_RELU2>(fmt, h, M, K, scale, act_out, q_out, q_t_out, amax_out,
                                                    sat_count, group_scales_out, group_rows, stream);
    }
}

extern "C" int fp8_quant_fused_batch(const fp8q_quant_args* args, int n, cudaStream_t stream) {
    if (!args) return FP8Q_ERR_NULL;
    if (n < 1 || n > FP8Q_BATCH_MAX) return FP8Q_ERR_SHAPE;
    BatchParams p = {};
    p.n = 0;
    int64_t blocks = 0;
    for (int i = 0; i < n; ++i) {
        const fp8q_quant_args& a = args[i];
        if (a.group_scales_out) return FP8Q_ERR_UNSUPPORTED;  // per-tensor scales only
        const int st = check_quant_args(a.h, a.M, a.K, a.act, a.fmt, a.scale, a.act_out, a.q_out, a.q_t_out,
                                        a.amax_out, a.sat_count, nullptr, a.group_rows, a.flags);
        if (st != FP8Q_OK) return st;
        if (a.hq_out) {  // the pre-activation's E4M3 cache
            if (!a.scale_h) return FP8Q_ERR_NULL;
            if (!aligned16(a.hq_out) || (reinterpret_cast<uintptr_t>(a.scale_h) & 3u) ||
                (reinterpret_cast<uintptr_t>(a.amax_h) & 3u) || (reinterpret_cast<uintptr_t>(a.sat_h) & 7u))
                return FP8Q_ERR_ALIGN;
        }
        if (a.M == 0) continue;
        BatchEntry& e = p.e[p.n++];
        e.h = static_cast<const uint16_t*>(a.h);
        e.M = a.M;
        e.K = a.K;
        e.scale = a.scale;
        e.act_out = static_cast<uint16_t*>(a.act_out);
        e.q_out = static_cast<uint8_t*>(a.q_out);
        e.q_t_out = static_cast<uint8_t*>(a.q_t_out);
        e.amax_out = a.amax_out;
        e.sat_out = a.sat_count;
        e.hq_out = static_cast<uint8_t*>(a.hq_out);
        e.scale_h = a.scale_h;
        e.amax_h = a.amax_h;
        e.sat_h = a.sat_h;
        e.act = a.act;
        e.fmt = a.fmt;
        e.tiles_x = (a.K + kTile - 1) / kTile;
        e.nblocks = a.q_t_out ? e.tiles_x * ((a.M + kTile - 1) / kTile) : stream_blocks(a.M * a.K / 8, kBatchU);
        e.block0 = blocks;
        blocks += e.nblocks;
    }
    if (blocks > (int64_t(1) << 31) - 1) return FP8Q_ERR_SHAPE;
    if (!device_is_sm103()) return FP8Q_ERR_UNSUPPORTED;
    for (int i = 0; i < n; ++i) {
        const fp8q_quant_args& a = args[i];
        if (a.flags & FP8Q_ACCUMULATE) continue;
        if (a.amax_out && cudaMemsetAsync(a.amax_out, 0, sizeof(float), stream) != cudaSuccess) return FP8Q_ERR_CUDA;
        if (a.sat_count && cudaMemsetAsync(a.sat_count, 0, sizeof(unsigned long long), stream) != cudaSuccess)
            return FP8Q_ERR_CUDA;
        if (a.hq_out && a.amax_h && cudaMemsetAsync(a.amax_h, 0, sizeof(float), stream) != cudaSuccess)
            return FP8Q_ERR_CUDA;
        if (a.hq_out && a.sat_h && cudaMemsetAsync(a.sat_h, 0, sizeof(unsigned long long), stream) != cudaSuccess)
            return FP8Q_ERR_CUDA;
    }
    if (p.n == 0) return FP8Q_OK;
    bool hq = false;
    for (int i = 0; i < p.n; ++i) hq = hq || p.e[i].hq_out != nullptr;
    if (launch_pdl(hq ? quant_batch_kernel<true> : quant_batch_kernel<false>, dim3(static_cast<unsigned>(blocks)),
                   dim3(kThreads), 0, stream, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8Q_ERR_CUDA;
    }
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}
