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
// Every GEMM here is D[M,N] = A[M,K] . B[N,K]^T with A and B K-major:
//   forward: A = X_q [M,K],   B = W_q^T [N,K]
//   dgrad:   A = dY_q [M,N],  B = W_q [K,N]   (the contraction runs over N)
//   wgrad:   A = X_q^T [K,M], B = dY_q^T [N,M] (the contraction runs over the tokens)
// Epilogue modes besides the plain dequantise-and-store: the 1x128 / 128x128
// group promotion (GROUP), the activation quantize of the next layer's input
// (EQ: the up-projection), the activation backward dH = dX act'(H) (DACT), and
// the one-launch step's extra quantize warps (FUSED).
//
// CTA = 6 warps (10 with 8 epilogue warps), persistent over output tiles
// (static round robin):
//   warp 0     TMA producer: one elected lane streams A/B k-blocks (128 B of
//              K per row, 128-byte swizzle) into a STAGES-deep ring.
//   warp 1     MMA issuer: allocates TMEM; one lane issues 4 x
//              tcgen05.mma.kind::f8f6f4 (K=32) per k-block and commits each
//              stage back to the producer.
//   warps 2-5  epilogue: tcgen05.ld the FP32 accumulator (each warp its 32
//              TMEM lanes), scale by 1/(s_a s_b), round to BF16, store.
//              Group mode and the 384-wide tile add warps 6-9, a second
//              warp per lane quarter taking half of the columns.
// Two TMEM accumulators let the epilogue of tile i overlap the main loop of
// tile i+1 (group mode keeps four; the 384-wide tile has room for one).
//
// PAIR = true: a cluster of two CTAs on two SMs computes a 256 x BN tile with
// tcgen05.mma.cta_group::2 (M = 256).  Each CTA loads its own 128 rows of A
// and one half (BN/2 rows) of B, so each SM fills and reads half the B bytes
// of a 1-CTA 128 x BN tile; both CTAs' copies complete on the leader's
// barrier, the leader's single thread issues the MMAs, and its commits
// arrive on the barriers of both CTAs.  Each CTA's TMEM holds its 128 rows.
//
// Every mbarrier wait is bounded; on time-out the CTA sets FP8Q_DEV_TIMEOUT,
// waits (bounded) for its copies and MMAs in flight, frees TMEM and exits.
//
// "FP8 Training & Inference", FP8 Training Recipe also defines the weight
// gradient (E4M3 activation x E5M2 gradient); "Paradigma Details FP8 and
// Optimizer Tricks Behind NanoGPT Records", second paragraph, places the
// quantize in the epilogue of the computation that produces its input.
#include "common.cuh"
#include "gemm_parts.cuh"
#include "quant_ops.cuh"
#include "history_ops.cuh"
#include "../../include/fp8q_testing.h"

#include <algorithm>
#include <atomic>
#include <cudaTypedefs.h>
#include <mutex>

namespace fp8q {

namespace {

constexpr int kThreadsGemm = 192;  // 6 warps
constexpr int kEpiWarps = 4;
constexpr int kWideEpiWarps = 8;  // two warps per TMEM lane quarter, each half the columns

// Fused quantize (FUSED != 0): extra warps per CTA (warps 6, 7, ...) turn the
// BF16 pre-activation into the GEMM's E4M3 A operand, a few rows at a time.
// They share the SM's issue slots with the producer, the MMA issuer and the
// epilogue, and the GEMM loses time wherever they run (at 131072 x 6400 ->
// 1600 the step takes 0.81 ms with the quantize loop removed, 1.01 ms with
// its arithmetic but no loads or stores, 1.22 ms whole).  Two layouts:
//   FUSED == 1  the quantize is the longer part of the step (few output
//               columns per byte of H): 24 warps, 8 loads in flight each;
//   FUSED == 2  the GEMM is the longer part: 12 warps, of which the three on
//               the MMA issuer's scheduler (warp id % 4 == 1) stay idle, and
//               16 loads in flight each -- the same bytes in flight from 9
//               warps, none competing with the MMA issuer (at 131072 x 6400 ->
//               1600 on 400-wide tiles, 1.19 -> 1.11 ms with 12 working warps x
//               12 loads; 9 x 16 a further 1 %; 7 x 20 and 6 x 24 slower; and
//               slower where the quantize is the longer part: 0.217 -> 0.235
//               ms at 65536 x 3072 -> 768) -- and units of 4 rows instead of
//               16, about one batch of loads per thread per unit at K = 6400,
//               so the unit's closing barrier paces the warps (1.10 -> 1.05 ms
//               there; 1, 2, 3, 5, 8, 12 rows: 2.10, 1.35, 1.07, 1.09, 1.08,
//               1.09 ms; 8 rows at 65536 x 3072 -> 768 in layout 1: 0.215 ->
//               0.238 ms).
template <int FUSED>
struct QuantLayout {
    static constexpr int WARPS = FUSED == 2 ? 12 : 24;  // warps the CTA launches for the quantize
    static constexpr int SKIP = FUSED == 2 ? 1 : -1;    // the scheduler left to the GEMM (warp id % 4)
    static constexpr int BATCH = FUSED == 2 ? 16 : 8;   // 16-byte loads in flight per thread
    static constexpr int UNIT = FUSED == 2 ? 4 : 16;     // rows per quantize unit in the full rounds
    static constexpr int FIRST_SKIP = 6 + ((SKIP - 6) % 4 + 4) % 4;  // lowest idle warp id
    static constexpr int active_warps() {
        int n = 0;
        for (int w = 6; w < 6 + WARPS; ++w) n += (SKIP < 0 || w % 4 != SKIP) ? 1 : 0;
        return n;
    }
    static constexpr int ACTIVE = active_warps();  // warps that quantize
    static constexpr int THREADS = ACTIVE * 32;
    // the thread's index among the quantize threads that work, or -1
    __device__ static int index(int warp, int lane) {
        if (SKIP >= 0 && warp % 4 == SKIP) return -1;
        const int idle_below = (SKIP >= 0 && warp > FIRST_SKIP) ? (warp - FIRST_SKIP + 3) / 4 : 0;
        return (warp - 6 - idle_below) * 32 + lane;
    }
};

// Epilogue warps: 8 where the epilogue is exposed -- group mode (a promotion
// per 128-long K slice; 12 and 16 on its 192- and 256-wide tiles, 64 columns
// per warp) and the 384-wide tile (one accumulator, so its drain is
// not hidden behind the next tile; 17.2 -> 16.4 us at 8192 x 3072 -> 768) --
// else 4 (8 would take a stage of the operand ring: 87.6 -> 92.6 us at 65536
// rows with 256-wide tiles) -- and the activation-quantize epilogue (EQ),
// whose per-element work is several times a plain epilogue's.
template <int BN, bool GROUP, int FUSED, bool EQ = false>
constexpr int epi_warps() {
    // group mode on 192 / 256-wide tiles: three / four promotion warps per lane quarter, 64 columns each
    return GROUP && BN == 256 ? 16 : GROUP && BN == 192 ? 12
         : !FUSED && (GROUP || EQ || (BN > 256 && BN != 400)) ? kWideEpiWarps : kEpiWarps;
}

template <int BN, bool GROUP, int FUSED, bool EQ = false>
constexpr int gemm_threads() {
    return kThreadsGemm + (FUSED ? QuantLayout<FUSED>::WARPS * 32 : 0) + (epi_warps<BN, GROUP, FUSED, EQ>() - kEpiWarps) * 32;
}

// Operands of the fused quantize.  ready[b] counts the rows of 128-row block b
// whose E4M3 codes are written; the GEMM's producer loads a tile's A rows once
// its block is complete.  Work is handed out by tickets: a CTA's quantize warps
// take the next row unit from q_next, and each epilogue warp the next weight
// unit from w_next, so only CTAs that are running claim work and no wait can
// depend on a CTA that has not been scheduled.  With w set, the epilogue warps
// first cast the weight W [K,N] into the GEMM's B operand W_q^T [N,K] (and
// W_q [K,N]); w_ready counts finished weight units and every producer waits
// for all w_units of them before its first B load.  The CTA that finishes
// last resets ready, w_ready, done and both ticket counters, so the workspace
// is zero again for the next launch, and then runs the delayed-scale history
// updates of X and W on the final amax values.
struct FusedArgs {
    const uint4* h;               // H [M,K] BF16, 8 elements per 16 bytes
    uint4* act_out;               // [M,K] BF16 activation copy, or nullptr
    uint2* x_q;                   // [M,K] E4M3: the GEMM's A operand
    float* amax_out;              // or nullptr; zero at the launch
    unsigned long long* sat_out;  // or nullptr; zero at the launch
    unsigned* ready;              // [nblocks], zero at the launch
    int act;                      // fp8q_act
    int64_t nblocks;              // ceil(M / 128)
    unsigned* done;               // CTAs finished; zero at the launch
    unsigned* q_next;             // next quantize ticket; zero at the launch
    unsigned* w_next;             // next weight-unit ticket; zero at the launch
    const uint4* w;               // W [K,N] BF16, or nullptr (W_q^T is then an input)
    const float* scale_w;         // W's scale (the GEMM's scale_b)
    uint8_t* wt_q;                // [N,K] E4M3, written when w is set
    uint8_t* w_q;                 // [K,N] E4M3 or nullptr
    float* amax_w;                // or nullptr; zero at the launch
    unsigned long long* sat_w;    // or nullptr: W's saturations; zero at the launch
    int64_t wn;                   // N
    unsigned* w_ready;            // weight units finished; zero at the launch
    unsigned w_units;             // weight units of the launch: (K / 8) * ceil(N / 256)
    HistoryArgs hx, hw;           // delayed-scale updates the last CTA runs (history == nullptr: none)
};

// The activation-quantize epilogue (EQ): the GEMM output is the pre-activation
// H of the next layer's quantize.  Per element: h = BF16(acc / (s_a s_b)),
// a = act(h), a_bf = BF16(a), q = E4M3(a_bf * s_h); amax = max |a_bf| and the
// saturation count, as in the standalone quantize.
struct EpiQuantArgs {
    const float* scale_h;           // E4M3 scale of the activation
    float* amax_out;                // or nullptr
    unsigned long long* sat_out;    // or nullptr
    int act;                        // fp8q_act
    int has_h, has_act;             // store H (through tmD) / the activation (through tmE1)
};

// Shared memory the operand ring and the epilogue staging share by default;
// the 256-wide group tile, whose staging is single-buffered, takes all but the
// barrier area, the alignment slack and 512 bytes for the kernel's static
// shared memory.
constexpr int kRingTotal = 220 * 1024;
constexpr int kGroupRingTotal = 232448 - 256 - 1024 - 512;

template <int BN, bool PAIR, int EPI = kEpiWarps, int ACC = (2 * BN <= 512 ? 2 : 1),
          int STAGE_PER_WARP = 2 * kEpiChunkBytes, int RING_TOTAL = kRingTotal>
struct Cfg {
    // A tile wider than 256 columns takes two MMAs per k-step (N <= 256 each)
    // into one accumulator; B then arrives as one box per MMA.  The 400-wide
    // pair tile (four tiles across N = 1600) splits unevenly: 192 + 208
    // columns, so each MMA's N is a multiple of 16 and each CTA's share of
    // its B rows (96, 104) a whole number of 8-row swizzle atoms.
    static constexpr int NSPLIT = BN > 256 ? 2 : 1;
    static constexpr int MMA_N = BN == 400 ? 192 : BN / NSPLIT;  // the first MMA's N
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // rows of B this CTA loads
    static constexpr int B_BOX = B_ROWS * MMA_N / BN;  // rows of B in the first TMA box
    // MMA j: its N, first accumulator / output column, this CTA's B rows
    // (one TMA box) and their offset in the stage's B area
    static constexpr int split_n(int j) { return j == 0 ? MMA_N : BN - MMA_N; }
    static constexpr int split_col(int j) { return j == 0 ? 0 : MMA_N; }
    static constexpr int split_rows(int j) { return j == 0 ? B_BOX : B_ROWS - B_BOX; }
    static constexpr int split_off(int j) { return j == 0 ? 0 : B_BOX * BK; }
    static constexpr int ACCS = ACC;                   // TMEM accumulators (512 columns)
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = B_ROWS * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TX_BYTES = STAGE_BYTES * (PAIR ? 2 : 1);  // bytes one stage's barrier awaits
    static constexpr int EPI_WARPS = EPI;
    static constexpr int EPI_STAGE = STAGE_PER_WARP;          // store staging per epilogue warp
    static constexpr int EPI_BYTES = EPI * STAGE_PER_WARP;
    static constexpr int RING_BUDGET = RING_TOTAL - EPI_BYTES;
    static constexpr int STAGES = RING_BUDGET / STAGE_BYTES < 8 ? RING_BUDGET / STAGE_BYTES : 8;
    static constexpr int TMEM_COLS = (ACCS * BN <= 256) ? 256 : 512;  // power of 2
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES + 1024;  // + alignment slack
    static constexpr int MMA_M = PAIR ? 2 * BM : BM;
    static constexpr int TILE_M = MMA_M;                              // output rows per tile
    static constexpr int EPI_ARRIVALS = EPI * (PAIR ? 2 : 1);         // per accumulator drain
    static_assert((BN % 32 == 0 && BN >= 64 && BN <= 384) || (BN == 400 && PAIR),
                  "BN: multiple of 32 in [64, 384], or the 400-wide pair tile");
    static_assert(split_n(0) % 16 == 0 && split_n(0) <= 256 && split_n(NSPLIT - 1) % 16 == 0 &&
                      split_n(NSPLIT - 1) <= 256, "MMA N: multiple of 16, at most 256");
    static_assert(split_rows(0) % 8 == 0 && split_rows(NSPLIT - 1) % 8 == 0, "B boxes: whole 8-row swizzle atoms");
    static_assert(B_BYTES % 1024 == 0, "stage tiles stay 1024-byte aligned");
    static_assert(STAGES >= 2, "at least a double-buffered ring");
    static_assert(ACCS >= 1 && ACCS * BN <= 512, "accumulators fit TMEM's 512 columns");
    static_assert((2 * STAGES + 2 * ACCS + 1) * 8 + 16 <= BAR_BYTES, "barrier area");
    static_assert(SMEM_BYTES <= 232448, "dynamic shared memory per CTA");
};

// Group mode promotes every 128-long K slice, so it keeps as many
// accumulators as TMEM holds: the MMAs run up to three slices ahead (one at
// 192 and 256 wide).  Its stores come once per tile; on the 256-wide tile
// each warp stages them in one 2 KB block and the operand ring takes the
// rest, 4 stages instead of 3 (85.5 against 93.7 us at 16384 x 4096 -> 1024;
// at 192 wide a fifth stage did not pay for the single staging block).
// EQ (the activation-quantize epilogue) stages two outputs per warp: the
// activation (BF16) and the E4M3 codes (64-column boxes), each double-buffered;
// H, when asked for, goes through the activation's buffer first.
// DACT (the activation backward in the dgrad epilogue) adds a load buffer for
// every 32-column chunk of H in the tile (BN / 16 KB) and one mbarrier: 5 KB +
// BN / 16 KB per warp, keeping each warp's buffers 1024-byte aligned.
template <int BN, bool GROUP, bool PAIR, int FUSED, bool EQ = false, int DACT = 0>
using KernelCfg = Cfg<BN, PAIR, epi_warps<BN, GROUP, FUSED, EQ>(), GROUP ? 512 / BN : (2 * BN <= 512 ? 2 : 1),
                      EQ ? 4 * kEpiChunkBytes : DACT ? (5 + BN / 16) * 1024 : GROUP && BN == 256 ? kEpiChunkBytes : 2 * kEpiChunkBytes,
                      (GROUP && BN == 256) || BN == 400 ? kGroupRingTotal : kRingTotal>;

// Bounded wait until a GPU-scope counter reaches `need` (acquire).
__device__ __forceinline__ bool wait_ready(const unsigned* counter, unsigned need, volatile int* abort_flag,
                                           int* status) {
    if (ld_acquire(counter) >= need) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(64);
        if (ld_acquire(counter) >= need) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kTimeoutNs) {
            *abort_flag = 1;
            if (status) atomicOr(status, FP8Q_DEV_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ uint4 act8_any(int act, uint4 x, uint32_t& amax2) {
    if (act == FP8Q_ACT_RELU2) return act8<FP8Q_ACT_RELU2>(x, amax2);
    if (act == FP8Q_ACT_RELU) return act8<FP8Q_ACT_RELU>(x, amax2);
    return act8<FP8Q_ACT_IDENTITY>(x, amax2);
}

// 16 accumulator columns of one row (this lane's) to D [M,N] BF16 with two
// 16-byte stores.  c0 and N are multiples of 16, so the columns lie wholly
// inside D or wholly past it, and the stores are aligned.
__device__ __forceinline__ void epi_store_tail16(uint16_t* d, uint32_t taddr, float inv, int64_t row, int64_t c0,
                                                 int64_t M, int64_t N) {
    uint32_t r[16];
    tmem_ld_x16_sync(taddr, r);
    if (row >= M || c0 >= N) return;
    uint32_t p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) p[j] = cvt_bf16x2(__uint_as_float(r[2 * j]) * inv, __uint_as_float(r[2 * j + 1]) * inv);
    uint4* dst = reinterpret_cast<uint4*>(d + row * N + c0);
    dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
    dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
}

// One unit of the fused quantize: rows [r0, r1) by all quantize threads of
// the CTA, then one thread publishes the rows with a release add to the count
// of each 128-row block they touch.  The quantize warps share their SM with
// the GEMM's warps, whose issue slots they take, so the per-element work is
// kept short: ReLU^2 as two packed BF16 instructions per pair, the scale as
// one packed float32 multiply per pair, and the saturation count taken once
// per batch of loads -- exactly, through sat_count8, only when the
// batch's largest magnitude can saturate.
template <int FUSED, int ACT>
__device__ __forceinline__ void fused_rows_body(const FusedArgs& fz, float s, int64_t r0, int64_t r1, int64_t K,
                                                int qt, uint32_t& amax2, uint32_t& nsat) {
    using L = QuantLayout<FUSED>;
    const int64_t c_end = r1 * (K / 8);
    for (int64_t c0 = r0 * (K / 8) + qt; c0 < c_end; c0 += int64_t(L::THREADS) * L::BATCH) {
        uint4 x[L::BATCH];
#pragma unroll
        for (int j = 0; j < L::BATCH; ++j) {
            const int64_t c = c0 + int64_t(j) * L::THREADS;
            x[j] = c < c_end ? ld_stream_v4(fz.h + c) : make_uint4(0, 0, 0, 0);
        }
        uint32_t bm2 = 0;  // this batch's magnitudes (act(0) = 0 for the padding)
#pragma unroll
        for (int j = 0; j < L::BATCH; ++j) x[j] = act8<ACT, true>(x[j], bm2);
        if (may_saturate<FP8Q_E4M3>(bm2, s)) {
#pragma unroll
            for (int j = 0; j < L::BATCH; ++j)
                if (c0 + int64_t(j) * L::THREADS < c_end) nsat += sat_count8<FP8Q_E4M3>(x[j], s);
        }
        amax2 = __vmaxu2(amax2, bm2);
#pragma unroll
        for (int j = 0; j < L::BATCH; ++j) {
            const int64_t c = c0 + int64_t(j) * L::THREADS;
            if (c < c_end) {
                if (fz.act_out) st_stream_v4(fz.act_out + c, x[j]);
                st_v2(fz.x_q + c, cast8_codes<FP8Q_E4M3>(x[j], s));
            }
        }
    }
}

template <int FUSED>
__device__ __forceinline__ void fused_quantize_rows(const FusedArgs& fz, float s, int64_t r0, int64_t r1,
                                                    int64_t K, int qt, uint32_t& amax2, uint32_t& nsat) {
    using L = QuantLayout<FUSED>;
    if (fz.act == FP8Q_ACT_RELU2) fused_rows_body<FUSED, FP8Q_ACT_RELU2>(fz, s, r0, r1, K, qt, amax2, nsat);
    else if (fz.act == FP8Q_ACT_RELU) fused_rows_body<FUSED, FP8Q_ACT_RELU>(fz, s, r0, r1, K, qt, amax2, nsat);
    else fused_rows_body<FUSED, FP8Q_ACT_IDENTITY>(fz, s, r0, r1, K, qt, amax2, nsat);
    // the unit's E4M3 codes are written by every quantize thread: order them
    // before the counts, which the producer reads before its TMA loads
    fence_proxy_async_global();
    named_barrier(1, L::THREADS);
    if (qt == 0) {
        for (int64_t b = r0 / BM; b * BM < r1; ++b) {
            const int64_t lo = b * BM > r0 ? b * BM : r0;
            const int64_t hi = (b + 1) * BM < r1 ? (b + 1) * BM : r1;
            red_release_add(fz.ready + b, static_cast<unsigned>(hi - lo));
        }
    }
}

// The last CTA's history update (once per launch: kept out of line).
__device__ __noinline__ void history_update_once(const HistoryArgs& a, const float* amax_new) {
    history_update_warp(a, amax_new);
}

// The weight cast of the fused kernel ("FP8 training: what it is and how it
// works", Step 4: the weight's 8-bit copy is cast from the master copy each
// step): W [K,N] BF16 -> W_q^T [N,K] (and W_q [K,N]) E4M3 with the scale s_w.
// The epilogue warps do it at the start of the kernel, while they would
// otherwise wait for their first accumulator.  A unit is 8 rows of W x 256
// columns, one warp, each lane 8 columns: the lane loads its 8 x 8 block row
// by row, casts it, and writes the block's transpose as 8 eight-byte pieces
// (8 consecutive k of one output row n).  A warp takes units by ticket
// (w_next), asking for the next one before it casts the current one, so the
// atomic's latency hides behind the loads.  Every epilogue warp then adds
// the number of units it cast to w_ready with release semantics, once (the
// producers wait for the whole weight, so one drain of the scattered stores
// per warp is enough).  The warp's max |W| goes to amax_w and its count of
// |v| > 448 to sat_w, one atomic each.
__device__ __forceinline__ void fused_cast_w(const FusedArgs& fz, int64_t K, int lane) {
    const int64_t N = fz.wn;
    const int64_t nbn = (N + 255) / 256;
    const unsigned units = fz.w_units;
    const float s = __ldg(fz.scale_w);
    uint32_t amax2w = 0, nsat = 0;
    unsigned cast = 0;
    unsigned u = 0;
    if (lane == 0) u = atomicAdd(fz.w_next, 1u);
    u = __shfl_sync(0xFFFFFFFFu, u, 0);
    while (u < units) {
        unsigned nxt = 0;
        if (lane == 0) nxt = atomicAdd(fz.w_next, 1u);
        const int64_t k0 = (int64_t(u) / nbn) * 8;
        const int64_t n = (int64_t(u) % nbn) * 256 + lane * 8;
        if (n < N) {
            uint4 x[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) x[r] = ld_stream_v4(fz.w + ((k0 + r) * N + n) / 8);
            uint2 q[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const uint4 a = act8<FP8Q_ACT_IDENTITY>(x[r], amax2w);
                q[r] = cast8<FP8Q_E4M3>(a, s, nsat);
                if (fz.w_q) st_v2(reinterpret_cast<uint2*>(fz.w_q + (k0 + r) * N + n), q[r]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t lo = 0, hi = 0;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    lo |= (((j < 4 ? q[r].x : q[r].y) >> (8 * (j & 3))) & 0xFFu) << (8 * r);
                    hi |= (((j < 4 ? q[r + 4].x : q[r + 4].y) >> (8 * (j & 3))) & 0xFFu) << (8 * r);
                }
                st_v2(reinterpret_cast<uint2*>(fz.wt_q + (n + j) * K + k0), make_uint2(lo, hi));
            }
        }
        ++cast;
        u = __shfl_sync(0xFFFFFFFFu, nxt, 0);
    }
    // the warp's codes, written by all lanes, are ordered before the count,
    // which every producer reads before its TMA loads of W_q^T
    fence_proxy_async_global();
    __syncwarp();
    if (lane == 0 && cast) red_release_add(fz.w_ready, cast);
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max16x2(amax2w));
    const uint32_t c = __reduce_add_sync(0xFFFFFFFFu, nsat);
    if (lane == 0 && fz.amax_w && m) atomicMax(reinterpret_cast<unsigned int*>(fz.amax_w), m << 16);
    if (lane == 0 && fz.sat_w && c) atomicAdd(fz.sat_w, static_cast<unsigned long long>(c));
}

// The quantize warps of the fused kernel.  Row units are handed out by
// ticket (q_next), in row order, so rows finish in order across the GPU and
// only running CTAs take work.  Tickets 0 .. full - 1 are units of L::UNIT
// rows; the rows after them (gridDim.x x UNIT rows or more when M allows) are
// split into gridDim.x equal units of at most UNIT + 1 rows, so the last
// units end together instead of one SM carrying a whole extra unit at the end.  One thread asks
// for the next ticket before the CTA quantizes the current unit; the unit's
// closing barrier publishes it to the other quantize threads.
template <int FUSED>
__device__ __forceinline__ void fused_quantize(const FusedArgs& fz, const float* scale, int64_t M, int64_t K) {
    using L = QuantLayout<FUSED>;
    __shared__ unsigned s_ticket[2];
    const int qt = L::index(threadIdx.x >> 5, threadIdx.x & 31);
    if (qt < 0) return;  // a warp the layout leaves idle
    const float s = __ldg(scale);
    uint32_t amax2 = 0, nsat = 0;
    const int64_t G = gridDim.x;
    const int64_t full = M / L::UNIT > G ? M / L::UNIT - G : 0;
    const int64_t share = (M - full * L::UNIT + G - 1) / G;
    const int64_t nunits = full + G;
    if (qt == 0) s_ticket[0] = atomicAdd(fz.q_next, 1u);
    named_barrier(1, L::THREADS);
    int par = 0;
    int64_t t = s_ticket[0];
    while (t < nunits) {
        if (qt == 0) s_ticket[par ^ 1] = atomicAdd(fz.q_next, 1u);
        int64_t r0, r1;
        if (t < full) {
            r0 = t * L::UNIT;
            r1 = r0 + L::UNIT;
        } else {
            r0 = full * L::UNIT + (t - full) * share;
            r1 = r0 + share < M ? r0 + share : M;
        }
        // fused_quantize_rows ends with a barrier of all quantize threads, after
        // which the next ticket is visible to all of them
        if (r0 < r1) fused_quantize_rows<FUSED>(fz, s, r0, r1, K, qt, amax2, nsat);
        else named_barrier(1, L::THREADS);
        par ^= 1;
        t = s_ticket[par];
    }
    __shared__ uint32_t s_amax[L::ACTIVE], s_sat[L::ACTIVE];
    uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max16x2(amax2));
    uint32_t c = __reduce_add_sync(0xFFFFFFFFu, nsat);
    if ((qt & 31) == 0) { s_amax[qt >> 5] = m; s_sat[qt >> 5] = c; }
    named_barrier(1, L::THREADS);
    if (qt == 0) {
        for (int w = 1; w < L::ACTIVE; ++w) { m = max(m, s_amax[w]); c += s_sat[w]; }
        if (fz.amax_out && m) atomicMax(reinterpret_cast<unsigned int*>(fz.amax_out), m << 16);
        if (fz.sat_out && c) atomicAdd(fz.sat_out, static_cast<unsigned long long>(c));
    }
}

// The activation-quantize epilogue (EQ) of one warp's 32 rows: the 64-column
// chunk pairs pair0, pair0 + pair_step, ... of the BN-wide accumulator (TMEM
// address taddr).  Per 32-column chunk: H = BF16(acc * inv), the activation
// (BF16) through a double-buffered 2 KB staging block (the 64-byte swizzle of
// epi_store_chunk) to one TMA store; the E4M3 codes of a pair fill one
// 64-column box (32 bytes of each 64-byte row per chunk), stored after the
// pair's second chunk.  Each chunk's stores are one bulk group, and a buffer
// is rewritten only after the group that last read it finished: activation
// buffers alternate with nchunk, E4M3 boxes with nq (E4M3 stores so far);
// between a box's store and its reuse there is always the group of the other
// box, so the wait for "at most one group pending" covers both.  H, when asked
// for, is staged in the activation buffer and stored (and drained) first.
// Boxes wholly outside D are skipped and counted nowhere.  amax2 / nsat
// collect this thread's maximum and saturations.
template <int BN>
__device__ __forceinline__ void epi_quant_tile(const CUtensorMap* tmH, const CUtensorMap* tmAct,
                                               const CUtensorMap* tmQ, const EpiQuantArgs& eq, uint8_t* warp_stage,
                                               int& nchunk, int& nq, int lane, uint32_t taddr, float inv, float s_h,
                                               int pair0, int pair_step, int64_t col_base, int64_t row0, int64_t M,
                                               int64_t N, uint32_t& amax2, uint32_t& nsat) {
    static_assert(BN % 64 == 0, "E4M3 boxes are 64 columns: whole chunk pairs");
    uint8_t* abuf = warp_stage;
    uint8_t* qbuf = warp_stage + 2 * kEpiChunkBytes;
    const int sw = (lane >> 1) & 3;
    if (row0 >= M) return;  // the warp's rows lie outside D
#pragma unroll 1
    for (int p = pair0; p < BN / 64; p += pair_step) {
        if (col_base + p * 64 >= N) break;  // this and the later pairs lie outside D
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            const int64_t col0 = col_base + p * 64 + half * 32;
            if (col0 >= N) break;
            uint32_t r[32];
            tmem_ld_x32_sync(taddr + static_cast<uint32_t>(p * 64 + half * 32), r);
            uint32_t hb[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                hb[j] = cvt_bf16x2(__uint_as_float(r[2 * j]) * inv, __uint_as_float(r[2 * j + 1]) * inv);
            uint4 a4[4];
            uint2 q2[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                a4[g] = act8_any(eq.act, make_uint4(hb[4 * g], hb[4 * g + 1], hb[4 * g + 2], hb[4 * g + 3]), amax2);
                q2[g] = cast8<FP8Q_E4M3>(a4[g], s_h, nsat);
            }
            if (nchunk >= 2) {
                if (lane == 0) bulk_wait_group_read<1>();
                __syncwarp();
            }
            uint8_t* ab_s = abuf + (nchunk & 1) * kEpiChunkBytes;
            uint8_t* qb_s = qbuf + (nq & 1) * kEpiChunkBytes;
            if (eq.has_h) {
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    *reinterpret_cast<uint4*>(ab_s + lane * 64 + ((g ^ sw) << 4)) =
                        make_uint4(hb[4 * g], hb[4 * g + 1], hb[4 * g + 2], hb[4 * g + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(tmH, smem_u32(ab_s), static_cast<int32_t>(col0), static_cast<int32_t>(row0));
                    bulk_commit_group();
                    bulk_wait_group_read<0>();  // the buffer is free for the activation
                }
                __syncwarp();
            }
            if (eq.has_act) {
#pragma unroll
                for (int g = 0; g < 4; ++g) *reinterpret_cast<uint4*>(ab_s + lane * 64 + ((g ^ sw) << 4)) = a4[g];
            }
            *reinterpret_cast<uint4*>(qb_s + lane * 64 + (((2 * half) ^ sw) << 4)) =
                make_uint4(q2[0].x, q2[0].y, q2[1].x, q2[1].y);
            *reinterpret_cast<uint4*>(qb_s + lane * 64 + (((2 * half + 1) ^ sw) << 4)) =
                make_uint4(q2[2].x, q2[2].y, q2[3].x, q2[3].y);
            fence_proxy_async_smem();
            __syncwarp();
            const bool box_done = half == 1 || col0 + 32 >= N;  // the box's last chunk inside D
            if (lane == 0) {
                if (eq.has_act)
                    tma_store_2d(tmAct, smem_u32(ab_s), static_cast<int32_t>(col0), static_cast<int32_t>(row0));
                if (box_done)
                    tma_store_2d(tmQ, smem_u32(qb_s), static_cast<int32_t>(col0 - half * 32),
                                 static_cast<int32_t>(row0));
                bulk_commit_group();
            }
            if (box_done) ++nq;
            ++nchunk;
        }
    }
}

// The activation backward in the dgrad epilogue (DACT): for the chunks c0,
// c0 + step, ... of one warp's 32 rows of the accumulator,
//   dh = BF16( acc * inv * act'(h) ),  act'(h) = 2 max(h, 0) (ReLU^2),
//   (h > 0) (ReLU) or 1 (identity), h the BF16 pre-activation at the same spot.
// issue_h_loads asks TMA for all of the warp's H boxes of a tile (32 rows x 32
// columns each, in the 64-byte swizzle of the store staging, so lane r reads
// row r) on one mbarrier, before the warp waits for the accumulator: the loads
// land while the MMAs of the tile run.  ldn counts the warp's tiles of loads
// (the barrier's phase is ldn & 1); epi_dact_tile waits for them once.
// Returns false when a bounded wait gave up.
__device__ __forceinline__ void issue_h_loads(const CUtensorMap* tmH, uint8_t* lbuf, uint64_t* lbar, uint32_t& ldn,
                                              int lane, int nck, int c0, int step, int64_t col_base, int64_t row0,
                                              uint32_t box_bytes) {
    fence_proxy_async_smem();  // the buffers' last reads (the previous tile) come first
    __syncwarp();
    if (lane == 0) {
        const uint32_t bar = smem_u32(lbar);
        int n = 0;
        for (int c = c0; c < nck; c += step) ++n;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * box_bytes);
        for (int c = c0, i = 0; c < nck; c += step, ++i)
            tma_load_2d(smem_u32(lbuf + i * kEpiChunkBytes), tmH, bar, static_cast<int32_t>(col_base + c * 32),
                        static_cast<int32_t>(row0));
    }
    ++ldn;
}

// HFMT 1: H is BF16 (32 x 32 boxes, 64-byte swizzle); HFMT 2: H is the
// pre-activation's E4M3 cache (32 x 32-byte boxes, unswizzled: lane r's row
// is 32 contiguous codes), decoded exactly and multiplied by inv_h = 1 / s_h.
template <int BN, int HFMT>
__device__ __forceinline__ bool epi_dact_tile(const CUtensorMap* tmD, int act, uint8_t* warp_stage,
                                              const uint8_t* lbuf, uint64_t* lbar, int& nchunk, uint32_t& ldw,
                                              int lane, uint32_t taddr, float inv, float inv_h, int c0, int step,
                                              int64_t col_base, int64_t row0, int64_t M, int64_t N,
                                              volatile int* abort_flag, int* status) {
    const int sw = (lane >> 1) & 3;
    const bool ok = __all_sync(0xFFFFFFFFu, wait_phase(lbar, ldw & 1, abort_flag, status));
    if (!ok) return false;
    ++ldw;
#pragma unroll 1
    for (int c = c0, i = 0; c < BN / 32; c += step, ++i) {
        uint32_t r[32];
        tmem_ld_x32_sync(taddr + static_cast<uint32_t>(c * 32), r);
        float hv[32];
        if constexpr (HFMT == 2) {
            const uint8_t* hrow = lbuf + i * kEpiChunkBytes + lane * 32;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const uint4 q = *reinterpret_cast<const uint4*>(hrow + 16 * g);
                const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(qw[k] & 0xFFFFu));
                    const float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(qw[k] >> 16));
                    const int j = g * 16 + k * 4;
                    hv[j] = lo.x * inv_h;
                    hv[j + 1] = lo.y * inv_h;
                    hv[j + 2] = hi.x * inv_h;
                    hv[j + 3] = hi.y * inv_h;
                }
            }
        } else {
            const uint8_t* hrow = lbuf + i * kEpiChunkBytes + lane * 64;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint4 h = *reinterpret_cast<const uint4*>(hrow + ((g ^ sw) << 4));
                const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    hv[g * 8 + k * 2] = bf16lo_to_f32(hw[k]);
                    hv[g * 8 + k * 2 + 1] = bf16hi_to_f32(hw[k]);
                }
            }
        }
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float d = hv[j] > 0.0f ? (act == FP8Q_ACT_RELU2 ? 2.0f * hv[j] : 1.0f) : 0.0f;
            const float f = act == FP8Q_ACT_IDENTITY ? 1.0f : d;
            v[j] = __uint_as_float(r[j]) * inv * f;
        }
        epi_store_chunk(tmD, warp_stage, nchunk, lane, v, static_cast<int32_t>(col_base + c * 32),
                        static_cast<int32_t>(row0), M, N);
    }
    return true;
}

// GROUP = false: per-tensor scales, one accumulation per tile.
// GROUP = true : 1-CTA, BN = 128; each 128-long K slice is accumulated into a
//                fresh TMEM buffer and promoted into FP32 registers with its
//                own 1/(s_a[row, kb] * s_b[kb, n_blk]) by 8 epilogue warps
//                (two per TMEM lane quarter, 64 columns each), so the
//                promotion keeps pace with the MMAs.
// PAIR = true  : 2-SM tiles (see the file header); per-tensor scales only.
// FUSED = true : the fused quantize + GEMM (per-tensor scales): the extra
//                quantize warps produce A = X_q from H while the GEMM consumes
//                finished 128-row blocks.
template <int BN, bool GROUP, bool PAIR, int FUSED, bool EQ, int DACT>
__global__ void __launch_bounds__(gemm_threads<BN, GROUP, FUSED, EQ>(), 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmD,
                const float* __restrict__ scale_a, const float* __restrict__ scale_b,
                int64_t M, int64_t N, int64_t K, uint32_t idesc, int* __restrict__ status,
                int hold_loads, const FusedArgs fz, const __grid_constant__ CUtensorMap tmE1,
                const __grid_constant__ CUtensorMap tmE2, const EpiQuantArgs eq, uint16_t* __restrict__ d_raw) {
    using C = KernelCfg<BN, GROUP, PAIR, FUSED, EQ, DACT>;
    static_assert(!DACT || (!GROUP && !FUSED && !EQ), "the activation backward runs in the per-tensor dgrad epilogue");
    static_assert(!EQ || (!GROUP && !FUSED && BN % 64 == 0 && BN <= 256),
                  "the activation-quantize epilogue: per-tensor tiles of whole 64-column pairs, two accumulators");
    static_assert(!GROUP || ((BN == 128 || BN == 192 || BN == 256) && !PAIR), "group mode uses 1-CTA tiles, 128-256 wide");
    static_assert(!(GROUP && FUSED), "the fused quantize feeds the per-tensor GEMM");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* epi_stage = smem + C::STAGES * C::STAGE_BYTES;  // 1024-aligned: STAGE_BYTES is
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
            mbar_init(smem_u32(&full[s]), 1);
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
        if constexpr (C::MMA_N * C::NSPLIT != BN) tma_prefetch_desc(&tmB2);
        tma_prefetch_desc(&tmD);
        if constexpr (EQ) {
            tma_prefetch_desc(&tmE1);
            tma_prefetch_desc(&tmE2);
        }
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
    // the prologue above overlaps the previous kernel; operands, scales and
    // D are touched only after it has finished
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            if constexpr (FUSED) {
                // the weight cast of this launch is complete before any B load
                if (fz.w && !hold_loads) {
                    ok = wait_ready(fz.w_ready, fz.w_units, abort_flag, status);
                    fence_proxy_async_global();
                }
            }
            // hold_loads (test hook): issue nothing, so the MMA issuer's first wait runs out
            for (int64_t tile = first_tile; tile < num_tiles && ok && !hold_loads; tile += tile_stride) {
                const int32_t m0 = static_cast<int32_t>((tile / num_n) * C::TILE_M + rank * BM);
                const int32_t n0 = static_cast<int32_t>((tile % num_n) * BN);
                if constexpr (FUSED) {
                    // this tile's A rows exist once every unit of their block is quantized
                    if (m0 < M) {
                        const int64_t blk = m0 / BM;
                        const int64_t rows = M - blk * BM < BM ? M - blk * BM : BM;
                        const unsigned need = static_cast<unsigned>(rows);
                        if (!wait_ready(fz.ready + blk, need, abort_flag, status)) { ok = false; break; }
                        fence_proxy_async_global();
                    }
                }
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!wait_phase(&empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
                    uint8_t* sa = smem + stage * C::STAGE_BYTES;
                    if constexpr (PAIR) {
                        // both CTAs' copies complete on the leader's barrier
                        const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
                        if (leader) mbar_arrive_expect_tx(smem_u32(&full[stage]), C::TX_BYTES);
                        tma_load_2d_pair(smem_u32(sa), &tmA, fb, kb * BK, m0);
#pragma unroll
                        for (int j = 0; j < C::NSPLIT; ++j)
                            tma_load_2d_pair(smem_u32(sa + C::A_BYTES + C::split_off(j)),
                                             C::MMA_N * C::NSPLIT != BN && j ? &tmB2 : &tmB, fb, kb * BK,
                                             n0 + C::split_col(j) + static_cast<int32_t>(rank) * C::split_rows(j));
                    } else {
                        const uint32_t fb = smem_u32(&full[stage]);
                        mbar_arrive_expect_tx(fb, C::TX_BYTES);
                        tma_load_2d(smem_u32(sa), &tmA, fb, kb * BK, m0);
#pragma unroll
                        for (int j = 0; j < C::NSPLIT; ++j)
                            tma_load_2d(smem_u32(sa + C::A_BYTES + C::split_off(j)), &tmB, fb, kb * BK,
                                        n0 + C::split_col(j));
                    }
                    ++issued;
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // No copy may still be landing in shared memory when the CTA exits:
            // wait for the last (up to STAGES) loads.  In a pair the leader's
            // barriers also count the peer's bytes.
            if (!PAIR || leader) {
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
        // -------------------------------------------------------- MMA issuer
        if (lane == 0 && (!PAIR || leader)) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t tile = first_tile; tile < num_tiles && ok; tile += tile_stride) {
                if (!GROUP) {
                    if (!wait_phase(&tempty[acc], acc_phase ^ 1u, abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                }
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (GROUP) {
                        if (!wait_phase(&tempty[acc], acc_phase ^ 1u, abort_flag, status)) { ok = false; break; }
                        tc_fence_after();
                    }
                    if (!wait_phase(&full[stage], phase, abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                    const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        const uint32_t accumulate = GROUP ? (k > 0) : (kb > 0 || k > 0);
                        const uint64_t ad = smem_desc_k_sw128(a_addr + k * UMMA_K);
#pragma unroll
                        for (int j = 0; j < C::NSPLIT; ++j) {
                            const uint64_t bd = smem_desc_k_sw128(b_addr + C::split_off(j) + k * UMMA_K);
                            const uint32_t dj = d_tmem + static_cast<uint32_t>(C::split_col(j));
                            const uint32_t idj = j == 0 ? idesc : idesc_with_n(idesc, C::split_n(j));
                            if constexpr (PAIR) mma_f8f6f4_pair(dj, ad, bd, idj, accumulate);
                            else mma_f8f6f4(dj, ad, bd, idj, accumulate);
                        }
                    }
                    // the stage is free (in both CTAs of a pair) once these MMAs finish
                    if constexpr (PAIR) mma_commit_pair_mc(smem_u32(&empty[stage]), 0x3);
                    else mma_commit(smem_u32(&empty[stage]));
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                    if (GROUP) {
                        if constexpr (PAIR) mma_commit_pair_mc(smem_u32(&tfull[acc]), 0x3);
                        else mma_commit(smem_u32(&tfull[acc]));
                        next_acc<C::ACCS>(acc, acc_phase);
                    }
                }
                if (!GROUP && ok) {
                    // accumulator ready for the epilogue(s)
                    if constexpr (PAIR) mma_commit_pair_mc(smem_u32(&tfull[acc]), 0x3);
                    else mma_commit(smem_u32(&tfull[acc]));
                    next_acc<C::ACCS>(acc, acc_phase);
                }
            }
            // all MMAs of this thread complete before TMEM is released
            if constexpr (PAIR) mma_commit_pair(smem_u32(drain));
            else mma_commit(smem_u32(drain));
            wait_phase_drain(drain, 0);
        }
    } else if (FUSED && warp >= 2 + kEpiWarps) {
        // ---------------------------------------------------- fused quantize
        if constexpr (FUSED) fused_quantize<FUSED>(fz, scale_a, M, K);
    } else {
        // ---------------------------------------------------------- epilogue
        if constexpr (FUSED) {
            if (fz.w) fused_cast_w(fz, K, lane);
        } else {
            // fp8_gemm_fwd_update: the step's delayed-scale updates, by one warp of
            // the first CTA while its first accumulator fills (the amax values
            // are final: the casts completed before pdl_wait returned).  They
            // write the other scale slot, never the scales this GEMM reads.
            if (blockIdx.x == 0 && warp == 2) {
                if (fz.hx.history) history_update_once(fz.hx, fz.amax_out);
                if (fz.hw.history) history_update_once(fz.hw, fz.amax_w);
            }
        }
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        // drained accumulators are reported to the leader's barrier
        const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(&tempty[0]), 0) : smem_u32(&tempty[0]);
        uint8_t* warp_stage = epi_stage + (warp - 2) * C::EPI_STAGE;
        int nq = 0;                        // EQ: E4M3 boxes stored by this warp
        uint32_t eq_amax2 = 0, eq_nsat = 0;  // EQ: this thread's maximum and saturations
        const float s_h = EQ ? __ldg(eq.scale_h) : 1.0f;
        // DACT: this warp's H load buffers (after its store staging) and their barrier
        uint8_t* lbuf = warp_stage + 2 * kEpiChunkBytes;
        uint64_t* lbar = reinterpret_cast<uint64_t*>(warp_stage + 2 * kEpiChunkBytes + (BN / 32) * kEpiChunkBytes);
        uint32_t ldn = 0, ldw = 0;  // DACT: tiles of H loads issued / consumed by this warp
        if constexpr (DACT) {
            if (lane == 0) {
                mbar_init(smem_u32(lbar), 1);
                fence_mbar_init();
            }
            __syncwarp();
        }
        int nchunk = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        float inv = 1.0f;
        if (!GROUP) inv = 1.0f / (__ldg(scale_a) * __ldg(scale_b));
        const float inv_h = DACT == 2 ? 1.0f / __ldg(eq.scale_h) : 1.0f;  // the E4M3 cache's dequantisation
        const int64_t kg = K / BK;                    // group mode: K % 128 == 0
        const int64_t ng = (N + 127) / 128;
        for (int64_t tile = first_tile; tile < num_tiles && ok; tile += tile_stride) {
            const int64_t m_blk = tile / num_n, n_blk = tile % num_n;
            const int64_t row0 = m_blk * C::TILE_M + rank * BM + q * 32;  // this warp's first row
            const int64_t row = row0 + lane;
            if constexpr (!GROUP) {
                // DACT: the first chunk's H is on its way while the accumulator fills
                if constexpr (DACT)
                    issue_h_loads(&tmE1, lbuf, lbar, ldn, lane, BN / 32, (warp - 2) / 4, C::EPI_WARPS / 4,
                                  n_blk * BN, row0, DACT == 2 ? 32 * 32 : kEpiChunkBytes);
                ok = wait_phase(&tfull[acc], acc_phase, abort_flag, status);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                tc_fence_after();
                if constexpr (EQ) {
                    epi_quant_tile<BN>(&tmD, &tmE1, &tmE2, eq, warp_stage, nchunk, nq, lane,
                                       tmem_base + lane_base + static_cast<uint32_t>(acc * BN), inv, s_h,
                                       (warp - 2) / 4, C::EPI_WARPS / 4, n_blk * BN, row0, M, N, eq_amax2, eq_nsat);
                }
                if constexpr (DACT) {
                    ok = epi_dact_tile<BN, DACT>(&tmD, eq.act, warp_stage, lbuf, lbar, nchunk, ldw, lane,
                                           tmem_base + lane_base + static_cast<uint32_t>(acc * BN), inv, inv_h,
                                           (warp - 2) / 4, C::EPI_WARPS / 4, n_blk * BN, row0, M, N, abort_flag,
                                           status);
                }
                // with 8 epilogue warps the two warps of a lane quarter take alternate chunks
#pragma unroll 1
                for (int c = (warp - 2) / 4; c < ((EQ || DACT) ? 0 : BN / 32); c += C::EPI_WARPS / 4) {
                    uint32_t r[32];
                    tmem_ld_x32_sync(tmem_base + lane_base + static_cast<uint32_t>(acc * BN + c * 32), r);
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * inv;
                    epi_store_chunk(&tmD, warp_stage, nchunk, lane, v, static_cast<int32_t>(n_blk * BN + c * 32),
                                    static_cast<int32_t>(row0), M, N);
                }
                if constexpr (BN % 32 == 16) {
                    // the last 16 columns (the 400-wide tile): no 32-column box fits
                    // them without covering the next tile's columns, so each lane
                    // stores its row's 32 bytes directly
                    if ((warp - 2) / 4 == (BN / 32) % (C::EPI_WARPS / 4))
                        epi_store_tail16(d_raw, tmem_base + lane_base + static_cast<uint32_t>(acc * BN + BN - 16), inv,
                                         row, n_blk * BN + BN - 16, M, N);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR) mbar_arrive_cluster(tempty0 + 8u * acc);
                    else mbar_arrive(tempty0 + 8u * acc);
                }
                next_acc<C::ACCS>(acc, acc_phase);
            } else {
                // warp (warp - 2) / 4 of its lane quarter promotes columns cbase..cbase + GC - 1,
                // all in one 128-column block of B's scales
                constexpr int GC = BN / (C::EPI_WARPS / 4);
                // x32 TMEM loads per wait (1 or 2); with 12 or 16 warps (a 128- or 96-register
                // cap) x16 loads, one per wait, so the 64 sums and one load fit without spills
                constexpr bool X16 = C::EPI_WARPS > 8;
                constexpr int LDB = X16 ? 1 : GC > 64 ? 1 : GC / 32;
                constexpr int LDW = X16 ? 16 : 32;  // columns per load
                // packed FP32 FMAs (half the promotion's FMA instructions) up to 12
                // warps; at 16 warps (a 96-register cap) their register pairs spill more
                // than they save (85.5 -> 97.2 us at 16384 x 4096 -> 1024)
                constexpr bool PACKED = C::EPI_WARPS <= 12;
                static_assert(!GROUP || (GC <= 128 && 128 % GC == 0), "a warp's columns share one block scale");
                const int cbase = ((warp - 2) / 4) * GC;
                const int64_t nb_raw = (n_blk * BN + cbase) / 128;
                const int64_t nb = nb_raw < ng ? nb_raw : ng - 1;  // columns past N are never stored
                float sum[GC];
#pragma unroll
                for (int j = 0; j < GC; ++j) sum[j] = 0.0f;
                const int64_t srow = row < M ? row : M - 1;
                // up to 12 warps the two scales of a slice are loaded two slices
                // ahead, so the promotion never waits on a load once its
                // accumulator is ready (131072 x 6400 -> 1600 on the 192-wide
                // tile: 1523 -> 1335 us); the 16-warp tile (a 96-register cap)
                // spills the extra registers and keeps the loads in the slice
                constexpr bool PREFETCH = C::EPI_WARPS <= 12;
                const float* sa_p = scale_a + srow * kg;
                const float* sb_p = scale_b + nb;
                float sa0 = 1.0f, sb0 = 1.0f, sa1 = 1.0f, sb1 = 1.0f;
                if constexpr (PREFETCH) {
                    sa0 = __ldg(sa_p);
                    sb0 = __ldg(sb_p);
                    if (num_kb > 1) {
                        sa1 = __ldg(sa_p + 1);
                        sb1 = __ldg(sb_p + ng);
                    }
                }
                for (int kb = 0; kb < num_kb; ++kb) {
                    float ginv;
                    if constexpr (PREFETCH) {
                        ginv = 1.0f / (sa0 * sb0);
                        sa0 = sa1;
                        sb0 = sb1;
                        if (kb + 2 < num_kb) {
                            sa1 = __ldg(sa_p + kb + 2);
                            sb1 = __ldg(sb_p + (kb + 2) * ng);
                        }
                    } else {
                        ginv = 1.0f / (__ldg(sa_p + kb) * __ldg(sb_p + kb * ng));
                    }
                    ok = wait_phase(&tfull[acc], acc_phase, abort_flag, status);
                    ok = __all_sync(0xFFFFFFFFu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    if constexpr (X16) {
#pragma unroll
                        for (int l = 0; l < GC / LDW; ++l) {
                            uint32_t r16[16];
                            tmem_ld_x16_sync(tmem_base + lane_base + static_cast<uint32_t>(acc * BN + cbase + l * 16), r16);
                            if (l + 1 == GC / LDW) {
                                // the accumulator is in registers: the MMA may reuse it
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(tempty0 + 8u * acc);
                            }
                            if constexpr (PACKED) {
#pragma unroll
                                for (int j = 0; j < 16; j += 2)
                                    fma_f32x2(sum[l * 16 + j], sum[l * 16 + j + 1], r16[j], r16[j + 1], ginv);
                            } else {
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    sum[l * 16 + j] = fmaf(__uint_as_float(r16[j]), ginv, sum[l * 16 + j]);
                            }
                        }
                    }
#pragma unroll
                    for (int c0 = 0; c0 < (X16 ? 0 : GC / 32); c0 += LDB) {
                        uint32_t r[LDB][32];
                        const uint32_t ta = tmem_base + lane_base + static_cast<uint32_t>(acc * BN + cbase + c0 * 32);
                        if constexpr (LDB == 2) tmem_ld_2x32_sync(ta, ta + 32, r[0], r[1]);
                        else tmem_ld_x32_sync(ta, r[0]);
                        if (c0 + LDB == GC / 32) {
                            // the accumulator is in registers: the MMA may reuse it
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) {
                                if constexpr (PAIR) mbar_arrive_cluster(tempty0 + 8u * acc);
                                else mbar_arrive(tempty0 + 8u * acc);
                            }
                        }
#pragma unroll
                        for (int b = 0; b < LDB; ++b)
#pragma unroll
                            for (int j = 0; j < 32; j += 2)
                                fma_f32x2(sum[(c0 + b) * 32 + j], sum[(c0 + b) * 32 + j + 1], r[b][j], r[b][j + 1], ginv);
                    }
                    next_acc<C::ACCS>(acc, acc_phase);
                }
                if (!ok) break;
#pragma unroll
                for (int c = 0; c < GC / 32; ++c) {
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = sum[c * 32 + j];
                    // one staging block per warp: these stores come once per tile
                    epi_store_chunk<C::EPI_STAGE / kEpiChunkBytes>(&tmD, warp_stage, nchunk, lane, v,
                                    static_cast<int32_t>(n_blk * BN + cbase + c * 32), static_cast<int32_t>(row0), M, N);
                }
            }
        }
        if constexpr (DACT) {
            // no H load may still be landing in shared memory when the CTA exits
            while (ldw < ldn) {
                wait_phase_drain(lbar, ldw & 1);
                ++ldw;
            }
        }
        // every store has finished reading shared memory (the writes to D
        // complete on their own and are visible when the grid finishes)
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        if constexpr (EQ) {
            const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max16x2(eq_amax2));
            const uint32_t c = __reduce_add_sync(0xFFFFFFFFu, eq_nsat);
            if (lane == 0) {
                // a non-negative float orders like its bit pattern
                if (eq.amax_out && m) atomicMax(reinterpret_cast<unsigned int*>(eq.amax_out), m << 16);
                if (eq.sat_out && c) atomicAdd(eq.sat_out, static_cast<unsigned long long>(c));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (FUSED) {
        // every wait of this CTA on the counters is over and its amax / count
        // atomics are done: the last CTA to get here resets the counters for
        // the next launch and pushes the final amax values into the histories
        __shared__ int s_last_cta;
        if (threadIdx.x == 0) {
            int last = 0;
            if (fz.done) {
                __threadfence();
                last = atomicAdd(fz.done, 1u) == gridDim.x - 1;
                if (last) __threadfence();
            }
            s_last_cta = last;
        }
        __syncthreads();
        if (s_last_cta && warp == 0) {
            for (int64_t b = lane; b < fz.nblocks; b += 32) fz.ready[b] = 0u;
            if (lane == 0) {
                *fz.w_ready = 0u;
                *fz.q_next = 0u;
                *fz.w_next = 0u;
                *fz.done = 0u;
            }
            if (fz.hx.history) history_update_once(fz.hx, fz.amax_out);
            if (fz.hw.history) history_update_once(fz.hw, fz.amax_w);
        }
    }
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
// E4M3 output Q [rows, cols]: box = 64 bytes x 32 rows, 64-byte swizzle (stores).
bool make_q_out_map(CUtensorMap* map, void* base, int64_t rows, int64_t cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// E4M3 input [rows, cols] read by the epilogue: box = 32 bytes x 32 rows, no swizzle.
bool make_q_in_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

std::atomic<int> g_hold_loads{0};   // fp8q_gemm_test_hold_loads
std::atomic<int> g_fused_grid{0};   // fp8q_test_set_fused_grid: CTAs of the fused kernel, 0 = one per SM

struct LaunchInfo {
    cudaError_t attr_err = cudaSuccess;
    int max_clusters = 0;  // co-resident 2-CTA clusters (PAIR only)
};

template <int BN, bool GROUP, bool PAIR, int FUSED, bool EQ = false, int DACT = 0>
const LaunchInfo& launch_info() {
    using C = KernelCfg<BN, GROUP, PAIR, FUSED, EQ, DACT>;
    static LaunchInfo info;
    static std::once_flag once;
    std::call_once(once, [] {
        auto kern = fp8_gemm_kernel<BN, GROUP, PAIR, FUSED, EQ, DACT>;
        info.attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (PAIR && info.attr_err == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * sm_count());
            cfg.blockDim = dim3(gemm_threads<BN, GROUP, FUSED, EQ>());
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

// Outputs of the activation-quantize epilogue (EQ): d is H (or nullptr).
struct EpiQuantHost {
    void* act_out;  // BF16 [M,N] or nullptr
    void* q_out;    // E4M3 [M,N]
    EpiQuantArgs args;
};

template <int BN, bool GROUP, bool PAIR, int FUSED, bool EQ = false, int DACT = 0>
int launch_gemm(const void* a, const void* b, const float* sa, const float* sb, void* d, int64_t M,
                int64_t N, int64_t K, uint32_t afmt, uint32_t bfmt, int* status, cudaStream_t stream,
                const FusedArgs& fz, const EpiQuantHost* eqh = nullptr, const void* h_in = nullptr,
                int act = 0) {
    using C = KernelCfg<BN, GROUP, PAIR, FUSED, EQ, DACT>;
    const LaunchInfo& info = launch_info<BN, GROUP, PAIR, FUSED, EQ, DACT>();
    if (info.attr_err != cudaSuccess) return FP8Q_ERR_CUDA;
    alignas(64) CUtensorMap mapA, mapB, mapB2, mapD, mapE1, mapE2;
    if (!make_kmajor_map(&mapA, a, M, K, BM) || !make_kmajor_map(&mapB, b, N, K, C::B_BOX)) return FP8Q_ERR_CUDA;
    mapB2 = mapB;  // the second MMA's B box, where it differs from the first's
    if constexpr (C::MMA_N * C::NSPLIT != BN)
        if (!make_kmajor_map(&mapB2, b, N, K, C::split_rows(1))) return FP8Q_ERR_CUDA;
    EpiQuantArgs eq = {};
    if constexpr (EQ) {
        // every map handed to the kernel is a valid one: an output not asked
        // for takes the E4M3 map, which the kernel then never stores through
        eq = eqh->args;
        if (!make_q_out_map(&mapE2, eqh->q_out, M, N)) return FP8Q_ERR_CUDA;
        mapE1 = mapE2;
        mapD = mapE2;
        if (eqh->act_out && !make_out_map(&mapE1, eqh->act_out, M, N)) return FP8Q_ERR_CUDA;
        if (d && !make_out_map(&mapD, d, M, N)) return FP8Q_ERR_CUDA;
        eq.has_act = eqh->act_out != nullptr;
        eq.has_h = d != nullptr;
    } else {
        if (!make_out_map(&mapD, d, M, N)) return FP8Q_ERR_CUDA;
        mapE1 = mapD;
        mapE2 = mapD;
        if constexpr (DACT == 1) {
            // H [M,N] (BF16), loaded in the same 32 x 32 boxes the output is stored in
            if (!make_out_map(&mapE1, const_cast<void*>(h_in), M, N)) return FP8Q_ERR_CUDA;
            eq.act = act;
        }
        if constexpr (DACT == 2) {
            // H's E4M3 cache [M,N]: 32-byte x 32-row boxes, unswizzled
            if (!make_q_in_map(&mapE1, h_in, M, N)) return FP8Q_ERR_CUDA;
            eq.act = act;
            eq.scale_h = eqh ? eqh->args.scale_h : nullptr;
        }
    }
    const int64_t tiles = ((M + C::TILE_M - 1) / C::TILE_M) * ((N + BN - 1) / BN);
    const uint32_t idesc = idesc_f8(afmt, bfmt, C::MMA_M, C::MMA_N);
    auto kern = fp8_gemm_kernel<BN, GROUP, PAIR, FUSED, EQ, DACT>;
    if constexpr (PAIR) {
        if (info.max_clusters < 1) return FP8Q_ERR_CUDA;
        // the fused kernel takes every co-resident cluster (its CTAs take work
        // by ticket, so a grid larger or smaller than that is also correct)
        const int fg = g_fused_grid.load();
        const int clusters = static_cast<int>(FUSED ? (fg > 0 ? std::max(1, fg / 2) : info.max_clusters)
                                                    : std::min<int64_t>(tiles, info.max_clusters));
        const FusedArgs& f = fz;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(2 * clusters);
        cfg.blockDim = dim3(gemm_threads<BN, GROUP, FUSED, EQ>());
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        if (cudaLaunchKernelEx(&cfg, kern, mapA, mapB, mapB2, mapD, sa, sb, M, N, K, idesc, status,
                               g_hold_loads.load(), f, mapE1, mapE2, eq, static_cast<uint16_t*>(d)) != cudaSuccess) {
            (void)cudaGetLastError();
            return FP8Q_ERR_CUDA;
        }
    } else {
        // the fused kernel: one CTA per SM (its CTAs take work by ticket, so a
        // grid larger or smaller than that is also correct)
        const int fg = g_fused_grid.load();
        const int grid = static_cast<int>(FUSED ? (fg > 0 ? fg : sm_count()) : std::min<int64_t>(tiles, sm_count()));
        const FusedArgs& f = fz;
        if (launch_pdl(kern, dim3(grid), dim3(gemm_threads<BN, GROUP, FUSED, EQ>()), C::SMEM_BYTES, stream, mapA, mapB,
                       mapB2, mapD, sa, sb, M, N, K, idesc, status, g_hold_loads.load(), f, mapE1, mapE2, eq,
                       static_cast<uint16_t*>(d)) != cudaSuccess) {
            (void)cudaGetLastError();
            return FP8Q_ERR_CUDA;
        }
    }
    FP8Q_CHECK_LAUNCH();
    return FP8Q_OK;
}

// Tile shape.  A tile's time depends only weakly on its width (the tensor
// core is much less efficient on narrow tiles), so each candidate is scored
// as (tiles per SM or SM pair, rounded up) x its measured time per tile.  The
// per-tile times are relative to the 2-SM 256-wide tile, from sweeps of this
// kernel over the workloads' shapes on GB300 (K-bound runs, TFLOP/s per tile
// width); ties go to the earlier candidate.
struct Shape {
    bool pair;
    int bn;
};

// fp8q_gemm_set_tile: -1 = automatic, else (pair << 16) | bn
std::atomic<int> g_tile_override{-1};

Shape pick_shape(int64_t M, int64_t N, bool wide) {
    const int ov = g_tile_override.load(std::memory_order_relaxed);
    if (ov >= 0) {
        const bool pair = (ov >> 16) != 0;
        const int bn = ov & 0xFFFF;
        if (!pair || M > BM) return Shape{pair, bn};
        return Shape{false, bn == 224 || bn == 384 || bn == 400 ? 256 : bn};
    }
    struct Cand { bool pair; int bn; double t; };
    // {true, 384}: one accumulator, so its epilogue is not hidden; 1.70 measured
    // at 8192 x 3072 -> 768, where its 64 tiles fit one wave of 76 pairs.
    // {true, 400}: one accumulator too; 1.74 measured at 131072 x 6400 -> 1600,
    // where four of its tiles span N exactly (the 256-wide tile computes 1792
    // columns there and reads each A row block seven times instead of four)
    static constexpr Cand kCands[] = {
        {true, 256, 1.000}, {true, 224, 0.946}, {true, 192, 0.909}, {true, 160, 0.837}, {true, 128, 0.858},
        {false, 192, 0.897}, {false, 160, 0.834}, {false, 128, 0.843}, {false, 256, 1.102}, {true, 384, 1.700},
        {true, 400, 1.740},
    };
    const int64_t sms = sm_count();
    Shape best{false, 128};
    double best_cost = -1.0;
    for (const Cand& c : kCands) {
        if ((c.pair && M <= BM) || (c.bn == 384 && !wide)) continue;
        const int64_t tile_m = c.pair ? 2 * BM : BM;
        const int64_t units = c.pair ? sms / 2 : sms;
        const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + c.bn - 1) / c.bn);
        const double cost = static_cast<double>((tiles + units - 1) / units) * c.t;
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = Shape{c.pair, c.bn}; }
    }
    return best;
}

// Group-mode tile width (1-CTA tiles, four accumulators' worth of TMEM): 128
// with 8 promotion warps, 192 with 12 or 256 with 16 (64 columns per warp, so
// each warp stays inside one 128-column scale block).  Scored like pick_shape,
// with per-wave times relative to the 128-wide tile from sweeps of the three
// widths over the workloads' shapes on GB300 (8192 to 131072 rows, N 768 to
// 1600; 192 wide 1.19 - 1.25x, 256 wide 1.68 - 1.75x).  A tile override (0, 128), (0, 192) or (0, 256) pins it.
int pick_group_bn(int64_t M, int64_t N) {
    const int ov = g_tile_override.load(std::memory_order_relaxed);
    if (ov >= 0 && (ov >> 16) == 0 && ((ov & 0xFFFF) == 256 || (ov & 0xFFFF) == 192 || (ov & 0xFFFF) == 128))
        return ov & 0xFFFF;
    struct Cand { int bn; double t; };
    static constexpr Cand kCands[] = {{128, 1.000}, {192, 1.210}, {256, 1.720}};
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

template <int FUSED>
int gemm_dispatch_t(const void* a, const void* b, const float* sa, const float* sb, int group, void* d,
                    int64_t M, int64_t N, int64_t K, uint32_t afmt, uint32_t bfmt, int* status,
                    cudaStream_t stream, const FusedArgs& fz) {
    if constexpr (!FUSED) {
        if (group) {
            const int gbn = pick_group_bn(M, N);
            if (gbn == 256)
                return launch_gemm<256, true, false, false>(a, b, sa, sb, d, M, N, K, afmt, bfmt, status, stream, fz);
            if (gbn == 192)
                return launch_gemm<192, true, false, false>(a, b, sa, sb, d, M, N, K, afmt, bfmt, status, stream, fz);
            return launch_gemm<128, true, false, false>(a, b, sa, sb, d, M, N, K, afmt, bfmt, status, stream, fz);
        }
    }
    Shape s = pick_shape(M, N, !FUSED);
    if (FUSED && s.bn == 384) s.bn = 256;  // the one-launch step keeps two accumulators
#define FP8Q_LAUNCH(BNV, PR) \
    return launch_gemm<BNV, false, PR, FUSED>(a, b, sa, sb, d, M, N, K, afmt, bfmt, status, stream, fz)
    if constexpr (FUSED == 2) {
        // the GEMM-first layout is built for the pair tiles of the wide steps
        if (s.pair && s.bn == 400) FP8Q_LAUNCH(400, true);
        if (s.pair && s.bn == 256) FP8Q_LAUNCH(256, true);
        return gemm_dispatch_t<1>(a, b, sa, sb, group, d, M, N, K, afmt, bfmt, status, stream, fz);
    } else {
    if (s.pair) {
        switch (s.bn) {
            case 400: FP8Q_LAUNCH(400, true);
            case 384:
                if constexpr (!FUSED) FP8Q_LAUNCH(384, true);
                [[fallthrough]];
            case 256: FP8Q_LAUNCH(256, true);
            case 224: FP8Q_LAUNCH(224, true);
            case 192: FP8Q_LAUNCH(192, true);
            case 160: FP8Q_LAUNCH(160, true);
            default: FP8Q_LAUNCH(128, true);
        }
    }
    switch (s.bn) {
        case 256: FP8Q_LAUNCH(256, false);
        case 192: FP8Q_LAUNCH(192, false);
        case 160: FP8Q_LAUNCH(160, false);
        default: FP8Q_LAUNCH(128, false);
    }
    }
#undef FP8Q_LAUNCH
}

// The one-launch step's quantize layout (QuantLayout): GEMM-first where the
// GEMM is the longer part of the step.  Its 2 M N K FLOPs against the
// quantize's 5 M K bytes, at the rates the two kernels reach alone on GB300
// (about 3.7 PFLOP/s and 6.45 TB/s), make the GEMM longer once
// 2 N / 3.7e15 > 5 / 6.45e12, i.e. N above ~1430 (GPT-2-XL's 1600; GPT-2's
// 768 is quantize-first).  fp8q_test_set_fused_layout pins either one.
std::atomic<int> g_fused_layout{0};

int fused_dispatch(const void* x_q, const void* wt_q, const float* sx, const float* sw, void* y, int64_t M,
                   int64_t N, int64_t K, int* status, cudaStream_t stream, const FusedArgs& fz) {
    const int ov = g_fused_layout.load(std::memory_order_relaxed);
    const bool gemm_first = ov ? ov == 2 : 2.0 * static_cast<double>(N) * 6.45e12 > 5.0 * 3.7e15;
    if (gemm_first)
        return gemm_dispatch_t<2>(x_q, wt_q, sx, sw, 0, y, M, N, K, FP8Q_E4M3, FP8Q_E4M3, status, stream, fz);
    return gemm_dispatch_t<1>(x_q, wt_q, sx, sw, 0, y, M, N, K, FP8Q_E4M3, FP8Q_E4M3, status, stream, fz);
}

int gemm_dispatch(const void* a, const void* b, const float* sa, const float* sb, int group, void* d,
                  int64_t M, int64_t N, int64_t K, uint32_t afmt, uint32_t bfmt, int* status,
                  cudaStream_t stream) {
    return gemm_dispatch_t<0>(a, b, sa, sb, group, d, M, N, K, afmt, bfmt, status, stream, FusedArgs{});
}

int check_gemm_args(const void* a, const void* b, const float* sa, const float* sb, const void* d,
                    int64_t M, int64_t N, int64_t K, const int* status) {
    if (!b || !sa || !sb) return FP8Q_ERR_NULL;
    if ((!a || !d) && M != 0) return FP8Q_ERR_NULL;  // an empty A / D may have no storage
    if (M < 0 || N < 16 || K < 16 || N % 16 != 0 || K % 16 != 0) return FP8Q_ERR_SHAPE;
    if (M > (int64_t(1) << 31) - 2 * BM || N > (int64_t(1) << 31) - 256 || K > (int64_t(1) << 31) - BK)
        return FP8Q_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return FP8Q_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(sa) | reinterpret_cast<uintptr_t>(sb) |
         reinterpret_cast<uintptr_t>(status)) & 3u)
        return FP8Q_ERR_ALIGN;
    if (!device_is_sm103()) return FP8Q_ERR_UNSUPPORTED;
    return FP8Q_OK;
}

// Tile for the activation-quantize epilogue: whole 64-column pairs and two
// accumulators, so widths 128, 192 and 256, scored like pick_shape.  A tile
// override names one of these or is ignored.
Shape pick_shape_eq(int64_t M, int64_t N) {
    const int ov = g_tile_override.load(std::memory_order_relaxed);
    if (ov >= 0) {
        const bool pair = (ov >> 16) != 0;
        const int bn = ov & 0xFFFF;
        if (bn % 64 == 0 && bn <= 256) return Shape{pair && M > BM, bn};
    }
    struct Cand { bool pair; int bn; double t; };
    static constexpr Cand kCands[] = {{true, 256, 1.000}, {true, 192, 0.909}, {true, 128, 0.858},
                                      {false, 192, 0.897}, {false, 128, 0.843}, {false, 256, 1.102}};
    const int64_t sms = sm_count();
    Shape best{false, 128};
    double best_cost = -1.0;
    for (const Cand& c : kCands) {
        if (c.pair && M <= BM) continue;
        const int64_t tile_m = c.pair ? 2 * BM : BM;
        const int64_t units = c.pair ? sms / 2 : sms;
        const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + c.bn - 1) / c.bn);
        const double cost = static_cast<double>((tiles + units - 1) / units) * c.t;
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = Shape{c.pair, c.bn}; }
    }
    return best;
}

// Tile for the dgrad with the activation backward: the plain GEMM's widths
// except 384 and 160, scored like pick_shape.  A tile override names one of
// these or is ignored.
Shape pick_shape_dact(int64_t M, int64_t N) {
    const int ov = g_tile_override.load(std::memory_order_relaxed);
    if (ov >= 0) {
        const bool pair = (ov >> 16) != 0;
        const int bn = ov & 0xFFFF;
        if (bn == 128 || bn == 192 || bn == 256 || (pair && bn == 224)) return Shape{pair && M > BM, bn == 224 && M <= BM ? 256 : bn};
    }
    struct Cand { bool pair; int bn; double t; };
    static constexpr Cand kCands[] = {{true, 256, 1.000}, {true, 224, 0.946}, {true, 192, 0.909}, {true, 128, 0.858},
                                      {false, 192, 0.897}, {false, 128, 0.843}, {false, 256, 1.102}};
    const int64_t sms = sm_count();
    Shape best{false, 128};
    double best_cost = -1.0;
    for (const Cand& c : kCands) {
        if (c.pair && M <= BM) continue;
        const int64_t tile_m = c.pair ? 2 * BM : BM;
        const int64_t units = c.pair ? sms / 2 : sms;
        const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + c.bn - 1) / c.bn);
        const double cost = static_cast<double>((tiles + units - 1) / units) * c.t;
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = Shape{c.pair, c.bn}; }
    }
    return best;
}

template <int HFMT>
int launch_dact(const Shape& s, const void* a, const void* b, const float* sa, const float* sb, void* d, int64_t M,
                int64_t N, int64_t K, const void* h, int act, int* status, cudaStream_t stream,
                const EpiQuantHost* eqh = nullptr) {
#define FP8Q_LAUNCH_DACT(BNV, PR) \
    return launch_gemm<BNV, false, PR, false, false, HFMT>(a, b, sa, sb, d, M, N, K, FP8Q_E5M2, FP8Q_E4M3, status, \
                                                           stream, FusedArgs{}, eqh, h, act)
    if (s.pair) {
        if (s.bn == 256) FP8Q_LAUNCH_DACT(256, true);
        if (s.bn == 224) FP8Q_LAUNCH_DACT(224, true);
        if (s.bn == 192) FP8Q_LAUNCH_DACT(192, true);
        FP8Q_LAUNCH_DACT(128, true);
    }
    if (s.bn == 256) FP8Q_LAUNCH_DACT(256, false);
    if (s.bn == 192) FP8Q_LAUNCH_DACT(192, false);
    FP8Q_LAUNCH_DACT(128, false);
#undef FP8Q_LAUNCH_DACT
}

int launch_eq(const Shape& s, const void* a, const void* b, const float* sa, const float* sb, void* h,
              int64_t M, int64_t N, int64_t K, int* status, cudaStream_t stream, const EpiQuantHost& e) {
#define FP8Q_LAUNCH_EQ(BNV, PR) \
    return launch_gemm<BNV, false, PR, false, true>(a, b, sa, sb, h, M, N, K, FP8Q_E4M3, FP8Q_E4M3, status, stream, \
                                                    FusedArgs{}, &e)
    if (s.pair) {
        if (s.bn == 256) FP8Q_LAUNCH_EQ(256, true);
        if (s.bn == 192) FP8Q_LAUNCH_EQ(192, true);
        FP8Q_LAUNCH_EQ(128, true);
    }
    if (s.bn == 256) FP8Q_LAUNCH_EQ(256, false);
    if (s.bn == 192) FP8Q_LAUNCH_EQ(192, false);
    FP8Q_LAUNCH_EQ(128, false);
#undef FP8Q_LAUNCH_EQ
}

}  // namespace

}  // namespace fp8q

using namespace fp8q;

extern "C" void fp8q_gemm_test_hold_loads(int on) { g_hold_loads.store(on != 0 ? 1 : 0); }

extern "C" int fp8q_test_gemm_tile(int64_t M, int64_t N, int fused, int* pair, int* bn) {
    if (!pair || !bn) return FP8Q_ERR_NULL;
    if (M < 1 || N < 16) return FP8Q_ERR_SHAPE;
    Shape s = pick_shape(M, N, !fused);
    if (fused && s.bn == 384) s.bn = 256;  // as gemm_dispatch_t does for the one-launch step
    *pair = s.pair ? 1 : 0;
    *bn = s.bn;
    return FP8Q_OK;
}

extern "C" int fp8q_test_set_fused_layout(int layout) {
    if (layout < 0 || layout > 2) return FP8Q_ERR_UNSUPPORTED;
    g_fused_layout.store(layout);
    return FP8Q_OK;
}

extern "C" int fp8q_test_set_fused_grid(int ctas) {
    if (ctas < 0 || ctas > 65535) return FP8Q_ERR_SHAPE;
    g_fused_grid.store(ctas);
    return FP8Q_OK;
}

extern "C" int fp8q_gemm_set_tile(int pair, int bn) {
    if (pair == -1) {
        g_tile_override.store(-1);
        return FP8Q_OK;
    }
    const bool ok1 = pair == 0 && (bn == 128 || bn == 160 || bn == 192 || bn == 256);
    const bool ok2 = pair == 1 && (bn == 128 || bn == 160 || bn == 192 || bn == 224 || bn == 256 || bn == 384 || bn == 400);
    if (!ok1 && !ok2) return FP8Q_ERR_UNSUPPORTED;
    g_tile_override.store((pair << 16) | bn);
    return FP8Q_OK;
}

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

extern "C" int fp8_gemm_fwd_update(const void* x_q, const void* wt_q, const float* scale_x, const float* scale_w,
                                   void* y, int64_t M, int64_t N, int64_t K, float* amax_x,
                                   const fp8q_history_args* hist_x, float* amax_w, const fp8q_history_args* hist_w,
                                   int* status, cudaStream_t stream) {
    FusedArgs fz = {};
    int st = FP8Q_OK;
    const fp8q_history_args* hs[2] = {hist_x, hist_w};
    float* amax[2] = {amax_x, amax_w};
    HistoryArgs* out[2] = {&fz.hx, &fz.hw};
    for (int i = 0; i < 2; ++i) {
        if (!hs[i]) continue;
        st = check_history(hs[i], amax[i], out[i]);
        if (st != FP8Q_OK) return st;
        // the update writes the next step's scale: never one this GEMM reads
        if (hs[i]->scale_out == scale_x || hs[i]->scale_out == scale_w) return FP8Q_ERR_SHAPE;
        if (hs[i]->amax_clear && (hs[i]->amax_clear == amax[0] || hs[i]->amax_clear == amax[1])) return FP8Q_ERR_SHAPE;
    }
    st = check_gemm_args(x_q, wt_q, scale_x, scale_w, y, M, N, K, status);
    if (st != FP8Q_OK) return st;
    if (M == 0) return (hist_x || hist_w) ? FP8Q_ERR_SHAPE : FP8Q_OK;  // the updates ride on the launch
    fz.amax_out = amax_x;
    fz.amax_w = amax_w;
    return gemm_dispatch_t<0>(x_q, wt_q, scale_x, scale_w, 0, y, M, N, K, FP8Q_E4M3, FP8Q_E4M3, status,
                                  stream, fz);
}

extern "C" int fp8_gemm_dgrad(const void* dy_q, const void* w_q, const float* scale_dy, const float* scale_w,
                              void* dx, int64_t M, int64_t N, int64_t K, int* status, cudaStream_t stream) {
    // D = dX [M,K], A = dY [M,N] (contraction N), B = W [K,N]
    int st = check_gemm_args(dy_q, w_q, scale_dy, scale_w, dx, M, K, N, status);
    if (st != FP8Q_OK) return st;
    if (M == 0) return FP8Q_OK;
    return gemm_dispatch(dy_q, w_q, scale_dy, scale_w, 0, dx, M, K, N, FP8Q_E5M2, FP8Q_E4M3, status, stream);
}

extern "C" int fp8_upproj_fwd(const void* x_q, const void* wt_q, const float* scale_x, const float* scale_w,
                              int act, const float* scale_h, void* h_out, void* act_out, void* h_q,
                              float* amax_out, unsigned long long* sat_count, int64_t M, int64_t N, int64_t K,
                              unsigned flags, int* status, cudaStream_t stream) {
    if (flags & ~static_cast<unsigned>(FP8Q_ACCUMULATE)) return FP8Q_ERR_UNSUPPORTED;
    if (act < FP8Q_ACT_IDENTITY || act > FP8Q_ACT_RELU2) return FP8Q_ERR_UNSUPPORTED;
    if (scale_h == nullptr) return FP8Q_ERR_NULL;
    if (!aligned16(h_out) || !aligned16(act_out) || (reinterpret_cast<uintptr_t>(amax_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(sat_count) & 7u) || (reinterpret_cast<uintptr_t>(scale_h) & 3u))
        return FP8Q_ERR_ALIGN;
    // D = the E4M3 copy [M,N] (required); H and the activation copy are optional
    int st = check_gemm_args(x_q, wt_q, scale_x, scale_w, h_q, M, N, K, status);
    if (st != FP8Q_OK) return st;
    if (!(flags & FP8Q_ACCUMULATE)) {
        if (amax_out && cudaMemsetAsync(amax_out, 0, sizeof(float), stream) != cudaSuccess) return FP8Q_ERR_CUDA;
        if (sat_count && cudaMemsetAsync(sat_count, 0, sizeof(unsigned long long), stream) != cudaSuccess)
            return FP8Q_ERR_CUDA;
    }
    if (M == 0) return FP8Q_OK;
    const EpiQuantHost e{act_out, h_q, EpiQuantArgs{scale_h, amax_out, sat_count, act, 0, 0}};
    return launch_eq(pick_shape_eq(M, N), x_q, wt_q, scale_x, scale_w, h_out, M, N, K, status, stream, e);
}

extern "C" int fp8_gemm_dgrad_act(const void* dy_q, const void* w_q, const float* scale_dy, const float* scale_w,
                                  const void* h, int act, void* dh, int64_t M, int64_t N, int64_t K, int* status,
                                  cudaStream_t stream) {
    // D = dH [M,K], A = dY [M,N] (contraction N), B = W [K,N]; H [M,K] read in the epilogue
    if (act < FP8Q_ACT_IDENTITY || act > FP8Q_ACT_RELU2) return FP8Q_ERR_UNSUPPORTED;
    if (h == nullptr && M != 0) return FP8Q_ERR_NULL;
    if (!aligned16(h)) return FP8Q_ERR_ALIGN;
    int st = check_gemm_args(dy_q, w_q, scale_dy, scale_w, dh, M, K, N, status);
    if (st != FP8Q_OK) return st;
    if (M == 0) return FP8Q_OK;
    return launch_dact<1>(pick_shape_dact(M, K), dy_q, w_q, scale_dy, scale_w, dh, M, K, N, h, act, status, stream);
}

extern "C" int fp8_gemm_dgrad_act_q(const void* dy_q, const void* w_q, const float* scale_dy, const float* scale_w,
                                    const void* h_q, const float* scale_h, int act, void* dh, int64_t M, int64_t N,
                                    int64_t K, int* status, cudaStream_t stream) {
    // D = dH [M,K], A = dY [M,N] (contraction N), B = W [K,N]; H's E4M3 cache [M,K] read in the epilogue
    if (act < FP8Q_ACT_IDENTITY || act > FP8Q_ACT_RELU2) return FP8Q_ERR_UNSUPPORTED;
    if ((h_q == nullptr && M != 0) || scale_h == nullptr) return FP8Q_ERR_NULL;
    if (!aligned16(h_q) || (reinterpret_cast<uintptr_t>(scale_h) & 3u)) return FP8Q_ERR_ALIGN;
    int st = check_gemm_args(dy_q, w_q, scale_dy, scale_w, dh, M, K, N, status);
    if (st != FP8Q_OK) return st;
    if (M == 0) return FP8Q_OK;
    EpiQuantHost e{};
    e.args.scale_h = scale_h;
    return launch_dact<2>(pick_shape_dact(M, K), dy_q, w_q, scale_dy, scale_w, dh, M, K, N, h_q, act, status, stream,
                          &e);
}

extern "C" int fp8_gemm_wgrad(const void* x_q_t, const void* dy_q_t, const float* scale_x,
                              const float* scale_dy, void* dw, int64_t M, int64_t N, int64_t K, int* status,
                              cudaStream_t stream) {
    // D = dW [K,N], A = X_q^T [K,M], B = dY_q^T [N,M] (contraction M)
    int st = check_gemm_args(x_q_t, dy_q_t, scale_x, scale_dy, dw, K, N, M, status);
    if (st != FP8Q_OK) return st;
    if (K == 0) return FP8Q_OK;
    return gemm_dispatch(x_q_t, dy_q_t, scale_x, scale_dy, 0, dw, K, N, M, FP8Q_E4M3, FP8Q_E5M2, status, stream);
}

extern "C" size_t fp8_downproj_workspace_bytes(int64_t M) {
    if (M <= 0) return 0;
    const size_t blocks = static_cast<size_t>((M + BM - 1) / BM);
    return ((blocks + 4) * sizeof(unsigned) + 255) / 256 * 256;  // ready[blocks], w_ready, done, q_next, w_next
}

namespace {

FusedArgs fused_args(const void* h, int act, void* act_out, void* x_q, float* amax_out,
                     unsigned long long* sat_count, unsigned* ws, int64_t M) {
    FusedArgs fz = {};
    fz.h = static_cast<const uint4*>(h);
    fz.act_out = static_cast<uint4*>(act_out);
    fz.x_q = static_cast<uint2*>(x_q);
    fz.amax_out = amax_out;
    fz.sat_out = sat_count;
    fz.act = act;
    fz.nblocks = (M + BM - 1) / BM;
    fz.ready = ws;
    fz.w_ready = ws + fz.nblocks;
    fz.done = ws + fz.nblocks + 1;
    fz.q_next = ws + fz.nblocks + 2;
    fz.w_next = ws + fz.nblocks + 3;
    return fz;
}

}  // namespace

extern "C" int fp8_downproj_fwd(const void* h, const void* wt_q, int64_t M, int64_t N, int64_t K, int act,
                                const float* scale_x, const float* scale_w, void* act_out, void* x_q,
                                float* amax_out, unsigned long long* sat_count, void* y, void* workspace,
                                size_t workspace_bytes, int* status, cudaStream_t stream) {
    return fp8_downproj_fwd_ex(h, nullptr, const_cast<void*>(wt_q), M, N, K, act, scale_x, scale_w, act_out, x_q,
                               amax_out, sat_count, nullptr, nullptr, nullptr, y, workspace, workspace_bytes,
                               nullptr, nullptr, 0u, status, stream);
}

namespace {

}  // namespace

extern "C" int fp8_downproj_fwd_ex(const void* h, const void* w, void* wt_q, int64_t M, int64_t N, int64_t K,
                                   int act, const float* scale_x, const float* scale_w, void* act_out, void* x_q,
                                   float* amax_x, unsigned long long* sat_count, void* w_q, float* amax_w,
                                   unsigned long long* sat_w, void* y,
                                   void* workspace, size_t workspace_bytes, const fp8q_history_args* hist_x,
                                   const fp8q_history_args* hist_w, unsigned flags, int* status,
                                   cudaStream_t stream) {
    if (flags & ~static_cast<unsigned>(FP8Q_ACCUMULATE)) return FP8Q_ERR_UNSUPPORTED;
    if (act < FP8Q_ACT_IDENTITY || act > FP8Q_ACT_RELU2) return FP8Q_ERR_UNSUPPORTED;
    if ((!h || !x_q || !workspace) && M != 0) return FP8Q_ERR_NULL;
    if (!aligned16(h) || !aligned16(act_out) || !aligned16(w) || !aligned16(w_q) ||
        (reinterpret_cast<uintptr_t>(workspace) & 3u) || (reinterpret_cast<uintptr_t>(amax_x) & 3u) ||
        (reinterpret_cast<uintptr_t>(amax_w) & 3u) || (reinterpret_cast<uintptr_t>(sat_count) & 7u) ||
        (reinterpret_cast<uintptr_t>(sat_w) & 7u))
        return FP8Q_ERR_ALIGN;
    if (workspace_bytes < fp8_downproj_workspace_bytes(M)) return FP8Q_ERR_SHAPE;
    // weight units are counted in 32 bits: (K / 8) * ceil(N / 256) of them
    if (w && (K / 8) * ((N + 255) / 256) > (int64_t(1) << 31)) return FP8Q_ERR_SHAPE;
    HistoryArgs hx = {}, hw = {};
    if (hist_w && !w) return FP8Q_ERR_NULL;  // W's amax exists only when the kernel casts W
    if (hist_x) {
        const int hs = check_history(hist_x, amax_x, &hx);
        if (hs != FP8Q_OK) return hs;
    }
    if (hist_w) {
        const int hs = check_history(hist_w, amax_w, &hw);
        if (hs != FP8Q_OK) return hs;
    }
    if ((hist_x || hist_w) && M == 0) return FP8Q_ERR_SHAPE;  // no kernel to run them in
    int st = check_gemm_args(x_q, wt_q, scale_x, scale_w, y, M, N, K, status);  // ends with the device check
    if (st != FP8Q_OK) return st;
    const bool zero = !(flags & FP8Q_ACCUMULATE);
    if (zero) {
        if (amax_x && cudaMemsetAsync(amax_x, 0, sizeof(float), stream) != cudaSuccess) return FP8Q_ERR_CUDA;
        if (sat_count && cudaMemsetAsync(sat_count, 0, sizeof(unsigned long long), stream) != cudaSuccess)
            return FP8Q_ERR_CUDA;
        if (w && amax_w && cudaMemsetAsync(amax_w, 0, sizeof(float), stream) != cudaSuccess) return FP8Q_ERR_CUDA;
        if (w && sat_w && cudaMemsetAsync(sat_w, 0, sizeof(unsigned long long), stream) != cudaSuccess)
            return FP8Q_ERR_CUDA;
    }
    if (M == 0) {
        // no GEMM: a weight to cast still is (the step's W_q^T and amax stay defined)
        if (!w) return FP8Q_OK;
        return fp8_quant_fused_ex(w, K, N, FP8Q_ACT_IDENTITY, FP8Q_E4M3, scale_w, nullptr, w_q, wt_q,
                                  amax_w, sat_w, nullptr, 1, FP8Q_ACCUMULATE, stream);
    }
    if (zero && cudaMemsetAsync(workspace, 0, fp8_downproj_workspace_bytes(M), stream) != cudaSuccess)
        return FP8Q_ERR_CUDA;
    FusedArgs fz = fused_args(h, act, act_out, x_q, amax_x, sat_count, static_cast<unsigned*>(workspace), M);
    if (w) {
        fz.w = static_cast<const uint4*>(w);
        fz.scale_w = scale_w;
        fz.wt_q = static_cast<uint8_t*>(wt_q);
        fz.w_q = static_cast<uint8_t*>(w_q);
        fz.amax_w = amax_w;
        fz.sat_w = sat_w;
        fz.wn = N;
        fz.w_units = static_cast<unsigned>((K / 8) * ((N + 255) / 256));
    }
    fz.hx = hx;
    fz.hw = hw;
    return fused_dispatch(x_q, wt_q, scale_x, scale_w, y, M, N, K, status, stream, fz);
}

// ---------------------------------------------------------------------------
// fp8_downproj_fwd_noalloc: the fused kernel with its counters in this
// library's own device memory, for callers that cannot allocate (see
// include/fp8q.h).  The array lives in the module's global memory on every
// device that loads the library, until the process exits.  In host code
// g_noalloc_ready only names the symbol: its device address comes from
// cudaGetSymbolAddress with the device current.  The address is looked up
// on every call rather than cached: after a device reset the module is
// loaded again in a new context, possibly at another address.

static __device__ __align__(256) unsigned g_noalloc_ready[FP8Q_NOALLOC_MAX_M / BM + 64];

static_assert(FP8Q_NOALLOC_MAX_M % BM == 0, "whole 128-row blocks");
static_assert(sizeof(g_noalloc_ready) == ((FP8Q_NOALLOC_MAX_M / BM + 4) * sizeof(unsigned) + 255) / 256 * 256,
              "the array is exactly the workspace of the largest M");

namespace {

// The array's device address on the current device.
int noalloc_scratch(unsigned** out) {
    unsigned* ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_ready) != cudaSuccess || !ptr) {
        (void)cudaGetLastError();
        return FP8Q_ERR_CUDA;
    }
    *out = ptr;
    return FP8Q_OK;
}

}  // namespace

extern "C" int fp8_downproj_fwd_noalloc(const void* h, const void* wt_q, int64_t M, int64_t N, int64_t K, int act,
                                        const float* scale_x, const float* scale_w, void* act_out, void* x_q,
                                        float* amax_out, unsigned long long* sat_count, void* y, int* status,
                                        cudaStream_t stream) {
    if (act < FP8Q_ACT_IDENTITY || act > FP8Q_ACT_RELU2) return FP8Q_ERR_UNSUPPORTED;
    if ((!h || !x_q) && M != 0) return FP8Q_ERR_NULL;
    if (!aligned16(h) || !aligned16(act_out) || (reinterpret_cast<uintptr_t>(amax_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(sat_count) & 7u))
        return FP8Q_ERR_ALIGN;
    if (M > FP8Q_NOALLOC_MAX_M) return FP8Q_ERR_SHAPE;  // more row blocks than the array counts
    int st = check_gemm_args(x_q, wt_q, scale_x, scale_w, y, M, N, K, status);  // ends with the device check
    if (st != FP8Q_OK) return st;
    unsigned* ready = nullptr;
    if (M != 0 && (st = noalloc_scratch(&ready)) != FP8Q_OK) return st;
    if (amax_out && cudaMemsetAsync(amax_out, 0, sizeof(float), stream) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (sat_count && cudaMemsetAsync(sat_count, 0, sizeof(unsigned long long), stream) != cudaSuccess)
        return FP8Q_ERR_CUDA;
    if (M == 0) return FP8Q_OK;
    // the array still holds what the previous call left (zero after a call that
    // ran to the end, but not after one that was cut short): start from zero
    if (cudaMemsetAsync(ready, 0, fp8_downproj_workspace_bytes(M), stream) != cudaSuccess) return FP8Q_ERR_CUDA;
    const FusedArgs fz = fused_args(h, act, act_out, x_q, amax_out, sat_count, ready, M);
    return fused_dispatch(x_q, wt_q, scale_x, scale_w, y, M, N, K, status, stream, fz);
}

extern "C" int fp8q_test_noalloc_fill(int byte, cudaStream_t stream) {
    unsigned* ptr = nullptr;
    const int st = noalloc_scratch(&ptr);
    if (st != FP8Q_OK) return st;
    if (cudaMemsetAsync(ptr, byte & 0xFF, sizeof(g_noalloc_ready), stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8Q_ERR_CUDA;
    }
    return FP8Q_OK;
}
