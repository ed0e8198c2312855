/*
 * fp8q_testing.h -- test and tuning hooks of libfp8q.so.  NOT part of the
 * down-projection's interface: a program that uses the library has no reason
 * to call these.  They exist so that the test suite can drive the failure
 * paths and the schedules that normal inputs never reach, and so that the
 * benchmark can pin a tile shape.
 *
 * Every hook is process-wide and changes what later launches of the library
 * do, for every caller in the process; each one is undone by calling it
 * again with its default (shown below).  Do not leave one set in a program
 * that shares the library with other code.
 */
#ifndef FP8Q_TESTING_H
#define FP8Q_TESTING_H

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fp8q_gemm_set_tile -- pin the GEMM tile shape (a tuning knob; "FP8 training:
 * what it is and how it works", Trade-offs and edge cases: tile size is a
 * tuning knob).  Affects later per-tensor fp8_gemm_fwd / fp8_gemm_dgrad /
 * fp8_gemm_wgrad calls.  The group-scaled GEMM takes the pins (0, 128),
 * (0, 192) and (0, 256) and ignores others.
 *   pair  -1: automatic choice (the default; bn ignored)
 *          0: one CTA per 128 x bn tile           bn in {128, 160, 192, 256}
 *          1: a CTA pair per 256 x bn tile (2-SM)  bn in {128, 160, 192, 224, 256, 384}
 *             (pairs are used only when M > 128; smaller M falls back to one CTA;
 *             384 is two 192-wide MMAs into one accumulator, plain GEMMs only:
 *             fp8_downproj_fwd takes 256 instead)
 * Returns FP8Q_ERR_UNSUPPORTED for any other combination (nothing changes).
 */
int fp8q_gemm_set_tile(int pair, int bn);

/*
 * fp8q_mx_set_tile -- pin the tile shape of fp8_gemm_mx (a tuning knob), or
 * (0, 0) for the automatic choice (the default):
 *   pair  0: one CTA per 128 x bn tile
 *         1: a CTA pair per 256 x bn tile (2-SM); used only when M > 128, else
 *            the 1-CTA tile of that width
 *   bn    128 or 256 (whole 128-row scale atoms of B per tile)
 * Returns FP8Q_ERR_UNSUPPORTED for any other combination (nothing changes).
 */
int fp8q_mx_set_tile(int pair, int bn);

/*
 * fp8q_gemm_test_hold_loads -- failure-path hook.  While on != 0, the GEMM
 * kernels launched afterwards issue no operand loads, so their first bounded
 * wait runs out (after about 2 s): the kernel ORs FP8Q_DEV_TIMEOUT into the
 * status word, releases its resources and exits, leaving the CUDA context
 * usable.  Default: 0.
 */
void fp8q_gemm_test_hold_loads(int on);

/*
 * fp8q_test_set_fused_grid -- launch the one-launch step kernels
 * (fp8_downproj_fwd, _ex, _noalloc) with `ctas` CTAs instead of one per SM
 * (rounded down to whole CTA pairs when the kernel runs on pairs).  The
 * kernel's CTAs take their quantize and weight-cast work by ticket, so any
 * grid gives the same results: a smaller one, and a larger one whose last
 * CTAs can only start once earlier ones have finished.  0 restores the
 * default.  Returns FP8Q_ERR_SHAPE unless 0 <= ctas <= 65535.
 */
int fp8q_test_set_fused_grid(int ctas);

/*
 * fp8q_test_set_fused_layout -- pin the layout of the one-launch step's
 * quantize warps: 1 = quantize-first (24 warps, 8 loads in flight each),
 * 2 = GEMM-first (9 working warps, none on the MMA issuer's scheduler, 16
 * loads in flight each, 4-row units; taken on 256- and 400-wide pair tiles only, else
 * layout 1), 0 = chosen by N (GEMM-first for N above ~1430, where the step's
 * GEMM outlasts its quantize).  The layouts give identical results.  Returns
 * FP8Q_ERR_UNSUPPORTED unless 0 <= layout <= 2.
 */
int fp8q_test_set_fused_layout(int layout);

/*
 * fp8q_test_gemm_tile -- the tile (*pair: 1 = 2-SM pair, 0 = one CTA; *bn:
 * its width) that the one-launch step (fused != 0) or fp8_gemm_fwd (fused ==
 * 0) takes at M x N under the current tile override, so a profile of a
 * smaller M can pin the full size's tile with fp8q_gemm_set_tile.  Needs a
 * device (the choice depends on its SM count).  Errors: FP8Q_ERR_NULL,
 * FP8Q_ERR_SHAPE (M < 1 or N < 16).
 */
int fp8q_test_gemm_tile(int64_t M, int64_t N, int fused, int* pair, int* bn);

/*
 * fp8q_test_noalloc_fill -- fill every byte of the static counter array of
 * fp8_downproj_fwd_noalloc on the current device with `byte` (stream-ordered
 * on `stream`), as a call that was cut short could leave it.  The next
 * fp8_downproj_fwd_noalloc call must clear what it uses before its kernel
 * starts; the test suite checks that it does.
 */
int fp8q_test_noalloc_fill(int byte, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_TESTING_H */
