/*
 * fp8q.h -- C ABI of libfp8q.so: the forward FP8 MLP down-projection on one
 * NVIDIA GB300 (sm_103a).
 *
 * The path, per training step:
 *   1. fp8_quant_fused      BF16 pre-activation H -> act(H) in registers ->
 *                           BF16 copy for backward + FP8 copy + amax
 *   2. fp8_gemm_fwd         Y = X_q W_q / (s_x s_w), FP32 accumulate, BF16 out
 *      (fp8_downproj_fwd    1 and 2 fused in one kernel)
 *      (fp8_downproj_fwd_ex the weight cast, 1, 2 and 3 in one kernel)
 *   3. amax_history_update  push this step's amax; scale for the next step
 *      (fp8_gemm_fwd_update 2 and 3 in one launch: the GEMM runs the updates)
 *   (fp8_gemm_dgrad         dX = dY_q W_q^T / (s_dy s_w), the gradient shape)
 *   (fp8_gemm_wgrad         dW = X_q^T dY_q / (s_x s_dy), the weight gradient)
 *   (fp8_upproj_fwd         the preceding up-projection with 1 in its epilogue)
 *   (fp8_gemm_dgrad_act     dgrad with the activation backward in its epilogue)
 *   (fp8_quant_mx,          MXFP8: 32-value blocks with power-of-two scales,
 *    fp8_gemm_mx             on the block-scaled tensor cores)
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers to caller-owned memory; the
 *    library allocates nothing, frees nothing and never synchronises.  Work is
 *    enqueued on `stream` (0 = the legacy default stream) and the call returns
 *    as soon as it is enqueued.
 *  - Matrices are row-major and densely packed (leading dimension = number of
 *    columns).  Tensor pointers must be 16-byte aligned.
 *  - FP8 tensors are raw bytes (E4M3 "fn" variant: max 448, no infinity;
 *    E5M2: IEEE-like, max 57344).  BF16 tensors are raw 16-bit patterns.
 *  - Scales are multipliers: q = FP8(x * s); dequantisation divides by s.
 *  - Return value: FP8Q_OK, or an fp8q_status describing the first argument
 *    error found (detected on the host, before anything is enqueued), or
 *    FP8Q_ERR_CUDA when a CUDA call or a launch fails.  Conditions only the
 *    GPU can see are OR-ed as FP8Q_DEV_* bits into the caller's optional
 *    device status word.  No call aborts the process or traps the GPU.
 *  - Test and tuning hooks are declared apart, in fp8q_testing.h.
 *
 * Sources (page title, section):
 *  [fused]  "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT
 *           Records", second paragraph -- one fused kernel writes the BF16
 *           copy needed for backward, emits the FP8 copy and keeps running
 *           maxima; the scale uses the previous step's maximum times a safety
 *           margin, so the large tensor is never reread.
 *  [scale]  "FP8 training: what it is and how it works", Step 2 -- scale =
 *           format max / amax; Step 1 -- E4M3 for activations and weights,
 *           E5M2 for gradients; Step 3 -- FP8 inputs, a wider running sum.
 *  [tiles]  same page, Trade-offs and edge cases -- amax computed online per
 *           1x128 activation tile and per 128x128 weight block.
 *  [mx]     same page, Trade-offs and edge cases -- MXFP8 (Blackwell): one
 *           power-of-two scale per block of 32 adjacent values.
 *  [gemms]  "FP8 Training & Inference", FP8 Training Recipe -- Y = X x W in
 *           E4M3; dX = dY x W^T with dY in E5M2 and W in E4M3; Per-Tensor
 *           Scaling for FP8 -- the scales are factored out of the matmul and
 *           the output is rescaled to BF16/FP32; Delayed Scaling -- use the
 *           previous iteration's maximum.
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8Q_OK = 0,
    FP8Q_ERR_NULL = 1,        /* a required pointer is NULL                       */
    FP8Q_ERR_ALIGN = 2,       /* a tensor pointer is not 16-byte aligned          */
    FP8Q_ERR_SHAPE = 3,       /* a size is out of range or breaks a multiple rule */
    FP8Q_ERR_UNSUPPORTED = 4, /* bad enum value, or the device is not sm_103      */
    FP8Q_ERR_CUDA = 5         /* a CUDA call or kernel launch failed              */
} fp8q_status;

/* Bits OR-ed into the optional device status word. */
#define FP8Q_DEV_TIMEOUT 1  /* a bounded wait inside the GEMM gave up; output invalid */
#define FP8Q_DEV_BAD_AMAX 2 /* history update kept the previous scale (amax 0/inf/NaN) */

typedef enum { FP8Q_E4M3 = 0, FP8Q_E5M2 = 1 } fp8q_format;
typedef enum { FP8Q_ACT_IDENTITY = 0, FP8Q_ACT_RELU = 1, FP8Q_ACT_RELU2 = 2 } fp8q_act;

/* Width of one scale group along the contraction dimension. */
#define FP8Q_GROUP 128

/*
 * fp8_quant_fused -- fused activation + BF16 copy + FP8 cast + amax  [fused]
 *
 * For every element of the BF16 tensor h [M,K]:
 *     a   = act(h)            ReLU(h) = h > 0 ? h : +0;  ReLU^2 = ReLU(h)^2
 *     abf = BF16(a)           round to nearest even          -> act_out[i,k]
 *     v   = float32(abf * s)                                  (s: see below)
 *     q   = FP8(v)            round to nearest even, saturate to +-max
 *                                                            -> q_out[i,k]
 *                                                            -> q_t_out[k,i]
 *     amax_out  = max |abf| over the tensor (exact: a BF16 value)
 *     sat_count = #{ |v| > format max }
 *
 * Scale modes:
 *   group_scales_out == NULL  per-tensor: s = *scale (device, 1 float; the
 *                             delayed scale of [fused]/[gemms]).
 *   group_scales_out != NULL  group mode [tiles]: blocks of group_rows x 128
 *                             elements (group_rows = 1: 1x128 activation
 *                             tiles; 128: 128x128 weight blocks).  Each block
 *                             gets s_g = float32(max / amax_g), 1 for an
 *                             all-zero block, clamped to FLT_MAX; written to
 *                             group_scales_out[ceil(M/group_rows), K/128].
 *                             `scale` is ignored (may be NULL).  K % 128 == 0.
 *
 * Arguments:
 *   h                 device [M,K] BF16, 16-byte aligned.  Required unless M == 0.
 *   M, K              M >= 0, K >= 16, K % 16 == 0.  M == 0 only zeroes
 *                     amax_out and sat_count.
 *   act, fmt          fp8q_act, fp8q_format.
 *   act_out           device [M,K] BF16 or NULL (W and dY casts skip it).
 *   q_out             device [M,K] FP8 or NULL.
 *   q_t_out           device [K,M] FP8 (transposed copy) or NULL; needs
 *                     M % 16 == 0.  Used for the weight: W [K,N] is cast to
 *                     W^T [N,K], the forward GEMM's K-major operand.
 *   amax_out          device float or NULL; zeroed by this call, stream-ordered.
 *   sat_count         device uint64 or NULL; zeroed by this call.
 *   stream            CUDA stream.
 * The tensors must not overlap each other.
 */
int fp8_quant_fused(const void* h, int64_t M, int64_t K, int act, int fmt,
                    const float* scale,
                    void* act_out, void* q_out, void* q_t_out,
                    float* amax_out, unsigned long long* sat_count,
                    float* group_scales_out, int group_rows,
                    cudaStream_t stream);

/* Flags of fp8_quant_fused_ex. */
#define FP8Q_ACCUMULATE 1 /* fold into amax_out / sat_count instead of zeroing them first */

/*
 * fp8_quant_fused_ex -- fp8_quant_fused with flags.
 *
 * FP8Q_ACCUMULATE: amax_out and sat_count are not zeroed; this call's
 * maximum and count are folded into the values already there.  A caller that
 * quantizes a tensor in row blocks (to overlap each block's GEMM with the
 * next block's quantize) zeroes on the first block and accumulates on the
 * rest, and the result equals one call over the whole tensor.  flags = 0 is
 * fp8_quant_fused.  Unknown flag bits give FP8Q_ERR_UNSUPPORTED.
 */
int fp8_quant_fused_ex(const void* h, int64_t M, int64_t K, int act, int fmt,
                       const float* scale,
                       void* act_out, void* q_out, void* q_t_out,
                       float* amax_out, unsigned long long* sat_count,
                       float* group_scales_out, int group_rows,
                       unsigned flags, cudaStream_t stream);

/*
 * fp8_quant_fused_batch -- several per-tensor fp8_quant_fused_ex calls in one
 * kernel launch  [fused][scale]
 *
 * The same per-element arithmetic as fp8_quant_fused ("Paradigma Details FP8
 * and Optimizer Tricks Behind NanoGPT Records", second paragraph; "FP8
 * training: what it is and how it works", Step 4: the weight's 8-bit copy is
 * cast from the master copy at every step), applied to n tensors by one grid:
 * the CTAs of args[0] come first, then those of args[1], and so on.  A
 * training step casts its weight (transposed copy, identity activation) and
 * quantizes its activation together, so the GEMM that follows waits on one
 * kernel instead of two.
 *   args[i]   the arguments of one fp8_quant_fused_ex call (fields of the same
 *             names and meaning); group_scales_out must be NULL (per-tensor
 *             scales only), flags 0 or FP8Q_ACCUMULATE.
 *   n         1 .. FP8Q_BATCH_MAX.
 * Results equal the n separate calls.  The tensors run concurrently, so no
 * entry may read what another entry writes, and outputs must not overlap.
 * Every entry is checked before anything is enqueued: the first failing
 * entry's status is returned and nothing runs.  amax_out / sat_count of an
 * entry without FP8Q_ACCUMULATE are zeroed (stream-ordered) before the launch.
 *
 * The pre-activation's FP8 cache ("FP8 training: what it is and how it
 * works", Trade-offs and edge cases: the activations kept for the backward
 * pass are stored in FP8): with hq_out set, the same pass also writes
 *     hq_out[i,k] = E4M3(float32(h[i,k] * s_h))   (h: the BF16 INPUT, before
 *                                                   the activation; s_h = *scale_h)
 * and folds max |h| into amax_h and #{|h * s_h| > 448} into sat_h (both
 * optional; zeroed first unless FP8Q_ACCUMULATE), so that a backward needing
 * act'(H) (fp8_gemm_dgrad_act_q) reads one byte per element instead of H's
 * two.  hq_out [M,K] bytes, 16-byte aligned; scale_h required with it.
 */
#define FP8Q_BATCH_MAX 4
typedef struct fp8q_quant_args {
    const void* h;
    int64_t M, K;
    int act, fmt;
    const float* scale;
    void* act_out;
    void* q_out;
    void* q_t_out;
    float* amax_out;
    unsigned long long* sat_count;
    float* group_scales_out;
    int group_rows;
    unsigned flags;
    void* hq_out;                   /* or NULL: the FP8 cache of the pre-activation (see below) */
    const float* scale_h;
    float* amax_h;
    unsigned long long* sat_h;
} fp8q_quant_args;
int fp8_quant_fused_batch(const fp8q_quant_args* args, int n, cudaStream_t stream);

/*
 * fp8_cast_f32 -- FP32 -> FP8, elementwise: q[i] = FP8(x[i])  [cast]
 *
 * The conversion every quantize call applies to its scaled value v = BF16(act(h))
 * * s ("FP8 training: what it is and how it works", Step 2: round to the nearest
 * representable value; Trade-offs and edge cases: saturate instead of
 * overflowing), exposed on its own so that it can be checked against the
 * formats' definition over all 2^32 inputs.  Round to nearest even; finite
 * values beyond the largest finite code and infinities give that code with the
 * input's sign (448 for E4M3, 57344 for E5M2); NaN gives a NaN code.
 *   x     device [n] float32, 16-byte aligned.
 *   q     device [n] bytes (E4M3 or E5M2 codes), 16-byte aligned.
 *   n     >= 0 (0: nothing is enqueued).
 *   fmt   FP8Q_E4M3 or FP8Q_E5M2.
 * Errors: FP8Q_ERR_SHAPE (n < 0), FP8Q_ERR_UNSUPPORTED (fmt, or not sm_103),
 * FP8Q_ERR_NULL, FP8Q_ERR_ALIGN, FP8Q_ERR_CUDA (launch).
 */
int fp8_cast_f32(const float* x, void* q, int64_t n, int fmt, cudaStream_t stream);

/*
 * fp8_gemm_fwd --Y = (X_q . W_q) / (s_x s_w), FP32 accumulation, BF16 out  [gemms][scale]
 *
 *   x_q     device [M,K] E4M3 (the activation, K contiguous).
 *   wt_q    device [N,K] E4M3: the weight W [K,N] stored transposed, i.e. the
 *           q_t_out of fp8_quant_fused run on W.
 *   scale_x, scale_w
 *           group_mode 0: device, 1 float each (the scales X and W were cast with).
 *           group_mode 1: scale_x = device [M, K/128] (1x128 tiles of X),
 *                         scale_w = device [K/128, ceil(N/128)] (128x128 blocks
 *                         of W [K,N]); each 128-long slice of the contraction
 *                         is rescaled by its own pair before it is added to the
 *                         FP32 sum.  Needs K % 128 == 0.
 *   y       device [M,N] BF16:  y[i,j] = BF16( (sum_k x[i,k] w[k,j]) / (s_x s_w) ).
 *   M, N, K M >= 0 (M == 0: nothing is enqueued; x_q and y may then be
 *           NULL); N >= 16, N % 16 == 0; K >= 16, K % 16 == 0.
 *   status  device int or NULL: FP8Q_DEV_TIMEOUT is OR-ed in if a bounded
 *           internal wait gives up (the kernel then exits cleanly; y is invalid).
 * Runs on tcgen05 tensor cores with TMA-fed shared-memory tiles; needs sm_103.
 */
int fp8_gemm_fwd(const void* x_q, const void* wt_q,
                 const float* scale_x, const float* scale_w, int group_mode,
                 void* y, int64_t M, int64_t N, int64_t K,
                 int* status, cudaStream_t stream);

/*
 * fp8_gemm_dgrad -- dX = (dY_q . W_q^T) / (s_dy s_w), FP32 accumulation, BF16 out  [gemms]
 *
 *   dy_q    device [M,N] E5M2 (the output gradient, N contiguous).
 *   w_q     device [K,N] E4M3: the weight in its own layout (q_out of
 *           fp8_quant_fused run on W).
 *   scale_dy, scale_w  device, 1 float each.
 *   dx      device [M,K] BF16:  dx[i,k] = BF16( (sum_n dy[i,n] w[k,n]) / (s_dy s_w) ).
 *   M, N, K M >= 0 (M == 0: nothing is enqueued); N >= 16, N % 16 == 0 (the
 *           contraction); K >= 16, K % 16 == 0.
 *   status  as for fp8_gemm_fwd.
 */
int fp8_gemm_dgrad(const void* dy_q, const void* w_q,
                   const float* scale_dy, const float* scale_w,
                   void* dx, int64_t M, int64_t N, int64_t K,
                   int* status, cudaStream_t stream);

/*
 * fp8_gemm_dgrad_act -- dH = dX * act'(H): the activation backward in the dgrad epilogue  [gemms][fused]
 *
 * dX = (dY_q . W_q^T) / (s_dy s_w) as in fp8_gemm_dgrad, multiplied in the
 * epilogue, while still in FP32, by the derivative of the activation at the
 * BF16 pre-activation H ("Paradigma Details FP8 and Optimizer Tricks Behind
 * NanoGPT Records", second paragraph: the activation whose BF16 copy the
 * forward keeps): act'(h) = 2 max(h, 0) for ReLU^2, (h > 0) for ReLU, 1 for
 * identity.  dX itself never reaches HBM.
 *   dy_q, w_q, scale_dy, scale_w, M, N, K, status  as for fp8_gemm_dgrad.
 *   h       device [M,K] BF16: the pre-activation (16-byte aligned).
 *   act     FP8Q_ACT_IDENTITY, FP8Q_ACT_RELU or FP8Q_ACT_RELU2.
 *   dh      device [M,K] BF16:  dh[i,k] = BF16( dX[i,k] (float32) * act'(h[i,k]) ).
 */
int fp8_gemm_dgrad_act(const void* dy_q, const void* w_q,
                       const float* scale_dy, const float* scale_w,
                       const void* h, int act, void* dh, int64_t M, int64_t N, int64_t K,
                       int* status, cudaStream_t stream);

/*
 * fp8_gemm_dgrad_act_q -- fp8_gemm_dgrad_act with the pre-activation read from
 * its FP8 cache  [gemms][fused]
 *
 * "FP8 training: what it is and how it works", Trade-offs and edge cases: the
 * activations kept for the backward pass are stored in FP8.  H is not kept in
 * BF16: the forward's quantize (fp8q_quant_args.hq_out) wrote h_q =
 * E4M3(float32(h * s_h)), and the derivative is taken at its dequantised value
 *     h~ = dec(h_q) * float32(1 / s_h)        (float32)
 *     dh[i,k] = BF16( dX[i,k] (float32) * act'(h~) ),  act' as in
 *     fp8_gemm_dgrad_act (2 max(h~, 0), (h~ > 0), or 1)
 * so the epilogue reads one byte per element of H instead of two.
 *   dy_q, w_q, scale_dy, scale_w, act, dh, M, N, K, status  as for fp8_gemm_dgrad_act.
 *   h_q      device [M,K] E4M3 (16-byte aligned).
 *   scale_h  device float: the scale h_q was cast with.
 */
int fp8_gemm_dgrad_act_q(const void* dy_q, const void* w_q, const float* scale_dy, const float* scale_w,
                         const void* h_q, const float* scale_h, int act, void* dh, int64_t M, int64_t N, int64_t K,
                         int* status, cudaStream_t stream);

/*
 * fp8_gemm_wgrad -- dW = (X_q^T . dY_q) / (s_x s_dy), FP32 accumulation, BF16 out  [gemms]
 *
 * The weight gradient of the same layer ("FP8 Training & Inference", FP8
 * Training Recipe: the weight-gradient GEMM takes the E4M3 activation and the
 * E5M2 output gradient).  Both operands are contracted over the M tokens, so
 * both come as their transposed, token-contiguous copies: q_t_out of
 * fp8_quant_fused run on H (the activation) and on dY.
 *   x_q_t   device [K,M] E4M3: the activation's transposed copy.
 *   dy_q_t  device [N,M] E5M2: the output gradient's transposed copy.
 *   scale_x, scale_dy  device, 1 float each.
 *   dw      device [K,N] BF16:  dw[k,n] = BF16( (sum_m x[m,k] dy[m,n]) / (s_x s_dy) ).
 *   M, N, K M >= 16, M % 16 == 0 (the contraction); N >= 16, N % 16 == 0;
 *           K >= 0 (K == 0: nothing is enqueued).
 *   status  as for fp8_gemm_fwd.
 */
int fp8_gemm_wgrad(const void* x_q_t, const void* dy_q_t,
                   const float* scale_x, const float* scale_dy,
                   void* dw, int64_t M, int64_t N, int64_t K,
                   int* status, cudaStream_t stream);

/*
 * fp8_upproj_fwd -- the up-projection GEMM with the activation quantize in its epilogue  [fused][gemms]
 *
 * "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records", second
 * paragraph: the activation and the cast run while the preceding computation
 * still holds its output in registers.  Here that computation is the FP8
 * up-projection H = X_q . W_q / (s_x s_w) itself, so H reaches HBM only if
 * asked for.  Per element of the [M,N] output:
 *   h = BF16(acc / (s_x s_w));  a = act(h) (float32);  a_bf = BF16(a);
 *   h_q = E4M3(float32(a_bf * s_h)) (round to nearest even, saturating);
 *   amax = max |a_bf|;  sat_count += (|a_bf * s_h| > 448)
 * -- fp8_quant_fused applied to the GEMM's BF16 output, without storing it.
 *   x_q, wt_q, scale_x, scale_w   as for fp8_gemm_fwd (per-tensor scales).
 *   act      FP8Q_ACT_IDENTITY, FP8Q_ACT_RELU or FP8Q_ACT_RELU2.
 *   scale_h  device, 1 float: s_h, the activation's (delayed) scale.
 *   h_out    device [M,N] BF16 or NULL: H itself.
 *   act_out  device [M,N] BF16 or NULL: the activation copy kept for backward.
 *   h_q      device [M,N] E4M3 (required): the next GEMM's operand.
 *   amax_out, sat_count  device float / uint64 or NULL; zeroed by the call
 *            (stream-ordered) unless flags has FP8Q_ACCUMULATE.
 *   M, N, K  as for fp8_gemm_fwd; the E4M3 rows are N bytes (N % 16 == 0).
 *   flags    0 or FP8Q_ACCUMULATE.
 *   status   as for fp8_gemm_fwd.
 */
int fp8_upproj_fwd(const void* x_q, const void* wt_q, const float* scale_x, const float* scale_w,
                   int act, const float* scale_h, void* h_out, void* act_out, void* h_q,
                   float* amax_out, unsigned long long* sat_count, int64_t M, int64_t N, int64_t K,
                   unsigned flags, int* status, cudaStream_t stream);

/*
 * fp8_downproj_fwd -- the fused quantize + forward GEMM in one kernel  [fused][gemms]
 *
 * Computes exactly what fp8_quant_fused(h, act, E4M3, scale_x, act_out, x_q,
 * amax_out, sat_count) followed by fp8_gemm_fwd(x_q, wt_q, scale_x, scale_w, y)
 * compute, in one persistent kernel: extra warps of every CTA quantize H a
 * few rows at a time and count finished rows per 128-row block in `workspace`;
 * the GEMM loads a tile's rows of x_q once their block is complete, so the
 * GEMM of early rows overlaps the quantize of later ones and the large tensor
 * is read once.  act_out, amax_out, sat_count may be NULL; x_q is required
 * (it is the GEMM's operand and the E4M3 copy).
 *   workspace  device scratch of at least fp8_downproj_workspace_bytes(M)
 *              bytes, 4-byte aligned, owned by the caller; zeroed by this call
 *              (stream-ordered), and left zero by the kernel when it
 *              finishes.  Two fused calls must not share it concurrently.
 * The kernel launches one CTA per SM.  Its CTAs take quantize (and weight
 * cast) work by ticket from counters in the workspace, so a CTA only ever
 * waits for work that a running CTA has taken: the kernel also completes
 * when other work holds some SMs and only part of its grid is resident.
 * Waits are bounded all the same (a wait that runs out sets
 * FP8Q_DEV_TIMEOUT).
 * Same shape, alignment and error rules as fp8_quant_fused / fp8_gemm_fwd.
 */
size_t fp8_downproj_workspace_bytes(int64_t M);
int fp8_downproj_fwd(const void* h, const void* wt_q, int64_t M, int64_t N, int64_t K, int act,
                     const float* scale_x, const float* scale_w,
                     void* act_out, void* x_q, float* amax_out, unsigned long long* sat_count,
                     void* y, void* workspace, size_t workspace_bytes,
                     int* status, cudaStream_t stream);

/*
 * fp8_downproj_fwd_ex -- the whole forward step's casts and GEMM in one kernel
 * [fused][gemms], with the weight cast folded in and no clearing ahead of it
 *
 * As fp8_downproj_fwd, plus:
 *   w        device W [K,N] BF16 (the master weight), or NULL.  When set, the
 *            kernel first casts it exactly as fp8_quant_fused(w, K, N,
 *            IDENTITY, E4M3, scale_w, q_out = w_q, q_t_out = wt_q, amax_out =
 *            amax_w) would ("FP8 training: what it is and how it works", Step
 *            4: the 8-bit weight copy is cast from the master copy every
 *            step), and the GEMM reads the W_q^T it wrote: wt_q is then an
 *            OUTPUT.  When NULL, wt_q is the GEMM's input as before and w_q,
 *            amax_w are ignored.
 *   w_q      device [K,N] E4M3 (the dgrad operand) or NULL.
 *   amax_w   device float or NULL: max |W|.
 *   sat_w    device uint64 or NULL: the weight cast's count of |W * s_w| >
 *            448, i.e. of values its scale saturated (the overflow test of
 *            detect-and-recompute).  Needs w, like amax_w.
 *   flags    0, or FP8Q_ACCUMULATE: nothing is zeroed before the kernel
 *            (amax_x, sat_count, amax_w, sat_w fold into their values; the workspace
 *            must already be zero -- zero-filled before first use, then kept
 *            zero by the kernel).  After a call that reported FP8Q_DEV_TIMEOUT
 *            the workspace may hold counts: zero it again.
 *   hist_x, hist_w  NULL, or the arguments of amax_history_update_ex for X
 *            (amax_new = amax_x) and for W (amax_new = amax_w; needs w): the
 *            last CTA of the kernel runs these updates on the final amax
 *            values, so a delayed-scaling step is this one launch.  The
 *            structs are read during the call only.  Need M > 0.
 * Results equal fp8_quant_fused_ex on W and H followed by fp8_gemm_fwd (and
 * amax_history_update_ex on X and W).  FP8Q_ERR_SHAPE also when W has more
 * than 2^31 units of 8 x 256 values.
 */
typedef struct fp8q_history_args {
    float* history;                 /* as amax_history_update_ex            */
    int L;
    int* head;
    float margin;
    int fmt;
    const float* scale_prev;        /* or NULL                               */
    float* scale_out;
    int* status;                    /* or NULL                               */
    float* amax_clear;              /* or NULL                               */
    unsigned long long* sat_clear;  /* or NULL                               */
} fp8q_history_args;
int fp8_downproj_fwd_ex(const void* h, const void* w, void* wt_q, int64_t M, int64_t N, int64_t K,
                        int act, const float* scale_x, const float* scale_w,
                        void* act_out, void* x_q, float* amax_x, unsigned long long* sat_count,
                        void* w_q, float* amax_w, unsigned long long* sat_w, void* y,
                        void* workspace, size_t workspace_bytes,
                        const fp8q_history_args* hist_x, const fp8q_history_args* hist_w,
                        unsigned flags, int* status, cudaStream_t stream);

/*
 * fp8_gemm_fwd_update -- fp8_gemm_fwd (per-tensor scales) that also runs the
 * step's delayed-scale updates  [gemms][scale]
 *
 * The same Y = (X_q . W_q) / (s_x s_w).  In addition, one warp of the first
 * CTA runs amax_history_update_ex with hist_x on amax_x and with hist_w on
 * amax_w while the first tile's products accumulate ("Paradigma Details FP8
 * and Optimizer Tricks Behind NanoGPT Records", second paragraph: the next
 * step's scale comes from this step's maximum, so it is computed beside this
 * step's GEMM and nothing waits for it).  The amax values must be final when
 * the GEMM starts (the casts that wrote them enqueued before it on `stream`).
 *   x_q, wt_q, scale_x, scale_w, y, M, N, K, status  as for fp8_gemm_fwd with
 *           group_mode 0.
 *   amax_x, hist_x / amax_w, hist_w  device float and the arguments of
 *           amax_history_update_ex for that tensor (amax_new = the float), or
 *           NULL history arguments for no update.  An update must write a
 *           scale other than scale_x and scale_w, and clear an amax other than
 *           amax_x and amax_w (the two-slot layout: this step's scales are
 *           read while the next step's are written).  The structs are read
 *           during the call only.
 * Results equal fp8_gemm_fwd followed by the amax_history_update_ex calls.
 * Errors: those of fp8_gemm_fwd and amax_history_update_ex; FP8Q_ERR_SHAPE
 * for an update that would write scale_x / scale_w or clear amax_x / amax_w,
 * or for M == 0 with an update (nothing is launched to run it).
 */
int fp8_gemm_fwd_update(const void* x_q, const void* wt_q,
                        const float* scale_x, const float* scale_w,
                        void* y, int64_t M, int64_t N, int64_t K,
                        float* amax_x, const fp8q_history_args* hist_x,
                        float* amax_w, const fp8q_history_args* hist_w,
                        int* status, cudaStream_t stream);

/*
 * fp8_downproj_fwd_noalloc -- fp8_downproj_fwd without a caller workspace
 *
 * No counterpart in the method's sources: a variant for callers that must
 * not allocate device memory.  Such callers include a plugin that a host
 * application hands only its input and output buffers (the host owns every
 * other byte of device memory under a fixed budget); code on a latency path,
 * where cudaFree (and, when the pool must grow, cudaMalloc) synchronizes the
 * whole device and stalls other streams; and code that runs while a stream is
 * being captured, where allocation calls are not allowed.
 *
 * Same arguments, results and error rules as fp8_downproj_fwd, minus
 * `workspace`: the kernel's counters (per-block ready counts, work tickets)
 * live in a fixed array of this library's own device memory
 * (FP8Q_NOALLOC_MAX_M / 128 + 64 counters, 8,448 bytes), which every device
 * that loads the library holds until the process exits.
 *   M > FP8Q_NOALLOC_MAX_M  -> FP8Q_ERR_SHAPE (use fp8_downproj_fwd)
 * The call allocates nothing: no cudaMalloc / cudaFree, no allocating
 * library routine.  Every call with M > 0 looks the array's address up
 * (cudaGetSymbolAddress, on the current device), so the address stays right
 * after a device reset, when the library's device code is loaded again in
 * a new context.  The first call on a device is also the one that loads that
 * code there if nothing else has: make it before any stream capture.  Every
 * call clears the counters it uses (stream-ordered) before its kernel
 * starts, since the array keeps what the previous call left.  All calls on a
 * device share the one array: calls that overlap on the GPU race on it and
 * give wrong results, so order them on one stream (or with events).
 */
#define FP8Q_NOALLOC_MAX_M 262144
int fp8_downproj_fwd_noalloc(const void* h, const void* wt_q, int64_t M, int64_t N, int64_t K, int act,
                             const float* scale_x, const float* scale_w,
                             void* act_out, void* x_q, float* amax_out, unsigned long long* sat_count,
                             void* y, int* status, cudaStream_t stream);

/*
 * fp8_quant_mx -- MXFP8 quantize: one power-of-two scale per 32 adjacent values  [mx]
 *
 * "FP8 training: what it is and how it works", Trade-offs and edge cases: the
 * microscaling recipe gives every block of 32 adjacent values its own scale,
 * and the scales are powers of two.  The pages fix neither which power of two
 * nor how it is stored; here (Step 2's scale = format max / amax, rounded
 * down so that no value of the block saturates):
 *     a = act(h), abf = BF16(a)                     as in fp8_quant_fused
 *     amax_b = max |abf| over the block
 *     s_b = 2^e, e = the largest integer with amax_b * 2^e <= fmt_max,
 *           clamped to [-127, 127]; e = 0 for an all-zero block
 *     q = FP8(float32(abf * s_b))                   (never saturates)
 *     scale byte = 127 - e: the biased 8-bit exponent of the dequantisation
 *           factor 1 / s_b, i.e. the E8M0 scale the block-scaled tensor-core
 *           MMA takes (2^(byte - 127) multiplies the block's codes)
 * Scale layout (both modes; the one fp8_gemm_mx reads): the scale bytes of a
 * block grid of R rows x KB blocks are stored in atoms of 128 rows x 4 blocks,
 * 512 bytes each -- the layout the block-scaled MMA's tensor-memory copy
 * takes, so one copy per 128 rows feeds a GEMM stage of 128 K values:
 *     byte of (row r, block b) = 512 * ((r / 128) * G + b / 4)
 *                                + 16 * (r % 32) + 4 * ((r / 32) % 4) + b % 4,
 *     G = ceil(KB / 4); size fp8_mx_scale_bytes(R, 32 * KB).
 * Blocks KB .. 4G - 1 of a row are padding and are written as 127; bytes of
 * rows past R in the last 128-row atom are left as they were.
 * Two modes, exactly one per call:
 *   rows:     blocks run along the rows of h [M,K] (K % 32 == 0, M * K / 32 <
 *             2^32): q_out [M,K] codes, sf_out the scale layout of the
 *             [M, K/32] grid, act_out [M,K] BF16 or NULL.  The activation X of
 *             the forward GEMM.
 *   columns:  blocks run down the columns of h [M,K] (M % 32 == 0), and the
 *             codes are written transposed: q_t_out [K,M], sf_t_out the scale
 *             layout of the [K, M/32] grid (block b of row k of the copy covers
 *             h[32b .. 32b + 31, k]).  The weight W [K_w, N_w] of the forward
 *             GEMM: its copy W_q^T [N_w, K_w] is the GEMM's K-major operand with
 *             blocks along K_w.  act_out must be NULL.
 *   amax_out, sat_count  device float / uint64 or NULL; zeroed by the call
 *             (sat_count counts |abf * s_b| > fmt_max: 0 for finite inputs).
 * Errors: FP8Q_ERR_UNSUPPORTED for both or neither mode, act_out in column
 * mode, a bad act or fmt, or no sm_103 device; FP8Q_ERR_NULL for a missing
 * output of the chosen mode; FP8Q_ERR_SHAPE for M < 0, (row mode) K < 32 or
 * K % 32 != 0, (column mode) M % 32 != 0, K < 16, K % 16 != 0 or
 * K > 4,194,240 (65535 tiles of 64 columns), (row mode) M * K / 32 >= 2^32;
 * FP8Q_ERR_ALIGN for tensors (scale arrays included) not 16-byte aligned.
 */
int fp8_quant_mx(const void* h, int64_t M, int64_t K, int act, int fmt, void* act_out, void* q_out,
                 uint8_t* sf_out, void* q_t_out, uint8_t* sf_t_out, float* amax_out,
                 unsigned long long* sat_count, cudaStream_t stream);

/*
 * fp8_gemm_mx -- the MXFP8 GEMM on the block-scaled tensor cores  [mx][gemms]
 *
 *   y[i,j] = BF16( sum_k dec(x_q[i,k]) 2^(sf_x[i, k/32] - 127)
 *                        dec(wt_q[j,k]) 2^(sf_w[j, k/32] - 127) )
 * with FP32 accumulation; the scales are applied by the MMA
 * (tcgen05.mma.kind::mxf8f6f4.block_scale), block by block.
 *   x_q     device [M,K] codes (fmt_x), K contiguous: the rows-mode output of
 *           fp8_quant_mx.
 *   sf_x    device scale bytes of x_q's [M, K/32] block grid in the tiled
 *           layout of fp8_quant_mx (fp8_mx_scale_bytes(M, K) bytes).
 *   wt_q    device [N,K] codes (fmt_w): the column-mode output of
 *           fp8_quant_mx run on W [K,N].
 *   sf_w    device scale bytes of wt_q's [N, K/32] grid, the same layout
 *           (fp8_mx_scale_bytes(N, K) bytes).
 *   y       device [M,N] BF16.
 *   M, N, K 0 <= M <= 2^31 - 256 (0: nothing is enqueued); N >= 16,
 *           N % 16 == 0; K >= 32, K % 32 == 0.
 *   fmt_x, fmt_w  FP8Q_E4M3 or FP8Q_E5M2.
 *   status  device int or NULL: FP8Q_DEV_TIMEOUT if a bounded wait gave up.
 * Errors: FP8Q_ERR_UNSUPPORTED for a bad format or no sm_103 device;
 * FP8Q_ERR_NULL for a missing pointer; FP8Q_ERR_SHAPE for the sizes above;
 * FP8Q_ERR_ALIGN for x_q, wt_q, y, sf_x or sf_w not 16-byte aligned.
 */
int fp8_gemm_mx(const void* x_q, const uint8_t* sf_x, const void* wt_q, const uint8_t* sf_w, void* y,
                int64_t M, int64_t N, int64_t K, int fmt_x, int fmt_w, int* status, cudaStream_t stream);

/*
 * fp8_mx_scale_bytes -- size of the MX scale layout  [mx]
 *
 * Bytes of the tiled scale layout (fp8_quant_mx) of a block grid of `rows`
 * rows x K/32 blocks: ceil(rows / 128) * ceil(K / 128) * 512.  Host only;
 * returns -1 for rows < 0, K < 0 or K % 32 != 0.
 */
int64_t fp8_mx_scale_bytes(int64_t rows, int64_t K);

/*
 * amax_history_update -- delayed per-tensor scale for the next step  [fused][gemms]
 *
 * history[0..L-1] (device floats) is a ring whose newest entry is
 * history[*head] (device int).  One call, in stream order:
 *     *head = (*head + 1) % L;  history[*head] = *amax_new;
 *     amax_ref = max(history[0..L-1]);
 *     s = float32( fmt_max / float32(margin * amax_ref) );
 *     *scale_out = s                 if amax_ref and s are positive and finite,
 *     otherwise *scale_out is left as it was and FP8Q_DEV_BAD_AMAX is OR-ed
 *     into *status (when status != NULL).
 * With L = 1 the scale depends on the previous step's amax alone.
 *   L         1 <= L <= 4096.
 *   margin    host float, positive and finite (multiplicative safety margin).
 *   fmt       fp8q_format (fmt_max = 448 or 57344).
 */
int amax_history_update(float* history, int L, int* head, const float* amax_new,
                        float margin, int fmt, float* scale_out, int* status,
                        cudaStream_t stream);

/*
 * amax_history_update_ex -- amax_history_update for a step that keeps its
 * scale, amax and saturation count in two alternating slots  [fused][gemms]
 *
 * The same update, plus, in the same launch:
 *   scale_prev  device float or NULL.  When the amax is unusable, *scale_out
 *               gets *scale_prev (the scale the step just used) instead of
 *               being left alone, so scale_out may be the other slot.
 *   amax_clear  device float or NULL: set to 0 (the next step's cast folds
 *               its maximum into it).  Must not be amax_new.
 *   sat_clear   device uint64 or NULL: set to 0.
 * amax_history_update(...) is amax_history_update_ex with the three NULL.
 */
int amax_history_update_ex(float* history, int L, int* head, const float* amax_new,
                           float margin, int fmt, const float* scale_prev, float* scale_out,
                           int* status, float* amax_clear, unsigned long long* sat_clear,
                           cudaStream_t stream);

/* Human-readable name of an fp8q_status value (static string). */
const char* fp8q_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int fp8q_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
