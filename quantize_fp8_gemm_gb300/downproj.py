"""Host-side driver of one FP8 down-projection step (device buffers + order of calls).

One training step of the forward FP8 MLP down-projection, as the pages lay it
out ("Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records",
second paragraph; "FP8 Training & Inference", FP8 Training Recipe and
Delayed Scaling):

    a7  W [K,N] BF16 -> W_q^T [N,K] E4M3 (+ W_q [K,N] for the gradient GEMM)
    a1-a5  H [M,K] BF16 -> ReLU^2 -> BF16 copy + X_q E4M3 + amax (+ saturations)
    a9  Y = X_q W_q / (s_x s_w)  -> BF16 [M,N]
    a6  push amax(X), amax(W) into their histories -> scales for the next step

Every step runs in libfp8q's kernels through the C ABI; this module only owns
the device buffers and issues the calls in order on the current stream.  The
scale a tensor was cast with stays in place until the history update at the
end of the step, so the GEMM dequantises with the scale actually used.
"""
from __future__ import annotations

import torch

from . import binding as B


# Default switch to the one-launch step (per-tensor scales).  On GB300 it beats
# the batched cast + GEMM pair from 16,384 rows (16384 x 4096 -> 1024: 100.0
# against 103.4 us; 16384 x 3072 -> 768: 70.6 against 72.0 us) and loses at
# 8192 (55.4 against 41.3 us at 8192 x 3072 -> 768).
FUSED_MIN_ROWS = 16384

RECOMPUTE_X, RECOMPUTE_W = 1, 2  # recompute_on_overflow(): which operand was cast again


class DelayedScale:
    """Device-resident delayed-scaling state of one tensor role.

    history [L] (ring, newest at ``head``), a status word for FP8Q_DEV_*
    flags, and two slots of (scale, amax, saturation count).  A step casts
    with the current slot's scale into the current slot's amax / count, and
    the GEMM dequantises with that scale, while the history update writes the
    next step's scale into the other slot; the two can therefore run
    concurrently.  ``update()`` also zeroes the other slot's amax and count,
    so the next step's cast can accumulate into them without clearing them
    first, and then makes the other slot current (a host-side switch).
    """

    def __init__(self, fmt: int, margin: float, history_len: int = 1, device="cuda"):
        self.fmt, self.margin, self.L = fmt, float(margin), int(history_len)
        self.history = torch.zeros(self.L, dtype=torch.float32, device=device)
        self.head = torch.zeros(1, dtype=torch.int32, device=device)
        self.scales = torch.ones(2, dtype=torch.float32, device=device)
        self.slot = 0
        self.amaxes = torch.zeros(2, dtype=torch.float32, device=device)
        self.sats = torch.zeros(2, dtype=torch.int64, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.clean = True  # the current slot's amax and count are zero

    @property
    def amax(self) -> torch.Tensor:
        """The amax the next cast writes (current slot)."""
        return self.amaxes[self.slot:self.slot + 1]

    @property
    def sat(self) -> torch.Tensor:
        """The saturation count the next cast writes (current slot)."""
        return self.sats[self.slot:self.slot + 1]

    @property
    def last_amax(self) -> torch.Tensor:
        """The amax the last update() pushed into the history."""
        return self.amaxes[1 - self.slot:2 - self.slot]

    @property
    def last_sat(self) -> torch.Tensor:
        """The saturation count of the cast before the last update()."""
        return self.sats[1 - self.slot:2 - self.slot]

    @property
    def scale(self) -> torch.Tensor:
        """The scale the next cast uses (a 1-element view of the current slot)."""
        return self.scales[self.slot:self.slot + 1]

    @property
    def last_scale(self) -> torch.Tensor:
        """The scale the cast before the last update() used."""
        return self.scales[1 - self.slot:2 - self.slot]

    def update(self) -> None:
        """Push this step's amax; write the next step's scale into the other
        slot (which first takes the current scale, kept if the amax is
        unusable) and make that slot current."""
        o = 1 - self.slot
        B.amax_history_update_ex(self.history, self.head, self.amax, self.margin, self.fmt, self.scales[o:o + 1],
                                 scale_prev=self.scale, status=self.status, amax_clear=self.amaxes[o:o + 1],
                                 sat_clear=self.sats[o:o + 1])
        self.slot ^= 1
        self.clean = True

    def kernel_update_args(self) -> "B.HistoryArgs":
        """The update() of this step as arguments for a kernel that runs it
        itself (fp8_downproj_fwd_ex); call advance() once it is enqueued."""
        o = 1 - self.slot
        return B.history_args(self.history, self.head, self.margin, self.fmt, self.scales[o:o + 1],
                              scale_prev=self.scale, status=self.status, amax_clear=self.amaxes[o:o + 1],
                              sat_clear=self.sats[o:o + 1])

    def advance(self) -> None:
        """The host side of update() when a kernel ran the update."""
        self.slot ^= 1
        self.clean = True

    def seed(self, amax: float) -> None:
        """Start the history from a known previous amax (e.g. a calibration pass)."""
        self.amax.fill_(float(amax))
        self.clean = False
        self.update()


class Fp8DownProj:
    """Buffers and call order for Y = fp8(act(H)) . fp8(W) -> BF16 on one GPU.

    group=False: per-tensor delayed scales for X and W.
    group=True : online 1x128 scales for X and 128x128 block scales for W
                 (needs K % 128 == 0 and N % 128 == 0).
    """

    def __init__(self, M: int, K: int, N: int, *, act: int = B.ACT_RELU2, margin: float = 2.0,
                 history_len: int = 1, group: bool = False, with_dgrad: bool = False,
                 keep_act: bool = True, chunks: int | None = None, fused: bool | None = None,
                 with_backward: bool = False, fp8_cache: bool = False, device="cuda"):
        self.M, self.K, self.N, self.act, self.group = M, K, N, act, group
        self.with_backward = with_backward
        if fp8_cache and not with_backward:
            raise ValueError("fp8_cache keeps the pre-activation for backward(): it needs with_backward")
        self.fp8_cache = fp8_cache
        if with_backward and (group or (chunks or 1) != 1 or fused):
            raise ValueError("backward() runs after the per-tensor one-block step (not fused, not grouped)")
        with_dgrad = with_dgrad or with_backward
        # The fused kernel (W cast + quantize + GEMM + history updates, one
        # launch) serves the per-tensor path in one block.  Measured per step
        # on GB300 (CUDA graph, L2 flushed): it wins on large batches (65,536 x
        # 3072 -> 768: 212 vs 259 us; 131,072 x 6400 -> 1600: 1227 vs 1437 us)
        # and loses at 8,192 rows (47.6 vs 40.6 us), where its last wave of
        # tiles, which waits for the last rows, is not hidden.
        if fused is None:
            fused = not group and (chunks or 1) == 1 and M >= FUSED_MIN_ROWS and not with_backward
        self.fused = fused
        if self.fused and (group or (chunks or 1) != 1):
            raise ValueError("the fused kernel runs the per-tensor path over the whole batch")
        if chunks is None:  # measured on GB300: overlapping row blocks does not pay off
            chunks = 1
        if chunks < 1 or M % chunks or (chunks > 1 and (M // chunks) % 256):
            raise ValueError("chunks must split M into row blocks that are multiples of 256")
        self.chunks = chunks
        dev = device
        self.x = DelayedScale(B.E4M3, margin, history_len, dev)
        self.w = DelayedScale(B.E4M3, margin, history_len, dev)
        self.act_bf16 = torch.empty(M, K, dtype=torch.bfloat16, device=dev) if keep_act else None
        self.x_q = torch.empty(M, K, dtype=torch.uint8, device=dev)
        self.wt_q = torch.empty(N, K, dtype=torch.uint8, device=dev)
        self.w_q = torch.empty(K, N, dtype=torch.uint8, device=dev) if with_dgrad else None
        self.y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        self.gemm_status = torch.zeros(1, dtype=torch.int32, device=dev)
        # recompute_on_overflow(): one-entry histories that turn this step's own
        # amax into a corrected scale, and the scratch amax / count of the re-cast
        self._fix_hist = torch.zeros(2, dtype=torch.float32, device=dev)
        self._fix_head = torch.zeros(2, dtype=torch.int32, device=dev)
        self._fix_scale = torch.ones(2, dtype=torch.float32, device=dev)
        self._fix_amax = torch.zeros(1, dtype=torch.float32, device=dev)
        self._fix_sat = torch.zeros(1, dtype=torch.int64, device=dev)
        self._fix_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.x_scale_used = None  # after recompute_on_overflow(): the scales X_q / W_q now carry
        self.w_scale_used = None
        # backward(): X_q^T cached by the forward's quantize, the gradient's
        # delayed scale (E5M2) and the outputs
        self.x_q_t = self.g = None
        if with_backward:
            self.x_q_t = torch.empty(K, M, dtype=torch.uint8, device=dev)
            self.g = DelayedScale(B.E5M2, margin, history_len, dev)
            self.dy_q = torch.empty(M, N, dtype=torch.uint8, device=dev)
            self.dy_q_t = torch.empty(N, M, dtype=torch.uint8, device=dev)
            self.dh = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
            self.dw = torch.empty(K, N, dtype=torch.bfloat16, device=dev)
        # fp8_cache: the pre-activation kept for backward in E4M3 under its own
        # delayed scale (written by the forward's quantize in the same pass)
        self.h_q = self.hs = None
        if fp8_cache:
            self.h_q = torch.empty(M, K, dtype=torch.uint8, device=dev)
            self.hs = DelayedScale(B.E4M3, margin, history_len, dev)
        self.workspace = None
        if self.fused:
            # zero-filled once; the fused kernel leaves it zero
            self.workspace = torch.zeros(max(1, B.fp8_downproj_workspace_bytes(M)), dtype=torch.uint8, device=dev)
        self._side = torch.cuda.Stream(device=dev)  # weight branch and history updates
        hi = torch.cuda.Stream.priority_range()[1]
        self._gemm = torch.cuda.Stream(device=dev, priority=hi)  # GEMM blocks, ahead of quantize blocks
        if group:
            if K % B.GROUP or N % B.GROUP:
                raise ValueError("group scales need K % 128 == 0 and N % 128 == 0")
            self.x_gscale = torch.empty(M, K // B.GROUP, dtype=torch.float32, device=dev)
            self.w_gscale = torch.empty(K // B.GROUP, N // B.GROUP, dtype=torch.float32, device=dev)

    @property
    def sat(self) -> torch.Tensor:
        """Saturation count of the most recent quantize of H."""
        return self.x.last_sat if self.x.clean else self.x.sat

    # -- a7 -------------------------------------------------------------------
    def cast_weight(self, W: torch.Tensor, scale: torch.Tensor | None = None) -> None:
        """W [K,N] BF16 -> W_q^T [N,K] (forward operand) and, if kept, W_q [K,N]."""
        scale = self.w.scale if scale is None else scale
        self.w.clean = False
        if self.group:
            B.fp8_quant_fused(W, B.ACT_IDENTITY, B.E4M3, None, q_out=self.w_q, q_t_out=self.wt_q,
                              amax_out=self.w.amax, group_scales_out=self.w_gscale,
                              group_rows=B.GROUP)
        else:
            B.fp8_quant_fused(W, B.ACT_IDENTITY, B.E4M3, scale, q_out=self.w_q,
                              q_t_out=self.wt_q, amax_out=self.w.amax, sat_count=self.w.sat)

    # -- a1-a5 ----------------------------------------------------------------
    def quantize(self, H: torch.Tensor, scale: torch.Tensor | None = None, rows=None) -> None:
        """Fused quantize of H (or of its row block rows = (r0, r1); blocks after
        the first fold into the amax / saturation count instead of resetting them)."""
        scale = self.x.scale if scale is None else scale
        r0, r1 = (0, self.M) if rows is None else rows
        flags = B.ACCUMULATE if r0 > 0 else 0
        self.x.clean = False
        act_out = None if self.act_bf16 is None else self.act_bf16[r0:r1]
        if self.group:
            B.fp8_quant_fused_ex(H[r0:r1], self.act, B.E4M3, None, act_out=act_out, q_out=self.x_q[r0:r1],
                                 amax_out=self.x.amax, sat_count=self.x.sat,
                                 group_scales_out=self.x_gscale[r0:r1], group_rows=1, flags=flags)
        else:
            B.fp8_quant_fused_ex(H[r0:r1], self.act, B.E4M3, scale, act_out=act_out,
                                 q_out=self.x_q[r0:r1], amax_out=self.x.amax, sat_count=self.x.sat,
                                 flags=flags)

    # -- a9 -------------------------------------------------------------------
    def gemm(self, scale_x: torch.Tensor | None = None, scale_w: torch.Tensor | None = None,
             rows=None) -> torch.Tensor:
        """Y = X_q W_q / (s_x s_w) for all rows, or for the row block rows = (r0, r1)."""
        scale_x = self.x.scale if scale_x is None else scale_x
        scale_w = self.w.scale if scale_w is None else scale_w
        r0, r1 = (0, self.M) if rows is None else rows
        if self.group:
            B.fp8_gemm_fwd(self.x_q[r0:r1], self.wt_q, self.x_gscale[r0:r1], self.w_gscale, self.y[r0:r1],
                           group_mode=1, status=self.gemm_status)
        else:
            B.fp8_gemm_fwd(self.x_q[r0:r1], self.wt_q, scale_x, scale_w, self.y[r0:r1],
                           status=self.gemm_status)
        return self.y

    def quantize_and_gemm(self, H: torch.Tensor, scale_x: torch.Tensor | None = None,
                          scale_w: torch.Tensor | None = None) -> torch.Tensor:
        """a1-a5 and a9 in the fused kernel (same results as quantize() then gemm())."""
        scale_x = self.x.scale if scale_x is None else scale_x
        scale_w = self.w.scale if scale_w is None else scale_w
        self.x.clean = False
        B.fp8_downproj_fwd(H, self.wt_q, scale_x, scale_w, self.x_q, self.y, self.workspace, act=self.act,
                           act_out=self.act_bf16, amax_out=self.x.amax, sat_count=self.x.sat,
                           status=self.gemm_status)
        return self.y

    # -- a6 -------------------------------------------------------------------
    def update_scales(self) -> None:
        if not self.group:
            self.x.update()
            self.w.update()

    def check_status(self) -> int:
        """Read and clear the device status words of the steps since the last
        check (this synchronises with the device).  Returns their OR: 0, or
        B.DEV_TIMEOUT (a bounded wait inside a GEMM ran out, so that step's Y is
        invalid) and/or B.DEV_BAD_AMAX (a history update kept the previous
        scale).  After a time-out the fused kernel's workspace may hold counts,
        so it is zeroed again here and the next step starts clean."""
        st = int(self.gemm_status.item()) | int(self.x.status.item()) | int(self.w.status.item())
        if st & B.DEV_TIMEOUT and self.workspace is not None:
            self.workspace.zero_()
        self.gemm_status.zero_()
        self.x.status.zero_()
        self.w.status.zero_()
        return st

    def step(self, H: torch.Tensor, W: torch.Tensor) -> torch.Tensor:
        """One forward step: cast W, fused quantize of H, FP8 GEMM, history updates.

        With ``fused`` (per-tensor scales only) the W cast, the quantize and
        the GEMM are one kernel (fp8_downproj_fwd_ex; see _step_fused).  With
        one row block the W cast and the quantize share one launch and the
        GEMM follows (_step_one_launch_cast).  Otherwise the batch is
        processed in ``chunks`` row blocks.  The current stream
        quantizes the blocks one after the other; a high-priority stream runs
        each block's GEMM as soon as that block is quantized, so the
        compute-bound GEMM of block i overlaps the memory-bound quantize of
        block i+1.  A side stream casts W and updates its history beside the
        first quantize, then updates the activation's history once the last
        block is quantized (the updates write the other scale slot, so they
        never race the GEMMs' reads).  All branches join the current stream."""
        self.x_scale_used = self.w_scale_used = None
        if self.fused:
            return self._step_fused(H, W)
        if not self.group and self.chunks == 1:
            return self._step_one_launch_cast(H, W)
        main, side, gs = torch.cuda.current_stream(), self._side, self._gemm
        sx, sw = self.x.scale, self.w.scale  # this step's slots
        side.wait_stream(main)
        w_ready = torch.cuda.Event()
        with torch.cuda.stream(side):
            self.cast_weight(W, sw)
            w_ready.record(side)
            if not self.group:
                self.w.update()
        gs.wait_stream(side)  # W_q^T ready (and everything before this step)
        block = self.M // self.chunks
        for i in range(self.chunks):
            rows = (i * block, (i + 1) * block)
            self.quantize(H, sx, rows)
            done = torch.cuda.Event()
            done.record(main)
            gs.wait_event(done)
            with torch.cuda.stream(gs):
                self.gemm(sx, sw, rows)
        if not self.group:
            side.wait_stream(main)  # every block quantized: this step's amax is final
            with torch.cuda.stream(side):
                self.x.update()
        main.wait_stream(gs)
        main.wait_stream(side)
        return self.y

    def _step_fused(self, H: torch.Tensor, W: torch.Tensor) -> torch.Tensor:
        """The per-tensor step as one kernel (fp8_downproj_fwd_ex): the W cast,
        the quantize of H and the GEMM, accumulating into this slot's amax /
        count (zeroed by the previous update()) with a workspace the kernel
        leaves zero, so nothing runs ahead of it; the kernel's last CTA also
        runs both history updates, so the step is one launch."""
        sx, sw = self.x.scale, self.w.scale
        flags = B.ACCUMULATE if (self.x.clean and self.w.clean) else 0
        B.fp8_downproj_fwd_ex(H, self.wt_q, sx, sw, self.x_q, self.y, self.workspace, w=W, w_q=self.w_q,
                              amax_w=self.w.amax, sat_w=self.w.sat, act=self.act, act_out=self.act_bf16, amax_out=self.x.amax,
                              sat_count=self.x.sat, hist_x=self.x.kernel_update_args(),
                              hist_w=self.w.kernel_update_args(), flags=flags, status=self.gemm_status)
        self.x.advance()
        self.w.advance()
        return self.y

    def _step_one_launch_cast(self, H: torch.Tensor, W: torch.Tensor) -> torch.Tensor:
        """The per-tensor step with separate quantize and GEMM kernels: the W cast
        and the quantize of H share one launch (fp8_quant_fused_batch), and the
        GEMM follows on the same stream, so its set-up overlaps the quantize's
        last CTAs.  Both casts accumulate into their slot's amax / count, which
        the previous update zeroed (no memset ahead of the cast).  The GEMM
        also runs both history updates (fp8_gemm_fwd_update: one warp of its
        first CTA, beside its first tile), so the step is two launches on one
        stream."""
        sx, sw = self.x.scale, self.w.scale
        hs = self.hs
        fx = B.ACCUMULATE if self.x.clean and (hs is None or hs.clean) else 0
        fw = B.ACCUMULATE if self.w.clean else 0
        cache = {} if hs is None else dict(hq_out=self.h_q, scale_h=hs.scale, amax_h=hs.amax, sat_h=hs.sat)
        B.fp8_quant_fused_batch([
            B.quant_args(W, B.ACT_IDENTITY, B.E4M3, sw, q_out=self.w_q, q_t_out=self.wt_q,
                         amax_out=self.w.amax, sat_count=self.w.sat, flags=fw),
            B.quant_args(H, self.act, B.E4M3, sx, act_out=self.act_bf16, q_out=self.x_q, q_t_out=self.x_q_t,
                         amax_out=self.x.amax, sat_count=self.x.sat, flags=fx, **cache),
        ])
        self.x.clean = self.w.clean = False
        B.fp8_gemm_fwd(self.x_q, self.wt_q, sx, sw, self.y, amax_x=self.x.amax, hist_x=self.x.kernel_update_args(),
                       amax_w=self.w.amax, hist_w=self.w.kernel_update_args(), status=self.gemm_status)
        self.x.advance()
        self.w.advance()
        if hs is not None:
            hs.clean = False
            hs.update()  # the cache's own delayed scale for the next step
        return self.y

    def capture(self, H: torch.Tensor, W: torch.Tensor, H_next: torch.Tensor | None = None,
                W_next: torch.Tensor | None = None) -> "StepGraph":
        """Capture the step as CUDA graphs on fixed buffers (see StepGraph)."""
        return StepGraph(self, H, W, H_next, W_next)

    def recompute_on_overflow(self, H: torch.Tensor, W: torch.Tensor) -> int:
        """Detect-and-recompute ("FP8 Training & Inference", Delayed Scaling:
        when the delayed scale is too large for this step's values, detect it
        and recompute with a corrected scale).  Call after step(H, W).  The
        casts saturate instead of producing infinities, so the overflow
        signal is a value past the format's maximum, which each cast counts on
        the device (the saturation counts of X and of W); the host reads the
        two counts back (one synchronisation) and does no arithmetic on them
        beyond "is it zero".  If the quantize of H saturated, H is cast again
        with the scale this step's own amax gives under the same rule,
        448 / fp32(margin * amax_t) (amax_history_update on a one-entry
        history; the act copy is unchanged and not rewritten); likewise W
        (both layouts) when its cast saturated.  The GEMM then runs
        again on the new operands.  The delayed-scale state is untouched: the
        history update of the step already holds amax_t, so the next step's
        scale accounts for it.  Returns RECOMPUTE_X | RECOMPUTE_W for what
        was cast again (0: nothing overflowed, Y stands); x_scale_used and
        w_scale_used name the scales X_q and W_q now carry.  Group scales are
        computed from each group's own values and never overflow: 0."""
        sx_prev, sw_prev = self.x.last_scale, self.w.last_scale
        self.x_scale_used, self.w_scale_used = sx_prev, sw_prev
        if self.group:
            return 0
        counts = torch.cat([self.x.last_sat, self.w.last_sat]).cpu()
        x_over, w_over = int(counts[0]) > 0, int(counts[1]) > 0
        if not (x_over or w_over):
            return 0
        redo = 0
        if x_over:
            sx = self._fix_scale[0:1]
            B.amax_history_update_ex(self._fix_hist[0:1], self._fix_head[0:1], self.x.last_amax, self.x.margin,
                                     B.E4M3, sx, scale_prev=sx_prev, status=self._fix_status)
            B.fp8_quant_fused_ex(H, self.act, B.E4M3, sx, q_out=self.x_q, q_t_out=self.x_q_t,
                                 amax_out=self._fix_amax, sat_count=self._fix_sat)
            self.x_scale_used = sx
            redo |= RECOMPUTE_X
        if w_over:
            sw = self._fix_scale[1:2]
            B.amax_history_update_ex(self._fix_hist[1:2], self._fix_head[1:2], self.w.last_amax, self.w.margin,
                                     B.E4M3, sw, scale_prev=sw_prev, status=self._fix_status)
            B.fp8_quant_fused(W, B.ACT_IDENTITY, B.E4M3, sw, q_out=self.w_q, q_t_out=self.wt_q,
                              amax_out=self._fix_amax)
            self.w_scale_used = sw
            redo |= RECOMPUTE_W
        self.gemm(self.x_scale_used, self.w_scale_used)
        return redo

    def backward(self, dY: torch.Tensor, H: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor]:
        """The down-projection's backward on the forward's FP8 operands ("FP8
        Training & Inference", FP8 Training Recipe: gradients in E5M2, weights
        and activations in E4M3), after step(H, W) and before the next step:

            dY [M,N] BF16 -> dY_q (E5M2, delayed scale) and dY_q^T, one pass
            dH = (dY_q . W_q^T) / (s_dy s_w) * act'(H)   -> [M,K] BF16 (dX never stored)
            dW = (X_q^T . dY_q) / (s_x s_dy)              -> [K,N] BF16
            push amax(dY) into the gradient's history

        X_q^T is the transposed copy the forward's quantize cached, W_q the
        weight's own layout; both carry the scales they were cast with (the
        recompute's, if recompute_on_overflow() ran).  H is the forward's BF16
        pre-activation; with fp8_cache it is not needed: act'(H) is taken at the
        E4M3 cache the forward wrote ("FP8 training: what it is and how it
        works", Trade-offs and edge cases: cached activations in FP8),
        dequantised with the scale it was cast with.  Needs with_backward.
        Returns views of (dH, dW)."""
        if not self.with_backward:
            raise RuntimeError("backward() needs Fp8DownProj(..., with_backward=True)")
        sx = self.x_scale_used if self.x_scale_used is not None else self.x.last_scale
        sw = self.w_scale_used if self.w_scale_used is not None else self.w.last_scale
        sdy = self.g.scale
        fl = B.ACCUMULATE if self.g.clean else 0
        B.fp8_quant_fused_ex(dY, B.ACT_IDENTITY, B.E5M2, sdy, q_out=self.dy_q, q_t_out=self.dy_q_t,
                             amax_out=self.g.amax, sat_count=self.g.sat, flags=fl)
        self.g.clean = False
        if self.fp8_cache:
            B.fp8_gemm_dgrad_act_q(self.dy_q, self.w_q, sdy, sw, self.h_q, self.hs.last_scale, self.dh, act=self.act,
                                   status=self.gemm_status)
        else:
            if H is None:
                raise ValueError("backward() needs the forward's pre-activation H (or fp8_cache=True)")
            B.fp8_gemm_dgrad_act(self.dy_q, self.w_q, sdy, sw, H, self.dh, act=self.act, status=self.gemm_status)
        B.fp8_gemm_wgrad(self.x_q_t, self.dy_q_t, sx, sdy, self.dw, status=self.gemm_status)
        self.g.update()
        return self.dh, self.dw

    def calibrate_backward(self, dY: torch.Tensor) -> None:
        """Bootstrap the gradient's delayed scale from a first dY (one amax pass),
        as calibrate() does for X and W."""
        if not self.with_backward:
            raise RuntimeError("calibrate_backward() needs Fp8DownProj(..., with_backward=True)")
        self.g.scales.fill_(1.0)
        B.fp8_quant_fused(dY, B.ACT_IDENTITY, B.E5M2, self.g.scale, q_out=self.dy_q, amax_out=self.g.amax)
        self.g.clean = False
        self.g.update()

    def calibrate(self, H: torch.Tensor, W: torch.Tensor) -> None:
        """Bootstrap the delayed scales from step 0's own tensors (one amax pass each).

        The casts run with a placeholder scale; only their amax is kept, and it
        seeds each history so step 0 already has a scale."""
        if self.group:
            return
        self.x.scales.fill_(1.0)
        self.w.scales.fill_(1.0)
        self.cast_weight(W)
        self.quantize(H)
        self.x.update()
        self.w.update()
        if self.hs is not None:  # the pre-activation cache's scale: an amax pass over H itself
            self.hs.scales.fill_(1.0)
            B.fp8_quant_fused(H, B.ACT_IDENTITY, B.E4M3, self.hs.scale, amax_out=self.hs.amax)
            self.hs.clean = False
            self.hs.update()


class StepGraph:
    """The down-projection step captured as CUDA graphs.

    All buffers are allocated beforehand, so a replay re-runs the same
    kernels on the same device pointers with no host work between them.
    Consecutive steps use alternating scale slots, so two graphs are
    captured (one per slot); ``replay()`` runs the one matching the current
    slot and switches slots, so replays and eager steps mix freely.  The
    graph for the slot current at capture reads H and W, the other H_next and
    W_next (default H and W), so a caller can fill one pair of buffers while
    the step reads the other (``buffer()`` names the pair the next replay
    reads).  The amax histories live in device memory, so replays carry the
    delayed scaling forward exactly as eager steps do.  Run at least one eager
    step first (it performs the one-time per-kernel set-up).
    """

    def __init__(self, dp: Fp8DownProj, H: torch.Tensor, W: torch.Tensor, H_next: torch.Tensor | None = None,
                 W_next: torch.Tensor | None = None):
        self.dp = dp
        self.slot0 = dp.x.slot  # the scale slot graph 0 reads; graph 1 reads the other
        self.graphs = []
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        for h, w in ((H, W), (H if H_next is None else H_next, W if W_next is None else W_next)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    self.y = dp.step(h, w)
            self.graphs.append(g)
        torch.cuda.current_stream().wait_stream(side)
        self._next = 0

    def buffer(self) -> int:
        """0 if the next replay reads (H, W), 1 if it reads (H_next, W_next)."""
        return self._next if self.dp.group else int(self.dp.x.slot != self.slot0)

    def replay(self) -> torch.Tensor:
        """Run one step: the graph whose scale slot is current, then switch
        the host-side slots as an eager step would."""
        dp = self.dp
        k = self.buffer()
        self.graphs[k].replay()
        self._next = k ^ 1
        if not dp.group:
            dp.x.slot ^= 1
            dp.w.slot ^= 1
        return self.y
