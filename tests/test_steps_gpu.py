"""Multi-step delayed scaling on the GPU against the oracle's recurrence.

Each step: the fused quantize runs with the scale the history produced, then
the history takes this step's amax.  Scales, amax, saturation counts and FP8
bytes must equal the oracle's bit for bit at every step ("Paradigma Details
FP8 and Optimizer Tricks Behind NanoGPT Records", second paragraph: previous
step's amax times a margin; "FP8 Training & Inference", Delayed Scaling).
"""
import numpy as np
import pytest
import torch

import oracle as O
from quantize_fp8_gemm_gb300 import binding as B
from quantize_fp8_gemm_gb300 import workloads as WL
from quantize_fp8_gemm_gb300 import downproj as dp_mod
from quantize_fp8_gemm_gb300.downproj import Fp8DownProj
from tests.parity import assert_gemm_close, dev_f32, dev_u8, host_bits16, host_u8

pytestmark = pytest.mark.gpu


class OracleRecurrence:
    """The oracle's side of the delayed-scaling loop for one tensor."""

    def __init__(self, L, margin, fmt=O.E4M3):
        self.hist = np.zeros(L, np.float32)
        self.head = 0
        self.scale = 1.0
        self.margin, self.fmt = margin, fmt

    def push(self, amax):
        st, self.hist, self.head, self.scale = O.history_update(self.hist, self.head, amax, self.margin,
                                                                self.fmt, self.scale)
        return st


@pytest.mark.parametrize("fused", [False, True])
def test_gpt2s_ten_steps_fresh_inputs(fused):
    """Ten steps with the separate quantize and GEMM kernels, and with the
    fused kernel (fp8_downproj_fwd) in their place."""
    w = WL.WORKLOADS["gpt2s"]
    W_bits = WL.w_down(w)
    H0 = WL.h_preact(w, 0)
    dp = Fp8DownProj(w.M, w.K, w.N, margin=w.margin, history_len=w.history_len, fused=fused)
    Wd = WL.bf16_tensor(W_bits).cuda()
    dp.calibrate(WL.bf16_tensor(H0).cuda(), Wd)
    ox, ow = OracleRecurrence(w.history_len, w.margin), OracleRecurrence(w.history_len, w.margin)
    ox.push(O.amax(H0, O.ACT_RELU2))
    ow.push(O.amax(W_bits, O.ACT_IDENTITY))
    rows = WL.sample_rows(w.M, 64, seed=11)
    for t in range(w.steps):
        h = WL.h_preact(w, t)
        sx_used, sw_used = float(dp.x.scale.item()), float(dp.w.scale.item())
        assert (sx_used, sw_used) == (ox.scale, ow.scale), f"step {t}"
        y = dp.step(WL.bf16_tensor(h).cuda(), Wd)
        torch.cuda.synchronize()
        rx = O.quant(h, O.ACT_RELU2, O.E4M3, ox.scale)
        assert np.array_equal(host_u8(dp.x_q), rx["q"]), f"step {t}: E4M3 codes"
        assert int(dp.sat.item()) == rx["sat"], f"step {t}: saturations"
        assert float(dp.x.history[0].item()) == rx["amax"], f"step {t}: amax"
        if t in (0, w.steps - 1):
            rw = O.quant(W_bits, O.ACT_IDENTITY, O.E4M3, ow.scale, want_act=False)
            Yr, S = O.gemm_fwd(rx["q"][rows], rw["q"], ox.scale, ow.scale)
            assert_gemm_close(y, Yr, S, rows=rows)
        ox.push(rx["amax"])
        ow.push(O.amax(W_bits, O.ACT_IDENTITY))
    assert int(dp.x.status.item()) == 0 and int(dp.gemm_status.item()) == 0


def test_gpt2s_batch_drift_and_saturation():
    """The GPT-2-small batch: 65,536 x 3072 -> 768, 20 steps with the std of H
    drifting 1.0 -> 1.5, driven through Fp8DownProj.step -- its default at this
    size is the one-launch step (fp8_downproj_fwd_ex: W cast, quantize, GEMM
    and both history updates in one kernel).  The delayed scale lags the
    drift by one step; the drift per step stays well inside the margin of 2,
    so the saturation count stays zero.  Every step: the full E4M3 tensor, the full BF16 activation copy, the amax,
    the saturation count and the next step's scales equal the oracle's
    recurrence bit for bit, and the count is zero whenever this step's amax
    stays below margin x the previous one.  Steps 0 and 19: Y within the GEMM
    tolerance on sampled rows, the first and last rows of several 128-row
    tiles among them."""
    w = WL.WORKLOADS["gpt2s_batch"]
    W_bits = WL.w_down(w)
    Wd = WL.bf16_tensor(W_bits).cuda()
    dp = Fp8DownProj(w.M, w.K, w.N, margin=w.margin, history_len=w.history_len)
    assert dp.fused
    H0 = WL.h_preact(w, 0, WL.drift_std(w, 0))
    dp.calibrate(WL.bf16_tensor(H0).cuda(), Wd)
    ox, ow = OracleRecurrence(w.history_len, w.margin), OracleRecurrence(w.history_len, w.margin)
    ox.push(O.amax(H0, O.ACT_RELU2))
    amax_w = O.amax(W_bits, O.ACT_IDENTITY)
    ow.push(amax_w)
    rw = None
    prev_amax = ox.hist[ox.head]
    rows = WL.sample_rows(w.M, 48, seed=12)
    for t in range(w.steps):
        h = WL.h_preact(w, t, WL.drift_std(w, t))
        assert (float(dp.x.scale.item()), float(dp.w.scale.item())) == (ox.scale, ow.scale), f"step {t}"
        y = dp.step(WL.bf16_tensor(h).cuda(), Wd)
        torch.cuda.synchronize()
        rx = O.quant(h, O.ACT_RELU2, O.E4M3, ox.scale)
        assert np.array_equal(host_u8(dp.x_q), rx["q"]), f"step {t}: E4M3 codes"
        assert np.array_equal(host_bits16(dp.act_bf16), rx["act"]), f"step {t}: BF16 activation copy"
        assert int(dp.sat.item()) == rx["sat"], f"step {t}: saturations"
        assert float(dp.x.history[0].item()) == rx["amax"], f"step {t}: amax"
        assert float(dp.w.history[0].item()) == amax_w, f"step {t}: amax of W"
        if t in (0, w.steps - 1):
            rw = O.quant(W_bits, O.ACT_IDENTITY, O.E4M3, ow.scale, want_act=False, want_qt=True)
            assert np.array_equal(host_u8(dp.wt_q), rw["q_t"]), f"step {t}: transposed E4M3 weight"
            Yr, S = O.gemm_fwd(rx["q"][rows], rw["q"], ox.scale, ow.scale)
            assert_gemm_close(y, Yr, S, rows=rows)
        if rx["amax"] < w.margin * prev_amax:
            assert rx["sat"] == 0
        prev_amax = rx["amax"]
        ox.push(rx["amax"])
        ow.push(amax_w)
        assert (float(dp.x.scale.item()), float(dp.w.scale.item())) == (ox.scale, ow.scale), f"step {t}: next scales"
    assert int(dp.x.status.item()) == 0 and int(dp.w.status.item()) == 0 and int(dp.gemm_status.item()) == 0


def test_checkpoint_resume_is_bit_identical():
    """The only state is the device history / head / scale: save after step 5,
    restore into a fresh instance, and steps 6-9 repeat bit for bit."""
    w = WL.WORKLOADS["gpt2s"]
    M, K, N = 1024, w.K, w.N
    W_bits = WL.w_down(w)
    Wd = WL.bf16_tensor(W_bits).cuda()
    hs = [WL.bf16_tensor(WL.h_preact(w, t)[:M]).cuda() for t in range(10)]
    a = Fp8DownProj(M, K, N, margin=w.margin, history_len=3)
    a.calibrate(hs[0], Wd)
    saved = None
    outs_a = []
    for t in range(10):
        y = a.step(hs[t], Wd).clone()
        if t == 5:
            saved = {k: (getattr(a, r).history.clone(), getattr(a, r).head.clone(), getattr(a, r).scale.clone())
                     for k, r in (("x", "x"), ("w", "w"))}
        if t > 5:
            outs_a.append((y, a.x_q.clone()))
    b = Fp8DownProj(M, K, N, margin=w.margin, history_len=3)
    for r in ("x", "w"):
        hist, head, scale = saved[r]
        getattr(b, r).history.copy_(hist)
        getattr(b, r).head.copy_(head)
        getattr(b, r).scale.copy_(scale)
    for i, t in enumerate(range(6, 10)):
        y = b.step(hs[t], Wd)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), outs_a[i][0].view(torch.int16))
        assert torch.equal(b.x_q, outs_a[i][1])


def test_graph_replay_matches_eager_steps():
    w = WL.WORKLOADS["gpt2s"]
    M, K, N = 2048, w.K, w.N
    Wd = WL.bf16_tensor(WL.w_down(w)).cuda()
    hs = [WL.bf16_tensor(WL.h_preact(w, t)[:M]).cuda() for t in range(4)]
    e = Fp8DownProj(M, K, N, margin=w.margin)
    g = Fp8DownProj(M, K, N, margin=w.margin)
    e.calibrate(hs[0], Wd)
    g.calibrate(hs[0], Wd)
    g.step(hs[0], Wd)  # one eager step on each before capture
    e.step(hs[0], Wd)
    buf = torch.empty_like(hs[0])
    graph = g.capture(buf, Wd)
    for t in range(1, 4):
        ye = e.step(hs[t], Wd)
        buf.copy_(hs[t])
        yg = graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(ye.view(torch.int16), yg.view(torch.int16)), f"step {t}"
        assert torch.equal(e.x.scale, g.x.scale)


@pytest.mark.parametrize("M", [2048, 65536])
def test_double_buffered_graph_matches_eager_steps(M):
    """capture(H, W, H_next, W_next): the two graphs read alternate buffer
    pairs (buffer() names the pair the next replay reads), so a caller can
    fill one while the other is in use.  Each step's H and W differ (W drifts
    too), at a two-launch size and a one-launch size; the replays equal eager
    steps on the same inputs bit for bit, and so do the delayed scales."""
    w = WL.WORKLOADS["gpt2s"]
    K, N = w.K, w.N
    g0 = torch.Generator(device="cuda").manual_seed(M)
    hs = [torch.randn(M, K, device="cuda", generator=g0).mul_(1.0 + 0.1 * t).to(torch.bfloat16) for t in range(5)]
    ws = [(torch.randn(K, N, device="cuda", generator=g0) * (0.02 + 0.002 * t)).to(torch.bfloat16) for t in range(5)]
    e = Fp8DownProj(M, K, N, margin=w.margin)
    g = Fp8DownProj(M, K, N, margin=w.margin)
    for dp in (e, g):
        dp.calibrate(hs[0], ws[0])
        dp.step(hs[0], ws[0])
    Hb = [torch.empty_like(hs[0]) for _ in range(2)]
    Wb = [torch.empty_like(ws[0]) for _ in range(2)]
    graph = g.capture(Hb[0], Wb[0], H_next=Hb[1], W_next=Wb[1])
    for t in range(1, 5):
        ye = e.step(hs[t], ws[t])
        b = graph.buffer()
        Hb[b].copy_(hs[t])
        Wb[b].copy_(ws[t])
        Hb[b ^ 1].zero_()  # the other pair must not be read
        Wb[b ^ 1].zero_()
        yg = graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(ye.view(torch.int16), yg.view(torch.int16)), f"step {t}"
        assert torch.equal(e.x.scale, g.x.scale) and torch.equal(e.w.scale, g.w.scale)


def test_check_status_recovers_after_a_timeout():
    """A one-launch step whose GEMM loads are held back (a test hook) gives up
    its bounded waits: check_status reports FP8Q_DEV_TIMEOUT and leaves the
    workspace zero, and the next step equals that of a run that never timed out
    (the quantize and the history updates of the failed step still ran)."""
    M, K, N = 4096, 3072, 768
    w = WL.WORKLOADS["gpt2s"]
    g = torch.Generator(device="cuda").manual_seed(21)
    H = [torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16) for _ in range(3)]
    W = (torch.randn(K, N, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    bad = Fp8DownProj(M, K, N, margin=w.margin, fused=True)
    good = Fp8DownProj(M, K, N, margin=w.margin, fused=True)
    for dp in (bad, good):
        dp.calibrate(H[0], W)
        dp.step(H[0], W)
    assert good.check_status() == 0 and bad.check_status() == 0
    B.fp8q_gemm_test_hold_loads(True)
    try:
        bad.step(H[1], W)
        torch.cuda.synchronize()
    finally:
        B.fp8q_gemm_test_hold_loads(False)
    good.step(H[1], W)
    assert bad.check_status() & B.DEV_TIMEOUT
    assert good.check_status() == 0
    assert int(bad.workspace.count_nonzero().item()) == 0
    assert torch.equal(bad.x.scale, good.x.scale) and torch.equal(bad.w.scale, good.w.scale)
    yb = bad.step(H[2], W).clone()
    yg = good.step(H[2], W).clone()
    torch.cuda.synchronize()
    assert bad.check_status() == 0
    assert torch.equal(yb.view(torch.int16), yg.view(torch.int16))


def test_bad_amax_keeps_scale_and_flags():
    hist = torch.zeros(1, device="cuda")
    head = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = torch.full((1,), 7.0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0.0, float("inf"), float("nan")):
        B.amax_history_update(hist, head, torch.tensor([bad], device="cuda"), 2.0, B.E4M3, scale, status=st)
        torch.cuda.synchronize()
        assert scale.item() == 7.0
        assert st.item() & B.DEV_BAD_AMAX
    # a ring of 4: window max and head match the oracle
    hist = torch.zeros(4, device="cuda")
    head = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = OracleRecurrence(4, 1.5)
    for a in [3.0, 100.0, 2.0, 0.5, 0.25, 0.125, 7.0]:
        B.amax_history_update(hist, head, torch.tensor([a], device="cuda"), 1.5, B.E4M3, scale)
        o.push(a)
        torch.cuda.synchronize()
        assert scale.item() == o.scale and int(head.item()) == o.head
        assert np.array_equal(hist.cpu().numpy(), o.hist)


@pytest.mark.parametrize("chunks", [2, 4])
def test_row_blocks_match_one_block(chunks):
    """Quantizing in row blocks (accumulating amax and saturations) with each
    block's GEMM overlapped gives exactly the one-block results."""
    w = WL.WORKLOADS["gpt2s"]
    M, K, N = 4096, w.K, w.N
    Wd = WL.bf16_tensor(WL.w_down(w)).cuda()
    hs = [WL.bf16_tensor(WL.h_preact(w, t)[:M]).cuda() for t in range(3)]
    one = Fp8DownProj(M, K, N, margin=w.margin, chunks=1)
    blk = Fp8DownProj(M, K, N, margin=w.margin, chunks=chunks)
    one.calibrate(hs[0], Wd)
    blk.calibrate(hs[0], Wd)
    for t in range(3):
        y1 = one.step(hs[t], Wd).clone()
        y2 = blk.step(hs[t], Wd)
        torch.cuda.synchronize()
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), f"step {t}: Y"
        assert torch.equal(one.x_q, blk.x_q) and torch.equal(one.act_bf16.view(torch.int16),
                                                             blk.act_bf16.view(torch.int16))
        assert one.sat.item() == blk.sat.item() and one.x.last_amax.item() == blk.x.last_amax.item()
        assert torch.equal(one.x.scale, blk.x.scale) and torch.equal(one.w.scale, blk.w.scale)


# Detect-and-recompute ("FP8 Training & Inference", Delayed Scaling: a scale
# too large for the step's values is detected and the step recomputed with a
# corrected scale).
def _scaled_bits(bits, factor):
    """BF16 bits of factor * x (a power of two: exact)."""
    return O.f32_to_bf16(O.bf16_to_f32(bits) * np.float32(factor))


def _recompute_fixture(M, fused=False):
    w = WL.WORKLOADS["gpt2s"]
    W_bits = WL.w_down(w)
    H0 = WL.h_preact(w, 0)[:M]
    dp = Fp8DownProj(M, w.K, w.N, margin=w.margin, fused=fused, with_dgrad=True)
    Wd = WL.bf16_tensor(W_bits).cuda()
    dp.calibrate(WL.bf16_tensor(H0).cuda(), Wd)
    y0 = dp.step(WL.bf16_tensor(H0).cuda(), Wd).clone()
    assert dp.recompute_on_overflow(WL.bf16_tensor(H0).cuda(), Wd) == 0
    return w, dp, W_bits, Wd, H0, y0


@pytest.mark.parametrize("fused", [False, True])
def test_recompute_after_activation_overflow(fused):
    """H grows 8x in one step (its ReLU^2 64x): the delayed scale saturates
    the cast; the recompute casts H again with 448 / fp32(margin * amax_t),
    whose codes, count and GEMM match the oracle's for that scale."""
    M = 2048
    w, dp, W_bits, Wd, H0, _ = _recompute_fixture(M, fused)
    H1 = _scaled_bits(H0, 8.0)
    H1d = WL.bf16_tensor(H1).cuda()
    dp.step(H1d, Wd)
    assert dp.recompute_on_overflow(H1d, Wd) == dp_mod.RECOMPUTE_X
    torch.cuda.synchronize()
    amax_t = O.amax(H1, O.ACT_RELU2)
    stale = O.quant(H1, O.ACT_RELU2, O.E4M3, float(dp.x.last_scale.item()), want_act=False)
    assert int(dp.x.last_sat.item()) == stale["sat"] > 0
    s_fix = O.delayed_scale(amax_t, w.margin, O.E4M3)
    assert float(dp.x_scale_used.item()) == s_fix
    rx = O.quant(H1, O.ACT_RELU2, O.E4M3, s_fix, want_act=False)
    assert np.array_equal(host_u8(dp.x_q), rx["q"])
    assert int(dp._fix_sat.item()) == rx["sat"] == 0
    s_w = float(dp.w_scale_used.item())
    rw = O.quant(W_bits, O.ACT_IDENTITY, O.E4M3, s_w, want_act=False)
    rows = WL.sample_rows(M, 64, seed=5)
    Yr, S = O.gemm_fwd(rx["q"][rows], rw["q"], s_fix, s_w)
    assert_gemm_close(dp.y, Yr, S, rows=rows)
    assert int(dp.gemm_status.item()) == 0 and int(dp._fix_status.item()) == 0


def test_recompute_after_weight_overflow():
    """W grows 16x in one step: both of its layouts are cast again with the
    corrected scale and the GEMM uses them."""
    M = 2048
    w, dp, W_bits, Wd, H0, _ = _recompute_fixture(M)
    W1 = _scaled_bits(W_bits, 16.0)
    W1d = WL.bf16_tensor(W1).cuda()
    H0d = WL.bf16_tensor(H0).cuda()
    dp.step(H0d, W1d)
    assert dp.recompute_on_overflow(H0d, W1d) == dp_mod.RECOMPUTE_W
    torch.cuda.synchronize()
    s_fix = O.delayed_scale(O.amax(W1, O.ACT_IDENTITY), w.margin, O.E4M3)
    assert float(dp.w_scale_used.item()) == s_fix
    rw = O.quant(W1, O.ACT_IDENTITY, O.E4M3, s_fix, want_act=False)
    assert np.array_equal(host_u8(dp.w_q), rw["q"])
    assert np.array_equal(host_u8(dp.wt_q), np.ascontiguousarray(rw["q"].T))
    s_x = float(dp.x_scale_used.item())
    rx = O.quant(H0, O.ACT_RELU2, O.E4M3, s_x, want_act=False)
    assert rx["sat"] == 0
    rows = WL.sample_rows(M, 64, seed=6)
    Yr, S = O.gemm_fwd(rx["q"][rows], rw["q"], s_x, s_fix)
    assert_gemm_close(dp.y, Yr, S, rows=rows)


def test_no_recompute_without_overflow():
    """A step within its scales: nothing is cast again and Y stands."""
    M = 2048
    w, dp, W_bits, Wd, H0, _ = _recompute_fixture(M)
    H1d = WL.bf16_tensor(WL.h_preact(w, 1)[:M]).cuda()
    y = dp.step(H1d, Wd).clone()
    q = dp.x_q.clone()
    assert dp.recompute_on_overflow(H1d, Wd) == 0
    torch.cuda.synchronize()
    assert torch.equal(dp.y.view(torch.int16), y.view(torch.int16)) and torch.equal(dp.x_q, q)


def _delayed(amax0, amax_now, sat_now):
    d = dp_mod.DelayedScale(B.E4M3, 2.0, 3, "cuda")
    d.seed(amax0)
    d.amax.fill_(amax_now)
    d.sat.fill_(sat_now)
    d.clean = False
    return d


@pytest.mark.parametrize("tile", [(-1, 0), (0, 128), (1, 256)])
@pytest.mark.parametrize("amax_x", [5.5, float("inf")])
def test_gemm_fwd_update_equals_gemm_then_updates(tile, amax_x):
    """fp8_gemm_fwd_update: the Y of fp8_gemm_fwd, and the histories, heads,
    next scales, cleared slots and status words of the two
    amax_history_update_ex calls (a non-finite amax keeps the previous scale
    and flags FP8Q_DEV_BAD_AMAX either way)."""
    M, K, N = 1000, 768, 512
    g = torch.Generator(device="cuda").manual_seed(3)
    xq = torch.randint(0, 120, (M, K), dtype=torch.uint8, device="cuda", generator=g)
    wt = torch.randint(0, 120, (N, K), dtype=torch.uint8, device="cuda", generator=g)
    xa, wa = _delayed(3.0, amax_x, 5), _delayed(0.1, 0.07, 0)
    xb, wb = _delayed(3.0, amax_x, 5), _delayed(0.1, 0.07, 0)
    ya = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    yb = torch.empty_like(ya)
    try:
        B.fp8q_gemm_set_tile(*tile)
        B.fp8_gemm_fwd(xq, wt, xa.scale, wa.scale, ya, amax_x=xa.amax, hist_x=xa.kernel_update_args(),
                       amax_w=wa.amax, hist_w=wa.kernel_update_args())
        xa.advance()
        wa.advance()
        B.fp8_gemm_fwd(xq, wt, xb.scale, wb.scale, yb)
        xb.update()
        wb.update()
        torch.cuda.synchronize()
    finally:
        B.fp8q_gemm_set_tile(-1)
    assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
    for a, b in ((xa, xb), (wa, wb)):
        assert a.slot == b.slot
        for f in ("history", "head", "scales", "amaxes", "sats", "status"):
            assert torch.equal(getattr(a, f), getattr(b, f)), f
    assert bool(int(xa.status.item()) & B.DEV_BAD_AMAX) == (amax_x == float("inf"))


def test_backward_after_a_step_against_the_oracle():
    """Fp8DownProj.backward after a forward step: dY cast to E5M2 with its
    delayed scale (both layouts bit for bit), dH = dgrad * act'(H) and
    dW = X_q^T dY_q from the forward's cached X_q^T, both within the GEMM
    tolerance of the oracle on sampled rows; the gradient's history takes
    amax(dY)."""
    w = WL.WORKLOADS["gpt2s"]
    M, K, N = 2048, w.K, w.N
    W_bits = WL.w_down(w)
    Wd = WL.bf16_tensor(W_bits).cuda()
    H0, H1 = WL.h_preact(w, 0)[:M], WL.h_preact(w, 1)[:M]
    rng = np.random.default_rng(8)
    dY0, dY1 = (WL.to_bf16_bits((rng.standard_normal((M, N)) * 1e-3).astype(np.float32)) for _ in range(2))
    dp = Fp8DownProj(M, K, N, margin=w.margin, with_backward=True)
    assert not dp.fused
    dp.calibrate(WL.bf16_tensor(H0).cuda(), Wd)
    dp.calibrate_backward(WL.bf16_tensor(dY0).cuda())
    H1d = WL.bf16_tensor(H1).cuda()
    dp.step(H1d, Wd)
    dh, dw = dp.backward(WL.bf16_tensor(dY1).cuda(), H1d)
    torch.cuda.synchronize()
    s_x, s_w = float(dp.x.last_scale.item()), float(dp.w.last_scale.item())
    s_dy = float(dp.g.last_scale.item())
    assert s_dy == O.delayed_scale(O.amax(dY0, O.ACT_IDENTITY), w.margin, O.E5M2)
    rx = O.quant(H1, O.ACT_RELU2, O.E4M3, s_x, want_act=False)
    rw = O.quant(W_bits, O.ACT_IDENTITY, O.E4M3, s_w, want_act=False)
    rd = O.quant(dY1, O.ACT_IDENTITY, O.E5M2, s_dy, want_act=False)
    assert np.array_equal(host_u8(dp.x_q_t), np.ascontiguousarray(rx["q"].T))
    assert np.array_equal(host_u8(dp.dy_q), rd["q"])
    assert np.array_equal(host_u8(dp.dy_q_t), np.ascontiguousarray(rd["q"].T))
    assert float(dp.g.history[0].item()) == rd["amax"]
    rows = WL.sample_rows(M, 48, seed=9)
    ref, S = O.gemm_dgrad_act(rd["q"], rw["q"], s_dy, s_w, H1, O.ACT_RELU2, rows=rows)
    assert_gemm_close(dh, ref, S, rows=rows)
    krows = WL.sample_rows(K, 48, seed=10)
    ref, S = O.gemm_wgrad(rx["q"], rd["q"], s_x, s_dy, rows=krows)
    assert_gemm_close(dw, ref, S, rows=krows)
    assert int(dp.gemm_status.item()) == 0


@pytest.mark.parametrize("act", [B.ACT_RELU2, B.ACT_RELU])
def test_backward_from_the_fp8_cache_against_the_oracle(act):
    """Fp8DownProj(fp8_cache=True): the forward's quantize also writes H in
    E4M3 under its own delayed scale (bit for bit the oracle's identity
    quantize of H with that scale; its amax is max |H|), the BF16 H is not
    kept, and the backward takes act'(H) at the dequantised cache: dH within
    the GEMM tolerance of the oracle's dgrad times act'(dec(h_q) / s_h); dW as
    before.  Two steps, so the cache's scale comes from the history."""
    w = WL.WORKLOADS["gpt2s"]
    M, K, N = 2048, w.K, w.N
    W_bits = WL.w_down(w)
    Wd = WL.bf16_tensor(W_bits).cuda()
    Hs = [WL.h_preact(w, t)[:M] for t in range(3)]
    rng = np.random.default_rng(18)
    dY0, dY1 = (WL.to_bf16_bits((rng.standard_normal((M, N)) * 1e-3).astype(np.float32)) for _ in range(2))
    dp = Fp8DownProj(M, K, N, act=act, margin=w.margin, with_backward=True, fp8_cache=True)
    dp.calibrate(WL.bf16_tensor(Hs[0]).cuda(), Wd)
    dp.calibrate_backward(WL.bf16_tensor(dY0).cuda())
    oh = OracleRecurrence(w.history_len, w.margin)
    oh.push(O.amax(Hs[0], O.ACT_IDENTITY))
    for t in (1, 2):
        assert float(dp.hs.scale.item()) == oh.scale
        dp.step(WL.bf16_tensor(Hs[t]).cuda(), Wd)
        torch.cuda.synchronize()
        rh = O.quant(Hs[t], O.ACT_IDENTITY, O.E4M3, oh.scale, want_act=False)
        assert np.array_equal(host_u8(dp.h_q), rh["q"]), f"step {t}: E4M3 cache of H"
        assert float(dp.hs.last_amax.item()) == O.amax(Hs[t], O.ACT_IDENTITY) == rh["amax"]
        assert int(dp.hs.last_sat.item()) == rh["sat"]
        s_h = oh.scale
        oh.push(rh["amax"])
    dh, dw = dp.backward(WL.bf16_tensor(dY1).cuda())
    torch.cuda.synchronize()
    s_x, s_w, s_dy = (float(t.item()) for t in (dp.x.last_scale, dp.w.last_scale, dp.g.last_scale))
    assert float(dp.hs.last_scale.item()) == s_h
    rx = O.quant(Hs[2], act, O.E4M3, s_x, want_act=False)
    rw = O.quant(W_bits, O.ACT_IDENTITY, O.E4M3, s_w, want_act=False)
    rd = O.quant(dY1, O.ACT_IDENTITY, O.E5M2, s_dy, want_act=False)
    rows = WL.sample_rows(M, 48, seed=19)
    ref, S = O.gemm_dgrad_act_q(rd["q"], rw["q"], s_dy, s_w, host_u8(dp.h_q), s_h, act, rows=rows)
    assert_gemm_close(dh, ref, S, rows=rows)
    krows = WL.sample_rows(K, 48, seed=20)
    ref, S = O.gemm_wgrad(rx["q"], rd["q"], s_x, s_dy, rows=krows)
    assert_gemm_close(dw, ref, S, rows=krows)
    assert int(dp.gemm_status.item()) == 0 and int(dp.hs.status.item()) == 0


@pytest.mark.parametrize("act", [B.ACT_RELU2, B.ACT_RELU, B.ACT_IDENTITY])
@pytest.mark.parametrize("pair,bn", [(-1, 0), (0, 128), (0, 192), (1, 256), (1, 224)])
def test_dgrad_act_from_the_fp8_cache_every_tile(act, pair, bn):
    """fp8_gemm_dgrad_act_q on ragged shapes with every tile the dispatcher
    offers, against the oracle over all rows; the cache holds codes of both
    signs, zeros and subnormals."""
    M, N, K = 300, 272, 400
    rng = np.random.default_rng(bn + act)
    dyq = O.fp8_encode((rng.standard_normal((M, N)) * 50).astype(np.float32), O.E5M2)
    wq = O.fp8_encode(rng.standard_normal((K, N)).astype(np.float32), O.E4M3)
    hq = rng.integers(0, 256, (M, K)).astype(np.uint8)
    hq[(hq & 0x7F) == 0x7F] = 0x00  # no NaN codes
    s_dy, s_w, s_h = 3.0, 5.0, 37.5
    dh = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        if pair >= 0:
            B.fp8q_gemm_set_tile(pair, bn)
        B.fp8_gemm_dgrad_act_q(dev_u8(dyq), dev_u8(wq), dev_f32(s_dy), dev_f32(s_w), dev_u8(hq), dev_f32(s_h), dh,
                               act=act, status=st)
        torch.cuda.synchronize()
    finally:
        B.fp8q_gemm_set_tile(-1)
    assert st.item() == 0
    ref, S = O.gemm_dgrad_act_q(dyq, wq, s_dy, s_w, hq, s_h, act)
    assert_gemm_close(dh, ref, S)


@pytest.mark.parametrize("N", [2304, 768])
def test_identity_activation_linear_layers(N):
    """The other GEMMs of a GPT-2-small block as FP8 layers (the QKV
    projection 768 -> 2304 and the attention output 768 -> 768): the same step
    with the identity activation, forward and backward against the oracle."""
    M, K = 1024, 768
    rng = np.random.default_rng(N)
    X = [WL.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32)) for _ in range(2)]
    W_bits = WL.to_bf16_bits((rng.standard_normal((K, N)) * 0.02).astype(np.float32))
    dY = WL.to_bf16_bits((rng.standard_normal((M, N)) * 1e-3).astype(np.float32))
    Wd = WL.bf16_tensor(W_bits).cuda()
    dp = Fp8DownProj(M, K, N, act=B.ACT_IDENTITY, margin=2.0, with_backward=True)
    dp.calibrate(WL.bf16_tensor(X[0]).cuda(), Wd)
    dp.calibrate_backward(WL.bf16_tensor(dY).cuda())
    X1 = WL.bf16_tensor(X[1]).cuda()
    y = dp.step(X1, Wd)
    dh, dw = dp.backward(WL.bf16_tensor(dY).cuda(), X1)
    torch.cuda.synchronize()
    s_x, s_w, s_dy = (float(t.item()) for t in (dp.x.last_scale, dp.w.last_scale, dp.g.last_scale))
    rx = O.quant(X[1], O.ACT_IDENTITY, O.E4M3, s_x)
    rw = O.quant(W_bits, O.ACT_IDENTITY, O.E4M3, s_w, want_act=False)
    rd = O.quant(dY, O.ACT_IDENTITY, O.E5M2, s_dy, want_act=False)
    assert np.array_equal(host_u8(dp.x_q), rx["q"])
    assert np.array_equal(host_bits16(dp.act_bf16), rx["act"])
    rows = WL.sample_rows(M, 32, seed=1)
    Yr, S = O.gemm_fwd(rx["q"][rows], rw["q"], s_x, s_w)
    assert_gemm_close(y, Yr, S, rows=rows)
    ref, S = O.gemm_dgrad_act(rd["q"], rw["q"], s_dy, s_w, X[1], O.ACT_IDENTITY, rows=rows)
    assert_gemm_close(dh, ref, S, rows=rows)
    krows = WL.sample_rows(K, 32, seed=2)
    ref, S = O.gemm_wgrad(rx["q"], rd["q"], s_x, s_dy, rows=krows)
    assert_gemm_close(dw, ref, S, rows=krows)
