"""The fused quantize + GEMM kernel (fp8_downproj_fwd) against the separate
fp8_quant_fused + fp8_gemm_fwd calls (bit for bit: same arithmetic, same GEMM
tiles) and against the oracle.  Shapes leave partial quantize units (a warp's
unit is 1 to 128 rows, depending on K), 128-row blocks and tiles; every tile
shape the dispatcher offers is pinned in turn."""
import numpy as np
import pytest
import torch

import oracle as O
from quantize_fp8_gemm_gb300 import binding as B
from quantize_fp8_gemm_gb300 import workloads as WL
from tests.parity import assert_gemm_close, dev_bf16, dev_f32, dev_u8, host_bits16, host_u8

pytestmark = pytest.mark.gpu

TILES = [(-1, 0), (0, 128), (0, 160), (0, 192), (0, 256), (1, 128), (1, 160), (1, 192), (1, 224), (1, 256),
         (1, 400)]


def _inputs(M, N, K, seed):
    rng = np.random.default_rng(seed)
    h = WL.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32) * np.float32(1.5))
    w = WL.to_bf16_bits(rng.standard_normal((K, N)).astype(np.float32) * np.float32(0.05))
    return h, w


def _run_both(h_bits, w_bits, act, sx, sw):
    M, K = h_bits.shape
    N = w_bits.shape[1]
    H = dev_bf16(h_bits)
    wt = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    B.fp8_quant_fused(dev_bf16(w_bits), B.ACT_IDENTITY, B.E4M3, dev_f32(sw), q_t_out=wt)
    s_x, s_w = dev_f32(sx), dev_f32(sw)
    out = {}
    for mode in ("separate", "fused"):
        a = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
        q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        amax = torch.full((1,), -1.0, device="cuda")
        sat = torch.full((1,), 99, dtype=torch.int64, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if mode == "separate":
            B.fp8_quant_fused(H, act, B.E4M3, s_x, act_out=a, q_out=q, amax_out=amax, sat_count=sat)
            B.fp8_gemm_fwd(q, wt, s_x, s_w, y, status=st)
        else:
            ws = torch.full((B.fp8_downproj_workspace_bytes(M),), 0x5A, dtype=torch.uint8, device="cuda")
            B.fp8_downproj_fwd(H, wt, s_x, s_w, q, y, ws, act=act, act_out=a, amax_out=amax, sat_count=sat,
                               status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        out[mode] = (a, q, y, amax.item(), sat.item(), wt)
    return out


@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("pair,bn", TILES)
def test_fused_equals_separate_calls(pair, bn, layout):
    """The one-launch step against the separate quantize and GEMM, bit for bit,
    on every tile and both layouts of its quantize warps (the GEMM-first layout
    exists on the 256- and 400-wide pair tiles; elsewhere the request falls back
    to the quantize-first one)."""
    try:
        B.fp8q_test_set_fused_layout(layout)
        if pair >= 0:
            B.fp8q_gemm_set_tile(pair, bn)
        for (M, N, K) in [(1000, 1600, 640), (300, 272, 400), (129, 144, 1600), (2048, 768, 3072), (16, 64, 96),
                          (1001, 160, 48), (130, 32, 16), (260, 1584, 272)]:
            h, w = _inputs(M, N, K, seed=M + N + K + bn)
            r = _run_both(h, w, B.ACT_RELU2, 20.0, 300.0)
            a1, q1, y1, am1, s1, _ = r["separate"]
            a2, q2, y2, am2, s2, _ = r["fused"]
            assert torch.equal(a1.view(torch.int16), a2.view(torch.int16)), (M, N, K)
            assert torch.equal(q1, q2), (M, N, K)
            assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), (M, N, K)
            assert (am1, s1) == (am2, s2)
    finally:
        B.fp8q_test_set_fused_layout(0)
        B.fp8q_gemm_set_tile(-1)


@pytest.mark.parametrize("act", [B.ACT_RELU2, B.ACT_RELU])
def test_fused_every_bf16_input(act):
    """The one-launch step's quantize (ReLU^2 as packed BF16 max and multiply)
    on every BF16 pattern, NaNs, +-0, subnormals and +-inf included: the BF16
    activation, the E4M3 codes, amax and the saturation count against the
    oracle."""
    M, K, N = 1024, 64, 32
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(M, K)
    H = dev_bf16(pats)
    wt = dev_u8(np.random.default_rng(5).integers(0, 0x7F, (N, K), dtype=np.uint8))  # finite E4M3 codes
    for s in (1.0, 3.0, 2.0 ** -20):
        a = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
        q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        amax = torch.zeros(1, device="cuda")
        sat = torch.zeros(1, dtype=torch.int64, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = torch.zeros(B.fp8_downproj_workspace_bytes(M), dtype=torch.uint8, device="cuda")
        B.fp8_downproj_fwd(H, wt, dev_f32(s), dev_f32(1.0), q, y, ws, act=act, act_out=a, amax_out=amax,
                           sat_count=sat, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        r = O.quant(pats, act, O.E4M3, np.float32(s))
        assert np.array_equal(host_bits16(a), r["act"]), s
        assert np.array_equal(host_u8(q), r["q"]), s
        assert amax.item() == r["amax"] and sat.item() == r["sat"], s


@pytest.mark.parametrize("act", [B.ACT_IDENTITY, B.ACT_RELU, B.ACT_RELU2])
def test_fused_against_oracle(act):
    M, N, K = 520, 384, 1024
    h, w = _inputs(M, N, K, seed=act)
    sx, sw = 12.5, 400.0
    r = _run_both(h, w, act, sx, sw)
    a, q, y, amax, sat, wt = r["fused"]
    ro = O.quant(h, act, O.E4M3, sx)
    rw = O.quant(w, O.ACT_IDENTITY, O.E4M3, sw, want_act=False)
    assert np.array_equal(host_u8(q), ro["q"])
    assert np.array_equal(a.view(torch.int16).cpu().numpy().view(np.uint16), ro["act"])
    assert amax == ro["amax"] and sat == ro["sat"]
    Yr, S = O.gemm_fwd(ro["q"], rw["q"], sx, sw)
    assert_gemm_close(y, Yr, S)


def test_fused_without_optional_outputs():
    M, N, K = 640, 256, 512
    h, w = _inputs(M, N, K, seed=5)
    H = dev_bf16(h)
    wt = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    B.fp8_quant_fused(dev_bf16(w), B.ACT_IDENTITY, B.E4M3, dev_f32(300.0), q_t_out=wt)
    q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(B.fp8_downproj_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    B.fp8_downproj_fwd(H, wt, dev_f32(20.0), dev_f32(300.0), q, y, ws)
    torch.cuda.synchronize()
    ro = O.quant(h, O.ACT_RELU2, O.E4M3, 20.0, want_act=False)
    assert np.array_equal(host_u8(q), ro["q"])


@pytest.mark.parametrize("pair,bn", [(-1, 0), (0, 192), (1, 256)])
def test_fused_weight_cast_equals_separate_calls(pair, bn):
    """fp8_downproj_fwd_ex with the master weight: the kernel's own W cast
    (W_q^T, W_q, amax_w) and the GEMM that reads it equal fp8_quant_fused on W
    followed by the separate quantize and GEMM, bit for bit.  Shapes leave a
    partial 256-column weight unit (N = 272, 144) and 8-row groups over K."""
    try:
        if pair >= 0:
            B.fp8q_gemm_set_tile(pair, bn)
        for (M, N, K) in [(1000, 272, 640), (2048, 768, 3072), (129, 144, 1600), (0, 272, 256)]:
            h, w = _inputs(max(M, 1), N, K, seed=M + N + K)
            h = h[:M]
            H, Wd = dev_bf16(h), dev_bf16(w)
            sx, sw = dev_f32(20.0), dev_f32(300.0)
            # separate: W cast, H quantize, GEMM
            wt1 = torch.empty(N, K, dtype=torch.uint8, device="cuda")
            wq1 = torch.empty(K, N, dtype=torch.uint8, device="cuda")
            aw1 = torch.zeros(1, device="cuda")
            B.fp8_quant_fused(Wd, B.ACT_IDENTITY, B.E4M3, sw, q_out=wq1, q_t_out=wt1, amax_out=aw1)
            a1 = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
            q1 = torch.empty(M, K, dtype=torch.uint8, device="cuda")
            y1 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            ax1, s1 = torch.zeros(1, device="cuda"), torch.zeros(1, dtype=torch.int64, device="cuda")
            B.fp8_quant_fused(H, B.ACT_RELU2, B.E4M3, sx, act_out=a1, q_out=q1, amax_out=ax1, sat_count=s1)
            if M:
                B.fp8_gemm_fwd(q1, wt1, sx, sw, y1)
            # one kernel, twice in a row on one workspace: flags 0, then ACCUMULATE on zeroed accumulators
            ws = torch.full((max(B.fp8_downproj_workspace_bytes(M), 256),), 0x5A, dtype=torch.uint8, device="cuda")
            for flags in (0, B.ACCUMULATE):
                wt2 = torch.full((N, K), 7, dtype=torch.uint8, device="cuda")
                wq2 = torch.empty(K, N, dtype=torch.uint8, device="cuda")
                aw2 = torch.full((1,), -1.0 if flags == 0 else 0.0, device="cuda")
                a2 = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
                q2 = torch.empty(M, K, dtype=torch.uint8, device="cuda")
                y2 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
                ax2 = torch.full((1,), -1.0 if flags == 0 else 0.0, device="cuda")
                s2 = torch.full((1,), 9 if flags == 0 else 0, dtype=torch.int64, device="cuda")
                st = torch.zeros(1, dtype=torch.int32, device="cuda")
                B.fp8_downproj_fwd_ex(H, wt2, sx, sw, q2, y2, ws, w=Wd, w_q=wq2, amax_w=aw2, act=B.ACT_RELU2,
                                      act_out=a2, amax_out=ax2, sat_count=s2, flags=flags, status=st)
                torch.cuda.synchronize()
                assert st.item() == 0
                assert torch.equal(wt1, wt2) and torch.equal(wq1, wq2) and aw1.item() == aw2.item(), (M, N, K)
                assert torch.equal(q1, q2) and torch.equal(a1.view(torch.int16), a2.view(torch.int16))
                assert ax1.item() == ax2.item() and s1.item() == s2.item()
                assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), (M, N, K, flags)
            assert int(ws[:B.fp8_downproj_workspace_bytes(M)].sum().item()) == 0, "the kernel leaves its counts at zero"
    finally:
        B.fp8q_gemm_set_tile(-1)


def test_fused_step_runs_history_updates():
    """The kernel's last CTA runs both delayed-scale updates: a good amax gives
    the oracle's next scale and clears the other slot's accumulators; an
    all-negative H under ReLU^2 (amax 0) keeps the previous scale and flags
    FP8Q_DEV_BAD_AMAX."""
    M, N, K = 600, 272, 512
    h, w = _inputs(M, N, K, seed=41)
    for bad in (False, True):
        hb = h.copy()
        if bad:
            hb = WL.to_bf16_bits(-np.abs(WL.bf16_tensor(h).float().numpy()) - 1.0)
        H, Wd = dev_bf16(hb), dev_bf16(w)
        scales_x = torch.tensor([20.0, 1.0], device="cuda")
        scales_w = torch.tensor([300.0, 1.0], device="cuda")
        hist_x, hist_w = torch.zeros(2, device="cuda"), torch.zeros(2, device="cuda")
        head_x, head_w = torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
        amax_x = torch.zeros(2, device="cuda")
        amax_w = torch.zeros(2, device="cuda")
        amax_x[1] = 5.0  # the other slot: must be cleared
        sats = torch.tensor([0, 77], dtype=torch.int64, device="cuda")
        st_x, st_w = torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
        wt = torch.empty(N, K, dtype=torch.uint8, device="cuda")
        q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(B.fp8_downproj_workspace_bytes(M), dtype=torch.uint8, device="cuda")
        hx = B.history_args(hist_x, head_x, 2.0, B.E4M3, scales_x[1:2], scale_prev=scales_x[0:1], status=st_x,
                            amax_clear=amax_x[1:2], sat_clear=sats[1:2])
        hw = B.history_args(hist_w, head_w, 2.0, B.E4M3, scales_w[1:2], scale_prev=scales_w[0:1], status=st_w,
                            amax_clear=amax_w[1:2])
        B.fp8_downproj_fwd_ex(H, wt, scales_x[0:1], scales_w[0:1], q, y, ws, w=Wd, amax_w=amax_w[0:1],
                              amax_out=amax_x[0:1], sat_count=sats[0:1], hist_x=hx, hist_w=hw,
                              flags=B.ACCUMULATE)
        torch.cuda.synchronize()
        ro = O.quant(hb, O.ACT_RELU2, O.E4M3, 20.0, want_act=False)
        rw_amax = O.amax(w, O.ACT_IDENTITY)
        assert amax_x[0].item() == ro["amax"] and amax_w[0].item() == rw_amax
        assert amax_x[1].item() == 0.0 and sats[1].item() == 0
        assert scales_w[1].item() == O.delayed_scale(rw_amax, 2.0, O.E4M3) and st_w.item() == 0
        assert int(head_x.item()) == 1 and hist_x[1].item() == ro["amax"]
        if bad:
            assert ro["amax"] == 0.0
            assert scales_x[1].item() == 20.0 and st_x.item() & B.DEV_BAD_AMAX
        else:
            assert scales_x[1].item() == O.delayed_scale(ro["amax"], 2.0, O.E4M3) and st_x.item() == 0
        assert int(ws.sum().item()) == 0


@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("ctas", [2, 37, 64, 400])
def test_fused_any_grid_gives_the_same_result(ctas, layout):
    """The one-launch step's CTAs take their quantize and weight-cast work by
    ticket, so no CTA waits on work held by a CTA that is not running.  A grid
    smaller than the SM count (2, 37, 64 CTAs) and one larger than the GPU
    holds at once (400 CTAs: the last ones can only start after earlier ones
    have finished) give the default grid's outputs bit for bit, and the
    workspace ends zero."""
    M, N, K = 2048, 768, 3072
    h, w = _inputs(M, N, K, seed=ctas)
    H, Wd = dev_bf16(h), dev_bf16(w)
    sx, sw = dev_f32(20.0), dev_f32(300.0)
    outs = []
    try:
        B.fp8q_test_set_fused_layout(layout)
        for grid in (0, ctas):
            B.fp8q_test_set_fused_grid(grid)
            o = dict(wt=torch.empty(N, K, dtype=torch.uint8, device="cuda"),
                     wq=torch.empty(K, N, dtype=torch.uint8, device="cuda"),
                     a=torch.empty(M, K, dtype=torch.bfloat16, device="cuda"),
                     q=torch.empty(M, K, dtype=torch.uint8, device="cuda"),
                     y=torch.empty(M, N, dtype=torch.bfloat16, device="cuda"),
                     aw=torch.zeros(1, device="cuda"), ax=torch.zeros(1, device="cuda"),
                     sx=torch.zeros(1, dtype=torch.int64, device="cuda"),
                     sw=torch.zeros(1, dtype=torch.int64, device="cuda"),
                     st=torch.zeros(1, dtype=torch.int32, device="cuda"),
                     ws=torch.zeros(B.fp8_downproj_workspace_bytes(M), dtype=torch.uint8, device="cuda"))
            B.fp8_downproj_fwd_ex(H, o["wt"], sx, sw, o["q"], o["y"], o["ws"], w=Wd, w_q=o["wq"], amax_w=o["aw"],
                                  sat_w=o["sw"], act=B.ACT_RELU2, act_out=o["a"], amax_out=o["ax"],
                                  sat_count=o["sx"], status=o["st"])
            torch.cuda.synchronize()
            assert o["st"].item() == 0 and int(o["ws"].sum().item()) == 0
            outs.append(o)
    finally:
        B.fp8q_test_set_fused_grid(0)
        B.fp8q_test_set_fused_layout(0)
    ref, got = outs
    for k in ("wt", "wq", "q", "aw", "ax", "sx", "sw"):
        assert torch.equal(ref[k], got[k]), k
    for k in ("a", "y"):
        assert torch.equal(ref[k].view(torch.int16), got[k].view(torch.int16)), k
    ro = O.quant(h, O.ACT_RELU2, O.E4M3, 20.0, want_act=False)
    assert np.array_equal(host_u8(got["q"]), ro["q"]) and got["sx"].item() == ro["sat"]


def test_fused_weight_saturation_count():
    """The kernel's weight cast counts the values its scale saturates (the
    overflow test of detect-and-recompute), like the standalone cast and the
    oracle: a scale with margin 2 saturates nothing, one 8x larger (margin
    0.25) exactly the oracle's count of values."""
    M, N, K = 512, 272, 640
    h, w = _inputs(M, N, K, seed=8)
    amax_w = O.amax(w, O.ACT_IDENTITY)
    for big in (False, True):
        s_w = O.delayed_scale(amax_w, 0.25 if big else 2.0, O.E4M3)
        sat_w = torch.full((1,), 5, dtype=torch.int64, device="cuda")
        sat_w2 = torch.full((1,), 5, dtype=torch.int64, device="cuda")
        wt = torch.empty(N, K, dtype=torch.uint8, device="cuda")
        q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(B.fp8_downproj_workspace_bytes(M), dtype=torch.uint8, device="cuda")
        B.fp8_downproj_fwd_ex(dev_bf16(h), wt, dev_f32(20.0), dev_f32(s_w), q, y, ws, w=dev_bf16(w),
                              sat_w=sat_w, act=B.ACT_RELU2)
        B.fp8_quant_fused(dev_bf16(w), B.ACT_IDENTITY, B.E4M3, dev_f32(s_w), q_t_out=torch.empty_like(wt),
                          sat_count=sat_w2)
        torch.cuda.synchronize()
        rw = O.quant(w, O.ACT_IDENTITY, O.E4M3, s_w, want_act=False)
        assert sat_w.item() == sat_w2.item() == rw["sat"]
        assert (rw["sat"] > 0) == big
