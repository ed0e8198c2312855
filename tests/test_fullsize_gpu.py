"""Parity at the workloads' full sizes, in the configuration the benchmark uses.

The fused quantize is checked element by element over the whole tensor (the
oracle runs on all host cores); the GEMMs on a seeded sample of output rows
that includes rows at 128-row tile edges, against the oracle's double GEMM.
"""
import numpy as np
import pytest
import torch

import oracle as O
from quantize_fp8_gemm_gb300 import binding as B
from quantize_fp8_gemm_gb300 import workloads as WL
from quantize_fp8_gemm_gb300.downproj import Fp8DownProj
from tests.parity import assert_gemm_close, dev_f32, host_u8

pytestmark = pytest.mark.gpu


def _forward_check(name, group=False, act=B.ACT_RELU2):
    w = WL.WORKLOADS[name]
    h_bits, w_bits = WL.h_preact(w, 0), WL.w_down(w)
    H, Wd = WL.bf16_tensor(h_bits).cuda(), WL.bf16_tensor(w_bits).cuda()
    dp = Fp8DownProj(w.M, w.K, w.N, act=act, margin=w.margin, group=group, keep_act=False)
    dp.calibrate(H, Wd)
    sx, sw = float(dp.x.scale.item()), float(dp.w.scale.item())
    y = dp.step(H, Wd)
    torch.cuda.synchronize()
    assert int(dp.gemm_status.item()) == 0
    rows = WL.sample_rows(w.M, 256, seed=w.seed)
    if group:
        rx = O.quant_group(h_bits, act, O.E4M3, 1, want_act=False)
        rw = O.quant_group(w_bits, O.ACT_IDENTITY, O.E4M3, 128, want_act=False, want_qt=True)
        assert np.array_equal(dp.x_gscale.cpu().numpy(), rx["scales"])
        assert np.array_equal(dp.w_gscale.cpu().numpy(), rw["scales"])
        sxa, swa = rx["scales"], rw["scales"]
    else:
        assert sx == O.delayed_scale(O.amax(h_bits, act), w.margin, O.E4M3)
        rx = O.quant(h_bits, act, O.E4M3, sx, want_act=False)
        rw = O.quant(w_bits, O.ACT_IDENTITY, O.E4M3, sw, want_act=False, want_qt=True)
        sxa, swa = sx, sw
    assert np.array_equal(host_u8(dp.x_q), rx["q"])
    assert np.array_equal(host_u8(dp.wt_q), rw["q_t"])
    assert int(dp.sat.item()) == rx["sat"]
    if group:
        Yr, S = O.gemm_fwd(rx["q"], rw["q"], sxa, swa, group=True, rows=rows)
    else:
        Yr, S = O.gemm_fwd(rx["q"], rw["q"], sxa, swa, rows=rows)
    assert_gemm_close(y, Yr, S, rows=rows)
    return rx, y


def test_gpt2s_forward():
    _forward_check("gpt2s")


def test_outlier_forward_per_tensor_and_group():
    """Per-tensor vs 1x128 group scales on the outlier workload: both in
    tolerance, and the group path flushes far fewer values to zero."""
    w = WL.WORKLOADS["outlier"]
    rt, _ = _forward_check("outlier", act=B.ACT_IDENTITY)
    rg, _ = _forward_check("outlier", group=True, act=B.ACT_IDENTITY)
    h_bits = WL.h_preact(w, 0)
    nz = O.bf16_to_f32(h_bits) != 0
    zt = np.mean((rt["q"] & 0x7F)[nz] == 0)
    zg = np.mean((rg["q"] & 0x7F)[nz] == 0)
    assert zg < zt


def test_gpt2xl_forward_dgrad_and_wgrad():
    """GPT-2-XL shape: H [131072, 6400] -> Y [131072, 1600]; dY [131072, 1600]
    in E5M2 -> dX = dY W^T [131072, 6400]; the transposed casts of the
    activation and of dY -> dW = X^T dY [6400, 1600]."""
    w = WL.WORKLOADS["gpt2xl"]
    h_bits, w_bits = WL.h_preact(w, 0), WL.w_down(w)
    H, Wd = WL.bf16_tensor(h_bits).cuda(), WL.bf16_tensor(w_bits).cuda()
    dp = Fp8DownProj(w.M, w.K, w.N, margin=w.margin, with_dgrad=True, keep_act=False)
    dp.calibrate(H, Wd)
    sx, sw = float(dp.x.scale.item()), float(dp.w.scale.item())
    y = dp.step(H, Wd)
    torch.cuda.synchronize()
    rows = WL.sample_rows(w.M, 128, seed=4)
    rx = O.quant(h_bits, O.ACT_RELU2, O.E4M3, sx, want_act=False)
    rw = O.quant(w_bits, O.ACT_IDENTITY, O.E4M3, sw, want_act=False, want_qt=True)
    assert np.array_equal(host_u8(dp.x_q), rx["q"])
    assert np.array_equal(host_u8(dp.wt_q), rw["q_t"])
    assert np.array_equal(host_u8(dp.w_q), rw["q"])
    Yr, S = O.gemm_fwd(rx["q"], rw["q"], sx, sw, rows=rows)
    assert_gemm_close(y, Yr, S, rows=rows)
    del y
    # the activation's transposed E4M3 copy (the weight gradient's operand), same scale
    xqt = torch.empty(w.K, w.M, dtype=torch.uint8, device="cuda")
    B.fp8_quant_fused(H, B.ACT_RELU2, B.E4M3, dev_f32(sx), q_t_out=xqt, amax_out=torch.zeros(1, device="cuda"))
    torch.cuda.synchronize()
    del H
    assert np.array_equal(host_u8(xqt), rx["q"].T)

    dy_bits = WL.dy_grad(w)
    s_dy = O.delayed_scale(O.amax(dy_bits, O.ACT_IDENTITY), w.margin, O.E5M2)
    dY = WL.bf16_tensor(dy_bits).cuda()
    dyq = torch.empty(w.M, w.N, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, device="cuda")
    B.fp8_quant_fused(dY, B.ACT_IDENTITY, B.E5M2, dev_f32(s_dy), q_out=dyq, amax_out=amax)
    rdy = O.quant(dy_bits, O.ACT_IDENTITY, O.E5M2, s_dy, want_act=False)
    assert np.array_equal(host_u8(dyq), rdy["q"])
    assert float(amax.item()) == rdy["amax"]
    dx = torch.empty(w.M, w.K, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.fp8_gemm_dgrad(dyq, dp.w_q, dev_f32(s_dy), dp.w.scale, dx, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    Dr, Sd = O.gemm_dgrad(rdy["q"], rw["q"], s_dy, sw, rows=rows)
    assert_gemm_close(dx, Dr, Sd, rows=rows)
    del dx

    dyqt = torch.empty(w.N, w.M, dtype=torch.uint8, device="cuda")
    B.fp8_quant_fused(dY, B.ACT_IDENTITY, B.E5M2, dev_f32(s_dy), q_t_out=dyqt, amax_out=amax)
    dw = torch.empty(w.K, w.N, dtype=torch.bfloat16, device="cuda")
    B.fp8_gemm_wgrad(xqt, dyqt, dev_f32(sx), dev_f32(s_dy), dw, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(host_u8(dyqt), rdy["q"].T)
    krows = WL.sample_rows(w.K, 48, seed=5)
    Wr, Sw = O.gemm_wgrad(rx["q"], rdy["q"], sx, s_dy, rows=krows)
    assert_gemm_close(dw, Wr, Sw, rows=krows)
