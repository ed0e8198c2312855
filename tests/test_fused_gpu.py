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
from tests.parity import assert_gemm_close, dev_bf16, dev_f32, host_u8

pytestmark = pytest.mark.gpu

TILES = [(-1, 0), (0, 128), (0, 160), (0, 192), (0, 256), (1, 128), (1, 160), (1, 192), (1, 224), (1, 256)]


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


@pytest.mark.parametrize("pair,bn", TILES)
def test_fused_equals_separate_calls(pair, bn):
    try:
        if pair >= 0:
            B.fp8q_gemm_set_tile(pair, bn)
        for (M, N, K) in [(1000, 1600, 640), (300, 272, 400), (129, 144, 1600), (2048, 768, 3072), (16, 64, 96),
                          (1001, 160, 48), (130, 32, 16)]:
            h, w = _inputs(M, N, K, seed=M + N + K + bn)
            r = _run_both(h, w, B.ACT_RELU2, 20.0, 300.0)
            a1, q1, y1, am1, s1, _ = r["separate"]
            a2, q2, y2, am2, s2, _ = r["fused"]
            assert torch.equal(a1.view(torch.int16), a2.view(torch.int16)), (M, N, K)
            assert torch.equal(q1, q2), (M, N, K)
            assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), (M, N, K)
            assert (am1, s1) == (am2, s2)
    finally:
        B.fp8q_gemm_set_tile(-1)


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
