"""Parity of the tcgen05 FP8 GEMMs (fp8_gemm_fwd, fp8_gemm_dgrad) with the
oracle's double-precision GEMM over the dequantised FP8 values.

Floating point: every output must satisfy
    |y_gpu - y_ref| <= ulp_bf16(y_ref) + 1e-5 * sum_k |a_ik b_kj| / (s_a s_b)
(tests/parity.py).  Operands are produced by the oracle's own encoder, so the
two sides share no code.
"""
import numpy as np
import pytest
import torch

import oracle as O
from quantize_fp8_gemm_gb300 import binding as B
from tests.parity import assert_gemm_close, dev_bf16, dev_f32, dev_u8

pytestmark = pytest.mark.gpu


def _codes(x, fmt):
    return O.fp8_encode(np.asarray(x, np.float32), fmt)


def rand_e4m3(shape, seed, scale=1.0):
    x = np.random.default_rng(seed).standard_normal(shape) * scale
    return _codes(x, O.E4M3)


def run_fwd(xq, wq, sx, sw, group=False):
    """xq [M,K], wq [K,N] (oracle layout); the GPU gets W^T [N,K]."""
    M, K = xq.shape
    N = wq.shape[1]
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.fp8_gemm_fwd(dev_u8(xq), dev_u8(np.ascontiguousarray(wq.T)), dev_f32(sx), dev_f32(sw), y,
                   group_mode=int(group), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return y


def test_matmul_worked_example_padded():
    """X = [1, 2], W = [[1,2,3,4],[5,6,7,8]] -> [11, 14, 17, 20], padded to 16 x 16."""
    x = np.zeros((1, 16)); x[0, :2] = [1, 2]
    w = np.zeros((16, 16)); w[0, :4] = [1, 2, 3, 4]; w[1, :4] = [5, 6, 7, 8]
    y = run_fwd(_codes(x, O.E4M3), _codes(w, O.E4M3), 1.0, 1.0)
    assert y[0, :4].float().cpu().tolist() == [11.0, 14.0, 17.0, 20.0]
    assert float(y[0, 4:].abs().max()) == 0.0


def test_small_integers_exact():
    """Integer-valued operands: the FP32 sum is exact, so Y is BF16(exact) bit for bit."""
    rng = np.random.default_rng(5)
    M, K, N = 150, 512, 272
    xi = rng.integers(-8, 9, (M, K))
    wi = rng.integers(-8, 9, (K, N))
    y = run_fwd(_codes(xi, O.E4M3), _codes(wi, O.E4M3), 1.0, 1.0)
    exact = torch.from_numpy((xi @ wi).astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(y.cpu().view(torch.int16), exact.view(torch.int16))


def test_tiny_workload():
    from quantize_fp8_gemm_gb300 import workloads as WL
    w = WL.WORKLOADS["tiny"]
    h = WL.h_preact(w)
    W = WL.w_down(w)
    sx = O.delayed_scale(w.prev_amax, w.margin, O.E4M3)
    rx = O.quant(h, O.ACT_RELU2, O.E4M3, sx)
    sw = O.delayed_scale(O.amax(W, O.ACT_IDENTITY), w.margin, O.E4M3)
    rw = O.quant(W, O.ACT_IDENTITY, O.E4M3, sw)
    Yr, S = O.gemm_fwd(rx["q"], rw["q"], sx, sw)
    y = run_fwd(rx["q"], rw["q"], sx, sw)
    assert_gemm_close(y, Yr, S)


@pytest.mark.parametrize("M,N,K", [
    (64, 64, 256), (128, 128, 128), (200, 272, 384), (129, 144, 1600), (300, 512, 16),
    (1, 16, 48), (513, 768, 3072), (1000, 1600, 640),
])
def test_fwd_shapes(M, N, K):
    xq = rand_e4m3((M, K), seed=M + N + K, scale=30.0)
    wq = rand_e4m3((K, N), seed=M * N + K, scale=30.0)
    sx, sw = 3.5, 0.75
    Yr, S = O.gemm_fwd(xq, wq, sx, sw)
    y = run_fwd(xq, wq, sx, sw)
    assert_gemm_close(y, Yr, S)


def run_dgrad_act(dyq, wq, sdy, sw, h_bits, act):
    M = dyq.shape[0]
    K = wq.shape[0]
    dh = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.fp8_gemm_dgrad_act(dev_u8(dyq), dev_u8(wq), dev_f32(sdy), dev_f32(sw), dev_bf16(h_bits), dh, act=act, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return dh


def _dgrad_act_operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    dyq = _codes(rng.standard_normal((M, N)) * 1000.0, O.E5M2)
    wq = rand_e4m3((K, N), seed=seed + 1, scale=50.0)
    h = O.f32_to_bf16((rng.standard_normal((M, K)) * 2.0).astype(np.float32))
    return dyq, wq, h


@pytest.mark.parametrize("act", [B.ACT_RELU2, B.ACT_RELU])
@pytest.mark.parametrize("M,N,K", [(130, 160, 272), (520, 768, 400), (300, 1600, 640), (64, 64, 3072)])
def test_dgrad_act_against_oracle(M, N, K, act):
    """dH = dX * act'(H) in the dgrad epilogue: within the GEMM tolerance of
    the oracle's double dX times act'(h) (S scaled by |act'(h)|)."""
    dyq, wq, h = _dgrad_act_operands(M, N, K, seed=M + N + K + act)
    ref, S = O.gemm_dgrad_act(dyq, wq, 1024.0, 5.0, h, {B.ACT_RELU2: O.ACT_RELU2, B.ACT_RELU: O.ACT_RELU}[act])
    assert_gemm_close(run_dgrad_act(dyq, wq, 1024.0, 5.0, h, act), ref, S)


@pytest.mark.parametrize("pair,bn", [(0, 128), (0, 192), (0, 256), (1, 128), (1, 192), (1, 224), (1, 256)])
def test_dgrad_act_identity_is_the_dgrad_on_every_tile(pair, bn):
    """With the identity the factor is 1: dH equals fp8_gemm_dgrad's dX bit for
    bit on the same tile, and ReLU^2 stays in tolerance, on a ragged problem."""
    M, N, K = 300, 272, 400
    dyq, wq, h = _dgrad_act_operands(M, N, K, seed=bn + pair)
    try:
        B.fp8q_gemm_set_tile(pair, bn)
        dh = run_dgrad_act(dyq, wq, 1024.0, 5.0, h, B.ACT_IDENTITY)
        dx = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
        B.fp8_gemm_dgrad(dev_u8(dyq), dev_u8(wq), dev_f32(1024.0), dev_f32(5.0), dx)
        torch.cuda.synchronize()
        assert torch.equal(dh.view(torch.int16), dx.view(torch.int16))
        ref, S = O.gemm_dgrad_act(dyq, wq, 1024.0, 5.0, h, O.ACT_RELU2)
        assert_gemm_close(run_dgrad_act(dyq, wq, 1024.0, 5.0, h, B.ACT_RELU2), ref, S)
    finally:
        B.fp8q_gemm_set_tile(-1)


def run_wgrad(xq, dyq, sx, sdy):
    """xq [M,K] E4M3, dyq [M,N] E5M2 (their own layouts); the GPU gets the
    transposed copies X_q^T [K,M] and dY_q^T [N,M]."""
    M, K = xq.shape
    N = dyq.shape[1]
    dw = torch.empty(K, N, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.fp8_gemm_wgrad(dev_u8(np.ascontiguousarray(xq.T)), dev_u8(np.ascontiguousarray(dyq.T)), dev_f32(sx),
                     dev_f32(sdy), dw, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return dw


@pytest.mark.parametrize("M,N,K", [(16, 16, 1), (272, 144, 129), (1008, 1600, 640), (4096, 768, 300),
                                   (6400, 160, 256)])
def test_wgrad_shapes(M, N, K):
    """dW = X^T dY (E4M3 x E5M2, contraction over the M tokens) against the oracle."""
    rng = np.random.default_rng(3 * M + N + K)
    xq = rand_e4m3((M, K), seed=M + K, scale=30.0)
    dyq = _codes(rng.standard_normal((M, N)) * 1000.0, O.E5M2)
    sx, sdy = 3.5, 2.0 ** 10
    Wr, S = O.gemm_wgrad(xq, dyq, sx, sdy)
    assert_gemm_close(run_wgrad(xq, dyq, sx, sdy), Wr, S)


def test_wgrad_small_integers_exact():
    """Integer-valued operands: the FP32 sums are exact, so dW is BF16(exact) bit for bit."""
    rng = np.random.default_rng(9)
    M, N, K = 512, 48, 40
    xi = rng.integers(-8, 9, (M, K))
    di = rng.integers(-6, 7, (M, N))
    dw = run_wgrad(_codes(xi, O.E4M3), _codes(di, O.E5M2), 1.0, 1.0)
    exact = torch.from_numpy((xi.T @ di).astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(dw.cpu().view(torch.int16), exact.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(130, 160, 272), (64, 1600, 512), (300, 256, 6400)])
def test_dgrad_shapes(M, N, K):
    rng = np.random.default_rng(M + N + K)
    dyq = _codes(rng.standard_normal((M, N)) * 1000.0, O.E5M2)
    wq = rand_e4m3((K, N), seed=K, scale=50.0)
    sdy, sw = 2.0 ** 10, 5.0
    Yr, S = O.gemm_dgrad(dyq, wq, sdy, sw)
    dx = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.fp8_gemm_dgrad(dev_u8(dyq), dev_u8(wq), dev_f32(sdy), dev_f32(sw), dx, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_gemm_close(dx, Yr, S)


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (300, 384, 512), (1, 256, 1024)])
def test_group_scaled_fwd(M, N, K):
    rng = np.random.default_rng(M * 3 + N + K)
    xq = rand_e4m3((M, K), seed=M + 1, scale=30.0)
    wq = rand_e4m3((K, N), seed=N + 2, scale=30.0)
    sx = (2.0 ** rng.uniform(-4, 4, (M, K // 128))).astype(np.float32)
    sw = (2.0 ** rng.uniform(-4, 4, (K // 128, N // 128))).astype(np.float32)
    Yr, S = O.gemm_fwd(xq, wq, sx, sw, group=True)
    y = run_fwd(xq, wq, sx, sw, group=True)
    assert_gemm_close(y, Yr, S)


GROUP_TILES = [(0, 128), (0, 192), (0, 256)]


@pytest.mark.parametrize("pair,bn", GROUP_TILES)
def test_group_scaled_every_tile(pair, bn):
    """Group-scaled forward on each group-mode tile (1-CTA, 128, 192 and 256 wide)
    over problems whose M and N leave partial tiles; N = 640 puts a 256-wide
    tile's last scale block past N."""
    try:
        B.fp8q_gemm_set_tile(pair, bn)
        for M, N, K in [(1000, 400, 384), (300, 768, 1152), (129, 144, 256), (257, 640, 128)]:
            rng = np.random.default_rng(M + 5 * N + K)
            xq = rand_e4m3((M, K), seed=M + 11, scale=30.0)
            wq = rand_e4m3((K, N), seed=N + 13, scale=30.0)
            ng = (N + 127) // 128
            sx = (2.0 ** rng.uniform(-4, 4, (M, K // 128))).astype(np.float32)
            sw = (2.0 ** rng.uniform(-4, 4, (K // 128, ng))).astype(np.float32)
            Yr, S = O.gemm_fwd(xq, wq, sx, sw, group=True)
            y = run_fwd(xq, wq, sx, sw, group=True)
            assert_gemm_close(y, Yr, S)
    finally:
        B.fp8q_gemm_set_tile(-1)


def test_constant_sign_long_contraction():
    """All-positive operands over K = 6400: the accumulation error does not cancel,
    which exposes a reduced-precision accumulator."""
    M, N, K = 128, 160, 6400
    rng = np.random.default_rng(77)
    xq = _codes(np.abs(rng.standard_normal((M, K))) * 100 + 1, O.E4M3)
    wq = _codes(np.abs(rng.standard_normal((K, N))) * 100 + 1, O.E4M3)
    Yr, S = O.gemm_fwd(xq, wq, 1.0, 1.0)
    y = run_fwd(xq, wq, 1.0, 1.0)
    assert_gemm_close(y, Yr, S)


TILES = [(0, 128), (0, 160), (0, 192), (0, 256), (1, 128), (1, 160), (1, 192), (1, 224), (1, 256), (1, 384),
         (1, 400)]


@pytest.mark.parametrize("pair,bn", TILES)
def test_every_tile_shape_on_ragged_problems(pair, bn):
    """Each tile shape (1-CTA and 2-SM pair, every width) on problems whose M, N
    and K all leave partial tiles: forward, dgrad and wgrad."""
    try:
        B.fp8q_gemm_set_tile(pair, bn)
        for M, N, K in [(1000, 1600, 640), (300, 272, 400), (129, 144, 1600), (513, 96, 48), (260, 1584, 272)]:
            xq = rand_e4m3((M, K), seed=M + 7 * N + K, scale=30.0)
            wq = rand_e4m3((K, N), seed=3 * M + N + K, scale=30.0)
            Yr, S = O.gemm_fwd(xq, wq, 2.5, 0.5)
            assert_gemm_close(run_fwd(xq, wq, 2.5, 0.5), Yr, S)
        M, N, K = 520, 160, 400
        rng = np.random.default_rng(pair * 1000 + bn)
        dyq = _codes(rng.standard_normal((M, N)) * 1000.0, O.E5M2)
        wq = rand_e4m3((K, N), seed=bn, scale=50.0)
        Dr, Sd = O.gemm_dgrad(dyq, wq, 1024.0, 5.0)
        dx = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
        B.fp8_gemm_dgrad(dev_u8(dyq), dev_u8(wq), dev_f32(1024.0), dev_f32(5.0), dx)
        torch.cuda.synchronize()
        assert_gemm_close(dx, Dr, Sd)
        xq = rand_e4m3((400, 300), seed=bn + 1, scale=30.0)
        dyq2 = _codes(rng.standard_normal((400, 144)) * 1000.0, O.E5M2)
        Wr, Sw = O.gemm_wgrad(xq, dyq2, 3.0, 1024.0)
        assert_gemm_close(run_wgrad(xq, dyq2, 3.0, 1024.0), Wr, Sw)
    finally:
        B.fp8q_gemm_set_tile(-1)


@pytest.mark.parametrize("pair,bn", [(0, 192), (1, 256)])
def test_bounded_wait_reports_timeout_and_context_survives(pair, bn):
    """With the loads held back nothing ever fills the MMA's first stage: the
    bounded wait runs out, the kernel reports FP8Q_DEV_TIMEOUT through the
    status word and exits, and the next GEMM on the same context is correct."""
    M, N, K = 512, 256, 256
    xq = rand_e4m3((M, K), seed=31, scale=30.0)
    wq = rand_e4m3((K, N), seed=32, scale=30.0)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        B.fp8q_gemm_set_tile(pair, bn)
        B.fp8q_gemm_test_hold_loads(True)
        B.fp8_gemm_fwd(dev_u8(xq), dev_u8(np.ascontiguousarray(wq.T)), dev_f32(1.0), dev_f32(1.0), y,
                       status=st)
        torch.cuda.synchronize()
        assert st.item() & B.DEV_TIMEOUT
    finally:
        B.fp8q_gemm_test_hold_loads(False)
        B.fp8q_gemm_set_tile(-1)
    Yr, S = O.gemm_fwd(xq, wq, 1.0, 1.0)
    assert_gemm_close(run_fwd(xq, wq, 1.0, 1.0), Yr, S)
