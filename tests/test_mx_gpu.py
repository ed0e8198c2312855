"""MXFP8 on the GPU against the oracle ("FP8 training: what it is and how it
works", Trade-offs and edge cases: one power-of-two scale per block of 32
adjacent values).

fp8_quant_mx: codes, scale bytes, the BF16 activation copy, amax and the
saturation count bit-exact against oref_quant_mx, in both modes (blocks along
the rows of X; blocks down the columns of W, written transposed), over values
spread across 40 binades, all-zero blocks, a lone outlier and BF16 subnormals.
fp8_gemm_mx: within the GEMM tolerance of the oracle's double sum over the
dequantised codes, for every tile (1-CTA and 2-SM pair, each width), ragged
M / N / K, both formats, and
block scales that differ from block to block on both operands; a structured
case (one non-zero 32-value block per row) checks that each MMA takes the
scale of its own block and row / column."""
import numpy as np
import pytest
import torch

import oracle as O
from quantize_fp8_gemm_gb300 import binding as B
from quantize_fp8_gemm_gb300 import workloads as WL
from tests.parity import assert_gemm_close, dev_bf16, dev_u8, host_bits16, host_u8, mx_scale_bytes, mx_tile, mx_untile

pytestmark = pytest.mark.gpu


def _spread(rng, M, K, decades=20):
    """Normals with a per-row and per-32-block power-of-two spread, a zero block,
    a lone outlier and a block of BF16 subnormals."""
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-decades, decades, (M, 1))).astype(np.float32)
    x *= np.exp2(rng.integers(-6, 7, (M, K // 32))).repeat(32, axis=1).astype(np.float32)
    x[0, :32] = 0.0
    if M > 1:
        x[1, 5] = 3.0e4
    if M > 2 and K >= 64:
        x[2, 32:64] = rng.standard_normal(32).astype(np.float32) * np.float32(1e-39)
    return WL.to_bf16_bits(x)


def _quant_rows(h_bits, act, fmt):
    M, K = h_bits.shape
    q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    sf = torch.full((mx_scale_bytes(M, K // 32),), 0xAA, dtype=torch.uint8, device="cuda")
    a = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    amax = torch.full((1,), -1.0, device="cuda")
    sat = torch.full((1,), 7, dtype=torch.int64, device="cuda")
    B.fp8_quant_mx(dev_bf16(h_bits), act, fmt, act_out=a, q_out=q, sf_out=sf, amax_out=amax, sat_count=sat)
    torch.cuda.synchronize()
    return q, sf, a, amax.item(), sat.item()


def _quant_cols(w_bits, fmt):
    R, C = w_bits.shape
    qt = torch.empty(C, R, dtype=torch.uint8, device="cuda")
    sft = torch.full((mx_scale_bytes(C, R // 32),), 0xAA, dtype=torch.uint8, device="cuda")
    amax = torch.full((1,), -1.0, device="cuda")
    B.fp8_quant_mx(dev_bf16(w_bits), B.ACT_IDENTITY, fmt, q_t_out=qt, sf_t_out=sft, amax_out=amax)
    torch.cuda.synchronize()
    return qt, sft, amax.item()


@pytest.mark.parametrize("act,fmt", [(B.ACT_RELU2, B.E4M3), (B.ACT_IDENTITY, B.E4M3), (B.ACT_RELU, B.E5M2),
                                     (B.ACT_IDENTITY, B.E5M2)])
@pytest.mark.parametrize("M,K", [(300, 640), (5, 32), (1024, 4096), (129, 96), (130, 224)])
def test_quant_mx_rows_against_oracle(act, fmt, M, K):
    rng = np.random.default_rng(M * 7 + K + act * 3 + fmt)
    h = _spread(rng, M, K)
    q, sf, a, amax, sat = _quant_rows(h, act, fmt)
    r = O.quant_mx(h, act, fmt)
    got, pad = mx_untile(host_u8(sf), M, K // 32, pad=True)
    assert np.array_equal(got, r["exps"]), "scale bytes"
    assert (pad == 127).all(), "padding blocks of the scale layout"
    assert np.array_equal(host_u8(q), r["q"]), "codes"
    assert np.array_equal(host_bits16(a), r["act"]), "BF16 activation copy"
    assert amax == r["amax"] and sat == r["sat"] == 0


@pytest.mark.parametrize("fmt", [B.E4M3, B.E5M2])
@pytest.mark.parametrize("R,C", [(640, 272), (32, 16), (6400, 1600), (96, 48), (160, 144)])
def test_quant_mx_columns_against_oracle(fmt, R, C):
    """W [R,C] -> W_q^T [C,R] with one scale per 32 rows of a column: the oracle's
    row-block quantize of W^T."""
    rng = np.random.default_rng(R + C + fmt)
    w = _spread(rng, C, R, decades=8).T.copy()  # [R,C]; blocks of 32 down its columns
    qt, sft, amax = _quant_cols(w, fmt)
    r = O.quant_mx(np.ascontiguousarray(w.T), O.ACT_IDENTITY, fmt, want_act=False)
    got, pad = mx_untile(host_u8(sft), C, R // 32, pad=True)
    assert np.array_equal(got, r["exps"]), "scale bytes"
    assert (pad == 127).all(), "padding blocks of the scale layout"
    assert np.array_equal(host_u8(qt), r["q"]), "transposed codes"
    assert amax == r["amax"]


def _scales(sf_tiled, rows, KB):
    """The oracle's block scales s_b = 2^(127 - byte) (the byte is 1/s_b's exponent) of a
    tiled scale buffer's [rows, KB] grid."""
    return np.ldexp(1.0, 127 - mx_untile(host_u8(sf_tiled), rows, KB).astype(np.int64)).astype(np.float32)


TILES = [(0, 0), (0, 128), (0, 256), (1, 128), (1, 256)]


@pytest.mark.parametrize("pair,bn", TILES)
@pytest.mark.parametrize("M,N,K", [(300, 272, 640), (128, 128, 128), (1000, 1600, 1280), (77, 16, 32), (513, 400, 96),
                                   (2125, 1024, 1024)])
def test_gemm_mx_against_oracle(pair, bn, M, N, K):
    """Ragged M / N / K for every tile; 2-SM pair tiles whose second CTA's rows
    lie partly or wholly past M (M = 300, 2125); K = 96 (three blocks per row:
    the scale atoms' padding block is read) and K = 1280 (ten); M <= 128 takes
    the 1-CTA tile of the pinned width; 2125 x 1024 gives every CTA or pair
    several tiles, so the stage ring and the accumulators wrap."""
    rng = np.random.default_rng(M + N + K + bn + pair)
    h = _spread(rng, M, K, decades=6)
    w = _spread(rng, N, K, decades=6).T.copy()  # W [K,N]
    q, sf, _, _, _ = _quant_rows(h, B.ACT_RELU2, B.E4M3)
    qt, sft, _ = _quant_cols(w, B.E4M3)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        B.fp8q_mx_set_tile(pair, bn)
        B.fp8_gemm_mx(q, sf, qt, sft, y, status=st)
        torch.cuda.synchronize()
    finally:
        B.fp8q_mx_set_tile(0, 0)
    assert st.item() == 0
    xq, xs = host_u8(q), _scales(sf, M, K // 32)
    wq, ws = np.ascontiguousarray(host_u8(qt).T), _scales(sft, N, K // 32)
    Yr, S = O.gemm_mx(xq, xs, wq, ws)
    assert_gemm_close(y, Yr, S)


@pytest.mark.parametrize("fmt_x,fmt_w", [(B.E5M2, B.E4M3), (B.E4M3, B.E5M2), (B.E5M2, B.E5M2)])
def test_gemm_mx_formats(fmt_x, fmt_w):
    M, N, K = 384, 256, 512
    rng = np.random.default_rng(11 + fmt_x * 2 + fmt_w)
    h = _spread(rng, M, K, decades=4)
    w = _spread(rng, N, K, decades=4).T.copy()
    q, sf, _, _, _ = _quant_rows(h, B.ACT_IDENTITY, fmt_x)
    qt, sft, _ = _quant_cols(w, fmt_w)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    B.fp8_gemm_mx(q, sf, qt, sft, y, fmt_x=fmt_x, fmt_w=fmt_w)
    torch.cuda.synchronize()
    Yr, S = O.gemm_mx(host_u8(q), _scales(sf, M, K // 32), np.ascontiguousarray(host_u8(qt).T),
                      _scales(sft, N, K // 32), fmt_x=fmt_x, fmt_w=fmt_w)
    assert_gemm_close(y, Yr, S)


@pytest.mark.parametrize("pair,bn", TILES[1:])
def test_gemm_mx_each_block_takes_its_own_scale(pair, bn):
    """Codes 1.0 in a single 32-value block per row of X (block j = row % (K/32))
    and per column of W (block j' = column % (K/32)), all other codes 0, and a
    different random scale byte for every block of both operands: Y[i,n] is
    32 * 2^(sx[i,j] - 127) * 2^(sw[n,j] - 127) where the two blocks meet, else
    0 -- exact, so any scale taken from the wrong row, column or block shows
    (with pair tiles: from the other CTA's rows or the other half of B)."""
    M, N, K = 256, 384, 256
    KB = K // 32
    rng = np.random.default_rng(bn + pair)
    one = 0x38  # E4M3 1.0
    xq = np.zeros((M, K), np.uint8)
    wq_t = np.zeros((N, K), np.uint8)
    for i in range(M):
        j = i % KB
        xq[i, 32 * j:32 * j + 32] = one
    for n in range(N):
        j = (n // 3) % KB
        wq_t[n, 32 * j:32 * j + 32] = one
    sx = rng.integers(118, 137, (M, KB)).astype(np.uint8)
    sw = rng.integers(118, 137, (N, KB)).astype(np.uint8)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    try:
        B.fp8q_mx_set_tile(pair, bn)
        B.fp8_gemm_mx(dev_u8(xq), dev_u8(mx_tile(sx)), dev_u8(wq_t), dev_u8(mx_tile(sw)), y)
        torch.cuda.synchronize()
    finally:
        B.fp8q_mx_set_tile(0, 0)
    got = y.float().cpu().numpy().astype(np.float64)
    want = np.zeros((M, N))
    for i in range(M):
        for n in range(N):
            j = i % KB
            if (n // 3) % KB == j:
                want[i, n] = 32.0 * np.ldexp(1.0, int(sx[i, j]) - 127 + int(sw[n, j]) - 127)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} outputs differ; first {tuple(bad[0])}: got {got[tuple(bad[0])]}, want {want[tuple(bad[0])]}"


@pytest.mark.parametrize("name", ["outlier", "gpt2xl"])
def test_mx_workload_shapes(name):
    """The outlier workload (16384 x 4096 -> 1024, 1 in 4096 entries at +-1e5)
    and the GPT-2-XL shape (131072 x 6400 -> 1600) through the MX path: the
    full tensors' codes and scale bytes bit-exact, Y in tolerance on sampled
    rows (tile edges among them)."""
    w = WL.WORKLOADS[name]
    h = WL.h_preact(w)
    wb = WL.w_down(w)
    q, sf, a, amax, sat = _quant_rows(h, B.ACT_RELU2, B.E4M3)
    qt, sft, _ = _quant_cols(wb, B.E4M3)
    r = O.quant_mx(h, O.ACT_RELU2, O.E4M3, want_act=False)
    assert np.array_equal(mx_untile(host_u8(sf), w.M, w.K // 32), r["exps"]) and np.array_equal(host_u8(q), r["q"])
    assert amax == r["amax"] and sat == 0
    rw = O.quant_mx(np.ascontiguousarray(wb.T), O.ACT_IDENTITY, O.E4M3, want_act=False)
    assert np.array_equal(mx_untile(host_u8(sft), w.N, w.K // 32), rw["exps"])
    assert np.array_equal(host_u8(qt), rw["q"])
    y = torch.empty(w.M, w.N, dtype=torch.bfloat16, device="cuda")
    B.fp8_gemm_mx(q, sf, qt, sft, y)
    torch.cuda.synchronize()
    rows = WL.sample_rows(w.M, 24, seed=44)
    Yr, S = O.gemm_mx(r["q"], r["scales"], np.ascontiguousarray(rw["q"].T), rw["scales"], rows=rows)
    assert_gemm_close(y, Yr, S, rows=rows)
