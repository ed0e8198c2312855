"""Pins of the oracle's MX (microscaling) functions: every block of 32
adjacent values gets its own power-of-two scale ("FP8 training: what it is
and how it works", Trade-offs and edge cases).  The scale is read as Step 2's
format max / amax rounded down to a power of two; these tests pin that
reading, the quantize's reduction to the per-tensor quantize, the property the
pages give for small blocks (an outlier changes only its own block), and the
GEMM's exact sums on small integers.  The GPU path (fp8_quant_mx, fp8_gemm_mx) is
tested against these functions in tests/test_mx_gpu.py."""
import numpy as np
import pytest

import oracle as O
from quantize_fp8_gemm_gb300 import workloads as WL


def _f32_next_up(x):
    return float(np.nextafter(np.float32(x), np.float32(np.inf)))


def test_mx_scale_closed_forms():
    assert O.mx_scale(448.0, O.E4M3) == 1.0
    assert O.mx_scale(1.0, O.E4M3) == 256.0             # 256 <= 448 < 512
    assert O.mx_scale(1.75, O.E4M3) == 256.0            # 1.75 * 256 = 448 exactly: still in range
    assert O.mx_scale(_f32_next_up(1.75), O.E4M3) == 128.0
    assert O.mx_scale(0.0, O.E4M3) == 1.0               # an all-zero block
    assert O.mx_scale(1.0, O.E5M2) == 32768.0           # 32768 <= 57344 < 65536
    assert O.mx_scale(1.75, O.E5M2) == 32768.0          # 1.75 * 32768 = 57344
    assert O.mx_scale(1e-38, O.E4M3) == 2.0 ** 127      # clamped to the 8-bit exponent range
    assert O.mx_scale(3.0e38, O.E4M3) == 2.0 ** -120    # 3e38 * 2^-120 = 226 <= 448 < 451


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_mx_scale_is_the_largest_power_of_two_in_range(fmt):
    rng = np.random.default_rng(fmt)
    fmax = O.fp8_max(fmt)
    amax = (2.0 ** rng.uniform(-60, 60, 4000) * rng.uniform(1, 2, 4000)).astype(np.float32)
    for a in amax:
        s = O.mx_scale(float(a), fmt)
        m, _ = np.frexp(s)
        assert m == 0.5                                  # a power of two
        assert float(a) * s <= fmax < float(a) * 2 * s


@pytest.mark.parametrize("act,fmt", [(O.ACT_RELU2, O.E4M3), (O.ACT_IDENTITY, O.E5M2)])
def test_quant_mx_equals_per_tensor_when_block_maxima_agree(act, fmt):
    """Every block holds the same largest magnitude, so every block scale is the
    same power of two and the MX quantize is the per-tensor quantize with it."""
    rng = np.random.default_rng(3)
    M, K = 24, 256
    x = rng.uniform(-1.5, 1.5, (M, K)).astype(np.float32)
    x[:, ::32] = 2.0                                     # each block's maximum (ReLU^2: 4.0)
    h = WL.to_bf16_bits(x)
    r = O.quant_mx(h, act, fmt)
    s = O.mx_scale(O.amax(h, act), fmt)
    assert np.all(r["scales"] == s)
    p = O.quant(h, act, fmt, s)
    assert np.array_equal(r["q"], p["q"]) and np.array_equal(r["act"], p["act"])
    assert r["amax"] == p["amax"] and r["sat"] == p["sat"] == 0


def test_quant_mx_never_saturates_and_exponent_bytes_invert_the_scales():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((64, 512)) * 2.0 ** rng.integers(-20, 20, (64, 1))).astype(np.float32)
    x[5, 77] = 3.0e5
    x[9, 0:32] = 0.0                                     # an all-zero block
    r = O.quant_mx(WL.to_bf16_bits(x), O.ACT_IDENTITY, O.E4M3)
    assert r["sat"] == 0
    assert r["scales"][9, 0] == 1.0 and np.all(r["q"][9, 0:32] == 0)
    inv = np.ldexp(1.0, r["exps"].astype(np.int64) - 127)
    assert np.array_equal(inv, 1.0 / r["scales"].astype(np.float64))


def test_quant_mx_outlier_changes_only_its_block():
    """A single large value changes the scale and codes of its own 32-value
    block and of no other (the pages' argument for small groups)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((16, 256)).astype(np.float32)
    h0 = WL.to_bf16_bits(x)
    x[7, 100] = 1.0e4
    h1 = WL.to_bf16_bits(x)
    r0, r1 = O.quant_mx(h0, O.ACT_IDENTITY, O.E4M3), O.quant_mx(h1, O.ACT_IDENTITY, O.E4M3)
    diff = r0["scales"] != r1["scales"]
    assert diff.sum() == 1 and diff[7, 100 // 32]
    block = np.zeros_like(r0["q"], dtype=bool)
    block[7, 96:128] = True
    assert np.array_equal(r0["q"][~block], r1["q"][~block])


def test_gemm_mx_equals_per_tensor_when_scales_agree():
    rng = np.random.default_rng(6)
    M, K, N = 20, 128, 24
    xq = O.fp8_encode(rng.standard_normal((M, K)).astype(np.float32) * 30, O.E4M3)
    wq = O.fp8_encode(rng.standard_normal((K, N)).astype(np.float32) * 30, O.E4M3)
    sx = np.full((M, K // 32), 8.0, np.float32)
    sw = np.full((N, K // 32), 0.25, np.float32)
    Y, S = O.gemm_mx(xq, sx, wq, sw)
    Yp, Sp = O.gemm_fwd(xq, wq, 8.0, 0.25)
    assert np.array_equal(Y, Yp) and np.array_equal(S, Sp)


def test_gemm_mx_small_integers_exact():
    """Integer operands and power-of-two block scales: every term and partial
    sum is a short dyadic rational, so the double sum is exact and equals the
    block-wise integer products divided by their scales."""
    rng = np.random.default_rng(7)
    M, K, N = 12, 160, 10
    xi = rng.integers(-8, 9, (M, K))
    wi = rng.integers(-8, 9, (K, N))
    sx = (2.0 ** rng.integers(-3, 4, (M, K // 32))).astype(np.float32)
    sw = (2.0 ** rng.integers(-3, 4, (N, K // 32))).astype(np.float32)
    Y, _ = O.gemm_mx(O.fp8_encode(xi.astype(np.float32), O.E4M3), sx,
                     O.fp8_encode(wi.astype(np.float32), O.E4M3), sw)
    ref = np.zeros((M, N))
    for b in range(K // 32):
        part = xi[:, 32 * b:32 * (b + 1)] @ wi[32 * b:32 * (b + 1), :]
        ref += part / (sx[:, b:b + 1].astype(np.float64) * sw[:, b][None, :].astype(np.float64))
    assert np.array_equal(Y, ref)
