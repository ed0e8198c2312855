"""Pins for the CPU oracle: each oracle function is tied to something other than
itself -- values the pages print (tests/golden/), closed forms, exhaustive sweeps
over all FP8 codes, or an independent library routine (torch's float8 and bf16
conversions, numpy's matmul).  No GPU is used.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O


def rel_close(a, b, tol):
    return abs(a - b) <= tol * abs(b)


# ----------------------------------------------------------------------------
# FP8 format constants ("FP8 training: what it is and how it works", Step 1/2;
# "FP8 Training & Inference", FP8 Formats, Exercise 1)
# ----------------------------------------------------------------------------
def _finite_positive_values(fmt):
    codes = np.arange(128, dtype=np.uint8)
    v = O.fp8_decode(codes, fmt)
    return codes[np.isfinite(v)], v[np.isfinite(v)]


def test_e4m3_constants(golden):
    g = golden("fp8_formats.txt")
    codes, vals = _finite_positive_values(O.E4M3)
    assert vals.max() == g["e4m3.max"] == O.fp8_max(O.E4M3)
    one = int(np.where(vals == 1.0)[0][0])
    assert vals[one + 1] - 1.0 == g["e4m3.gap_after_one"]
    smallest = vals[vals > 0].min()
    assert round(smallest, 6) == g["e4m3.min_subnormal"]
    assert smallest == 2.0 ** -9
    # smallest normal: the first code with a nonzero exponent field
    assert O.fp8_decode(np.array([0x08], np.uint8), O.E4M3)[0] == g["e4m3.min_normal"]
    binade = vals[(vals >= 1.0) & (vals < 2.0)]
    assert binade.size == g["e4m3.values_per_binade"]


def test_e5m2_constants(golden):
    g = golden("fp8_formats.txt")
    codes, vals = _finite_positive_values(O.E5M2)
    assert vals.max() == g["e5m2.max"] == O.fp8_max(O.E5M2)
    one = int(np.where(vals == 1.0)[0][0])
    assert vals[one + 1] - 1.0 == g["e5m2.gap_after_one"]
    smallest = vals[vals > 0].min()
    assert round(smallest, 6) == g["e5m2.min_nonzero"]
    binade = vals[(vals >= 1.0) & (vals < 2.0)]
    assert binade.size == g["e5m2.values_per_binade"]
    assert O.fp8_max(O.E5M2) / O.fp8_max(O.E4M3) == g["range_ratio_e5m2_over_e4m3"]


# ----------------------------------------------------------------------------
# Exhaustive sweep over all 256 codes of each format
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_all_codes_decode_encode(fmt):
    codes = np.arange(256, dtype=np.uint8)
    v = O.fp8_decode(codes, fmt)
    nan_codes = set(codes[np.isnan(v)].tolist())
    inf_codes = set(codes[np.isinf(v)].tolist())
    if fmt == O.E4M3:
        assert nan_codes == {0x7F, 0xFF} and not inf_codes
    else:
        assert nan_codes == {0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF}
        assert inf_codes == {0x7C, 0xFC}
    # sign symmetry
    pos, neg = v[:128], v[128:]
    fin = np.isfinite(pos)
    assert np.array_equal(-pos[fin], neg[fin])
    # positive finite values strictly increase with the code
    pv = pos[fin]
    assert np.all(np.diff(pv) > 0)
    # every finite code round-trips (including -0 -> 0x80)
    fc = codes[np.isfinite(v)]
    back = O.fp8_encode(v[np.isfinite(v)].astype(np.float32), fmt)
    assert np.array_equal(back, fc)
    assert O.fp8_encode(np.array([-0.0], np.float32), fmt)[0] == 0x80


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_midpoints_round_to_even(fmt):
    codes, vals = _finite_positive_values(fmt)
    lo, hi = vals[:-1], vals[1:]
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.all(mid.astype(np.float64) == (lo + hi) / 2)  # midpoints are exact in f32
    got = O.fp8_encode(mid, fmt)
    even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    assert np.array_equal(got, even)
    above = np.nextafter(mid, np.float32(np.inf))
    below = np.nextafter(mid, np.float32(0))
    assert np.array_equal(O.fp8_encode(above, fmt), codes[1:])
    assert np.array_equal(O.fp8_encode(below, fmt), codes[:-1])
    # negative side mirrors
    assert np.array_equal(O.fp8_encode(-mid, fmt), even | 0x80)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_saturation_and_specials(fmt):
    mx = O.fp8_max(fmt)
    maxc = 0x7E if fmt == O.E4M3 else 0x7B
    vals = np.array([mx, mx * 1.01, mx * 1e6, np.inf, -mx * 3, -np.inf, 3.4e38], np.float32)
    got = O.fp8_encode(vals, fmt)
    assert got.tolist() == [maxc, maxc, maxc, maxc, maxc | 0x80, maxc | 0x80, maxc]
    assert O.fp8_encode(np.array([np.nan], np.float32), fmt)[0] == 0x7F
    # underflow: half the smallest subnormal ties to +-0; just above goes up
    tiny = 2.0 ** (-9 if fmt == O.E4M3 else -16)
    t = np.array([tiny / 2, -tiny / 2, np.nextafter(np.float32(tiny / 2), np.float32(1))],
                 np.float32)
    assert O.fp8_encode(t, fmt).tolist() == [0x00, 0x80, 0x01]


@pytest.mark.parametrize("fmt,tdtype", [(O.E4M3, torch.float8_e4m3fn), (O.E5M2, torch.float8_e5m2)])
def test_encoder_matches_torch_in_range(fmt, tdtype):
    """Independent library routine: torch's float8 cast is round-to-nearest-even
    inside the finite range (it does not saturate, so only |v| <= max is used)."""
    mx = O.fp8_max(fmt)
    rng = np.random.default_rng(123)
    # random float32 bit patterns whose magnitude falls in [0, max]
    bits = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= mx)]
    # plus dense coverage of the subnormal / normal boundary and of every bf16 value
    dense = np.linspace(-4 * 2.0 ** -6, 4 * 2.0 ** -6, 20001, dtype=np.float32)
    allbf16 = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    allbf16 = allbf16[np.isfinite(allbf16) & (np.abs(allbf16) <= mx)]
    v = np.concatenate([v, dense, allbf16, allbf16 * np.float32(0.37)])
    ours = O.fp8_encode(v, fmt)
    theirs = torch.from_numpy(v).to(tdtype).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


# ----------------------------------------------------------------------------
# BF16 ("Pretraining at scale", 4a)
# ----------------------------------------------------------------------------
def test_bf16_worked_example(golden):
    g = golden("bf16_example.txt")
    b = int(O.f32_to_bf16(np.array([g["x"]], np.float32))[0])
    assert b >> 15 == g["bf16.sign"]
    assert (b >> 7) & 0xFF == g["bf16.exponent_field"]
    assert b & 0x7F == g["bf16.fraction_field"]
    assert float(O.bf16_to_f32(np.array([b], np.uint16))[0]) == g["bf16.value"]
    one_next = float(O.bf16_to_f32(np.array([0x3F81], np.uint16))[0])
    assert one_next - 1.0 == g["bf16.eps"]


def test_bf16_matches_torch():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=500_000, dtype=np.uint64).astype(np.uint32)
    extra = np.array([0x3F808000, 0x3F818000, 0x7F7FFFFF, 0x7F7F8000, 0x00008000,
                      0x80008000, 0x00000001, 0x7F800000, 0xFF800000], np.uint32)
    v = np.concatenate([bits, extra]).view(np.float32)
    v = v[~np.isnan(v)]
    ours = O.f32_to_bf16(v)
    theirs = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


# ----------------------------------------------------------------------------
# Scale and cast ("FP8 training: what it is and how it works", Step 2;
# "FP8 Training & Inference", Exercise 2)
# ----------------------------------------------------------------------------
def test_scaling_worked_example(golden):
    g = golden("scaling_example.txt")
    s = O.delayed_scale(g["amax"], 1.0, O.E4M3)
    assert s == g["scale"]
    v = np.float32(g["x"]) * np.float32(s)
    assert round(float(v), 6) == g["scaled"]
    code = O.fp8_encode(np.array([v], np.float32), O.E4M3)
    r = O.fp8_decode(code, O.E4M3)[0]
    assert r == g["rounded"]
    back = r / s
    assert round(back, 5) == g["returned"]
    assert round(abs(back - g["x"]) / g["x"] * 100, 2) == g["rel_error_percent"]
    assert O.delayed_scale(g["ex2.amax"], 1.0, O.E4M3) == g["ex2.scale"]


# ----------------------------------------------------------------------------
# The outlier experiment ("FP8 training: what it is and how it works",
# Step 2, Worked example, Follow-up questions)
# ----------------------------------------------------------------------------
def _outlier_stats(outlier, tile):
    x = np.random.default_rng(0).standard_normal(4096)
    x[0] = outlier
    x32 = x.astype(np.float32)
    y = np.empty_like(x)
    v_all = np.empty(4096, np.float32)
    span = 4096 if tile is None else tile
    for t0 in range(0, 4096, span):
        seg = x32[t0:t0 + span]
        am = float(np.max(np.abs(seg)))
        s = O.delayed_scale(am, 1.0, O.E4M3) if tile is None else O.group_scale(am, O.E4M3)
        v = seg * np.float32(s)
        v_all[t0:t0 + span] = v
        y[t0:t0 + span] = O.fp8_decode(O.fp8_encode(v, O.E4M3), O.E4M3) / s
    xo, yo, vo = x[1:], y[1:], v_all[1:]
    return {
        "zero": 100 * np.mean(yo == 0),
        "sub": 100 * np.mean(np.abs(vo) < 2.0 ** -6),
        "rms": 100 * math.sqrt(np.mean((yo - xo) ** 2) / np.mean(xo ** 2)),
        "scale": O.delayed_scale(float(np.max(np.abs(x32))), 1.0, O.E4M3),
    }


def test_outlier_experiment(golden):
    g = golden("outlier_experiment.txt")
    t = _outlier_stats(1e5, None)
    assert round(t["scale"], 5) == g["outlier.1e5.scale"]
    assert round(t["zero"], 2) == g["outlier.1e5.zero_percent"]
    assert round(t["sub"], 2) == g["outlier.1e5.subnormal_percent"]
    assert round(t["rms"], 2) == g["outlier.1e5.rms_tensor_percent"]
    tl = _outlier_stats(1e5, 128)
    assert round(tl["rms"], 2) == g["outlier.1e5.rms_tile_percent"]
    assert round(_outlier_stats(1e4, None)["zero"], 2) == g["outlier.1e4.zero_percent"]
    for o in (1e1, 1e2, 1e3):
        for tile in (None, 128):
            assert abs(_outlier_stats(o, tile)["rms"] - g["floor_percent_below_1e4"]) < 0.15
    # "any value below about 0.22 rounds to zero" at 1e5: half the smallest
    # subnormal divided by the scale
    assert round(2.0 ** -10 / t["scale"], 2) == g["zero_threshold_1e5"]


# ----------------------------------------------------------------------------
# Activation + fused quantize
# ----------------------------------------------------------------------------
def test_activation_closed_forms():
    assert O.act(3.0, O.ACT_RELU2) == 9.0
    assert O.act(-2.0, O.ACT_RELU2) == 0.0
    assert O.act(-2.0, O.ACT_RELU) == 0.0
    assert O.act(2.5, O.ACT_RELU) == 2.5
    assert math.copysign(1.0, O.act(-0.0, O.ACT_RELU2)) == 1.0
    assert O.act(-7.25, O.ACT_IDENTITY) == -7.25
    assert O.act(1e20, O.ACT_RELU2) == math.inf  # float32 overflow
    assert O.act(float("nan"), O.ACT_RELU2) == 0.0


def _rand_bf16(shape, seed, std=1.0):
    x = (np.random.default_rng(seed).standard_normal(shape) * std).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quant_per_tensor_against_torch():
    """act_out and q against torch's bf16/float8 casts of the same float32 values."""
    h = _rand_bf16((37, 256), 5)
    s = 56.0
    r = O.quant(h, O.ACT_RELU2, O.E4M3, s, want_qt=True)
    hf = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float()
    a = torch.where(hf > 0, hf, torch.zeros_like(hf)) ** 2  # exact in float32
    abf = a.to(torch.bfloat16)
    assert np.array_equal(r["act"], abf.view(torch.int16).numpy().view(np.uint16))
    v = abf.float() * s
    v_in = v.clamp(-448, 448)  # torch does not saturate; the oracle does
    qt = v_in.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(r["q"], qt)
    assert np.array_equal(r["q_t"], r["q"].T)
    assert r["amax"] == float(abf.float().abs().max())
    assert r["sat"] == int((v.abs() > 448).sum())


def test_quant_identity_e5m2_and_sat_closed_form():
    """With scale 1 and identity, v = h exactly: sat is #{|h| > max}."""
    vals = np.array([1.0, -60000.0, 57344.0, 70000.0, -1e-9, 0.0, 3.0e38, -448.0], np.float32)
    h = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    h = np.tile(h, 2).reshape(2, 8)
    r = O.quant(h, O.ACT_IDENTITY, O.E5M2, 1.0)
    hv = O.bf16_to_f32(h).astype(np.float64)
    assert r["sat"] == int(np.sum(np.abs(hv) > 57344.0))
    r4 = O.quant(h, O.ACT_IDENTITY, O.E4M3, 1.0)
    assert r4["sat"] == int(np.sum(np.abs(hv) > 448.0))
    assert r4["amax"] == float(np.max(np.abs(hv)))


def test_quant_tiny_saturation_closed_form():
    """Tiny workload: prev amax 4, margin 2 -> s = 448/8 = 56; ReLU^2 values
    saturate iff bf16(h^2) * 56 > 448, i.e. bf16(h^2) > 8."""
    s = O.delayed_scale(4.0, 2.0, O.E4M3)
    assert s == 56.0
    h = _rand_bf16((64, 256), 0)
    r = O.quant(h, O.ACT_RELU2, O.E4M3, s)
    hv = O.bf16_to_f32(h).astype(np.float64)
    sq = torch.from_numpy(np.where(hv > 0, hv, 0.0).astype(np.float32) ** 2).to(torch.bfloat16)
    assert r["sat"] == int((sq.double() > 8.0).sum())
    # expected count is near P(h > sqrt 8) * M * K
    p = 0.5 * math.erfc(math.sqrt(8) / math.sqrt(2))
    assert abs(r["sat"] - p * 64 * 256) < 5 * math.sqrt(p * 64 * 256) + 1


def test_quant_group_invariants():
    h = _rand_bf16((5, 512), 11)
    h[2, 128:256] = 0  # an all-zero group -> scale 1, codes 0
    r = O.quant_group(h, O.ACT_RELU2, O.E4M3, 1, want_qt=True)
    dec = O.fp8_decode(r["q"], O.E4M3).reshape(5, 4, 128)
    mx = np.max(np.abs(dec), axis=2)
    a = O.bf16_to_f32(r["act"]).reshape(5, 4, 128).astype(np.float64)
    am = np.max(np.abs(a), axis=2)
    for i in range(5):
        for g in range(4):
            if am[i, g] > 0:
                assert mx[i, g] == 448.0  # each group's largest value lands on 448
                assert r["scales"][i, g] == np.float32(448.0 / np.float32(am[i, g]))
            else:
                assert r["scales"][i, g] == 1.0 and mx[i, g] == 0.0
    assert np.array_equal(r["q_t"], r["q"].T)
    # a 1x128 group is per-tensor quantisation of that slice with its own scale
    for i in range(5):
        for g in range(4):
            sl = h[i:i + 1, g * 128:(g + 1) * 128]
            rr = O.quant(sl, O.ACT_RELU2, O.E4M3, float(r["scales"][i, g]))
            assert np.array_equal(rr["q"][0], r["q"][i, g * 128:(g + 1) * 128])


def test_quant_group_blocks_128x128():
    h = _rand_bf16((300, 256), 12)
    r = O.quant_group(h, O.ACT_IDENTITY, O.E4M3, 128)
    assert r["scales"].shape == (3, 2)
    hv = np.abs(O.bf16_to_f32(h).astype(np.float64))
    for rb in range(3):
        for cb in range(2):
            blk = hv[rb * 128:(rb + 1) * 128, cb * 128:(cb + 1) * 128]
            assert r["scales"][rb, cb] == np.float32(448.0 / np.float32(blk.max()))


def test_amax_calibration_matches_quant():
    h = _rand_bf16((33, 96), 13, std=3.0)
    assert O.amax(h, O.ACT_RELU2) == O.quant(h, O.ACT_RELU2, O.E4M3, 1.0)["amax"]


# ----------------------------------------------------------------------------
# Delayed scaling history ("Paradigma Details FP8 ...", second paragraph;
# "FP8 Training & Inference", Delayed Scaling)
# ----------------------------------------------------------------------------
def test_history_previous_step_times_margin():
    st, hist, head, s = O.history_update(np.zeros(1, np.float32), 0, 4.0, 2.0, O.E4M3, 1.0)
    assert (st, head, s) == (0, 0, 56.0)
    st, hist, head, s = O.history_update(hist, head, 3.2, 1.0, O.E4M3, s)
    assert s == 140.0  # L = 1: only the previous step counts


def test_history_ring_window():
    hist, head, s = np.zeros(3, np.float32), 2, 1.0
    seq = [8.0, 1.0, 2.0, 0.5, 0.25]
    refs = []
    for a in seq:
        st, hist, head, s = O.history_update(hist, head, a, 1.0, O.E4M3, s)
        refs.append(448.0 / s)
    # max over the last three pushes
    assert refs == [8.0, 8.0, 8.0, 2.0, 2.0]
    assert head == (2 + len(seq)) % 3


def test_history_keeps_scale_on_bad_amax():
    for bad in (0.0, float("inf"), float("nan")):
        st, hist, head, s = O.history_update(np.zeros(1, np.float32), 0, bad, 2.0, O.E4M3, 7.0)
        assert st == 1 and s == 7.0
    # E5M2 uses its own maximum
    assert O.delayed_scale(4.0, 2.0, O.E5M2) == 57344.0 / 8.0


# ----------------------------------------------------------------------------
# GEMMs ("Pretraining at scale", 3c worked example; "FP8 Training & Inference",
# FP8 Training Recipe and Per-Tensor Scaling)
# ----------------------------------------------------------------------------
def _codes(vals, fmt):
    return O.fp8_encode(np.asarray(vals, np.float32), fmt)


def test_gemm_matmul_worked_example(golden):
    g = golden("matmul_example.txt")
    X = _codes([g["x"]], O.E4M3)
    W = _codes([g["w.row0"], g["w.row1"]], O.E4M3)
    Y, S = O.gemm_fwd(X, W, 1.0, 1.0)
    assert Y[0].tolist() == g["y"]
    # the row split of the page: partial sums from each row of W add up
    p1, _ = O.gemm_fwd(X[:, :1], W[:1], 1.0, 1.0)
    p2, _ = O.gemm_fwd(X[:, 1:], W[1:], 1.0, 1.0)
    assert p1[0].tolist() == [1, 2, 3, 4] and p2[0].tolist() == [10, 12, 14, 16]
    assert (p1 + p2)[0].tolist() == g["y"]


def test_gemm_against_numpy_and_scales():
    rng = np.random.default_rng(21)
    M, K, N = 19, 256, 40
    X = rng.integers(0, 256, (M, K), dtype=np.uint8)
    W = rng.integers(0, 256, (K, N), dtype=np.uint8)
    X[(X & 0x7F) == 0x7F] = 0x3C  # drop NaN codes
    W[(W & 0x7F) == 0x7F] = 0x30
    Xd, Wd = O.fp8_decode(X, O.E4M3), O.fp8_decode(W, O.E4M3)
    Y, S = O.gemm_fwd(X, W, 1.0, 1.0)
    ref = Xd @ Wd
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-9)
    assert np.allclose(S, np.abs(Xd) @ np.abs(Wd), rtol=1e-12, atol=1e-9)
    Y2, _ = O.gemm_fwd(X, W, 2.0, 0.25)
    assert np.allclose(Y2, ref / 0.5, rtol=1e-12, atol=1e-9)
    rows = np.array([3, 0, 18], np.int64)
    Yr, _ = O.gemm_fwd(X, W, 1.0, 1.0, rows=rows)
    assert np.array_equal(Yr, Y[rows])


def test_gemm_small_integers_exact_and_identity():
    rng = np.random.default_rng(22)
    Xi = rng.integers(-8, 9, (7, 32))
    Wi = rng.integers(-8, 9, (32, 9))
    Y, _ = O.gemm_fwd(_codes(Xi, O.E4M3), _codes(Wi, O.E4M3), 1.0, 1.0)
    assert np.array_equal(Y, (Xi @ Wi).astype(np.float64))
    I = _codes(np.eye(32), O.E4M3)
    Xc = _codes(rng.standard_normal((7, 32)), O.E4M3)
    Yi, _ = O.gemm_fwd(Xc, I, 4.0, 1.0)
    assert np.array_equal(Yi, O.fp8_decode(Xc, O.E4M3) / 4.0)


def test_gemm_dgrad_is_dy_times_w_transposed():
    rng = np.random.default_rng(23)
    M, N, K = 11, 64, 48
    dY = _codes(rng.standard_normal((M, N)) * 100, O.E5M2)
    W = _codes(rng.standard_normal((K, N)), O.E4M3)
    dX, S = O.gemm_dgrad(dY, W, 3.0, 5.0)
    ref = O.fp8_decode(dY, O.E5M2) @ O.fp8_decode(W, O.E4M3).T / 15.0
    assert np.allclose(dX, ref, rtol=1e-12, atol=1e-12)
    # same as the forward on the transposed weight with an E5M2 left operand
    Yf, _ = O.gemm_fwd(dY, np.ascontiguousarray(W.T), 3.0, 5.0, fmt_x=O.E5M2)
    assert np.allclose(dX, Yf, rtol=1e-13, atol=1e-13)


def test_gemm_wgrad_is_x_transposed_times_dy():
    """dW = X^T dY: exact on small integers (exactly representable in E4M3 and
    E5M2, so the sums are exact) against numpy's integer matmul, numpy's matmul
    of the decoded operands otherwise, and row selection."""
    rng = np.random.default_rng(24)
    M, K, N = 40, 24, 33
    Xi = rng.integers(-8, 9, (M, K))
    Di = rng.integers(-6, 7, (M, N))
    dW, S = O.gemm_wgrad(_codes(Xi, O.E4M3), _codes(Di, O.E5M2), 1.0, 1.0)
    assert np.array_equal(dW, (Xi.T @ Di).astype(np.float64))
    assert np.array_equal(S, (np.abs(Xi).T @ np.abs(Di)).astype(np.float64))
    X = _codes(rng.standard_normal((M, K)) * 50, O.E4M3)
    D = _codes(rng.standard_normal((M, N)) * 1e3, O.E5M2)
    dW, _ = O.gemm_wgrad(X, D, 4.0, 0.5)
    ref = O.fp8_decode(X, O.E4M3).T @ O.fp8_decode(D, O.E5M2) / 2.0
    assert np.allclose(dW, ref, rtol=1e-12, atol=1e-12)
    rows = np.array([5, 0, 23], np.int64)
    dWr, _ = O.gemm_wgrad(X, D, 4.0, 0.5, rows=rows)
    assert np.array_equal(dWr, dW[rows])


def test_dgrad_act_closed_forms():
    """dH = dX * act'(H): identity reduces to the dgrad; ReLU gates it by h > 0
    (so -0, 0 and negatives give 0); ReLU^2 scales it by 2h; rows select."""
    rng = np.random.default_rng(25)
    M, N, K = 9, 48, 20
    dY = _codes(rng.standard_normal((M, N)) * 100, O.E5M2)
    W = _codes(rng.standard_normal((K, N)), O.E4M3)
    dX, S = O.gemm_dgrad(dY, W, 2.0, 8.0)
    hv = rng.standard_normal((M, K)).astype(np.float32)
    hv[0, :4] = [0.0, -0.0, -1.0, 3.0]
    h = O.f32_to_bf16(hv)
    d0, s0 = O.gemm_dgrad_act(dY, W, 2.0, 8.0, h, O.ACT_IDENTITY)
    assert np.array_equal(d0, dX) and np.array_equal(s0, S)
    hf = O.bf16_to_f32(h).astype(np.float64)
    d1, _ = O.gemm_dgrad_act(dY, W, 2.0, 8.0, h, O.ACT_RELU)
    assert np.array_equal(d1, np.where(hf > 0, dX, 0.0))
    assert np.array_equal(d1[0, :3], [0.0, 0.0, 0.0]) and d1[0, 3] == dX[0, 3]
    d2, s2 = O.gemm_dgrad_act(dY, W, 2.0, 8.0, h, O.ACT_RELU2)
    assert np.array_equal(d2, np.where(hf > 0, 2.0 * hf * dX, 0.0))
    assert np.array_equal(s2, S * np.where(hf > 0, 2.0 * hf, 0.0))
    rows = np.array([4, 0], np.int64)
    dr, _ = O.gemm_dgrad_act(dY, W, 2.0, 8.0, h, O.ACT_RELU2, rows=rows)
    assert np.array_equal(dr, d2[rows])


def _pow2_step(h: np.ndarray) -> np.ndarray:
    """delta = 2^(floor(log2|h|) - 8): h is a BF16 value (8 significant bits), so
    h +- delta has at most 10 and its square at most 20 -- both exact in float32,
    which is what the oracle's forward activation computes in."""
    return np.exp2(np.floor(np.log2(np.abs(h))) - 8.0)


@pytest.mark.parametrize("which", [O.ACT_RELU2, O.ACT_RELU, O.ACT_IDENTITY])
def test_act_grad_is_the_derivative_of_the_forward_activation(which):
    """act_grad against a central difference of the oracle's own forward
    activation O.act (pinned separately by its closed forms), computed in
    float64: (act(h + d) - act(h - d)) / 2d.  For the quadratic ReLU^2 and the
    piecewise-linear ReLU / identity the central difference has no truncation
    error once |h| > d, and with d a power of two 2^-8 |h| every evaluation is
    exact, so the two must agree bit for bit over a sweep of BF16 values of
    both signs across 60 binades.  A derivative taken as h instead of 2h, as
    2 relu(h)^2, or at the activation's output instead of its input fails."""
    rng = np.random.default_rng(26)
    mags = np.exp2(rng.uniform(-30, 30, 3000)) * rng.uniform(1.0, 2.0, 3000)
    hv = (mags * rng.choice([-1.0, 1.0], 3000)).astype(np.float32)
    hb = O.f32_to_bf16(hv)
    h = O.bf16_to_f32(hb).astype(np.float64)
    d = _pow2_step(h)
    fd = np.array([(O.act(float(x + e), which) - O.act(float(x - e), which)) / (2.0 * e)
                   for x, e in zip(h, d)], dtype=np.float64)
    g = O.act_grad(hb, which)
    assert np.array_equal(g, fd)
    # one-sided differences where the activation has its kink: at h = +0 and
    # -0 the right difference of ReLU^2 is d (-> 0) and of ReLU is 1, the left
    # one 0; the oracle takes the forward's own comparison h > 0 there, i.e.
    # the left derivative 0 for both, and 1 for the identity
    e = 2.0 ** -20
    for z in (0.0, -0.0):
        zb = O.f32_to_bf16(np.array([z], np.float32))
        left = (O.act(z, which) - O.act(z - e, which)) / e
        right = (O.act(z + e, which) - O.act(z, which)) / e
        assert O.act_grad(zb, which)[0] == left
        assert right == {O.ACT_RELU2: e, O.ACT_RELU: 1.0, O.ACT_IDENTITY: 1.0}[which]
    # far into the negative half the activation is flat (ReLU, ReLU^2)
    neg = O.f32_to_bf16(np.array([-1.0, -3.5e-30, -6.0e20], np.float32))
    want = 1.0 if which == O.ACT_IDENTITY else 0.0
    assert np.array_equal(O.act_grad(neg, which), [want] * 3)


def test_act_grad_at_the_fp8_cache():
    """act_grad_q dequantises the E4M3 cache and then is act_grad: on H values
    that lie on the E4M3 grid divided by a power-of-two scale the cache is
    exact and the two agree bit for bit; the scale divides (a code cast with
    s_h = 4 is a quarter of its value); and against values off the grid the
    cached derivative differs from the exact one by at most the E4M3
    rounding of s_h h (half a code step: 2^-4 relative for normals)."""
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]                # no NaN codes
    vals = O.fp8_decode(codes, O.E4M3)
    for s_h in (1.0, 4.0, 0.125):
        h = O.f32_to_bf16((vals / s_h).astype(np.float32))  # exact: E4M3 values have 4 significant bits
        for which in (O.ACT_RELU2, O.ACT_RELU, O.ACT_IDENTITY):
            assert np.array_equal(O.act_grad_q(codes, s_h, which), O.act_grad(h, which))
    assert O.act_grad_q(np.array([0x38], np.uint8), 4.0, O.ACT_RELU2)[0] == 0.5   # 1.0 / 4, times 2
    rng = np.random.default_rng(27)
    hv = (rng.standard_normal((50, 100)) * 2.0).astype(np.float32)
    hb = O.f32_to_bf16(hv)
    s_h = O.delayed_scale(O.amax(hb, O.ACT_IDENTITY), 2.0, O.E4M3)
    q = O.quant(hb, O.ACT_IDENTITY, O.E4M3, s_h)["q"]
    exact, cached = O.act_grad(hb, O.ACT_RELU2), O.act_grad_q(q, s_h, O.ACT_RELU2)
    big = np.abs(O.bf16_to_f32(hb).astype(np.float64)) * s_h >= 2.0 ** -6   # normal E4M3 range
    assert np.all(np.abs(cached - exact)[big] <= exact[big] * 2.0 ** -4 + 1e-12)
    assert np.array_equal(cached > 0, (O.fp8_decode(q, O.E4M3) > 0))


def test_group_gemm_reductions():
    """Group mode: equal scales reduce to per-tensor; power-of-two scales that
    differ per row, per 128-slice of K and per 128-block of N reduce to numpy's
    matmul of exactly rescaled operands (catches a transposed scale index)."""
    rng = np.random.default_rng(24)
    M, K, N = 6, 384, 200
    X = _codes(rng.standard_normal((M, K)), O.E4M3)
    W = _codes(rng.standard_normal((K, N)), O.E4M3)
    kg, ng = K // 128, (N + 127) // 128
    Yp, _ = O.gemm_fwd(X, W, 3.0, 7.0)
    Yg, _ = O.gemm_fwd(X, W, np.full((M, kg), 3.0), np.full((kg, ng), 7.0), group=True)
    assert np.allclose(Yg, Yp, rtol=1e-13, atol=1e-13)
    sx = 2.0 ** rng.integers(-3, 4, (M, kg)).astype(np.float64)
    sw = 2.0 ** rng.integers(-3, 4, (kg, ng)).astype(np.float64)
    Xd = O.fp8_decode(X, O.E4M3) / np.repeat(sx, 128, axis=1)
    Wd = O.fp8_decode(W, O.E4M3) / np.repeat(np.repeat(sw, 128, axis=0), 128, axis=1)[:, :N]
    Yg2, _ = O.gemm_fwd(X, W, sx.astype(np.float32), sw.astype(np.float32), group=True)
    assert np.allclose(Yg2, Xd @ Wd, rtol=1e-12, atol=1e-12)
