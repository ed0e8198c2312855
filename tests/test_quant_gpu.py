"""Parity of the fused quantize kernel (fp8_quant_fused) with the CPU oracle.

FP8 codes, BF16 activation copies, amax, group scales and saturation counts
are integer/byte results: they must match the oracle bit-exactly.  Both sides
take the FP8 decision on the same float32 value v = float32(BF16(act(h)) * s).
"""
import numpy as np
import pytest
import torch

import oracle as O
from quantize_fp8_gemm_gb300 import binding as B
from quantize_fp8_gemm_gb300 import workloads as WL
from tests.parity import dev_bf16, dev_f32, host_bits16, host_u8

pytestmark = pytest.mark.gpu


def _rand_bits(M, K, seed, std=1.0):
    x = np.random.default_rng(seed).standard_normal((M, K)).astype(np.float32) * np.float32(std)
    return WL.to_bf16_bits(x)


def run_quant(h_bits, act, fmt, scale, *, want_act=True, want_q=True, want_qt=False, group_rows=None):
    M, K = h_bits.shape
    h = dev_bf16(h_bits)
    act_out = torch.empty(M, K, dtype=torch.bfloat16, device="cuda") if want_act else None
    q = torch.empty(M, K, dtype=torch.uint8, device="cuda") if want_q else None
    qt = torch.empty(K, M, dtype=torch.uint8, device="cuda") if want_qt else None
    amax = torch.full((1,), -1.0, device="cuda")
    sat = torch.full((1,), 12345, dtype=torch.int64, device="cuda")
    gs = None
    if group_rows is not None:
        gs = torch.empty((M + group_rows - 1) // group_rows, K // 128, dtype=torch.float32, device="cuda")
        B.fp8_quant_fused(h, act, fmt, None, act_out=act_out, q_out=q, q_t_out=qt, amax_out=amax,
                          sat_count=sat, group_scales_out=gs, group_rows=group_rows)
    else:
        B.fp8_quant_fused(h, act, fmt, dev_f32(scale), act_out=act_out, q_out=q, q_t_out=qt,
                          amax_out=amax, sat_count=sat)
    torch.cuda.synchronize()
    return {
        "act": host_bits16(act_out) if want_act else None,
        "q": host_u8(q) if want_q else None,
        "q_t": host_u8(qt) if want_qt else None,
        "amax": float(amax.item()),
        "sat": int(sat.item()),
        "scales": gs.cpu().numpy() if gs is not None else None,
    }


def assert_same(gpu, ref, keys):
    for k in keys:
        if isinstance(ref[k], np.ndarray):
            bad = np.argwhere(gpu[k] != ref[k])
            assert bad.size == 0, f"{k}: {len(bad)} mismatches, first at {bad[0]}: gpu={gpu[k][tuple(bad[0])]} ref={ref[k][tuple(bad[0])]}"
        else:
            assert gpu[k] == ref[k], f"{k}: gpu={gpu[k]} ref={ref[k]}"


def test_tiny_workload_bit_exact():
    w = WL.WORKLOADS["tiny"]
    h = WL.h_preact(w)
    # the delayed scale from previous amax 4.0 and margin 2.0, computed on the GPU
    ds_hist = torch.zeros(1, device="cuda")
    head = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = torch.ones(1, device="cuda")
    B.amax_history_update(ds_hist, head, dev_f32(w.prev_amax), w.margin, B.E4M3, scale)
    s = float(scale.item())
    assert s == O.delayed_scale(w.prev_amax, w.margin, O.E4M3) == 56.0
    g = run_quant(h, B.ACT_RELU2, B.E4M3, s)
    r = O.quant(h, O.ACT_RELU2, O.E4M3, s)
    assert_same(g, r, ["act", "q", "amax", "sat"])
    assert g["sat"] > 0  # h > sqrt(8) saturates at this scale


@pytest.mark.parametrize("M,K", [(1, 16), (3, 48), (37, 256), (130, 384), (1000, 272), (2048, 1024)])
@pytest.mark.parametrize("act", [B.ACT_IDENTITY, B.ACT_RELU, B.ACT_RELU2])
@pytest.mark.parametrize("fmt", [B.E4M3, B.E5M2])
def test_per_tensor_shapes(M, K, act, fmt):
    h = _rand_bits(M, K, seed=M * 7 + K, std=2.0)
    s = 37.5 if fmt == B.E4M3 else 3000.0
    g = run_quant(h, act, fmt, s)
    r = O.quant(h, act, fmt, s)
    assert_same(g, r, ["act", "q", "amax", "sat"])


@pytest.mark.parametrize("fmt", [B.E4M3, B.E5M2])
def test_every_bf16_input(fmt):
    """All non-NaN BF16 patterns (incl. +-0, subnormals, +-inf) under several scales."""
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = (allp.astype(np.uint32) << 16).view(np.float32)
    pats = allp[~np.isnan(f)]
    pad = (-pats.size) % 64
    pats = np.concatenate([pats, np.zeros(pad, np.uint16)]).reshape(-1, 64)
    for s in [1.0, 56.0, 140.0, 0.00448, 3.0, 1.0 / 3.0, 2.0 ** -20, 2.0 ** 20, 7.25, 1e-30, 3e30]:
        g = run_quant(pats, B.ACT_IDENTITY, fmt, s, want_act=False)
        r = O.quant(pats, O.ACT_IDENTITY, fmt, np.float32(s), want_act=False)
        assert_same(g, r, ["q", "amax", "sat"])


@pytest.mark.parametrize("act", [B.ACT_RELU2, B.ACT_RELU])
def test_every_bf16_input_through_the_activation(act):
    """Every BF16 pattern, NaNs, +-0, subnormals and +-inf included, through
    ReLU^2 and ReLU: the BF16 activation, the E4M3 codes, amax and the
    saturation count against the oracle, under scales that put the codes in
    every range."""
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(-1, 64)
    for s in [1.0, 3.0, 2.0 ** -20, 1e-30, 3e30]:
        g = run_quant(allp, act, B.E4M3, s)
        r = O.quant(allp, act, O.E4M3, np.float32(s))
        assert_same(g, r, ["act", "q", "amax", "sat"])


@pytest.mark.parametrize("fmt", [B.E4M3, B.E5M2])
def test_cast_every_fp32_pattern(fmt):
    """The kernels' FP32 -> FP8 conversion over all 2^32 float32 bit patterns
    against the oracle's encoder, written from the formats' definition: every
    non-NaN input gives the oracle's code bit for bit, every NaN a NaN code."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    chunk = 1 << 24
    workers = max(1, min(32, len(os.sched_getaffinity(0))))
    nan_codes = {0x7F, 0xFF} if fmt == B.E4M3 else {0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF}
    base = torch.arange(chunk, dtype=torch.int64, device="cuda")
    q = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    piece = chunk // workers

    def encode(x, lo):
        return O.fp8_encode(x[lo:lo + piece] if lo + piece < x.size else x[lo:], fmt)

    with ThreadPoolExecutor(workers) as ex:
        for c in range(1 << 8):
            start = c * chunk
            bits = (base + start).to(torch.int32) if start + chunk <= (1 << 31) else (base + start - (1 << 32)).to(torch.int32)
            B.fp8_cast_f32(bits.view(torch.float32), fmt, q)
            got = q.cpu().numpy()
            x = (np.arange(chunk, dtype=np.uint64) + start).astype(np.uint32).view(np.float32)
            want = np.concatenate(list(ex.map(lambda lo: encode(x, lo), range(0, chunk, piece))))
            nan = np.isnan(x)
            bad = (got != want) & ~nan
            assert not bad.any(), (f"chunk {c}: {int(bad.sum())} codes differ, first input bits "
                                   f"0x{int(x.view(np.uint32)[bad][0]):08x}: gpu 0x{int(got[bad][0]):02x} "
                                   f"oracle 0x{int(want[bad][0]):02x}")
            if nan.any():
                assert set(np.unique(got[nan]).tolist()) <= nan_codes, f"chunk {c}: a NaN gave a non-NaN code"


def test_cast_ragged_lengths():
    """fp8_cast_f32 on lengths that leave 1-3 values after the 4-wide steps."""
    rng = np.random.default_rng(11)
    for n in (1, 2, 3, 5, 4099, 1 << 16):
        x = (rng.standard_normal(n) * 300).astype(np.float32)
        for fmt in (B.E4M3, B.E5M2):
            got = B.fp8_cast_f32(torch.from_numpy(x).cuda(), fmt).cpu().numpy()
            assert np.array_equal(got, O.fp8_encode(x, fmt))


@pytest.mark.parametrize("M,K", [(1, 128), (5, 512), (333, 256), (4096, 3072)])
@pytest.mark.parametrize("act", [B.ACT_IDENTITY, B.ACT_RELU2])
def test_group_1x128(M, K, act):
    h = _rand_bits(M, K, seed=M + K, std=3.0)
    h[0, :128] = 0  # an all-zero group
    if M > 2:
        h[2, 128:129] = WL.to_bf16_bits(np.array([1e5], np.float32))  # an outlier
    g = run_quant(h, act, B.E4M3, None, group_rows=1)
    r = O.quant_group(h, act, O.E4M3, 1)
    assert_same(g, r, ["act", "q", "amax", "sat", "scales"])


@pytest.mark.parametrize("M,K", [(16, 16), (272, 160), (384, 256), (6400, 1600)])
def test_weight_cast_transposed(M, K):
    """W [K,N] -> W_q [K,N] and W_q^T [N,K] (here M plays K and K plays N)."""
    h = _rand_bits(M, K, seed=M * K, std=0.02)
    s = O.delayed_scale(O.amax(h, O.ACT_IDENTITY), 2.0, O.E4M3)
    g = run_quant(h, B.ACT_IDENTITY, B.E4M3, s, want_act=False, want_qt=True)
    r = O.quant(h, O.ACT_IDENTITY, O.E4M3, s, want_act=False, want_qt=True)
    assert_same(g, r, ["q", "q_t", "amax", "sat"])


@pytest.mark.parametrize("M,K", [(128, 128), (300, 384), (6400, 1024)])
def test_weight_blocks_128x128(M, K):
    h = _rand_bits(M, K, seed=M + 3 * K, std=0.02)
    h[5, 200 % K] = WL.to_bf16_bits(np.array([3.0], np.float32))[0]
    g = run_quant(h, B.ACT_IDENTITY, B.E4M3, None, want_act=False, want_qt=(M % 16 == 0), group_rows=128)
    r = O.quant_group(h, O.ACT_IDENTITY, O.E4M3, 128, want_act=False, want_qt=(M % 16 == 0))
    keys = ["q", "amax", "sat", "scales"] + (["q_t"] if M % 16 == 0 else [])
    assert_same(g, r, keys)


@pytest.mark.parametrize("mode", ["tensor", "relu2_act", "blocks_128x128", "groups_1x128"])
@pytest.mark.parametrize("M,K", [(2000, 10240), (2000, 5120)])
def test_large_tiled_grid_every_mode(mode, M, K):
    """Grids past two rounds of the register-landing tile kernel run the
    shared-memory one: 2000 x 10240 is 16 x 80 = 1280 tiles (a ragged last
    tile row), in each tiled mode, with the transposed copy.  2000 x 5120 is
    640 tiles: the register-landing kernel in two rounds (608 resident CTAs on
    GB300's 152 SMs), the ragged tile row in the second."""
    h = _rand_bits(M, K, seed=77, std=0.5)
    h[7, 300] = WL.to_bf16_bits(np.array([60.0], np.float32))[0]
    if mode == "tensor":
        g = run_quant(h, B.ACT_IDENTITY, B.E4M3, 4.0, want_act=False, want_qt=True)
        r = O.quant(h, O.ACT_IDENTITY, O.E4M3, 4.0, want_act=False, want_qt=True)
        keys = ["q", "q_t", "amax", "sat"]
    elif mode == "relu2_act":
        g = run_quant(h, B.ACT_RELU2, B.E5M2, 1000.0, want_qt=True)
        r = O.quant(h, O.ACT_RELU2, O.E5M2, 1000.0, want_qt=True)
        keys = ["act", "q", "q_t", "amax", "sat"]
    else:
        rows = 128 if mode == "blocks_128x128" else 1
        g = run_quant(h, B.ACT_IDENTITY, B.E4M3, None, want_act=False, want_qt=True, group_rows=rows)
        r = O.quant_group(h, O.ACT_IDENTITY, O.E4M3, rows, want_act=False, want_qt=True)
        keys = ["q", "q_t", "amax", "sat", "scales"]
    assert_same(g, r, keys)


def test_relu2_with_transposed_copy_and_act():
    """The tiled path with an activation and every output at once."""
    h = _rand_bits(256, 384, seed=9)
    g = run_quant(h, B.ACT_RELU2, B.E4M3, 20.0, want_qt=True)
    r = O.quant(h, O.ACT_RELU2, O.E4M3, 20.0, want_qt=True)
    assert_same(g, r, ["act", "q", "q_t", "amax", "sat"])


def test_empty_input_zeroes_amax():
    h = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    amax = torch.full((1,), 5.0, device="cuda")
    sat = torch.full((1,), 7, dtype=torch.int64, device="cuda")
    q = torch.empty(0, 64, dtype=torch.uint8, device="cuda")
    B.fp8_quant_fused(h, B.ACT_RELU2, B.E4M3, dev_f32(1.0), q_out=q, amax_out=amax, sat_count=sat)
    torch.cuda.synchronize()
    assert amax.item() == 0.0 and sat.item() == 0


def test_fused_equals_naive_three_pass():
    """The fused kernel and the unfused write/scan/cast passes give the same bytes
    when the cast uses the same scale."""
    h_bits = _rand_bits(512, 768, seed=4)
    h = dev_bf16(h_bits)
    a1 = torch.empty(512, 768, dtype=torch.bfloat16, device="cuda")
    q1 = torch.empty(512, 768, dtype=torch.uint8, device="cuda")
    amax1 = torch.zeros(1, device="cuda")
    sc = torch.zeros(1, device="cuda")
    B.fp8q_naive_act(h, B.ACT_RELU2, a1)
    B.fp8q_naive_amax(a1, amax1)
    B.fp8q_naive_cast(a1, B.E4M3, amax1, 2.0, q1, scale_out=sc)
    a2 = torch.empty_like(a1)
    q2 = torch.empty_like(q1)
    amax2 = torch.zeros(1, device="cuda")
    B.fp8_quant_fused(h, B.ACT_RELU2, B.E4M3, sc, act_out=a2, q_out=q2, amax_out=amax2)
    torch.cuda.synchronize()
    assert torch.equal(a1.view(torch.int16), a2.view(torch.int16))
    assert torch.equal(q1, q2)
    assert amax1.item() == amax2.item()
    assert sc.item() == O.delayed_scale(amax1.item(), 2.0, O.E4M3)


@pytest.mark.parametrize("name", ["gpt2s", "outlier"])
def test_full_size_workload_bit_exact(name):
    w = WL.WORKLOADS[name]
    h = WL.h_preact(w)
    s = 448.0 / (w.margin * 20.0)
    g = run_quant(h, B.ACT_RELU2, B.E4M3, s)
    r = O.quant(h, O.ACT_RELU2, O.E4M3, np.float32(s))
    assert_same(g, r, ["act", "q", "amax", "sat"])
    if name == "outlier":
        gg = run_quant(h, B.ACT_IDENTITY, B.E4M3, None, want_act=False, group_rows=1)
        rg = O.quant_group(h, O.ACT_IDENTITY, O.E4M3, 1, want_act=False)
        assert_same(gg, rg, ["q", "amax", "sat", "scales"])


def _outs(M, K, act=True, q=True, qt=False):
    return dict(a=torch.empty(M, K, dtype=torch.bfloat16, device="cuda") if act else None,
                q=torch.empty(M, K, dtype=torch.uint8, device="cuda") if q else None,
                qt=torch.empty(K, M, dtype=torch.uint8, device="cuda") if qt else None,
                amax=torch.full((1,), -1.0, device="cuda"),
                sat=torch.full((1,), 7, dtype=torch.int64, device="cuda"))


def test_batch_equals_separate_calls():
    """fp8_quant_fused_batch over a weight (identity, transposed and row-major
    copies), an activation (ReLU^2 + BF16 copy), a gradient (E5M2), an empty
    tensor and a ragged ReLU tensor: every output equals its own
    fp8_quant_fused call bit for bit, and ACCUMULATE folds into the values
    already there."""
    cases = [  # (M, K, act, fmt, scale, want act_out, want q_t_out, flags)
        (3072, 768, B.ACT_IDENTITY, B.E4M3, 2667.0, False, True, 0),
        (1000, 640, B.ACT_RELU2, B.E4M3, 20.0, True, False, 0),
        (0, 256, B.ACT_RELU, B.E4M3, 1.0, True, False, 0),
        (517, 48, B.ACT_RELU, B.E5M2, 9000.0, True, False, B.ACCUMULATE),
    ]
    ins, sep, bat, entries = [], [], [], []
    for i, (M, K, act, fmt, sc, wa, wqt, flags) in enumerate(cases):
        h = dev_bf16(_rand_bits(M, K, seed=100 + i, std=1.5))
        s = dev_f32(sc)
        r, b = _outs(M, K, wa, True, wqt), _outs(M, K, wa, True, wqt)
        if flags:
            for d in (r, b):
                d["amax"].fill_(0.5)
                d["sat"].fill_(3)
        B.fp8_quant_fused_ex(h, act, fmt, s, act_out=r["a"], q_out=r["q"], q_t_out=r["qt"], amax_out=r["amax"],
                             sat_count=r["sat"], flags=flags)
        entries.append(B.quant_args(h, act, fmt, s, act_out=b["a"], q_out=b["q"], q_t_out=b["qt"],
                                    amax_out=b["amax"], sat_count=b["sat"], flags=flags))
        ins.append((h, s))
        sep.append(r)
        bat.append(b)
    B.fp8_quant_fused_batch(entries)
    torch.cuda.synchronize()
    for (M, K, *_), r, b in zip(cases, sep, bat):
        for key in ("a", "q", "qt"):
            if r[key] is not None and M:
                assert torch.equal(r[key].view(torch.uint8), b[key].view(torch.uint8)), (M, K, key)
        assert r["amax"].item() == b["amax"].item() and r["sat"].item() == b["sat"].item(), (M, K)
    assert sep[2]["amax"].item() == 0.0 and sep[2]["sat"].item() == 0  # empty entry: zeroed
    assert sep[3]["amax"].item() >= 0.5 and sep[3]["sat"].item() >= 3  # accumulated


def test_batch_against_oracle():
    """The step's pair (W transposed cast + H ReLU^2 quantize) in one launch, against the oracle."""
    w_bits = _rand_bits(384, 272, seed=7, std=0.05)
    h_bits = _rand_bits(300, 384, seed=8, std=1.2)
    sw, sx = 3000.0, 25.0
    W, H = dev_bf16(w_bits), dev_bf16(h_bits)
    wt = torch.empty(272, 384, dtype=torch.uint8, device="cuda")
    o = _outs(300, 384)
    aw = torch.zeros(1, device="cuda")
    B.fp8_quant_fused_batch([
        B.quant_args(W, B.ACT_IDENTITY, B.E4M3, dev_f32(sw), q_t_out=wt, amax_out=aw),
        B.quant_args(H, B.ACT_RELU2, B.E4M3, dev_f32(sx), act_out=o["a"], q_out=o["q"], amax_out=o["amax"],
                     sat_count=o["sat"]),
    ])
    torch.cuda.synchronize()
    rw = O.quant(w_bits, O.ACT_IDENTITY, O.E4M3, sw, want_act=False)
    rx = O.quant(h_bits, O.ACT_RELU2, O.E4M3, sx)
    assert np.array_equal(host_u8(wt), rw["q"].T)
    assert aw.item() == rw["amax"]
    assert np.array_equal(host_u8(o["q"]), rx["q"])
    assert np.array_equal(host_bits16(o["a"]), rx["act"])
    assert o["amax"].item() == rx["amax"] and o["sat"].item() == rx["sat"]
