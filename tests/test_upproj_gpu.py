"""The up-projection with the activation quantize in its epilogue
(fp8_upproj_fwd) against the oracle.

The GEMM part decides H in the kernel's FP32 accumulation, so it is checked
like every GEMM (tests/parity.py: 1 BF16 ulp + 1e-5 * S of the oracle's
double-precision result).  The quantize part is a pure function of that H: the
activation copy, the E4M3 codes, amax and the saturation count must equal the
oracle's quantize of the kernel's own H bit for bit.  The H output is optional;
the runs that leave it out must give the same codes.
"""
import numpy as np
import pytest
import torch

import oracle as O
from quantize_fp8_gemm_gb300 import binding as B
from tests.parity import assert_gemm_close, dev_f32, dev_u8, host_bits16, host_u8

pytestmark = pytest.mark.gpu

ORACLE_ACT = {B.ACT_IDENTITY: O.ACT_IDENTITY, B.ACT_RELU: O.ACT_RELU, B.ACT_RELU2: O.ACT_RELU2}


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    xq = O.fp8_encode((rng.standard_normal((M, K)) * 3.0).astype(np.float32), O.E4M3)
    wq = O.fp8_encode((rng.standard_normal((K, N)) * 0.05).astype(np.float32), O.E4M3)
    return xq, wq


def run_upproj(xq, wq, sx, sw, sh, act, *, want_h=True, want_act=True, flags=0, amax=None, sat=None):
    M, K = xq.shape
    N = wq.shape[1]
    h = torch.empty(M, N, dtype=torch.bfloat16, device="cuda") if want_h else None
    a = torch.empty(M, N, dtype=torch.bfloat16, device="cuda") if want_act else None
    q = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    amax = torch.full((1,), -1.0, device="cuda") if amax is None else amax
    sat = torch.full((1,), 777, dtype=torch.int64, device="cuda") if sat is None else sat
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.fp8_upproj_fwd(dev_u8(xq), dev_u8(np.ascontiguousarray(wq.T)), dev_f32(sx), dev_f32(sw), dev_f32(sh), q,
                     act=act, h_out=h, act_out=a, amax_out=amax, sat_count=sat, flags=flags, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return {"h": h, "act": host_bits16(a) if want_act else None, "q": host_u8(q), "amax": float(amax.item()),
            "sat": int(sat.item())}


def check_against_oracle(xq, wq, sx, sw, sh, act):
    g = run_upproj(xq, wq, sx, sw, sh, act)
    Hr, S = O.gemm_fwd(xq, wq, sx, sw)
    assert_gemm_close(g["h"], Hr, S)
    ref = O.quant(host_bits16(g["h"]), ORACLE_ACT[act], O.E4M3, sh)
    for k in ("act", "q"):
        bad = np.argwhere(g[k] != ref[k])
        assert bad.size == 0, f"{k}: {len(bad)} mismatches, first at {tuple(bad[0])}"
    assert g["amax"] == ref["amax"] and g["sat"] == ref["sat"]
    return g, ref


@pytest.mark.parametrize("act", [B.ACT_RELU2, B.ACT_IDENTITY, B.ACT_RELU])
@pytest.mark.parametrize("M,N,K", [(129, 192, 256), (1000, 640, 768), (513, 3072, 768), (64, 64, 3072)])
def test_upproj_against_oracle(M, N, K, act):
    xq, wq = _operands(M, N, K, seed=M + N + K + act)
    # unit GEMM scales put H at a few units; s_h = 448 / 8 saturates the activations above 8
    g, ref = check_against_oracle(xq, wq, 1.0, 1.0, 56.0, act)
    if act == B.ACT_RELU2:
        assert ref["sat"] > 0


def test_optional_outputs_give_the_same_codes():
    """Without H, without the activation copy, or without both: the same E4M3
    codes, amax and saturation count."""
    xq, wq = _operands(700, 1024, 512, seed=5)
    full = run_upproj(xq, wq, 4.0, 64.0, 100.0, B.ACT_RELU2)
    for want_h, want_act in ((False, True), (True, False), (False, False)):
        part = run_upproj(xq, wq, 4.0, 64.0, 100.0, B.ACT_RELU2, want_h=want_h, want_act=want_act)
        assert np.array_equal(part["q"], full["q"])
        assert part["amax"] == full["amax"] and part["sat"] == full["sat"]
        if want_act:
            assert np.array_equal(part["act"], full["act"])


EQ_TILES = [(0, 128), (0, 192), (0, 256), (1, 128), (1, 192), (1, 256)]


@pytest.mark.parametrize("pair,bn", EQ_TILES)
def test_every_tile_on_ragged_problems(pair, bn):
    """Each tile of the epilogue on problems with partial tiles in M and N,
    including N = 400 (the last 64-column E4M3 box holds one chunk)."""
    try:
        B.fp8q_gemm_set_tile(pair, bn)
        for M, N, K in [(300, 400, 256), (1000, 144, 640), (257, 1088, 128)]:
            xq, wq = _operands(M, N, K, seed=3 * M + N + bn)
            check_against_oracle(xq, wq, 2.0, 32.0, 50.0, B.ACT_RELU2)
    finally:
        B.fp8q_gemm_set_tile(-1)


def test_accumulate_folds_into_amax_and_count():
    """FP8Q_ACCUMULATE: a second call folds its maximum and saturations into
    the first call's instead of resetting them."""
    xa, wq = _operands(256, 512, 256, seed=11)
    xb, _ = _operands(256, 512, 256, seed=12)
    amax = torch.zeros(1, device="cuda")
    sat = torch.zeros(1, dtype=torch.int64, device="cuda")
    ra = run_upproj(xa, wq, 1.0, 1.0, 56.0, B.ACT_RELU2, amax=amax, sat=sat)
    a1, s1 = ra["amax"], ra["sat"]
    rb = run_upproj(xb, wq, 1.0, 1.0, 56.0, B.ACT_RELU2, amax=amax, sat=sat, flags=B.ACCUMULATE)
    solo = run_upproj(xb, wq, 1.0, 1.0, 56.0, B.ACT_RELU2)
    assert s1 > 0 and solo["sat"] > 0
    assert rb["amax"] == max(a1, solo["amax"])
    assert rb["sat"] == s1 + solo["sat"]
