"""Host side of detect-and-recompute ("FP8 Training & Inference", Delayed
Scaling: a delayed scale too large for the step's values is detected and the
step recomputed with a corrected scale): the overflow decision, pinned to the
oracle's saturation count of the same cast."""
import numpy as np
import pytest

import oracle as O
from quantize_fp8_gemm_gb300 import binding as B
from quantize_fp8_gemm_gb300.downproj import fp8_overflow


def test_activation_overflow_is_any_saturation():
    assert fp8_overflow(0, 1.0, 1.0) == (False, False)
    assert fp8_overflow(1, 1.0, 1.0) == (True, False)
    assert fp8_overflow(10 ** 9, 1.0, 1.0)[0]


def test_weight_overflow_boundary():
    """448 itself is representable; the next FP32 product above it saturates."""
    up = float(np.nextafter(np.float32(1.0), np.float32(2.0)))
    assert fp8_overflow(0, 448.0, 1.0) == (False, False)
    assert fp8_overflow(0, 448.0, up) == (False, True)
    assert fp8_overflow(0, 0.0, 3.0e38) == (False, False)
    assert fp8_overflow(0, 57344.0, 1.0, B.E5M2) == (False, False)
    assert fp8_overflow(0, 57344.0, up, B.E5M2) == (False, True)


@pytest.mark.parametrize("seed", range(6))
def test_weight_decision_matches_the_oracle_cast(seed):
    """For W and a scale near the edge, the decision equals 'the oracle's cast
    of W with that scale saturates at least one value'."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((64, 96)) * 0.05).astype(np.float32)
    bits = O.f32_to_bf16(W)
    amax = O.amax(bits, O.ACT_IDENTITY)
    edge = np.float32(448.0) / np.float32(amax)
    for s in (edge, np.nextafter(edge, np.float32(0)), np.nextafter(edge, np.float32(np.inf)), edge * 2, edge / 2):
        r = O.quant(bits, O.ACT_IDENTITY, O.E4M3, float(s), want_act=False)
        assert fp8_overflow(0, amax, float(s))[1] == (r["sat"] > 0), (seed, float(s))


@pytest.mark.parametrize("kw", [dict(fused=True), dict(group=True), dict(chunks=2)])
def test_backward_needs_the_one_block_per_tensor_step(kw):
    """backward() reads the X_q^T that the one-block per-tensor step caches; the
    constructor refuses the other step forms before it allocates anything."""
    from quantize_fp8_gemm_gb300.downproj import Fp8DownProj
    with pytest.raises(ValueError):
        Fp8DownProj(1024, 768, 768, with_backward=True, device="cpu", **kw)
