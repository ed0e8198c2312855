"""Host side of the step module: the constructor's refusals, checked before
any device memory is touched.  (The overflow decision of detect-and-recompute
is taken on the device, from the casts' saturation counts; its tests run on
the GPU.)"""
import pytest


@pytest.mark.parametrize("kw", [dict(fused=True), dict(group=True), dict(chunks=2)])
def test_backward_needs_the_one_block_per_tensor_step(kw):
    """backward() reads the X_q^T that the one-block per-tensor step caches; the
    constructor refuses the other step forms before it allocates anything."""
    from quantize_fp8_gemm_gb300.downproj import Fp8DownProj
    with pytest.raises(ValueError):
        Fp8DownProj(1024, 768, 768, with_backward=True, device="cpu", **kw)
