"""fp8_downproj_fwd_noalloc (the fused quantize + GEMM with its ready counts
in the library's static device array) against fp8_downproj_fwd (the same
kernel with a caller workspace).  Two no-alloc calls in a row, with different
inputs and a smaller M the second time, into the same output buffers: counts
left over from the first call would let the second call's GEMM load stale
codes, so a missing clear shows up as a mismatch.  The two entry points run
one kernel, so every output must agree bit for bit (inside the GEMM
tolerance of the other tests)."""
import numpy as np
import pytest
import torch

from quantize_fp8_gemm_gb300 import binding as B
from quantize_fp8_gemm_gb300 import workloads as WL
from tests.parity import dev_bf16, dev_f32

pytestmark = pytest.mark.gpu


def _outputs(M, N, K):
    return dict(a=torch.empty(M, K, dtype=torch.bfloat16, device="cuda"),
                q=torch.empty(M, K, dtype=torch.uint8, device="cuda"),
                y=torch.empty(M, N, dtype=torch.bfloat16, device="cuda"),
                amax=torch.full((1,), -1.0, device="cuda"),
                sat=torch.full((1,), 99, dtype=torch.int64, device="cuda"),
                st=torch.zeros(1, dtype=torch.int32, device="cuda"))


def _same(o, r, M):
    assert torch.equal(o["q"][:M], r["q"]), "E4M3 codes"
    assert torch.equal(o["a"][:M].view(torch.int16), r["a"].view(torch.int16)), "BF16 activation"
    assert torch.equal(o["y"][:M].view(torch.int16), r["y"].view(torch.int16)), "Y"
    assert o["amax"].item() == r["amax"].item() and o["sat"].item() == r["sat"].item()
    assert o["st"].item() == 0 and r["st"].item() == 0


def test_noalloc_matches_workspace_entry_two_calls():
    N, K = 272, 640
    rng = np.random.default_rng(2024)
    w_bits = WL.to_bf16_bits(rng.standard_normal((K, N)).astype(np.float32) * np.float32(0.05))
    wt = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    sw = dev_f32(300.0)
    B.fp8_quant_fused(dev_bf16(w_bits), B.ACT_IDENTITY, B.E4M3, sw, q_t_out=wt)
    sx = dev_f32(40.0)
    Mmax = 1000
    mine = _outputs(Mmax, N, K)  # shared by both no-alloc calls
    for M, std in ((1000, 1.5), (700, 2.5)):
        h = dev_bf16(WL.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32) * np.float32(std)))
        ref = _outputs(M, N, K)
        ws = torch.empty(B.fp8_downproj_workspace_bytes(M), dtype=torch.uint8, device="cuda")
        B.fp8_downproj_fwd(h, wt, sx, sw, ref["q"], ref["y"], ws, act=B.ACT_RELU2, act_out=ref["a"],
                           amax_out=ref["amax"], sat_count=ref["sat"], status=ref["st"])
        B.fp8_downproj_fwd_noalloc(h, wt, sx, sw, mine["q"][:M], mine["y"][:M], act=B.ACT_RELU2,
                                   act_out=mine["a"][:M], amax_out=mine["amax"], sat_count=mine["sat"],
                                   status=mine["st"])
        torch.cuda.synchronize()
        _same(mine, ref, M)
        assert ref["sat"].item() > 0  # the scale saturates some of these rows


def test_noalloc_rejects_rows_beyond_its_array():
    M, N, K = B.NOALLOC_MAX_M + 1, 16, 16
    h = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    wt = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.Fp8qError) as e:
        B.fp8_downproj_fwd_noalloc(h, wt, dev_f32(1.0), dev_f32(1.0), q, y)
    assert e.value.status == 3  # FP8Q_ERR_SHAPE
