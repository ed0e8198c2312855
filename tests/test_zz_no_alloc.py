"""fp8_downproj_fwd_noalloc -- the fused quantize + GEMM for callers that
cannot allocate device memory -- against fp8_downproj_fwd (the same kernel
with a caller workspace) and against the oracle.

The entry point keeps the kernel's counters in one static array of the
library.  Before each call here the array is filled with 0xFF bytes through a
test hook, as a call that was cut short could leave it: ready counts that
claim every row is quantized, work tickets past the end and a finished-CTA
count that never reaches the grid.  The entry point must clear what it uses
before its kernel starts, or the GEMM reads codes that are not written yet
and the outputs differ.  Two calls in a row, with different inputs and a
smaller M the second time, into the same output buffers; every output must
equal the workspace entry's bit for bit (inside the GEMM tolerance of the
other tests), and the first call's outputs also the oracle's."""
import numpy as np
import pytest
import torch

import oracle as O
from quantize_fp8_gemm_gb300 import binding as B
from quantize_fp8_gemm_gb300 import workloads as WL
from tests.parity import assert_gemm_close, dev_bf16, dev_f32, host_bits16, host_u8

pytestmark = pytest.mark.gpu


def _outputs(M, N, K):
    return dict(a=torch.full((M, K), 1.0, dtype=torch.bfloat16, device="cuda"),
                q=torch.full((M, K), 0x33, dtype=torch.uint8, device="cuda"),
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
    s_w, s_x = 300.0, 40.0
    sw, sx = dev_f32(s_w), dev_f32(s_x)
    B.fp8_quant_fused(dev_bf16(w_bits), B.ACT_IDENTITY, B.E4M3, sw, q_t_out=wt)
    Mmax = 1000
    mine = _outputs(Mmax, N, K)  # shared by both no-alloc calls
    for i, (M, std) in enumerate(((1000, 1.5), (700, 2.5))):
        h_bits = WL.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32) * np.float32(std))
        h = dev_bf16(h_bits)
        ref = _outputs(M, N, K)
        ws = torch.empty(B.fp8_downproj_workspace_bytes(M), dtype=torch.uint8, device="cuda")
        B.fp8_downproj_fwd(h, wt, sx, sw, ref["q"], ref["y"], ws, act=B.ACT_RELU2, act_out=ref["a"],
                           amax_out=ref["amax"], sat_count=ref["sat"], status=ref["st"])
        B.fp8q_test_noalloc_fill(0xFF)  # what a call cut short could leave behind
        B.fp8_downproj_fwd_noalloc(h, wt, sx, sw, mine["q"][:M], mine["y"][:M], act=B.ACT_RELU2,
                                   act_out=mine["a"][:M], amax_out=mine["amax"], sat_count=mine["sat"],
                                   status=mine["st"])
        torch.cuda.synchronize()
        _same(mine, ref, M)
        assert ref["sat"].item() > 0  # the scale saturates some of these rows
        if i == 0:
            ro = O.quant(h_bits, O.ACT_RELU2, O.E4M3, s_x)
            assert np.array_equal(host_u8(mine["q"][:M]), ro["q"])
            assert np.array_equal(host_bits16(mine["a"][:M]), ro["act"])
            assert mine["amax"].item() == ro["amax"] and mine["sat"].item() == ro["sat"]
            rw = O.quant(w_bits, O.ACT_IDENTITY, O.E4M3, s_w, want_act=False)
            rows = WL.sample_rows(M, 64, seed=31)
            Yr, S = O.gemm_fwd(ro["q"][rows], rw["q"], s_x, s_w)
            assert_gemm_close(mine["y"][:M], Yr, S, rows=rows)


def test_noalloc_rejects_rows_beyond_its_array():
    M, N, K = B.NOALLOC_MAX_M + 1, 16, 16
    h = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    wt = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.Fp8qError) as e:
        B.fp8_downproj_fwd_noalloc(h, wt, dev_f32(1.0), dev_f32(1.0), q, y)
    assert e.value.status == 3  # FP8Q_ERR_SHAPE
