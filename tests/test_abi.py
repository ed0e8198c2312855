"""The C ABI library builds, loads and exports every function include/*.h
declares; its host-side argument checks return the documented status codes.
No kernel is launched: with no sm_103 device visible, valid arguments end in
FP8Q_ERR_UNSUPPORTED, and invalid ones are rejected before any CUDA call.
The pointers passed here are never dereferenced on the host.
"""
import ctypes
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

INCLUDE = os.path.join(ROOT, "include")

OK, ERR_NULL, ERR_ALIGN, ERR_SHAPE, ERR_UNSUPPORTED, ERR_CUDA = range(6)


@pytest.fixture(scope="module")
def lib():
    from quantize_fp8_gemm_gb300 import build
    path = build.build()
    from quantize_fp8_gemm_gb300 import binding
    return binding.lib()


# which library exports the functions each header declares
HEADER_LIBS = {"fp8q.h": "libfp8q.so", "fp8q_testing.h": "libfp8q.so", "fp8q_naive.h": "libfp8q_naive.so"}


def declared_functions(header=None):
    names = []
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h") and (header is None or h == header):
            text = open(os.path.join(INCLUDE, h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_\s\*]*?\b([a-z][a-z0-9_]*)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for fn in ("fp8_quant_fused", "fp8_gemm_fwd", "fp8_gemm_dgrad", "amax_history_update"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    from quantize_fp8_gemm_gb300 import binding
    headers = sorted(h for h in os.listdir(INCLUDE) if h.endswith(".h"))
    assert set(headers) == set(HEADER_LIBS), "a header without a library to check it against"
    for h in headers:
        path = os.path.join(binding.PKG, HEADER_LIBS[h])
        out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
        exported = set(re.findall(r"\s[TW]\s+(\S+)$", out, re.M))
        dl = ctypes.CDLL(path)
        for fn in declared_functions(h):
            assert fn in exported, f"{fn} declared in include/{h} but not exported by {HEADER_LIBS[h]}"
            assert hasattr(dl, fn)


def test_product_library_holds_no_comparator(lib):
    """The unfused three-pass comparator lives in libfp8q_naive.so only."""
    from quantize_fp8_gemm_gb300 import binding
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True).stdout
    assert "fp8q_naive" not in out


def test_status_strings_and_version(lib):
    assert lib.fp8q_version() >= 100
    for s in range(6):
        assert lib.fp8q_status_string(s)


A = 1 << 20  # a 16-byte aligned fake device address (never dereferenced)


def quant(lib, h=A, M=64, K=256, act=2, fmt=0, scale=A, act_out=A, q=A, qt=None, amax=A, sat=A,
          gs=None, grows=1):
    return lib.fp8_quant_fused(h, M, K, act, fmt, scale, act_out, q, qt, amax, sat, gs, grows, None)


def test_quant_argument_checks(lib):
    assert quant(lib, h=None) == ERR_NULL
    assert quant(lib, scale=None) == ERR_NULL
    assert quant(lib, act=3) == ERR_UNSUPPORTED
    assert quant(lib, fmt=2) == ERR_UNSUPPORTED
    assert quant(lib, K=8) == ERR_SHAPE
    assert quant(lib, K=40) == ERR_SHAPE
    assert quant(lib, M=-1) == ERR_SHAPE
    assert quant(lib, qt=A, M=65) == ERR_SHAPE
    assert quant(lib, h=A + 8) == ERR_ALIGN
    assert quant(lib, q=A + 4) == ERR_ALIGN
    assert quant(lib, sat=A + 4) == ERR_ALIGN
    assert quant(lib, gs=A, K=192) == ERR_SHAPE
    assert quant(lib, gs=A, grows=2) == ERR_UNSUPPORTED
    # well-formed: only the device check remains, and there is no sm_103 here
    assert quant(lib) == ERR_UNSUPPORTED
    assert quant(lib, scale=None, gs=A, grows=128) == ERR_UNSUPPORTED


def gemm(lib, a=A, b=A, sa=A, sb=A, grp=0, d=A, M=128, N=256, K=512, st=None):
    return lib.fp8_gemm_fwd(a, b, sa, sb, grp, d, M, N, K, st, None)


def test_gemm_fwd_update_history_checks(lib):
    """fp8_gemm_fwd_update: the history arguments are checked first (by the
    rules of amax_history_update_ex, and against the scales and amax values
    the GEMM itself uses); a well-formed call then stops at the device check."""
    import ctypes
    from quantize_fp8_gemm_gb300 import binding
    H, S, AX, AW, CLR = A + 4096, A + 8192, A + 12288, A + 16384, A + 20480

    def hist(**kw):
        h = dict(history=H, L=4, head=A + 24576, margin=2.0, fmt=0, scale_prev=S, scale_out=A + 28672, status=None,
                 amax_clear=CLR, sat_clear=None)
        h.update(kw)
        return binding.HistoryArgs(*[h[f] for f, _ in binding.HistoryArgs._fields_])

    def call(hx=None, hw=None, sx=S, amax_x=AX):
        return lib.fp8_gemm_fwd_update(A, A, sx, A + 32768, A, 256, 256, 512, amax_x,
                                       None if hx is None else ctypes.byref(hx), AW,
                                       None if hw is None else ctypes.byref(hw), None, None)

    assert call(hist(history=None)) == ERR_NULL
    assert call(hist(L=0)) == ERR_SHAPE
    assert call(hist(fmt=7)) == ERR_UNSUPPORTED
    assert call(hist(margin=0.0)) == ERR_SHAPE
    assert call(hist(head=A + 2)) == ERR_ALIGN
    assert call(hist(scale_out=S)) == ERR_SHAPE           # would overwrite scale_x
    assert call(None, hist(scale_out=A + 32768)) == ERR_SHAPE  # would overwrite scale_w
    assert call(hist(amax_clear=AW)) == ERR_SHAPE         # would clear the other amax
    assert call(hist(), amax_x=None) == ERR_NULL
    assert call(hist(), hist(history=A + 36864, head=A + 40960, scale_out=A + 45056, amax_clear=A + 49152)) \
        == ERR_UNSUPPORTED
    assert call() == ERR_UNSUPPORTED


def test_gemm_argument_checks(lib):
    assert gemm(lib, a=None) == ERR_NULL
    assert gemm(lib, sb=None) == ERR_NULL
    assert gemm(lib, N=8) == ERR_SHAPE
    assert gemm(lib, N=24) == ERR_SHAPE
    assert gemm(lib, K=40) == ERR_SHAPE
    assert gemm(lib, M=-5) == ERR_SHAPE
    assert gemm(lib, d=A + 2) == ERR_ALIGN
    assert gemm(lib, st=A + 2) == ERR_ALIGN
    assert gemm(lib) == ERR_UNSUPPORTED
    dg = lib.fp8_gemm_dgrad
    assert dg(A, A, A, A, A, 128, 24, 256, None, None) == ERR_SHAPE      # contraction N % 16
    assert dg(A, A, A, A, None, 128, 32, 256, None, None) == ERR_NULL
    assert dg(A, A, A, A, A, 128, 32, 256, None, None) == ERR_UNSUPPORTED
    da = lib.fp8_gemm_dgrad_act
    da.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_void_p] + [ctypes.c_int64] * 3 + [ctypes.c_void_p] * 2
    da.restype = ctypes.c_int
    assert da(A, A, A, A, A, 3, A, 128, 32, 256, None, None) == ERR_UNSUPPORTED   # act
    assert da(A, A, A, A, None, 2, A, 128, 32, 256, None, None) == ERR_NULL       # h
    assert da(A, A, A, A, A + 8, 2, A, 128, 32, 256, None, None) == ERR_ALIGN     # h alignment
    assert da(A, A, A, A, A, 2, A, 128, 24, 256, None, None) == ERR_SHAPE         # contraction N % 16
    assert da(A, A, A, A, A, 2, A, 128, 32, 256, None, None) == ERR_UNSUPPORTED   # no sm_103 device here
    wg = lib.fp8_gemm_wgrad
    wg.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_void_p] * 2
    wg.restype = ctypes.c_int
    assert wg(A, A, A, A, A, 1000, 64, 256, None, None) == ERR_SHAPE     # contraction M % 16
    assert wg(A, A, A, A, A, 0, 64, 256, None, None) == ERR_SHAPE        # contraction M >= 16
    assert wg(A, A, A, A, A, 1024, 40, 256, None, None) == ERR_SHAPE     # N % 16
    assert wg(A, None, A, A, A, 1024, 64, 256, None, None) == ERR_NULL
    assert wg(A, A, A, A, A + 2, 1024, 64, 256, None, None) == ERR_ALIGN
    assert wg(A, A, A, A, A, 1024, 64, 256, None, None) == ERR_UNSUPPORTED


def test_upproj_argument_checks(lib):
    """fp8_upproj_fwd checks its arguments on the host, before any device work."""
    f = lib.fp8_upproj_fwd
    P, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [P, P, P, P, ctypes.c_int, P, P, P, P, P, P, i64, i64, i64, ctypes.c_uint, P, P]
    f.restype = ctypes.c_int

    def call(act=2, sh=A, h=None, a=None, q=A, amax=None, M=128, N=256, K=256, flags=0):
        return f(A, A, A, A, act, sh, h, a, q, amax, None, M, N, K, flags, None, None)

    assert call(act=3) == ERR_UNSUPPORTED
    assert call(flags=2) == ERR_UNSUPPORTED
    assert call(sh=None) == ERR_NULL
    assert call(q=None) == ERR_NULL
    assert call(a=A + 8) == ERR_ALIGN
    assert call(amax=A + 2) == ERR_ALIGN
    assert call(N=200) == ERR_SHAPE
    assert call(K=40) == ERR_SHAPE
    assert call() == ERR_UNSUPPORTED  # valid arguments, no sm_103 device here


def test_history_argument_checks(lib):
    f = lib.amax_history_update
    assert f(None, 1, A, A, 2.0, 0, A, None, None) == ERR_NULL
    assert f(A, 0, A, A, 2.0, 0, A, None, None) == ERR_SHAPE
    assert f(A, 5000, A, A, 2.0, 0, A, None, None) == ERR_SHAPE
    assert f(A, 1, A, A, 0.0, 0, A, None, None) == ERR_SHAPE
    assert f(A, 1, A, A, float("nan"), 0, A, None, None) == ERR_SHAPE
    assert f(A, 1, A, A, 2.0, 7, A, None, None) == ERR_UNSUPPORTED
    assert f(A, 1, A + 2, A, 2.0, 0, A, None, None) == ERR_ALIGN
    assert f(A, 4, A, A, 2.0, 0, A, None, None) == ERR_UNSUPPORTED


def test_binding_refuses_host_tensors(lib):
    import torch
    from quantize_fp8_gemm_gb300 import binding as B
    h = torch.zeros(16, 16, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        B.fp8_quant_fused(h, B.ACT_RELU2, B.E4M3, torch.ones(1))


def test_gemm_tile_knob_arguments(lib):
    assert lib.fp8q_gemm_set_tile(0, 96) == ERR_UNSUPPORTED
    assert lib.fp8q_gemm_set_tile(0, 224) == ERR_UNSUPPORTED
    assert lib.fp8q_gemm_set_tile(2, 128) == ERR_UNSUPPORTED
    assert lib.fp8q_gemm_set_tile(1, 224) == OK
    assert lib.fp8q_gemm_set_tile(1, 384) == OK
    assert lib.fp8q_gemm_set_tile(0, 384) == ERR_UNSUPPORTED
    assert lib.fp8q_gemm_set_tile(0, 160) == OK
    assert lib.fp8q_gemm_set_tile(-1, 0) == OK


def test_cast_f32_arguments(lib):
    """fp8_cast_f32 checks its arguments on the host, before any device work."""
    f = lib.fp8_cast_f32
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    good = ctypes.c_void_p(1 << 20)
    assert f(good, good, -1, 0, None) == ERR_SHAPE
    assert f(good, good, 16, 7, None) == ERR_UNSUPPORTED
    assert f(good, good, 0, 0, None) == OK  # nothing to do, nothing enqueued
    assert f(None, good, 16, 0, None) == ERR_NULL
    assert f(good, None, 16, 1, None) == ERR_NULL
    assert f(ctypes.c_void_p((1 << 20) + 4), good, 16, 0, None) == ERR_ALIGN
    assert f(good, ctypes.c_void_p((1 << 20) + 8), 16, 0, None) == ERR_ALIGN


def test_quant_ex_flags(lib):
    lib.fp8_quant_fused_ex.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                       ctypes.c_uint, ctypes.c_void_p]
    f = lambda flags: lib.fp8_quant_fused_ex(A, 64, 256, 2, 0, A, A, A, None, A, A, None, 1, flags, None)
    assert f(2) == ERR_UNSUPPORTED
    assert f(1) == ERR_UNSUPPORTED  # valid flags: only the missing sm_103 device is left
    assert f(0) == ERR_UNSUPPORTED
    assert lib.fp8_quant_fused_ex(None, 64, 256, 2, 0, A, A, A, None, A, A, None, 1, 1, None) == ERR_NULL


def test_fused_argument_checks(lib):
    f = lambda ws=A, wsb=1 << 20, h=A, M=256, act=2: lib.fp8_downproj_fwd(
        h, A, M, 128, 256, act, A, A, A, A, A, A, A, ws, wsb, None, None)
    lib.fp8_downproj_fwd.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                     ctypes.c_void_p]
    lib.fp8_downproj_workspace_bytes.argtypes = [ctypes.c_int64]
    lib.fp8_downproj_workspace_bytes.restype = ctypes.c_size_t
    assert lib.fp8_downproj_workspace_bytes(256) == 256
    assert lib.fp8_downproj_workspace_bytes(129 * 128) == 768
    assert f(ws=None) == ERR_NULL
    assert f(h=None) == ERR_NULL
    assert f(wsb=4) == ERR_SHAPE
    assert f(act=5) == ERR_UNSUPPORTED
    assert f(h=A + 8) == ERR_ALIGN
    assert f() == ERR_UNSUPPORTED  # no sm_103 device here


def test_ex_argument_checks(lib):
    """fp8_downproj_fwd_ex: the weight's saturation counter is checked like the other counters."""
    P, i64 = ctypes.c_void_p, ctypes.c_int64
    f = lib.fp8_downproj_fwd_ex
    f.argtypes = [P, P, P, i64, i64, i64, ctypes.c_int] + [P] * 11 + [ctypes.c_size_t, P, P, ctypes.c_uint, P, P]
    f.restype = ctypes.c_int

    def call(sat_w=A, w=A, flags=0, M=256):
        return f(A, w, A, M, 128, 256, 2, A, A, A, A, A, A, A, A, sat_w, A, A, 1 << 20, None, None, flags, None, None)

    assert call(sat_w=A + 4) == ERR_ALIGN
    assert call(flags=4) == ERR_UNSUPPORTED
    assert call() == ERR_UNSUPPORTED  # valid: only the missing sm_103 device is left


def test_testing_hooks_arguments(lib):
    assert lib.fp8q_test_set_fused_grid(-1) == ERR_SHAPE
    assert lib.fp8q_test_set_fused_grid(70000) == ERR_SHAPE
    assert lib.fp8q_test_set_fused_grid(5) == OK
    assert lib.fp8q_test_set_fused_grid(0) == OK
    assert lib.fp8q_test_set_fused_layout(3) == ERR_UNSUPPORTED
    assert lib.fp8q_test_set_fused_layout(-1) == ERR_UNSUPPORTED
    assert lib.fp8q_test_set_fused_layout(2) == OK
    assert lib.fp8q_test_set_fused_layout(0) == OK
    pair, bn = ctypes.c_int(-1), ctypes.c_int(-1)
    f = lib.fp8q_test_gemm_tile
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(1024, 1600, 1, None, ctypes.byref(bn)) == ERR_NULL
    assert f(1024, 1600, 1, ctypes.byref(pair), None) == ERR_NULL
    assert f(0, 1600, 0, ctypes.byref(pair), ctypes.byref(bn)) == ERR_SHAPE
    assert f(1024, 8, 0, ctypes.byref(pair), ctypes.byref(bn)) == ERR_SHAPE
    assert (pair.value, bn.value) == (-1, -1)  # untouched on error
    import torch
    if not torch.cuda.is_available():
        # no device: the static array has no address to look up
        assert lib.fp8q_test_noalloc_fill(0, None) == ERR_CUDA


def test_noalloc_argument_checks(lib):
    f = lambda M=256, h=A, act=2: lib.fp8_downproj_fwd_noalloc(h, A, M, 128, 256, act, A, A, A, A, A, A, A,
                                                               None, None)
    assert f(h=None) == ERR_NULL
    assert f(act=5) == ERR_UNSUPPORTED
    assert f(h=A + 8) == ERR_ALIGN
    assert f(M=262144 + 1) == ERR_SHAPE  # beyond the static array's row blocks
    assert f(M=262144) == ERR_UNSUPPORTED  # at the limit: only the missing sm_103 device is left


def test_batch_quant_argument_checks(lib):
    from quantize_fp8_gemm_gb300 import binding as B
    lib.fp8_quant_fused_batch.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    assert ctypes.sizeof(B.QuantArgs) == 128
    good = B.QuantArgs(A, 64, 256, 2, 0, A, A, A, None, A, A, None, 1, 0)
    arr = (B.QuantArgs * 2)(good, good)
    assert lib.fp8_quant_fused_batch(None, 1, None) == ERR_NULL
    assert lib.fp8_quant_fused_batch(arr, 0, None) == ERR_SHAPE
    assert lib.fp8_quant_fused_batch(arr, 5, None) == ERR_SHAPE
    arr[1].K = 40
    assert lib.fp8_quant_fused_batch(arr, 2, None) == ERR_SHAPE  # the second entry's own check
    arr[1].K = 256
    arr[1].group_scales_out = A
    assert lib.fp8_quant_fused_batch(arr, 2, None) == ERR_UNSUPPORTED  # per-tensor entries only
    arr[1].group_scales_out = None
    arr[1].flags = 2
    assert lib.fp8_quant_fused_batch(arr, 2, None) == ERR_UNSUPPORTED
    arr[1].flags = 1
    assert lib.fp8_quant_fused_batch(arr, 2, None) == ERR_UNSUPPORTED  # valid: no sm_103 device here


def test_mx_argument_checks(lib):
    """fp8_quant_mx / fp8_gemm_mx check their arguments on the host."""
    P, i64 = ctypes.c_void_p, ctypes.c_int64
    q = lib.fp8_quant_mx
    q.argtypes = [P, i64, i64, ctypes.c_int, ctypes.c_int] + [P] * 8
    q.restype = ctypes.c_int

    def quant(M=64, K=256, act=2, fmt=0, a=None, qo=A, sf=A, qt=None, sft=None):
        return q(A, M, K, act, fmt, a, qo, sf, qt, sft, None, None, None)

    assert quant(qo=None, sf=None) == ERR_UNSUPPORTED            # no mode
    assert quant(qt=A, sft=A) == ERR_UNSUPPORTED                 # both modes
    assert quant(qo=None, sf=None, qt=A, sft=A, a=A) == ERR_UNSUPPORTED  # act copy in column mode
    assert quant(sf=None) == ERR_NULL
    assert quant(K=48) == ERR_SHAPE                              # rows: K % 32
    assert quant(qo=None, sf=None, qt=A, sft=A, M=48) == ERR_SHAPE  # columns: M % 32
    assert quant(qo=None, sf=None, qt=A, sft=A, K=24) == ERR_SHAPE  # columns: K % 16
    assert quant(act=4) == ERR_UNSUPPORTED
    assert quant(a=A + 8) == ERR_ALIGN
    assert quant(sf=A + 4) == ERR_ALIGN                          # scale arrays: 16-byte aligned
    assert quant(qo=None, sf=None, qt=A, sft=A + 4) == ERR_ALIGN
    assert quant() == ERR_UNSUPPORTED                            # valid: no sm_103 device here
    assert quant(qo=None, sf=None, qt=A, sft=A, K=272) == ERR_UNSUPPORTED
    g = lib.fp8_gemm_mx
    g.argtypes = [P] * 5 + [i64] * 3 + [ctypes.c_int] * 2 + [P] * 2
    g.restype = ctypes.c_int

    def gemm(M=128, N=256, K=512, fx=0, fw=0, x=A, y=A, sfx=A, sfw=A):
        return g(x, sfx, A, sfw, y, M, N, K, fx, fw, None, None)

    assert gemm(fx=2) == ERR_UNSUPPORTED
    assert gemm(x=None) == ERR_NULL
    assert gemm(K=48) == ERR_SHAPE
    assert gemm(N=24) == ERR_SHAPE
    assert gemm(M=(1 << 31) - 255) == ERR_SHAPE                 # 32-bit TMA row coordinates of pair tiles
    assert quant(M=(1 << 27) + 1, K=1024) == ERR_SHAPE           # rows: 2^32 blocks or more
    assert gemm(y=A + 2) == ERR_ALIGN
    assert gemm(sfx=A + 4) == ERR_ALIGN and gemm(sfw=A + 8) == ERR_ALIGN
    assert gemm() == ERR_UNSUPPORTED
    assert lib.fp8q_mx_set_tile(0, 96) == ERR_UNSUPPORTED
    assert lib.fp8q_mx_set_tile(0, 192) == ERR_UNSUPPORTED      # B's scale atoms: whole 128-row blocks
    assert lib.fp8q_mx_set_tile(2, 128) == ERR_UNSUPPORTED
    assert lib.fp8q_mx_set_tile(1, 0) == ERR_UNSUPPORTED
    assert lib.fp8q_mx_set_tile(0, 128) == OK and lib.fp8q_mx_set_tile(1, 256) == OK
    assert lib.fp8q_mx_set_tile(0, 0) == OK


def test_mx_scale_layout_size(lib):
    """fp8_mx_scale_bytes: 512-byte atoms of 128 rows x 4 blocks of 32 values."""
    sb = lib.fp8_mx_scale_bytes
    sb.argtypes = [ctypes.c_int64, ctypes.c_int64]
    sb.restype = ctypes.c_int64
    assert sb(128, 128) == 512 and sb(1, 32) == 512 and sb(0, 64) == 0
    assert sb(129, 128) == 1024 and sb(128, 160) == 1024
    assert sb(131072, 6400) == 1024 * 50 * 512 and sb(1600, 6400) == 13 * 50 * 512
    assert sb(-1, 32) == -1 and sb(10, 48) == -1 and sb(10, -32) == -1
