"""CPU oracle for the forward FP8 MLP down-projection.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``quantize_fp8_gemm_gb300``) never imports, links or runs it.

This module is argument marshalling around ``oref.c`` (numpy arrays in,
numpy arrays out).  The arithmetic lives in the C file, except two plain numpy
steps stated where they are used (the weight gradient's transposed operand in
``gemm_wgrad``, the activation derivative in ``act_grad``); written from the
pages:

* "FP8 training: what it is and how it works" -- Step 1 (E4M3/E5M2), Step 2
  (scale = format max / amax), Step 3 (FP8 inputs, wide sums), Worked example
  and Trade-offs (1x128 / 128x128 groups, delayed scaling history).
* "FP8 Training & Inference" -- FP8 Formats, FP8 Training Recipe (three GEMMs),
  Per-Tensor Scaling, Delayed Scaling.
* "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records" -- the
  fused activation + quantize step with running maxima and a delayed,
  margin-multiplied scale.
* "Pretraining at scale", 4a -- BF16 rounding.

Parity pins (tests/test_oracle_pins.py, tests/test_oracle_mx_pins.py) tie each
function to printed values, closed forms, exhaustive code sweeps or an
independent library routine; the group-scale and MX GEMMs are pinned by
closed-form special cases and exact integer sums (see there).  The MX
functions (32-value blocks, power-of-two scales: "FP8 training: what it is
and how it works", Trade-offs and edge cases) are the reference of the
block-scaled GPU path (fp8_quant_mx, fp8_gemm_mx).
"""
import ctypes
import os

import numpy as np

from .build import build as _build

E4M3, E5M2 = 0, 1
ACT_IDENTITY, ACT_RELU, ACT_RELU2 = 0, 1, 2
GROUP = 128

_lib = None


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(_build())
        P = ctypes.c_void_p
        i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        L.oref_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oref_bf16_to_f32.restype = f32
        L.oref_f32_to_bf16.argtypes = [f32]
        L.oref_f32_to_bf16.restype = ctypes.c_uint16
        L.oref_f32_to_bf16_array.argtypes = [P, i64, P]
        L.oref_fp8_max.argtypes = [i32]
        L.oref_fp8_max.restype = f64
        L.oref_fp8_decode.argtypes = [ctypes.c_uint8, i32]
        L.oref_fp8_decode.restype = f64
        L.oref_fp8_encode.argtypes = [f32, i32]
        L.oref_fp8_encode.restype = ctypes.c_uint8
        L.oref_fp8_encode_array.argtypes = [P, i64, i32, P]
        L.oref_fp8_decode_array.argtypes = [P, i64, i32, P]
        L.oref_act.argtypes = [f32, i32]
        L.oref_act.restype = f32
        L.oref_delayed_scale.argtypes = [f32, f32, i32]
        L.oref_delayed_scale.restype = f32
        L.oref_history_update.argtypes = [P, i32, P, f32, f32, i32, P]
        L.oref_history_update.restype = i32
        L.oref_group_scale.argtypes = [f32, i32]
        L.oref_group_scale.restype = f32
        L.oref_quant.argtypes = [P, i64, i64, i32, i32, f32, P, P, P, P, P, i32]
        L.oref_quant_group.argtypes = [P, i64, i64, i32, i32, i32, P, P, P, P, P, P, i32]
        L.oref_amax.argtypes = [P, i64, i32]
        L.oref_amax.restype = f32
        L.oref_gemm_fwd.argtypes = [P, i32, P, i32, i64, i64, i64, P, P, i32, P, i64, P, P, i32]
        L.oref_mx_scale.argtypes = [f32, i32]
        L.oref_mx_scale.restype = f32
        L.oref_quant_mx.argtypes = [P, i64, i64, i32, i32, P, P, P, P, P, P, i32]
        L.oref_gemm_mx.argtypes = [P, i32, P, i32, i64, i64, i64, P, P, P, i64, P, P, i32]
        L.oref_gemm_dgrad.argtypes = [P, i32, P, i32, i64, i64, i64, f32, f32, P, i64, P, P, i32]
        L.oref_openmp_max_threads.restype = i32
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- scalars --
def bf16_to_f32(u16):
    u16 = _c(u16, np.uint16)
    return (u16.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oref_f32_to_bf16_array(_p(x), x.size, _p(out))
    return out


def fp8_max(fmt: int) -> float:
    return lib().oref_fp8_max(fmt)


def fp8_encode(v, fmt: int):
    v = _c(v, np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().oref_fp8_encode_array(_p(v), v.size, fmt, _p(out))
    return out


def fp8_decode(codes, fmt: int):
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().oref_fp8_decode_array(_p(c), c.size, fmt, _p(out))
    return out


def act(h: float, which: int) -> float:
    return lib().oref_act(float(h), which)


def delayed_scale(amax_ref: float, margin: float, fmt: int) -> float:
    return lib().oref_delayed_scale(amax_ref, margin, fmt)


def group_scale(amax_g: float, fmt: int) -> float:
    return lib().oref_group_scale(amax_g, fmt)


def history_update(history, head: int, amax_new: float, margin: float, fmt: int, scale: float):
    """One delayed-scaling step.  Returns (status, history', head', scale')."""
    h = _c(history, np.float32).copy()
    hd = ctypes.c_int(head)
    sc = ctypes.c_float(scale)
    st = lib().oref_history_update(_p(h), h.size, ctypes.byref(hd), amax_new, margin, fmt,
                                   ctypes.byref(sc))
    return st, h, hd.value, sc.value


# ------------------------------------------------------------------ tensors --
def quant(h_bf16, act_kind: int, fmt: int, scale: float, *, want_act=True, want_q=True,
          want_qt=False, nthreads=None):
    """Per-tensor fused quantize of a [M,K] BF16 tensor (uint16 bit patterns)."""
    h = _c(h_bf16, np.uint16)
    M, K = h.shape
    a = np.empty((M, K), np.uint16) if want_act else None
    q = np.empty((M, K), np.uint8) if want_q else None
    qt = np.empty((K, M), np.uint8) if want_qt else None
    amax = np.zeros(1, np.float32)
    sat = np.zeros(1, np.uint64)
    lib().oref_quant(_p(h), M, K, act_kind, fmt, float(scale), _p(a), _p(q), _p(qt),
                     _p(amax), _p(sat), nthreads or default_threads())
    return {"act": a, "q": q, "q_t": qt, "amax": float(amax[0]), "sat": int(sat[0])}


def quant_group(h_bf16, act_kind: int, fmt: int, group_rows: int, *, want_act=True,
                want_q=True, want_qt=False, nthreads=None):
    """Group-scaled quantize: blocks of group_rows x 128 (1 -> 1x128 tiles, 128 -> blocks)."""
    h = _c(h_bf16, np.uint16)
    M, K = h.shape
    assert K % GROUP == 0
    nbr = (M + group_rows - 1) // group_rows
    a = np.empty((M, K), np.uint16) if want_act else None
    q = np.empty((M, K), np.uint8) if want_q else None
    qt = np.empty((K, M), np.uint8) if want_qt else None
    scales = np.empty((nbr, K // GROUP), np.float32)
    amax = np.zeros(1, np.float32)
    sat = np.zeros(1, np.uint64)
    lib().oref_quant_group(_p(h), M, K, act_kind, fmt, group_rows, _p(a), _p(q), _p(qt),
                           _p(scales), _p(amax), _p(sat), nthreads or default_threads())
    return {"act": a, "q": q, "q_t": qt, "scales": scales, "amax": float(amax[0]),
            "sat": int(sat[0])}


def mx_scale(amax_b: float, fmt: int) -> float:
    """The power-of-two scale of one 32-value block (see oref_mx_scale)."""
    return lib().oref_mx_scale(amax_b, fmt)


def quant_mx(h_bf16, act_kind: int, fmt: int, *, want_act=True, nthreads=None):
    """MX quantize: one power-of-two scale per 32-value block of each row of the
    [M,K] BF16 tensor.  Returns q, act, scales [M, K/32] (float32 powers of
    two), exps [M, K/32] (the biased exponent bytes of 1 / scale), amax, sat."""
    h = _c(h_bf16, np.uint16)
    M, K = h.shape
    assert K % 32 == 0
    a = np.empty((M, K), np.uint16) if want_act else None
    q = np.empty((M, K), np.uint8)
    scales = np.empty((M, K // 32), np.float32)
    exps = np.empty((M, K // 32), np.uint8)
    amax = np.zeros(1, np.float32)
    sat = np.zeros(1, np.uint64)
    lib().oref_quant_mx(_p(h), M, K, act_kind, fmt, _p(a), _p(q), _p(scales), _p(exps), _p(amax), _p(sat),
                        nthreads or default_threads())
    return {"act": a, "q": q, "scales": scales, "exps": exps, "amax": float(amax[0]), "sat": int(sat[0])}


def gemm_mx(x_q, s_x, w_q, s_w, *, rows=None, fmt_x=E4M3, fmt_w=E4M3, nthreads=None):
    """Y = X x W over MX-dequantised FP8: X [M,K] with s_x [M, K/32], W [K,N]
    with s_w [N, K/32] (the blocks of W's columns).  Returns (Y, S)."""
    X = _c(x_q, np.uint8)
    W = _c(w_q, np.uint8)
    M, K = X.shape
    K2, N = W.shape
    assert K == K2 and K % 32 == 0
    sx = _c(s_x, np.float32)
    sw = _c(s_w, np.float32)
    assert sx.shape == (M, K // 32) and sw.shape == (N, K // 32)
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    Y = np.empty((rows.size, N), np.float64)
    S = np.empty((rows.size, N), np.float64)
    lib().oref_gemm_mx(_p(X), fmt_x, _p(W), fmt_w, M, N, K, _p(sx), _p(sw), _p(rows), rows.size, _p(Y), _p(S),
                       nthreads or default_threads())
    return Y, S


def amax(h_bf16, act_kind: int) -> float:
    h = _c(h_bf16, np.uint16)
    return lib().oref_amax(_p(h), h.size, act_kind)


def gemm_fwd(x_q, w_q, s_x, s_w, *, group=False, rows=None, fmt_x=E4M3, fmt_w=E4M3,
             nthreads=None):
    """Y = X x W over dequantised FP8; X [M,K], W [K,N] (row-major).  Returns (Y, S)."""
    X = _c(x_q, np.uint8)
    W = _c(w_q, np.uint8)
    M, K = X.shape
    K2, N = W.shape
    assert K == K2
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    sx = _c(np.atleast_1d(s_x), np.float32)
    sw = _c(np.atleast_1d(s_w), np.float32)
    Y = np.empty((rows.size, N), np.float64)
    S = np.empty((rows.size, N), np.float64)
    lib().oref_gemm_fwd(_p(X), fmt_x, _p(W), fmt_w, M, N, K, _p(sx), _p(sw), int(bool(group)),
                        _p(rows), rows.size, _p(Y), _p(S), nthreads or default_threads())
    return Y, S


def gemm_dgrad(dy_q, w_q, s_dy: float, s_w: float, *, rows=None, fmt_dy=E5M2, fmt_w=E4M3,
               nthreads=None):
    """dX = dY x W^T over dequantised FP8; dY [M,N], W [K,N].  Returns (dX, S)."""
    D = _c(dy_q, np.uint8)
    W = _c(w_q, np.uint8)
    M, N = D.shape
    K, N2 = W.shape
    assert N == N2
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    dX = np.empty((rows.size, K), np.float64)
    S = np.empty((rows.size, K), np.float64)
    lib().oref_gemm_dgrad(_p(D), fmt_dy, _p(W), fmt_w, M, N, K, float(s_dy), float(s_w),
                          _p(rows), rows.size, _p(dX), _p(S), nthreads or default_threads())
    return dX, S


def act_grad(h_bf16, act_kind: int):
    """d act(h) / dh at the BF16 values h (float64): ReLU^2 -> 2 max(h, 0), ReLU
    -> 1 where h > 0 else 0, identity -> 1 (the derivatives of the activations
    of "Paradigma Details FP8 and Optimizer Tricks Behind NanoGPT Records",
    second paragraph; h > 0 is the comparison the forward's ReLU uses)."""
    h = bf16_to_f32(_c(h_bf16, np.uint16)).astype(np.float64)
    if act_kind == ACT_RELU2:
        return np.where(h > 0, 2.0 * h, 0.0)
    if act_kind == ACT_RELU:
        return np.where(h > 0, 1.0, 0.0)
    return np.ones_like(h)


def act_grad_q(h_q, s_h: float, act_kind: int):
    """The activation derivative at the pre-activation cached in FP8 ("FP8
    training: what it is and how it works", Trade-offs and edge cases: the
    activations kept for the backward pass are stored in FP8): h~ =
    dec(h_q) / s_h, the E4M3 code of H dequantised with the scale it was cast
    with (float64, exact), then the derivative of act_grad at h~."""
    h = fp8_decode(_c(h_q, np.uint8), E4M3) / float(s_h)
    if act_kind == ACT_RELU2:
        return np.where(h > 0, 2.0 * h, 0.0)
    if act_kind == ACT_RELU:
        return np.where(h > 0, 1.0, 0.0)
    return np.ones_like(h)


def gemm_dgrad_act_q(dy_q, w_q, s_dy: float, s_w: float, h_q, s_h: float, act_kind: int, *, rows=None,
                     fmt_dy=E5M2, fmt_w=E4M3, nthreads=None):
    """gemm_dgrad_act with the pre-activation taken from its E4M3 cache h_q [M,K]
    (cast with the scale s_h): dH = (dY x W^T) * act'(dec(h_q) / s_h).
    Returns (dH, S): S is the dgrad's sum of |terms| times |act'|."""
    dX, S = gemm_dgrad(dy_q, w_q, s_dy, s_w, rows=rows, fmt_dy=fmt_dy, fmt_w=fmt_w, nthreads=nthreads)
    hq = _c(h_q, np.uint8)
    if rows is not None:
        hq = hq[_c(rows, np.int64)]
    g = act_grad_q(hq, s_h, act_kind)
    return dX * g, S * np.abs(g)


def gemm_dgrad_act(dy_q, w_q, s_dy: float, s_w: float, h_bf16, act_kind: int, *, rows=None, fmt_dy=E5M2,
                   fmt_w=E4M3, nthreads=None):
    """The activation backward through the down-projection's dgrad:
    dH = (dY x W^T) * act'(H) over dequantised FP8, dY [M,N], W [K,N], H [M,K]
    BF16.  Returns (dH, S): S is the dgrad's sum of |terms| times |act'(H)|."""
    dX, S = gemm_dgrad(dy_q, w_q, s_dy, s_w, rows=rows, fmt_dy=fmt_dy, fmt_w=fmt_w, nthreads=nthreads)
    h = _c(h_bf16, np.uint16)
    if rows is not None:
        h = h[_c(rows, np.int64)]
    g = act_grad(h, act_kind)
    return dX * g, S * np.abs(g)


def gemm_wgrad(x_q, dy_q, s_x: float, s_dy: float, *, rows=None, fmt_x=E4M3, fmt_dy=E5M2,
               nthreads=None):
    """dW = X^T x dY over dequantised FP8 ("FP8 Training & Inference", FP8
    Training Recipe: the weight gradient of the E4M3 activation and the E5M2
    output gradient); X [M,K], dY [M,N] in their own layouts, contracted over
    the M tokens.  rows: the rows k of dW to compute.  Returns (dW, S): S is
    sum_m |x[m,k] dy[m,n]| / (s_x s_dy)."""
    X = _c(x_q, np.uint8)
    D = _c(dy_q, np.uint8)
    assert X.shape[0] == D.shape[0]
    # dW[k, n] = sum_m X^T[k, m] dY[m, n]: the plain GEMM with X^T as its first operand
    return gemm_fwd(np.ascontiguousarray(X.T), D, s_x, s_dy, rows=rows, fmt_x=fmt_x, fmt_w=fmt_dy,
                    nthreads=nthreads)


def openmp_threads() -> int:
    return lib().oref_openmp_max_threads()
