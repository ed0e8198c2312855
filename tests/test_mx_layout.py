"""The MX scale layout (include/fp8q.h, fp8_quant_mx): 512-byte atoms of 128
rows x 4 blocks, byte of (row r, block b) at 512 ((r / 128) G + b / 4) +
16 (r % 32) + 4 ((r / 32) % 4) + b % 4, G = ceil(KB / 4).  The tests' own
helpers that undo it (tests/parity.py) are checked here against that formula
byte by byte, and the library's size function against the helpers, on the
CPU (the library's size call needs no device)."""
import ctypes

import numpy as np
import pytest

from tests.parity import mx_scale_bytes, mx_tile, mx_untile


@pytest.fixture(scope="module")
def lib():
    from quantize_fp8_gemm_gb300 import binding, build
    build.build()
    return binding.lib()

SHAPES = [(1, 1), (5, 3), (31, 4), (128, 4), (129, 5), (300, 20), (1000, 40), (257, 9)]


@pytest.mark.parametrize("rows,KB", SHAPES)
def test_tile_places_every_byte_by_the_formula(rows, KB):
    rng = np.random.default_rng(rows * 31 + KB)
    x = rng.integers(0, 256, (rows, KB)).astype(np.uint8)
    t = mx_tile(x)
    G = -(-KB // 4)
    assert t.size == mx_scale_bytes(rows, KB) == -(-rows // 128) * G * 512
    for r in range(rows):
        for b in range(KB):
            off = 512 * ((r // 128) * G + b // 4) + 16 * (r % 32) + 4 * ((r // 32) % 4) + b % 4
            assert t[off] == x[r, b]
    got, pad = mx_untile(t, rows, KB, pad=True)
    assert np.array_equal(got, x)
    assert (pad == 127).all()


def test_every_byte_of_an_atom_is_used_once():
    """One full atom: the 512 offsets of 128 rows x 4 blocks are a permutation."""
    x = np.arange(512, dtype=np.int64).reshape(128, 4)
    G = 1
    offs = sorted(512 * ((r // 128) * G + b // 4) + 16 * (r % 32) + 4 * ((r // 32) % 4) + b % 4
                  for r in range(128) for b in range(4))
    assert offs == list(range(512))
    t = mx_tile((x % 256).astype(np.uint8))
    assert t.size == 512


def test_library_size_function_matches(lib):
    sb = lib.fp8_mx_scale_bytes
    sb.argtypes = [ctypes.c_int64, ctypes.c_int64]
    sb.restype = ctypes.c_int64
    for rows, KB in SHAPES + [(131072, 200), (1600, 200), (16384, 128)]:
        assert sb(rows, 32 * KB) == mx_scale_bytes(rows, KB) == mx_tile(np.zeros((rows, KB), np.uint8)).size
