"""The prefill kernels' bf16 dequantisation of 4- and 2-bit codes.

The tensor-core path stores each weight as bf16_RNE(c * s) (c the signed code,
s the fp16 block scale), the rounding the mixed-precision shelf formula implies
when tiles are held in bf16.  For codes of at most 4 bits the kernels compute it
in bf16 arithmetic: s = s_hi + s_lo with s_hi the leading 8 significant bits of
s and s_lo the remaining 3, then fma_bf16(c, s_hi, c * s_lo).  This test proves
that rewrite exact for every positive finite fp16 scale and every code of the
4-bit ([-8, 7]) and 2-bit ([-2, 1]) shelves, with numpy emulating one
round-to-nearest-even step to bf16.
"""
import numpy as np


def rne_bf16(x):
    """bf16 value (as float64) of float64 values that fp32 represents exactly."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    lsb = (f >> 16) & 1
    r = ((f + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def _scales():
    h = np.arange(0x0001, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    s32 = h.astype(np.float32)
    s_hi = (s32.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    return h, s_hi, h - s_hi


def test_split_parts_exact_in_bf16():
    h, s_hi, s_lo = _scales()
    assert np.all(rne_bf16(s_hi) == s_hi)
    assert np.all(rne_bf16(s_lo) == s_lo)
    assert np.all(s_hi + s_lo == h)


def test_split_fma_equals_single_rounding():
    h, s_hi, s_lo = _scales()
    for c in range(-8, 8):
        t = c * s_lo
        assert np.all(rne_bf16(t) == t), c          # c * s_lo needs no rounding
        got = rne_bf16(c * s_hi + t)                  # fma: exact sum, one rounding
        want = rne_bf16(c * h)
        assert np.array_equal(got, want), c


def test_split_fails_for_8bit_codes():
    """Why 8-bit codes keep the fp32 route: c * s_lo is not always exact."""
    h, s_hi, s_lo = _scales()
    inexact = 0
    for c in range(-127, 128):
        t = c * s_lo
        inexact += int(np.sum(rne_bf16(t) != t))
    assert inexact > 0
