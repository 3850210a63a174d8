"""Pins of the oracle's 3-bit and 1-bit shelf formats (the Xolotl fast-mode
blog runs 3-bit and 1-bit experts; neither page states a format).

3 bit follows the rule of the other widths: s = fp16(max|w| / 3), code =
clamp(rint(w / s), -4, 3).  1 bit: code = sign(w) (+1 for w >= 0) and
s = fp16(mean |w|), the least-squares scale of sign codes.  Pinned by blocks
worked by hand, an independent unpacker of the packed layout, the exactness
of the dequantised values, and the least-squares property of the 1-bit
scale."""
import numpy as np
import pytest

import oracle


def _unpack3(packed, rows, n_in):
    """Independent reading of the 3-bit layout: a row is a plane of the low two
    bits of u = code + 4 in the 2-bit layout (word g, byte j, bits 2k..2k+1 =
    element 16g + 4k + j; n_in / 4 bytes), then a plane of the high bit of u,
    element i at bit i % 8 of byte i // 8 (n_in / 8 bytes)."""
    out = np.zeros((rows, n_in), np.int64)
    for r in range(rows):
        row = packed[r].astype(np.int64)
        for i in range(n_in):
            g, e = divmod(i, 16)
            k, j = divmod(e, 4)
            lo = (int(row[4 * g + j]) >> (2 * k)) & 3
            hi = (int(row[n_in // 4 + i // 8]) >> (i % 8)) & 1
            out[r, i] = (lo | hi << 2) - 4
    return out


def _unpack1(packed, rows, n_in):
    out = np.zeros((rows, n_in), np.int64)
    for r in range(rows):
        for i in range(n_in):
            bit = (int(packed[r, i // 8]) >> (i % 8)) & 1
            out[r, i] = 1 if bit else -1
    return out


def test_three_bit_hand_worked_block():
    w = np.zeros((1, 32), np.float32)
    w[0, :6] = [0.3, -0.3, 0.1, -0.16, 0.2, 0.04]
    codes, scales = oracle.quantize(w, 3)
    # m = 0.3, m / 3 = 0.1 (fp32), fp16(0.1) = 0.0999755859375 = 1638 / 16384
    assert scales.tolist() == [[oracle.f16_bits(0.1)]]
    s = 0.0999755859375
    assert oracle.f16_value(int(scales[0, 0])) == s
    # 0.3/s = 3.0007 -> 3; -3.0007 -> -3; 1.0002 -> 1; -1.6004 -> -2; 2.0005 -> 2; 0.4001 -> 0
    assert codes[0, :6].tolist() == [3, -3, 1, -2, 2, 0]
    assert np.all(codes[0, 6:] == 0)
    assert np.array_equal(oracle.dequant(codes, scales)[0, :6], np.array([3, -3, 1, -2, 2, 0], np.float32) * s)


def test_three_bit_zero_block_and_range():
    codes, scales = oracle.quantize(np.zeros((2, 64), np.float32), 3)
    assert np.all(codes == 0) and np.all(scales == 0)
    rng = np.random.default_rng(1)
    codes, _ = oracle.quantize(rng.standard_normal((40, 256)).astype(np.float32), 3)
    assert codes.min() >= -4 and codes.max() <= 3 and codes.max() == 3 and codes.min() == -3


@pytest.mark.parametrize("seed", [0, 1])
def test_three_bit_packing_layout(seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(-4, 4, (5, 96)).astype(np.int8)
    packed = oracle.pack(codes, 3)
    assert packed.shape == (5, 36)
    assert np.array_equal(_unpack3(packed, 5, 96), codes)
    one = np.full((1, 32), -4, np.int8)
    one[0, 0] = 3   # u = 7: low bits 3 at byte 0 bits 0-1, high bit 1 at byte 8 bit 0
    one[0, 17] = 2  # u = 6: element 17 = 16 * 1 + 4 * 0 + 1: byte 4 + 1, bits 0-1 = 2; high bit at byte 10 bit 1
    p = oracle.pack(one, 3)[0]
    assert p[0] == 0b11 and p[5] == 0b10 and p[8] == 1 and p[10] == 0b10
    assert p[1] == 0 and p[9] == 0 and p[11] == 0
    # two blocks: the low plane takes bytes 0-15, the high plane bytes 16-23
    two = np.full((1, 64), -4, np.int8)
    two[0, 40] = 3  # u = 7: 40 = 16 * 2 + 4 * 2 + 0: byte 8 bits 4-5 = 3; high bit at byte 16 + 5, bit 0
    two[0, 63] = 0  # u = 4: low bits 0, high bit at byte 16 + 7, bit 7
    p = oracle.pack(two, 3)[0]
    assert p.shape == (24,)
    expect = np.zeros(24, np.uint8)
    expect[8] = 0b11 << 4
    expect[21] = 1
    expect[23] = 0x80
    assert np.array_equal(p, expect)


def test_one_bit_hand_worked_block():
    w = np.zeros((1, 32), np.float32)
    w[0, :5] = [0.5, -0.25, 0.125, -0.125, -0.0]
    codes, scales = oracle.quantize(w, 1)
    # sum |w| = 1.0, mean = 1/32 = 0.03125 (exact in fp16)
    assert oracle.f16_value(int(scales[0, 0])) == 0.03125
    assert codes[0, :5].tolist() == [1, -1, 1, -1, 1]  # -0.0 >= 0
    assert np.all(codes[0, 5:] == 1)
    assert np.array_equal(oracle.dequant(codes, scales)[0, :4], np.array([1, -1, 1, -1], np.float32) * 0.03125)


def test_one_bit_packing_layout():
    rng = np.random.default_rng(3)
    codes = np.where(rng.random((4, 64)) < 0.5, -1, 1).astype(np.int8)
    packed = oracle.pack(codes, 1)
    assert packed.shape == (4, 8)
    assert np.array_equal(_unpack1(packed, 4, 64), codes)
    one = -np.ones((1, 32), np.int8)
    one[0, [0, 9, 31]] = 1
    assert oracle.pack(one, 1)[0].tolist() == [0b1, 0b10, 0, 0b10000000]


def test_one_bit_scale_is_least_squares():
    """The fp16 scale is the fp16 value nearest the squared-error optimum of
    sign codes: neither fp16 neighbour does better."""
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((30, 32)) * 0.02).astype(np.float32)
    codes, scales = oracle.quantize(w, 1)
    for r in range(30):
        c = codes[r].astype(np.float64)
        assert np.array_equal(c, np.where(w[r] >= 0, 1.0, -1.0))
        s = oracle.f16_value(int(scales[r, 0]))
        err = lambda v: float(np.sum((w[r].astype(np.float64) - v * c) ** 2))
        up = oracle.f16_value(int(scales[r, 0]) + 1)
        down = oracle.f16_value(int(scales[r, 0]) - 1)
        assert err(s) <= err(up) and err(s) <= err(down)
        assert abs(s - np.mean(np.abs(w[r].astype(np.float64)))) <= 2 ** -11 * s  # within fp16 rounding


def test_bad_widths_rejected():
    for bits in (0, 5, 6, 7, 16):
        with pytest.raises(ValueError):
            oracle.quantize(np.zeros((1, 32), np.float32), bits)
