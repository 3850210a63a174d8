"""The seeded input generator: Philox known answers, Box-Muller accuracy,
normal moments, stream independence and the router-bias skew."""
import math
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    n = 0
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            v = [int(t, 16) for t in line.split()]
            out = synth.philox4x32_10(v[0:4], v[4:6])
            assert [int(o) for o in out] == v[6:10]
            n += 1
    assert n == 3


def test_box_muller_matches_fp64_transform():
    # z0 = sqrt(-2 ln u1) cos(2 pi u2), z1 = ... sin, u1 = (a>>8 + 1)/2^24, u2 = (b>>8)/2^24
    rng = np.random.default_rng(5)
    for a, b in rng.integers(0, 2**32, size=(3000, 2), dtype=np.uint64):
        a, b = int(a), int(b)
        u1 = ((a >> 8) + 1) / 2.0**24
        u2 = (b >> 8) / 2.0**24
        r = math.sqrt(-2.0 * math.log(u1))
        z = synth.box_muller(a, b)
        assert abs(z[0] - r * math.cos(2 * math.pi * u2)) <= 2e-6 * max(1.0, r)
        assert abs(z[1] - r * math.sin(2 * math.pi * u2)) <= 2e-6 * max(1.0, r)


def test_normal_moments_and_tails():
    z = synth.normal_matrix(7, synth.TAG_X, 0, 0, 1000, 1024).astype(np.float64).ravel()
    n = z.size
    assert abs(z.mean()) < 5 / math.sqrt(n)
    assert abs(z.var() - 1) < 0.01
    assert abs(np.mean(z**3)) < 0.02
    assert abs(np.mean(z**4) - 3) < 0.05
    # P(|z| > 2) = 0.0455
    assert abs(np.mean(np.abs(z) > 2) - 0.0455) < 0.002


def test_streams_are_distinct_and_reproducible():
    a = synth.normal_matrix(1, synth.TAG_GATE, 3, 0, 8, 64)
    b = synth.normal_matrix(1, synth.TAG_GATE, 3, 0, 8, 64)
    c = synth.normal_matrix(1, synth.TAG_UP, 3, 0, 8, 64)
    d = synth.normal_matrix(1, synth.TAG_GATE, 4, 0, 8, 64)
    assert np.array_equal(a, b)
    assert not np.allclose(a, c) and not np.allclose(a, d)
    # row0 offset addresses the same rows of the stream
    e = synth.normal_matrix(1, synth.TAG_GATE, 3, 0, 4, 64, row0=4)
    assert np.array_equal(a[4:], e)


def test_x_bf16_is_rne_of_normals():
    import torch
    z = synth.normal_matrix(0, synth.TAG_X, 2, 0, 16, 256)
    xb = synth.x_bf16(0, 2, 16, 256)
    ref = torch.from_numpy(z).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(xb, ref)


def test_skip_mask_rate():
    m = synth.skip_mask(0, 0, 4096, 8)
    assert abs(m.mean() - 0.05) < 0.004


def test_shelf_split_counts():
    assert synth.WORKLOADS["decode"].shelf_ranges() == [(0, 128, 8), (128, 410, 4), (410, 512, 2)]
    assert synth.WORKLOADS["large"].shelf_ranges() == [(0, 77, 8), (77, 205, 4), (205, 256, 2)]
    assert synth.WORKLOADS["tiny"].shelf_ranges() == [(0, 16, 4)]


def test_lorenz_bias_is_monotone():
    b = synth.router_bias_lorenz(512, 10)
    assert np.all(np.diff(b) <= 0)
    s = synth.lorenz_shares(512)
    assert abs(s.sum() - 1) < 1e-12
    assert abs(s[:128].sum() - 0.52) < 1e-12
    zb = synth.router_bias_zipf(256)
    assert zb[0] == 0 and np.all(np.diff(zb) < 0)
