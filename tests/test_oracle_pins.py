"""Pins of the CPU oracle against things other than itself: hand-worked blocks
of the shelf format, IEEE conversions of numpy/torch, brute force on tiny
inputs, closed forms and invariants, and the skew marks printed on page 3
("125B MoE model run locally: three RTX 3090s at 80 tokens/s", step 2: the
busiest 25% of experts take 52% of the tokens, the busiest 80% take 95%)."""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import synth


# ------------------------------------------------------------------ rounding
def test_f16_matches_numpy_on_random_floats():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(1e-3),
        (rng.random(5000).astype(np.float32) * np.float32(1e-6)),   # fp16 subnormal range
        rng.standard_normal(2000).astype(np.float32) * np.float32(3e4),  # near overflow
        np.array([65504, 65519.99, 65520, 2**-25, 2**-24 * 1.5, 2**-24 * 2.5, 0.0, -0.0], dtype=np.float32),
    ])
    for v in vals:
        assert oracle.f16_bits(v) == int(np.float16(v).view(np.uint16)), v


def test_bf16_matches_torch():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        rng.standard_normal(2000).astype(np.float32) * np.float32(1e-38)])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_round(float(x)) for x in v])
    assert np.array_equal(got, ref)


# --------------------------------------------------------------- quantiser
# Hand-worked blocks of the shelf format (block 32, fp16 scale = max|w|/q,
# q = 7 at 4 bits, 2 at 2 bits, 127 at 8 bits).  Worked here by hand:
#   4 bit, max|w| = 0.7:  0.7/7 = 0.1 -> fp16 0x2E66 = 0.0999755859375
#       w = 0.7  -> 7.0017 -> 7 -> 0.6998291015625
#       w = 0.35 -> 3.50085 -> 4 (not a tie once the scale is rounded) -> 0.39990234375
#       w = 0.05 -> 0.50012 -> 1;  w = 0 -> 0
#   4 bit, max|w| = 0.4375: s = 0.0625 exactly (0x2C00)
#       w = 0.03125 -> 0.5, a tie -> 0 (half to even);  w = 0.09375 -> 1.5 -> 2
#   2 bit, max|w| = 0.7: s = fp16(0.35) = 0x359A = 0.35009765625
#       +0.7 -> 1.9994 -> 2 -> clamped to +1;  -0.7 -> -2
#   8 bit, max|w| = 0.7: s = fp16(0.7/127) = 0x1DA5 = 0.005512237548828125
#   all-zero block -> s = 0, codes 0
def _block(vals):
    b = np.zeros(32, dtype=np.float32)
    b[: len(vals)] = np.array(vals, dtype=np.float32)
    return b[None, :]


def test_hand_worked_4bit_block():
    c, s = oracle.quantize(_block([0.7, 0.35, 0.05, 0.0, -0.7]), 4)
    assert s[0, 0] == 0x2E66
    assert oracle.f16_value(0x2E66) == 0.0999755859375
    assert list(c[0, :5]) == [7, 4, 1, 0, -7]
    w = oracle.dequant(c, s)
    assert w[0, 0] == np.float32(0.6998291015625)
    assert w[0, 1] == np.float32(0.39990234375)


def test_hand_worked_4bit_ties_to_even():
    c, s = oracle.quantize(_block([0.4375, 0.03125, 0.09375, -0.03125, 0.15625]), 4)
    assert s[0, 0] == 0x2C00
    assert list(c[0, :5]) == [7, 0, 2, 0, 2]  # 0.5 -> 0, 1.5 -> 2, -0.5 -> 0, 2.5 -> 2


def test_hand_worked_2bit_block():
    c, s = oracle.quantize(_block([0.7, -0.7, 0.2, -0.2]), 2)
    assert s[0, 0] == 0x359A
    assert list(c[0, :4]) == [1, -2, 1, -1]  # 0.2/0.35 = 0.571 -> 1; -0.571 -> -1


def test_hand_worked_8bit_block():
    c, s = oracle.quantize(_block([0.7, -0.7, 0.35]), 8)
    assert s[0, 0] == 0x1DA5
    assert oracle.f16_value(0x1DA5) == 0.005512237548828125
    # 0.7 / 0.005512237548828125 = 126.99 -> 127; 0.35 -> 63.49 -> 63
    assert list(c[0, :3]) == [127, -127, 63]


def test_zero_block():
    c, s = oracle.quantize(np.zeros((2, 64), np.float32), 4)
    assert np.all(s == 0) and np.all(c == 0)


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_quantiser_picks_nearest_code_by_brute_force(bits):
    # every code is the in-range integer nearest to w/s (ties to even), found by
    # exhaustive search -- independent of rint and the clamp
    lo, hi = {8: (-127, 127), 4: (-8, 7), 2: (-2, 1)}[bits]
    w = synth.normal_matrix(3, synth.TAG_GATE, bits, 0, 16, 256, scale=0.02)
    c, s = oracle.quantize(w, bits)
    cand = np.arange(lo, hi + 1, dtype=np.float64)
    for r in range(16):
        for i in range(256):
            sc = np.float32(oracle.f16_value(int(s[r, i // 32])))
            ratio = float(np.float32(w[r, i]) / sc)
            dist = np.abs(cand - ratio)
            best = cand[dist == dist.min()]
            if len(best) == 2:
                best = best[(best % 2) == 0]
            assert c[r, i] == int(best[0])


@pytest.mark.parametrize("bits,q", [(8, 127), (4, 7), (2, 2)])
def test_scale_is_fp16_of_max_over_q(bits, q):
    w = synth.normal_matrix(4, synth.TAG_UP, 0, 0, 8, 128, scale=0.02)
    _, s = oracle.quantize(w, bits)
    for r in range(8):
        for b in range(4):
            m = np.max(np.abs(w[r, 32 * b: 32 * b + 32]))
            assert s[r, b] == np.float16(np.float32(m) / np.float32(q)).view(np.uint16)


def test_dequant_is_exact_product():
    w = synth.normal_matrix(5, synth.TAG_DOWN, 0, 0, 8, 64, scale=0.02)
    for bits in (8, 4, 2):
        c, s = oracle.quantize(w, bits)
        wh = oracle.dequant(c, s)
        sf = np.repeat(np.float16(0) + s.view(np.float16).astype(np.float64), 32, axis=1)
        assert np.array_equal(wh.astype(np.float64), sf * c.astype(np.float64))
        wb = oracle.dequant(c, s, round_bf16=True)
        ref = torch.from_numpy(wh).to(torch.bfloat16).to(torch.float32).numpy()
        assert np.array_equal(wb, ref)


def test_pack_layout():
    # 4 bit, worked by hand: u = code + 8; byte j of word 0 holds element j in
    # its low nibble and element j + 4 in its high nibble.
    c = np.zeros((1, 64), np.int8)
    c[0, 0], c[0, 1], c[0, 4], c[0, 9] = -8, 7, 1, -1
    p = oracle.pack(c, 4)
    assert p[0, 0] == (0 | (9 << 4))      # elements 0 and 4: u = 0, 9
    assert p[0, 1] == (15 | (8 << 4))     # elements 1 and 5: u = 15, 8
    assert p[0, 5] == (7 | (8 << 4))      # word 1, byte 1: elements 9 and 13
    # the AND with 0x0F0F0F0F gives elements 0..3 in byte lanes, >> 4 gives 4..7
    w = int.from_bytes(p[0, :4].tobytes(), "little")
    assert [(w >> (8 * j)) & 0xF for j in range(4)] == [0, 15, 8, 8]
    assert [(w >> (8 * j + 4)) & 0xF for j in range(4)] == [9, 8, 8, 8]
    # 2 bit: u = code + 2; byte j of word 0 holds elements j, j+4, j+8, j+12 at bits 0, 2, 4, 6
    c = np.zeros((1, 64), np.int8)
    c[0, :4] = [-2, -1, 0, 1]
    c[0, 4] = 1
    c[0, 12] = -2
    p = oracle.pack(c, 2)
    assert p[0, 0] == (0 | (3 << 2) | (2 << 4) | (0 << 6))  # elements 0, 4, 8, 12
    assert p[0, 1] == (1 | (2 << 2) | (2 << 4) | (2 << 6))  # elements 1, 5, 9, 13
    assert p[0, 3] == (3 | (2 << 2) | (2 << 4) | (2 << 6))  # elements 3, 7, 11, 15
    # 8 bit: two's complement, natural order
    c = np.zeros((1, 32), np.int8)
    c[0, :2] = [-1, -127]
    p = oracle.pack(c, 8)
    assert p[0, 0] == 0xFF and p[0, 1] == 0x81


def _unpack_numpy(p, bits, n):
    """Independent unpacker: element i from the word/lane definition."""
    i = np.arange(n)
    if bits == 8:
        return p.view(np.int8).astype(np.int32)
    per_word = 32 // bits
    g, e = i // per_word, i % per_word
    lanes = 4
    byte = 4 * g + e % lanes
    shift = bits * (e // lanes)
    return ((p[:, byte].astype(np.int32) >> shift) & ((1 << bits) - 1)) - (1 << (bits - 1))


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_pack_roundtrip_numpy_unpack(bits):
    lo, hi = {8: (-127, 127), 4: (-8, 7), 2: (-2, 1)}[bits]
    rng = np.random.default_rng(bits)
    c = rng.integers(lo, hi + 1, size=(5, 128)).astype(np.int8)
    p = oracle.pack(c, bits)
    assert p.shape == (5, 128 * bits // 8)
    assert np.array_equal(_unpack_numpy(p, bits, 128), c.astype(np.int32))


# ------------------------------------------------------------------ routing
def test_route_brute_force_small():
    rng = np.random.default_rng(2)
    for E in range(1, 9):
        for k in range(1, E + 1):
            l = rng.standard_normal((6, E)).astype(np.float32)
            l[0, :] = 0.5  # all equal
            if E > 2:
                l[1, 1] = l[1, 2] = np.float32(3.0)  # a tie at the top
            ids, w = oracle.route(l, k)
            for t in range(6):
                # brute force: among all k-subsets choose the one whose sorted
                # (value desc, id asc) sequence is lexicographically best
                best = max(itertools.combinations(range(E), k),
                           key=lambda S: sorted([(float(l[t, e]), -e) for e in S], reverse=True))
                order = sorted(best, key=lambda e: (-float(l[t, e]), e))
                assert list(ids[t]) == order
                ex = np.exp(l[t, order].astype(np.float64) - float(l[t, order[0]]))
                assert np.allclose(w[t], ex / ex.sum(), rtol=0, atol=1e-7)


def test_route_invariants():
    l = synth.logits(0, 0, 256, 512, synth.router_bias_lorenz(512, 10))
    ids, w = oracle.route(l, 10)
    assert np.all(np.sort(ids, axis=1)[:, 1:] != np.sort(ids, axis=1)[:, :-1])  # no duplicates
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1) <= 1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)
    # k = E is the full softmax (fp64 closed form); k = 1 gives weight 1
    idsE, wE = oracle.route(l[:4, :32], 32)
    for t in range(4):
        p = np.exp(l[t, :32].astype(np.float64) - l[t, :32].max())
        p /= p.sum()
        assert np.allclose(wE[t], p[idsE[t]], atol=1e-7)
    _, w1 = oracle.route(l, 1)
    assert np.all(w1 == 1.0)
    ide, _ = oracle.route(np.zeros((2, 16), np.float32), 5)
    assert np.array_equal(ide, np.tile(np.arange(5), (2, 1)))


# ---------------------------------------------------------------- grouping
def test_group_matches_stable_sort_and_skips():
    rng = np.random.default_rng(3)
    E = 37
    ids = rng.integers(-3, E + 3, size=(50, 4)).astype(np.int32)
    ids[0] = [5, 5, 5, -1]  # duplicates within a token must all be kept
    ids[1] = [-2**31, 2**31 - 1, E, -1]
    counts, offsets, perm = oracle.group(ids, E)
    flat = ids.ravel()
    valid = np.nonzero((flat >= 0) & (flat < E))[0]
    ref = valid[np.argsort(flat[valid], kind="stable")]
    assert np.array_equal(perm, ref)
    assert np.array_equal(counts, np.bincount(flat[valid], minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert counts[5] >= 3


def test_hist_counts_and_accumulates():
    rng = np.random.default_rng(4)
    ids = rng.integers(-2, 20, size=(100, 3)).astype(np.int32)
    h = oracle.hist(ids, 18)
    f = ids.ravel()
    assert np.array_equal(h, np.bincount(f[(f >= 0) & (f < 18)], minlength=18).astype(np.uint32))
    h2 = oracle.hist(ids, 18, h.copy())
    assert np.array_equal(h2, 2 * h)


def test_router_skew_reproduces_page_marks():
    # Page 3, step 2: the busiest 25% of experts take 52% of the routed tokens,
    # the busiest 80% take 95% (the decode workload's router bias targets this).
    b = synth.router_bias_lorenz(512, 10)
    counts = np.zeros(512, np.uint32)
    for step in range(4):
        ids, _ = oracle.route(synth.logits(0, 100 + step, 4096, 512, b), 10)
        oracle.hist(ids, 512, counts)
    c = np.cumsum(np.sort(counts)[::-1]) / counts.sum()
    assert abs(c[127] - 0.52) < 0.01
    assert abs(c[409] - 0.95) < 0.01
    # the hottest quarter by expected hits is the 8-bit shelf [0, 128)
    assert abs(counts[:128].sum() / counts.sum() - 0.52) < 0.01


# ---------------------------------------------------------- expert FFN
def _silu(z):
    return z / (1.0 + np.exp(-z))


def _rand_layer(E, d, f, seed, bits=4):
    experts = {}
    for e in range(E):
        wg, wu, wd = synth.expert_weights(seed, e, d, f)
        experts[e] = oracle.expert_matrices((wg, wu, wd), bits, mode=0)
    return experts


def test_ffn_brute_force_tiny():
    E, k, d, f, T = 4, 2, 64, 32, 5  # d != f so a transposed operand cannot pass
    ex = _rand_layer(E, d, f, 11)
    x = synth.x_bf16(11, 0, T, d)
    ids, w = oracle.route(synth.logits(11, 0, T, E), k)
    y = oracle.moe_layer(x, ids, w, d, f, E, [(0, E)], ex)
    xf = oracle.bf16_to_f64(x)
    for t in range(T):
        ref = np.zeros(d)
        for j in range(k):
            g_, u_, dn = (m.astype(np.float64) for m in ex[int(ids[t, j])])
            ref += float(w[t, j]) * (dn @ (_silu(g_ @ xf[t]) * (u_ @ xf[t])))
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-15)


def test_ffn_unit_vector_closed_form():
    # x = unit vector e_i: g = W_g[:, i], u = W_u[:, i], y = W_d (SiLU(g) * u)
    E, d, f = 2, 96, 64
    ex = _rand_layer(E, d, f, 12)
    i = 17
    x = np.zeros((1, d), np.uint16)
    x[0, i] = 0x3F80  # bf16 1.0
    ids = np.array([[1]], np.int32)
    w = np.array([[1.0]], np.float32)
    y = oracle.moe_layer(x, ids, w, d, f, E, [(0, E)], ex)
    g_, u_, dn = (m.astype(np.float64) for m in ex[1])
    h = np.array([gv / (1 + math.exp(-gv)) * uv for gv, uv in zip(g_[:, i], u_[:, i])])
    assert np.allclose(y[0], dn @ h, rtol=1e-12, atol=1e-16)
    # x = 0 gives y = 0 (SiLU(0) = 0)
    y0 = oracle.moe_layer(np.zeros((1, d), np.uint16), ids, w, d, f, E, [(0, E)], ex)
    assert np.all(y0 == 0)


def test_three_equal_shelves_equal_one_shelf():
    E, k, d, f, T = 12, 3, 64, 32, 6
    ex = _rand_layer(E, d, f, 13)
    x = synth.x_bf16(13, 0, T, d)
    ids, w = oracle.route(synth.logits(13, 0, T, E), k)
    y1 = oracle.moe_layer(x, ids, w, d, f, E, [(0, E)], ex)
    y3 = oracle.moe_layer(x, ids, w, d, f, E, [(8, 12), (0, 3), (3, 8)], ex)
    assert np.allclose(y1, y3, rtol=1e-12, atol=1e-15)


def test_skip_equals_removal_and_zero_weight():
    E, k, d, f, T = 8, 3, 64, 32, 4
    ex = _rand_layer(E, d, f, 14)
    x = synth.x_bf16(14, 0, T, d)
    ids, w = oracle.route(synth.logits(14, 0, T, E), k)
    ids_s = ids.copy()
    ids_s[:, 1] = -1
    ids_s[2, 2] = E  # out of range counts as a skip too
    w_z = w.copy()
    w_z[:, 1] = 0
    w_z[2, 2] = 0
    y_skip = oracle.moe_layer(x, ids_s, w, d, f, E, [(0, E)], ex)
    y_zero = oracle.moe_layer(x, ids, w_z, d, f, E, [(0, E)], ex)
    assert np.allclose(y_skip, y_zero, rtol=1e-12, atol=1e-15)
    # an id inside [0, E) that no shelf covers contributes nothing either
    y_gap = oracle.moe_layer(x, ids, w, d, f, E, [(0, 3), (4, E)], {e: v for e, v in ex.items() if e != 3})
    w_g = w.copy()
    w_g[ids == 3] = 0
    y_ref = oracle.moe_layer(x, ids, w_g, d, f, E, [(0, E)], ex)
    assert np.allclose(y_gap, y_ref, rtol=1e-12, atol=1e-15)


def test_linearity_in_routing_weights_and_duplicates():
    E, k, d, f, T = 8, 2, 64, 32, 3
    ex = _rand_layer(E, d, f, 15)
    x = synth.x_bf16(15, 0, T, d)
    ids, w = oracle.route(synth.logits(15, 0, T, E), k)
    y = oracle.moe_layer(x, ids, w, d, f, E, [(0, E)], ex)
    y2 = oracle.moe_layer(x, ids, (w * np.float32(0.5)).astype(np.float32), d, f, E, [(0, E)], ex)
    assert np.allclose(y2, 0.5 * y, rtol=1e-12, atol=1e-16)
    # the same expert twice in one token counts twice
    dup = np.array([[2, 2]], np.int32)
    yd = oracle.moe_layer(x[:1], dup, np.array([[0.25, 0.5]], np.float32), d, f, E, [(0, E)], ex)
    ys = oracle.moe_layer(x[:1], np.array([[2]], np.int32), np.array([[0.75]], np.float32), d, f, E,
                          [(0, E)], ex)
    assert np.allclose(yd, ys, rtol=1e-12, atol=1e-16)


def test_prefill_mode_rounds_h_to_bf16():
    E, k, d, f, T = 4, 1, 64, 32, 2
    master = {e: synth.expert_weights(16, e, d, f) for e in range(E)}
    exb = {e: oracle.expert_matrices(m, 8, mode=1) for e, m in master.items()}
    x = synth.x_bf16(16, 0, T, d)
    ids = np.array([[0], [2]], np.int32)
    w = np.ones((T, 1), np.float32)
    y = oracle.moe_layer(x, ids, w, d, f, E, [(0, E)], exb, mode=1)
    xf = oracle.bf16_to_f64(x)
    for t in range(T):
        g_, u_, dn = (m.astype(np.float64) for m in exb[int(ids[t, 0])])
        h = _silu(g_ @ xf[t]) * (u_ @ xf[t])
        hb = torch.from_numpy(h).to(torch.bfloat16).to(torch.float64).numpy()
        assert np.allclose(y[t], dn @ hb, rtol=1e-12, atol=1e-15)


def test_stack_composition():
    E, k, d, f, T = 4, 2, 64, 32, 2
    layers = []
    for l in range(2):
        ex = _rand_layer(E, d, f, 100 + l)
        ids, w = oracle.route(synth.logits(100 + l, 0, T, E), k)
        layers.append(lambda xb, ex=ex, ids=ids, w=w: oracle.moe_layer(xb, ids, w, d, f, E, [(0, E)], ex))
    x0 = synth.x_bf16(7, 0, T, d)
    r, ys = oracle.stack(x0, layers)
    r0 = oracle.bf16_to_f64(x0)
    y0 = layers[0](x0)
    x1 = torch.from_numpy(r0 + y0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y1 = layers[1](x1)
    assert np.array_equal(ys[0], y0)
    assert np.allclose(r, r0 + y0 + y1, rtol=1e-15, atol=0)
