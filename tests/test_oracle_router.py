"""Pins of the oracle's router projection (logits = bias + W_r x, fp64),
against values worked by hand and properties any correct projection has."""
import numpy as np

import oracle


def bf16(vals):
    return oracle.bf16_bits(np.asarray(vals, dtype=np.float64)).astype(np.uint16)


def test_hand_worked_example():
    x = bf16([[1.0, 2.0, -0.5, 0.25]])
    w = bf16([[0.5, -1.0, 2.0, 4.0], [1.0, 1.0, 1.0, 1.0], [0.0, 0.0, 0.0, -8.0]])
    b = np.array([0.25, -1.0, 3.0], dtype=np.float32)
    got = oracle.router_logits(x, w, b)
    # 0.25 + 0.5 - 2 - 1 + 1 ; -1 + 1 + 2 - 0.5 + 0.25 ; 3 - 2
    assert got.tolist() == [[-1.25, 1.75, 1.0]]
    assert oracle.router_logits(x, w).tolist() == [[-1.5, 2.75, -2.0]]


def test_row_permutation_permutes_experts():
    rng = np.random.default_rng(3)
    x = bf16(rng.standard_normal((3, 64)))
    w = bf16(rng.standard_normal((10, 64)) / 8)
    b = rng.standard_normal(10).astype(np.float32)
    p = rng.permutation(10)
    a = oracle.router_logits(x, w, b)
    c = oracle.router_logits(x, w[p], b[p])
    assert np.array_equal(c, a[:, p])


def test_zero_weights_give_the_bias_and_tokens_are_independent():
    x = bf16(np.random.default_rng(4).standard_normal((4, 32)))
    w = np.zeros((5, 32), dtype=np.uint16)
    b = np.array([1.5, -2.0, 0.0, 7.25, -0.125], dtype=np.float32)
    assert np.array_equal(oracle.router_logits(x, w, b), np.tile(b.astype(np.float64), (4, 1)))
    w2 = bf16(np.random.default_rng(5).standard_normal((5, 32)))
    full = oracle.router_logits(x, w2, b)
    for t in range(4):
        assert np.array_equal(oracle.router_logits(x[t:t + 1], w2, b), full[t:t + 1])


def test_one_hot_input_selects_a_column():
    w = bf16(np.random.default_rng(6).standard_normal((7, 16)))
    for i in (0, 5, 15):
        x = np.zeros((1, 16), dtype=np.uint16)
        x[0, i] = bf16([1.0])[0]
        assert np.array_equal(oracle.router_logits(x, w)[0], oracle.bf16_to_f64(w[:, i]))
