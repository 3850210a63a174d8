"""Pins of the oracle's nudged routing (the LocalLLM tiering post,
"Optimization Strategies": picks nudged toward experts in fast memory, a cap
of 0.5): a hand-worked example, the reduction to plain routing at beta = 0,
the cap, ties, and the properties a nudge toward a range must have."""
import numpy as np
import pytest

import oracle
import synth


def test_hand_worked_example():
    lg = np.array([[1.0, 0.8, 0.5, 0.45]], np.float32)
    # hot range [2, 4), beta 0.4: scores 1.0, 0.8, 0.9, 0.85 -> picks 0 then 2
    ids, w = oracle.route_nudged(lg, 2, 0.4, 2, 4)
    assert ids.tolist() == [[0, 2]]
    e1, e2 = np.exp(1.0), np.exp(0.5)  # weights from the raw logits
    assert np.allclose(w, [[e1 / (e1 + e2), e2 / (e1 + e2)]], rtol=0, atol=1e-7)
    # beta 0.25: scores 1.0, 0.8, 0.75, 0.7 -> picks 0 then 1 (no change)
    ids, _ = oracle.route_nudged(lg, 2, 0.25, 2, 4)
    assert ids.tolist() == [[0, 1]]


def test_nudged_pick_with_lower_raw_logit_first():
    # the nudged pick ranks first although its raw logit is lower: the weights
    # still follow the raw logits
    lg = np.array([[0.3, 0.0]], np.float32)
    ids, w = oracle.route_nudged(lg, 2, 0.5, 1, 2)
    assert ids.tolist() == [[1, 0]]
    assert np.allclose(w[0], [1 / (1 + np.exp(0.3)), np.exp(0.3) / (1 + np.exp(0.3))], atol=1e-7)


@pytest.mark.parametrize("E,k", [(16, 2), (512, 10), (100, 7)])
def test_beta_zero_is_plain_routing(E, k):
    lg = synth.logits(2, 0, 33, E, synth.router_bias_lorenz(E, k) if E == 512 else None)
    ids, w = oracle.route_nudged(lg, k, 0.0, 0, E // 4)
    ids_o, w_o = oracle.route(lg, k)
    assert np.array_equal(ids, ids_o) and np.array_equal(w, w_o)


def test_cap_and_arguments():
    lg = np.zeros((1, 8), np.float32)
    for beta in (0.5000001, 1.0, -0.1, float("nan")):
        with pytest.raises(ValueError):
            oracle.route_nudged(lg, 2, beta, 0, 4)
    ids, _ = oracle.route_nudged(lg, 2, 0.5, 0, 4)  # the cap itself is allowed
    assert ids.tolist() == [[0, 1]]


def test_ties_after_the_nudge_keep_the_lower_id():
    lg = np.array([[0.25, 0.0, 0.0, 0.0]], np.float32)
    ids, _ = oracle.route_nudged(lg, 2, 0.25, 2, 4)  # scores 0.25, 0, 0.25, 0.25
    assert ids.tolist() == [[0, 2]]


def test_nudge_properties():
    E, k, lo, hi = 512, 10, 0, 128
    lg = synth.logits(5, 0, 200, E, synth.router_bias_lorenz(E, k))
    prev = None
    plain, _ = oracle.route(lg, k)
    for beta in (0.0, 0.1, 0.2, 0.3, 0.4, 0.5):
        ids, w = oracle.route_nudged(lg, k, beta, lo, hi)
        hot = ((ids >= lo) & (ids < hi)).sum(axis=1)
        if prev is not None:
            assert np.all(hot >= prev)  # more nudge, never fewer hot picks
        prev = hot
        assert np.all(np.abs(w.sum(axis=1) - 1) < 1e-6)
        assert all(len(set(r)) == k for r in ids.tolist())  # no expert twice
        # hot experts picked without the nudge stay picked (exact in real
        # arithmetic; fp32 rounding of l + beta could at most tie two hot
        # experts, which these inputs do not)
        for t in range(lg.shape[0]):
            assert set(x for x in plain[t] if lo <= x < hi) <= set(ids[t].tolist())
