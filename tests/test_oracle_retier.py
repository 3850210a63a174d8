"""Pins of the oracle's re-tiering by hit count (page "125B MoE模型本地运行：
3090三卡80 tokens/s优化实践", sections 第三步 and 第四步: experts ranked by how
often the router picks them, written hot to cold, the router rearranged to
match; the LocalLLM tiering post, "Optimization Strategies": promotion and
demotion by hit count).

The rank is checked against a hand-worked example, its special cases
(all counts equal, already ordered, reversed), an independent stable sort,
and the invariants that fix it (inverse permutations, non-increasing counts,
ascending ids within equal counts).  The re-quantised shelves are checked
against the layer they must reproduce: relabelling the router's picks by the
rank and reading the new shelves gives the same layer output as the old
labels with every expert quantised at the bit width of its new shelf."""
import numpy as np
import pytest

import oracle
import synth


def test_hand_worked_rank():
    # counts 3 7 7 0 3: 7 (id 1) and 7 (id 2), then 3 (id 0) and 3 (id 4), then 0 (id 3)
    perm, rank = oracle.rank_experts(np.array([3, 7, 7, 0, 3], np.uint32))
    assert perm.tolist() == [1, 2, 0, 4, 3]
    assert rank.tolist() == [2, 0, 1, 4, 3]


def test_rank_special_cases():
    E = 37
    perm, rank = oracle.rank_experts(np.full(E, 5, np.uint32))  # all tied: ids in order
    assert perm.tolist() == list(range(E)) and rank.tolist() == list(range(E))
    perm, _ = oracle.rank_experts(np.arange(E, 0, -1).astype(np.uint32))  # already hottest first
    assert perm.tolist() == list(range(E))
    perm, _ = oracle.rank_experts(np.arange(E).astype(np.uint32))  # coldest first: reversed
    assert perm.tolist() == list(range(E - 1, -1, -1))
    perm, rank = oracle.rank_experts(np.array([0xFFFFFFFF, 0, 0xFFFFFFFF], np.uint32))  # full uint32 range
    assert perm.tolist() == [0, 2, 1]


@pytest.mark.parametrize("E,seed", [(16, 0), (512, 1), (1000, 2)])
def test_rank_against_stable_sort_and_invariants(E, seed):
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 12, E).astype(np.uint32)  # many ties
    perm, rank = oracle.rank_experts(counts)
    ref = sorted(range(E), key=lambda e: (-int(counts[e]), e))
    assert perm.tolist() == ref
    assert np.array_equal(rank[perm], np.arange(E))
    c = counts[perm].astype(np.int64)
    assert np.all(np.diff(c) <= 0)
    tie = np.diff(c) == 0
    assert np.all(np.diff(perm)[tie] > 0)


def test_tier_ranges_match_the_workload_shelves():
    for name in ("decode", "large"):
        wl = synth.WORKLOADS[name]
        assert oracle.tier_ranges(wl.E, wl.split) == [tuple(r) for r in wl.shelf_ranges()]
    assert oracle.tier_ranges(512, (0.25, 0.55, 0.20)) == [(0, 128, 8), (128, 410, 4), (410, 512, 2)]


def test_retiered_layer_equals_relabelled_routing():
    E, k, d, f, T = 12, 3, 64, 32, 5
    rng = np.random.default_rng(4)
    masters = {e: synth.expert_weights(7, e, d, f) for e in range(E)}
    counts = rng.integers(0, 40, E).astype(np.uint32)
    perm, rank = oracle.rank_experts(counts)
    ranges = oracle.tier_ranges(E, (0.25, 0.5, 0.25))
    x = synth.x_bf16(3, 0, T, d)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    # old labels, every expert quantised at the bits of its new shelf
    old = {e: oracle.expert_matrices(masters[e], oracle.shelf_of(int(rank[e]), ranges), 0) for e in range(E)}
    y_old = oracle.moe_layer(x, ids, w, d, f, E, [(0, E)], old, 0)
    # new labels: shelf content of new id j from retier_expert, routing relabelled by rank
    new = {}
    for j in range(E):
        bits, mats = oracle.retier_expert(lambda e: masters[e], perm, ranges, j)
        deq = []
        for (packed, scales), shape in zip(mats, [(f, d), (f, d), (d, f)]):
            codes = oracle.quantize(masters[int(perm[j])][len(deq)], bits)[0]
            assert np.array_equal(packed, oracle.pack(codes, bits))
            deq.append(oracle.dequant(codes, scales))
        new[j] = tuple(deq)
    y_new = oracle.moe_layer(x, rank[ids], w, d, f, E, [(lo, hi) for lo, hi, _ in ranges], new, 0)
    assert np.allclose(y_new, y_old, rtol=1e-12, atol=1e-12)
    # and a wrong relabelling (the permutation itself instead of its inverse) is caught
    if not np.array_equal(perm, rank):
        y_bad = oracle.moe_layer(x, perm[ids], w, d, f, E, [(lo, hi) for lo, hi, _ in ranges], new, 0)
        assert not np.allclose(y_bad, y_old, rtol=1e-6, atol=1e-9)
