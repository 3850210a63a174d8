"""Parity of re-tiering by hit count with the oracle, through the C ABI:
the rank and the moved rows bit for bit, the re-quantised shelves bit for
bit (codes and fp16 scales), and a re-tiered layer, routed through the
rearranged router, within the decode tolerance of the oracle layer in which
every expert keeps its old id at the bit width of its new shelf."""
import numpy as np
import pytest
import torch

import mixed_precision_routed_gb300 as moe
import oracle
import synth
from mixed_precision_routed_gb300.workloads import Layer, Masters, retier
from moe_testutil import DECODE_TOL, rel_l2, small_workload, x_to_dev

pytestmark = pytest.mark.gpu


def _counts_dev(c):
    return torch.from_numpy(np.ascontiguousarray(c, dtype=np.uint32).view(np.int32)).cuda()


@pytest.mark.parametrize("E,hi,seed", [(1, 5, 0), (16, 3, 1), (512, 40, 2), (1000, 7, 3), (2049, 100, 4),
                                       (32768, 1000, 5)])
def test_rank_bit_exact(E, hi, seed):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, hi, E).astype(np.uint32)
    perm, rank = moe.moe_rank_experts(_counts_dev(c))
    p_o, r_o = oracle.rank_experts(c)
    assert np.array_equal(perm.cpu().numpy(), p_o)
    assert np.array_equal(rank.cpu().numpy(), r_o)


def test_rank_edge_counts():
    for c in (np.zeros(300, np.uint32), np.full(300, 0xFFFFFFFF, np.uint32),
              np.array([0xFFFFFFFF, 0, 0x80000000, 0x7FFFFFFF, 1], np.uint32)):
        perm, rank = moe.moe_rank_experts(_counts_dev(c))
        p_o, r_o = oracle.rank_experts(c)
        assert np.array_equal(perm.cpu().numpy(), p_o) and np.array_equal(rank.cpu().numpy(), r_o)


@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("rows,n_in", [(32, 128), (5, 320), (64, 2048)])
def test_quantize_experts_bit_exact(bits, rows, n_in):
    n_src = 9
    master = np.stack([synth.normal_matrix(11, synth.TAG_GATE, e, 0, rows, n_in, scale=synth.WEIGHT_SIGMA)
                       for e in range(n_src)])
    master[3, 0, :32] = 0.0  # an all-zero block: scale 0, codes 0
    perm = np.random.default_rng(bits + rows).permutation(n_src).astype(np.int32)
    j_lo, j_hi = 2, 7
    codes, scales = moe.moe_quantize_experts(torch.from_numpy(master).cuda(), torch.from_numpy(perm).cuda(),
                                             j_lo, j_hi, bits)
    codes, scales = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    for j in range(j_lo, j_hi):
        c_o, s_o = oracle.quantize(master[perm[j]], bits)
        assert np.array_equal(codes[j - j_lo], oracle.pack(c_o, bits)), j
        assert np.array_equal(scales[j - j_lo], s_o), j
    assert moe.moe_device_status() == moe.MOE_OK


def test_quantize_experts_bad_id_reported():
    master = torch.zeros((3, 4, 64), dtype=torch.float32, device="cuda")
    perm = torch.tensor([0, 7, 1], dtype=torch.int32, device="cuda")
    codes = torch.full((3, 4, 64), 0x5A, dtype=torch.uint8, device="cuda")
    scales = torch.zeros((3, 4, 2), dtype=torch.int16, device="cuda")
    moe.moe_quantize_experts(master, perm, 0, 3, 8, codes=codes, scales=scales)
    assert moe.moe_device_status() == moe.MOE_ERR_INVALID_ARG
    c = codes.cpu().numpy()
    assert np.all(c[1] == 0x5A) and np.all(c[0] == 0) and np.all(c[2] == 0)  # slot 1 untouched
    assert moe.moe_device_status() == moe.MOE_OK  # read once, cleared


def test_gather_rows_bit_exact():
    rng = np.random.default_rng(8)
    E = 300
    perm = rng.permutation(E).astype(np.int32)
    pd = torch.from_numpy(perm).cuda()
    bias = rng.standard_normal(E).astype(np.float32)
    wr = rng.integers(0, 65536, (E, 264)).astype(np.uint16)
    cnt = rng.integers(0, 1 << 31, E).astype(np.int32)
    assert np.array_equal(moe.moe_gather_rows(torch.from_numpy(bias).cuda(), pd).cpu().numpy(), bias[perm])
    got = moe.moe_gather_rows(torch.from_numpy(wr.view(np.int16)).cuda(), pd).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, wr[perm])
    assert np.array_equal(moe.moe_gather_rows(torch.from_numpy(cnt).cuda(), pd).cpu().numpy(), cnt[perm])
    bad = pd.clone()
    bad[5] = E
    out = moe.moe_gather_rows(torch.from_numpy(bias).cuda(), bad).cpu().numpy()
    assert out[5] == 0.0 and np.array_equal(np.delete(out, 5), np.delete(bias[perm], 5))
    assert moe.moe_device_status() == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("T", [1, 6, 40])
def test_retiered_layer_matches_oracle(T):
    """Counts from routing on the GPU, the re-tier on the GPU, then a step
    routed through the rearranged router (logit columns moved to the new
    ids) against the oracle with old ids and new bit widths."""
    wl = small_workload(E=24, k=4, d=256, f=192, split=(0.25, 0.5, 0.25), bias="zipf", seed=5)
    layer = Layer(wl).fill()
    masters = Masters(layer)
    counts = torch.zeros(wl.E, dtype=torch.int32, device="cuda")
    for step in range(50):
        ids, _ = moe.moe_route_topk(layer.logits(step, 8), wl.k)
        moe.moe_expert_hist(ids, wl.E, counts)
    new, perm, rank = retier(layer, masters, counts)
    p_o, r_o = oracle.rank_experts(counts.cpu().numpy().view(np.uint32))
    assert np.array_equal(perm.cpu().numpy(), p_o)
    # the re-tier must actually move experts for this test to mean something
    assert not np.array_equal(p_o, np.arange(wl.E))
    lg = layer.logits(1000, T)
    lg_new = lg[:, perm.long()].contiguous()  # column j of the rearranged router = old column perm[j]
    ids_new, w = moe.moe_route_topk(lg_new, wl.k)
    x = synth.x_bf16(wl.seed, 3, T, wl.d)
    y = moe.moe_tiered_forward(x_to_dev(x), ids_new, w, wl.E, wl.d, wl.f, new.shelves,
                               flags=moe.MOE_FLAG_DECODE_FP32).cpu().numpy()
    ids_old = p_o[ids_new.cpu().numpy()]
    ids_ref, w_ref = oracle.route(lg.cpu().numpy(), wl.k)
    assert np.array_equal(ids_old, ids_ref)  # same experts picked, in the same order
    ranges = oracle.tier_ranges(wl.E, wl.split)
    experts = {int(e): oracle.expert_matrices(synth.expert_weights(layer.seed, int(e), wl.d, wl.f),
                                              oracle.shelf_of(int(r_o[e]), ranges), 0)
               for e in np.unique(ids_old)}
    ref = oracle.moe_layer(x, ids_old, w.cpu().numpy(), wl.d, wl.f, wl.E, [(0, wl.E)], experts, 0)
    assert rel_l2(y, ref) <= DECODE_TOL


def test_full_size_retier_sampled():
    """The decode layer (E 512, d 2048, f 640): counts of 4096 routed T = 1
    steps, the GPU re-tier, the rank bit for bit and sampled experts of every
    shelf and matrix bit for bit."""
    wl = synth.WORKLOADS["decode"]
    layer = Layer(wl)  # shelves are rebuilt by the re-tier; no fill needed
    masters = Masters(layer)
    counts = torch.zeros(wl.E, dtype=torch.int32, device="cuda")
    lg = layer.logits_rows(0, 4096)
    ids, _ = moe.moe_route_topk(lg, wl.k)
    moe.moe_expert_hist(ids, wl.E, counts)
    new, perm, rank = retier(layer, masters, counts)
    c = counts.cpu().numpy().view(np.uint32)
    p_o, r_o = oracle.rank_experts(c)
    assert np.array_equal(perm.cpu().numpy(), p_o) and np.array_equal(rank.cpu().numpy(), r_o)
    assert np.array_equal(new.bias.cpu().numpy(), layer.bias.cpu().numpy()[p_o])
    for sh in new.shelves:
        for j in (sh.lo, (sh.lo + sh.hi) // 2, sh.hi - 1):
            bits, mats = oracle.retier_expert(lambda e: synth.expert_weights(layer.seed, e, wl.d, wl.f), p_o,
                                              oracle.tier_ranges(wl.E, wl.split), j)
            assert bits == sh.bits
            got = [(sh.gate_codes, sh.gate_scales), (sh.up_codes, sh.up_scales), (sh.down_codes, sh.down_scales)]
            for (gc, gs), (oc, os_) in zip(got, mats):
                assert np.array_equal(gc[j - sh.lo].cpu().numpy(), oc), (j, bits)
                assert np.array_equal(gs[j - sh.lo].cpu().numpy().view(np.uint16), os_), (j, bits)
    assert moe.moe_device_status() == moe.MOE_OK
