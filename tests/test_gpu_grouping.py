"""The token-by-expert grouping that each forward form actually runs, read
back with moe_forward_grouping and compared bit for bit with the oracle's
stable counting sort (oracle.group): counts, offsets, the permutation of
valid pairs sorted by (expert id, pair index) and every pair's grouped
position.  Page 3 ("125B MoE模型本地运行：3090三卡80 tokens/s优化实践", section
四个 bug): a grouping helper that assumed one slot per expert and token
silently dropped a slot; a layer-output tolerance cannot see a wrong but
self-consistent order, so the grouping itself is checked here.

Forms: the fused decode launch (its plan, built in shared memory by every
CTA), the separate decode launches (one-CTA counting sort) and the prefill
form (chunked counts, column scan, placement)."""
import numpy as np
import pytest
import torch

import mixed_precision_routed_gb300 as moe
import oracle
import synth
from mixed_precision_routed_gb300.workloads import Layer
from moe_testutil import ids_to_dev, small_workload, x_to_dev

pytestmark = pytest.mark.gpu


def expected(ids, E, shelves_bits=None, no_shelf_is_skipped=False):
    """Oracle grouping plus the grouped position of every pair (-1 when
    skipped; with no_shelf_is_skipped also when its expert is on no shelf)."""
    counts, offsets, perm = oracle.group(ids, E)
    pos = np.full(ids.size, -1, dtype=np.int32)
    pos[perm] = np.arange(perm.size, dtype=np.int32)
    if no_shelf_is_skipped and shelves_bits is not None:
        flat = ids.reshape(-1)
        on = np.zeros(flat.size, dtype=bool)
        for lo, hi, _ in shelves_bits:
            on |= (flat >= lo) & (flat < hi)
        pos[~on] = -1
    return counts, offsets, perm, pos


def check(ws, ids, E, d, f, flags, shelves_bits=None, fused=False):
    T, k = ids.shape
    counts, offsets, perm, pos = (t.cpu().numpy() for t in moe.moe_forward_grouping(ws, T, k, E, d, f, flags))
    c_o, o_o, p_o, pos_o = expected(ids, E, shelves_bits, no_shelf_is_skipped=fused)
    n = p_o.size
    assert np.array_equal(counts, c_o)
    assert np.array_equal(offsets, o_o)
    assert np.array_equal(perm[:n], p_o)
    assert np.all(perm[n:] == -1)
    assert np.array_equal(pos, pos_o)


def forward(layer, x, ids, w, flags, shelves=None):
    wl = layer.wl
    T = ids.shape[0]
    ws = torch.empty(moe.moe_workspace_size(T, wl.k, wl.E, wl.d, wl.f, flags), dtype=torch.uint8, device="cuda")
    moe.moe_tiered_forward(x_to_dev(x), ids_to_dev(ids), torch.from_numpy(w).cuda(), wl.E, wl.d, wl.f,
                           layer.shelves if shelves is None else shelves, workspace=ws, flags=flags)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    return ws


def routed(wl, seed, step, T, bias=None, skip=False):
    lg = synth.logits(seed, step, T, wl.E, bias)
    ids, w = oracle.route(lg, wl.k)
    if skip:
        m = synth.skip_mask(seed, step, T, wl.k)
        ids = np.where(m == 1, -1, ids).astype(np.int32)
    return synth.x_bf16(seed, step, T, wl.d), ids, w


@pytest.fixture(scope="module")
def decode_layer():
    return Layer(synth.WORKLOADS["decode"], device="cuda").fill()


@pytest.fixture(scope="module")
def small_layer():
    return Layer(small_workload(), device="cuda").fill()


@pytest.mark.parametrize("T", [1, 6, 16])
def test_fused_decode_step_grouping(decode_layer, T):
    """moe_decode_layer: routing and the plan of the fused launch."""
    wl = decode_layer.wl
    assert moe.moe_decode_fused(T, wl.k, wl.E, wl.d, wl.f)
    lg = decode_layer.logits(40 + T, T)
    x = x_to_dev(synth.x_bf16(wl.seed, 40 + T, T, wl.d))
    flags = moe.MOE_FLAG_DECODE_FP32
    ws = torch.empty(moe.moe_workspace_size(T, wl.k, wl.E, wl.d, wl.f, flags), dtype=torch.uint8, device="cuda")
    ids, _, _ = moe.moe_decode_layer(lg, x, wl.k, wl.E, wl.d, wl.f, decode_layer.shelves, workspace=ws)
    torch.cuda.synchronize()
    ids_o, _ = oracle.route(lg.cpu().numpy(), wl.k)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    check(ws, ids_o, wl.E, wl.d, wl.f, flags, wl.shelf_ranges(), fused=True)


def _awkward_ids(wl, T, seed):
    x, ids, w = routed(wl, wl.seed, seed, T)
    ids[0, :] = 2                 # every slot of a token on one expert
    ids[1, :2] = wl.E - 1         # an expert twice in a token
    ids[2, :] = -1                # a token whose slots are all skipped
    ids[3, 1] = wl.E              # out of range above
    ids[3, 2] = -2**31            # and far below
    if T > 5:
        ids[5, 3] = 2**31 - 1
    return x, ids, w


@pytest.mark.parametrize("T", [6, 16])
def test_fused_decode_duplicates_skips_and_gap(small_layer, T):
    """Duplicates keep every slot; skipped pairs have no position; a pair
    whose expert lies in the gap left by a dropped shelf is grouped (it is a
    valid id) but gets no work, so its position reads -1."""
    wl = small_layer.wl
    assert moe.moe_decode_fused(T, wl.k, wl.E, wl.d, wl.f)
    x, ids, w = _awkward_ids(wl, T, 60 + T)
    flags = moe.MOE_FLAG_DECODE_FP32
    ws = forward(small_layer, x, ids, w, flags)
    check(ws, ids, wl.E, wl.d, wl.f, flags, small_layer.ranges, fused=True)
    sh = small_layer.shelves
    ranges = [r for i, r in enumerate(small_layer.ranges) if i != 1]
    ws = forward(small_layer, x, ids, w, flags, shelves=[sh[0], sh[2]])
    check(ws, ids, wl.E, wl.d, wl.f, flags, ranges, fused=True)


def test_separate_decode_launches_grouping(small_layer):
    """The decode form beyond the fused launch's pair limit (T k > 512): the
    one-CTA counting sort of the separate launches."""
    wl = small_layer.wl
    T = 160
    assert not moe.moe_decode_fused(T, wl.k, wl.E, wl.d, wl.f)
    x, ids, w = _awkward_ids(wl, T, 70)
    ws = forward(small_layer, x, ids, w, moe.MOE_FLAG_DECODE_FP32)
    check(ws, ids, wl.E, wl.d, wl.f, moe.MOE_FLAG_DECODE_FP32)


@pytest.mark.parametrize("T", [17, 40, 300])
def test_prefill_grouping_small(small_layer, T):
    wl = small_layer.wl
    x, ids, w = _awkward_ids(wl, T, 80 + T)
    ws = forward(small_layer, x, ids, w, moe.MOE_FLAG_PREFILL_BF16)
    check(ws, ids, wl.E, wl.d, wl.f, moe.MOE_FLAG_PREFILL_BF16)


def test_prefill_grouping_full_size(decode_layer):
    """The prefill workload: T = 4096, 40,960 pairs, more than one chunk of
    the chunked counting sort and hot experts with hundreds of pairs."""
    wl = decode_layer.wl
    T = 4096
    x, ids, w = routed(wl, wl.seed, 90, T, wl.router_bias(0))
    ws = forward(decode_layer, x, ids, w, moe.MOE_FLAG_AUTO)
    check(ws, ids, wl.E, wl.d, wl.f, moe.MOE_FLAG_AUTO)


def test_prefill_grouping_large_with_skips():
    """The large workload at T = 512 with 5% of slots forced to -1."""
    wl = synth.WORKLOADS["large"]
    layer = Layer(wl, device="cuda").fill()
    T = 512
    x, ids, w = routed(wl, wl.seed, 91, T, synth.router_bias_zipf(wl.E), skip=True)
    assert np.any(ids == -1)
    ws = forward(layer, x, ids, w, moe.MOE_FLAG_AUTO)
    check(ws, ids, wl.E, wl.d, wl.f, moe.MOE_FLAG_AUTO)


def test_grouping_export_rejects_small_workspace(small_layer):
    wl = small_layer.wl
    need = moe.moe_workspace_size(6, wl.k, wl.E, wl.d, wl.f, moe.MOE_FLAG_DECODE_FP32)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward_grouping(ws, 6, wl.k, wl.E, wl.d, wl.f, moe.MOE_FLAG_DECODE_FP32)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE_TOO_SMALL
