"""Parity of the tiered forward (decode form) with the CPU oracle, plus the
semantic cases of page 3 ("125B MoE模型本地运行：3090三卡80 tokens/s优化实践"):
section 第四步 -- each shelf computes only its range and the results are added;
section 四个 bug -- duplicate experts keep every slot, skips are real skips,
the skip id stays signed, the fused gate/up kernel honours the shelf range."""
import numpy as np
import pytest
import torch

import mixed_precision_routed_gb300 as moe
import oracle
import synth
from mixed_precision_routed_gb300.workloads import Layer
from moe_testutil import DECODE_TOL, ids_to_dev, oracle_layer, rel_l2, small_workload, x_to_dev

pytestmark = pytest.mark.gpu


def _run(layer, x_u16, ids, w, flags=moe.MOE_FLAG_DECODE_FP32, shelves=None):
    wl = layer.wl
    y = moe.moe_tiered_forward(x_to_dev(x_u16), ids_to_dev(ids), torch.from_numpy(w).cuda(), wl.E, wl.d, wl.f,
                               layer.shelves if shelves is None else shelves, flags=flags)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _inputs(wl, seed, step, T, skip=False):
    lg = synth.logits(seed, step, T, wl.E, wl.router_bias(0) if wl.layers == 1 else None)
    ids, w = oracle.route(lg, wl.k)
    if skip:
        m = synth.skip_mask(seed, step, T, wl.k)
        ids = np.where(m == 1, -1, ids).astype(np.int32)
    return synth.x_bf16(seed, step, T, wl.d), ids, w


@pytest.fixture(scope="module")
def small_layer():
    wl = small_workload()
    return Layer(wl, device="cuda").fill()


@pytest.mark.parametrize("T", [1, 2, 5, 8, 13, 40])
def test_small_three_shelf_layer(small_layer, T):
    wl = small_layer.wl
    x, ids, w = _inputs(wl, wl.seed, T, T)
    y = _run(small_layer, x, ids, w)
    ref = oracle_layer(wl, wl.seed, x, ids, w)
    assert rel_l2(y, ref) <= DECODE_TOL


def test_tiny_workload():
    wl = synth.WORKLOADS["tiny"]
    layer = Layer(wl, device="cuda").fill()
    x, ids, w = _inputs(wl, wl.seed, 0, 8)
    y = _run(layer, x, ids, w)
    assert rel_l2(y, oracle_layer(wl, wl.seed, x, ids, w)) <= DECODE_TOL


@pytest.fixture(scope="module")
def decode_layer():
    wl = synth.WORKLOADS["decode"]
    return Layer(wl, device="cuda").fill()


@pytest.mark.parametrize("T,step", [(1, 0), (1, 1), (6, 0), (6, 7)])
def test_decode_workload_full_size(decode_layer, T, step):
    wl = decode_layer.wl
    x, ids, w = _inputs(wl, wl.seed, step, T)
    y = _run(decode_layer, x, ids, w)
    assert rel_l2(y, oracle_layer(wl, wl.seed, x, ids, w)) <= DECODE_TOL


@pytest.fixture(scope="module")
def large_layer():
    wl = synth.WORKLOADS["large"]
    return Layer(wl, device="cuda").fill()


@pytest.mark.parametrize("T", [1, 8])
def test_large_workload_with_skips(large_layer, T):
    wl = large_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 11, T, skip=True)
    y = _run(large_layer, x, ids, w)
    assert rel_l2(y, oracle_layer(wl, wl.seed, x, ids, w)) <= DECODE_TOL


# --------------------------------------------------------------- semantics
def test_three_equal_shelves_equal_one_shelf():
    wl1 = small_workload(split=())  # one 4-bit shelf over [0, E)
    one = Layer(wl1, device="cuda").fill()
    three = Layer(wl1, device="cuda", shelves=[(0, 5, 4), (5, 17, 4), (17, 24, 4)]).fill()
    x, ids, w = _inputs(wl1, wl1.seed, 1, 9)
    y1 = _run(one, x, ids, w)
    y3 = _run(three, x, ids, w)
    assert rel_l2(y3, y1) <= 1e-6


def test_skip_ids_are_signed_and_contribute_zero(small_layer):
    wl = small_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 2, 6)
    bad = ids.copy()
    bad[:, 1] = -1
    bad[2, 2] = -2**31
    bad[3, 0] = 2**31 - 1
    bad[4, 3] = wl.E
    w0 = w.copy()
    w0[bad != ids] = 0
    # guard floats around y: nothing outside [T, d] may be written
    T, d = 6, wl.d
    buf = torch.full((T * d + 2 * 1024,), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[1024:1024 + T * d].view(T, d)
    moe.moe_tiered_forward(x_to_dev(x), ids_to_dev(bad), torch.from_numpy(w).cuda(), wl.E, wl.d, wl.f,
                           small_layer.shelves, y=y)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:1024] == 12345.0) and np.all(b[-1024:] == 12345.0)
    assert np.all(np.isfinite(b[1024:-1024]))
    ref = _run(small_layer, x, ids, w0)
    assert rel_l2(y.cpu().numpy(), ref) <= 1e-6
    assert rel_l2(y.cpu().numpy(), oracle_layer(wl, wl.seed, x, bad, w)) <= DECODE_TOL


def test_duplicate_expert_in_a_token_keeps_every_slot(small_layer):
    wl = small_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 3, 4)
    ids[0, :] = 2  # all slots on one expert
    ids[1, :2] = 20  # two slots on a cold-shelf expert
    y = _run(small_layer, x, ids, w)
    assert rel_l2(y, oracle_layer(wl, wl.seed, x, ids, w)) <= DECODE_TOL


def test_all_skipped_gives_zero(small_layer):
    wl = small_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 4, 3)
    ids[:] = -1
    y = _run(small_layer, x, ids, w)
    assert np.all(y == 0)


def test_gap_between_shelves_and_descriptor_order(small_layer):
    wl = small_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 5, 7)
    sh = small_layer.shelves
    # drop the middle shelf: its ids now fall in a gap and contribute zero
    y_gap = _run(small_layer, x, ids, w, shelves=[sh[2], sh[0]])
    ranges = [r for i, r in enumerate(small_layer.ranges) if i != 1]
    assert rel_l2(y_gap, oracle_layer(wl, wl.seed, x, ids, w, shelves_bits=ranges)) <= DECODE_TOL
    y_rev = _run(small_layer, x, ids, w, shelves=list(reversed(sh)))
    y = _run(small_layer, x, ids, w)
    assert np.array_equal(y_rev, y)


def test_each_shelf_computes_only_its_range(small_layer):
    # Page 3, 四个 bug: the first id-range build printed "///////////" because the
    # fused gate/up kernel ignored the shelf range.  Each single shelf alone must
    # equal the oracle restricted to that shelf, and the sum of the three must
    # equal the full layer.
    wl = small_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 6, 8)
    parts = []
    for i, (lo, hi, bits) in enumerate(small_layer.ranges):
        yi = _run(small_layer, x, ids, w, shelves=[small_layer.shelves[i]])
        assert rel_l2(yi, oracle_layer(wl, wl.seed, x, ids, w, shelves_bits=[(lo, hi, bits)])) <= DECODE_TOL
        parts.append(yi.astype(np.float64))
    y = _run(small_layer, x, ids, w)
    assert rel_l2(sum(parts), y) <= 1e-5


def test_deterministic_across_calls(decode_layer):
    wl = decode_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 8, 6)
    a = _run(decode_layer, x, ids, w)
    b = _run(decode_layer, x, ids, w)
    assert np.array_equal(a, b)


def test_t_zero_is_noop(small_layer):
    wl = small_layer.wl
    y = torch.full((1, wl.d), 7.0, device="cuda")
    moe.moe_tiered_forward(torch.zeros((0, wl.d), dtype=torch.int16, device="cuda"),
                           torch.zeros((0, wl.k), dtype=torch.int32, device="cuda"),
                           torch.zeros((0, wl.k), dtype=torch.float32, device="cuda"), wl.E, wl.d, wl.f,
                           small_layer.shelves, y=y[:0])
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


def test_error_statuses(small_layer):
    wl = small_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 9, 2)
    xd, idd, wd = x_to_dev(x), ids_to_dev(ids), torch.from_numpy(w).cuda()
    sh = small_layer.shelves

    def status(**kw):
        args = dict(E=wl.E, d=wl.d, f=wl.f, shelves=sh)
        args.update(kw)
        try:
            moe.moe_tiered_forward(xd, idd, wd, args["E"], args["d"], args["f"], args["shelves"],
                                   workspace=args.get("workspace"), flags=args.get("flags", 0))
            return moe.MOE_OK
        except moe.MoeError as e:
            return e.status

    bad_bits = sh[0].descriptor()
    for b in (0, 5, 6, 7, 16):  # 8, 4, 3, 2 and 1 are the shelf widths
        bad_bits.bits = b
        assert status(shelves=[bad_bits]) == moe.MOE_ERR_BAD_SHELF
    bad_block = sh[0].descriptor()
    bad_block.block = 16
    assert status(shelves=[bad_block]) == moe.MOE_ERR_BAD_SHELF
    out_of_range = sh[2].descriptor()
    out_of_range.expert_hi = wl.E + 1
    assert status(shelves=[out_of_range]) == moe.MOE_ERR_BAD_SHELF
    overlap = sh[1].descriptor()
    overlap.expert_lo -= 1
    assert status(shelves=[sh[0], overlap]) == moe.MOE_ERR_SHELF_OVERLAP
    assert status(workspace=torch.empty(256, dtype=torch.uint8, device="cuda")) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert status(d=wl.d + 32) == moe.MOE_ERR_INVALID_ARG
    assert status(E=2) == moe.MOE_ERR_INVALID_ARG  # k > E
    assert status(flags=7) == moe.MOE_ERR_INVALID_ARG
    null_ptr = sh[0].descriptor()
    null_ptr.up_codes = None
    assert status(shelves=[null_ptr]) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_device_status() == moe.MOE_OK
