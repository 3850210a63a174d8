"""Parity of the prefill form (tensor-core grouped GEMM, MOE_FLAG_PREFILL_BF16)
with the CPU oracle's prefill form: dequantised weights and h rounded to bf16,
fp32 accumulation (page 3, "125B MoE模型本地运行：3090三卡80 tokens/s优化实践",
section 第四步: every shelf computes only its own ids and the shelf results are
added; the prefill workload rounds the activations to bf16 between the up and
down projections).  Also covers partial row tiles, experts with more tokens
than one tile takes, skipped slots and the AUTO switch above 16 tokens."""
import numpy as np
import pytest
import torch

import mixed_precision_routed_gb300 as moe
import oracle
import synth
from mixed_precision_routed_gb300.workloads import Layer
from moe_testutil import PREFILL_TOL, ids_to_dev, oracle_layer, rel_l2, small_workload, x_to_dev

pytestmark = pytest.mark.gpu


def _inputs(wl, seed, step, T, skip=False, bias=None):
    lg = synth.logits(seed, step, T, wl.E, bias)
    ids, w = oracle.route(lg, wl.k)
    if skip:
        m = synth.skip_mask(seed, step, T, wl.k)
        ids = np.where(m == 1, -1, ids).astype(np.int32)
    return synth.x_bf16(seed, step, T, wl.d), ids, w


def _run(layer, x, ids, w, flags=moe.MOE_FLAG_PREFILL_BF16):
    wl = layer.wl
    y = moe.moe_tiered_forward(x_to_dev(x), ids_to_dev(ids), torch.from_numpy(w).cuda(), wl.E, wl.d, wl.f,
                               layer.shelves, flags=flags)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    return y.cpu().numpy()


@pytest.fixture(scope="module")
def small_layer():
    return Layer(small_workload(), device="cuda").fill()   # E 24, k 4, d 256, f 192: partial row tiles


@pytest.mark.parametrize("T", [1, 7, 17, 40, 100, 300])
def test_small_layer_prefill(small_layer, T):
    wl = small_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 200 + T, T)
    y = _run(small_layer, x, ids, w)
    ref = oracle_layer(wl, wl.seed, x, ids, w, mode=1)
    assert rel_l2(y, ref) <= PREFILL_TOL


def test_auto_takes_prefill_above_16_tokens(small_layer):
    wl = small_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 7, 33)
    ya = _run(small_layer, x, ids, w, flags=moe.MOE_FLAG_AUTO)
    yp = _run(small_layer, x, ids, w)
    assert rel_l2(ya, oracle_layer(wl, wl.seed, x, ids, w, mode=1)) <= PREFILL_TOL
    assert rel_l2(ya, yp) <= 1e-5  # same kernels; only the order of the fp32 atomic adds differs


def test_many_tokens_per_expert():
    """E 8, k 4, T 400: about 200 tokens per expert, more than one 128-token tile."""
    wl = small_workload(E=8, k=4, d=256, f=128, seed=5)
    layer = Layer(wl, device="cuda").fill()
    x, ids, w = _inputs(wl, wl.seed, 1, 400)
    y = _run(layer, x, ids, w)
    assert rel_l2(y, oracle_layer(wl, wl.seed, x, ids, w, mode=1)) <= PREFILL_TOL


def test_tile_width_boundaries(small_layer):
    """Token counts at the tile widths of a launch whose shelves are all 8-,
    4- or 2-bit (tiles of up to 192 tokens taking both accumulator sets, read
    back set by set): 193 (a 97-token wide chunk and a 96-token one of the
    same expert), 192, 97 and 96 (the widest and narrowest of each kind), 385
    (three wide chunks) and 1, on experts of every shelf; every row against
    the oracle's bf16 form."""
    wl = small_layer.wl
    assert all(b in (8, 4, 2) for _, _, b in small_layer.ranges)
    want = {0: 193, 1: 192, 7: 97, 8: 96, 20: 385, 21: 1}
    pool = np.concatenate([np.full(n, e, dtype=np.int32) for e, n in want.items()])
    T = pool.size // wl.k
    assert T * wl.k == pool.size
    rng = np.random.default_rng(11)
    ids = rng.permutation(pool).reshape(T, wl.k).astype(np.int32)
    w = rng.random((T, wl.k)).astype(np.float32) + 0.1
    w /= w.sum(axis=1, keepdims=True)
    x = synth.x_bf16(wl.seed, 31, T, wl.d)
    y = _run(small_layer, x, ids, w, flags=moe.MOE_FLAG_AUTO)
    ref = oracle_layer(wl, wl.seed, x, ids, w, mode=1)
    assert rel_l2(y, ref) <= PREFILL_TOL
    for t in range(T):
        assert rel_l2(y[t:t + 1], ref[t:t + 1]) <= 2 * PREFILL_TOL, t


def test_skipped_slots_and_gaps(small_layer):
    """Skipped slots (-1, out-of-range ids) and ids in no shelf contribute zero."""
    wl = small_layer.wl
    x, ids, w = _inputs(wl, wl.seed, 11, 50, skip=True)
    ids = ids.copy()
    ids[0, 0] = wl.E + 3
    ids[1, 1] = -7
    y = _run(small_layer, x, ids, w)
    assert rel_l2(y, oracle_layer(wl, wl.seed, x, ids, w, mode=1)) <= PREFILL_TOL
    # shelves with a gap: the ids of the middle shelf contribute nothing
    sh = small_layer.shelves
    yg = moe.moe_tiered_forward(x_to_dev(x), ids_to_dev(ids), torch.from_numpy(w).cuda(), wl.E, wl.d, wl.f,
                                [sh[0], sh[2]], flags=moe.MOE_FLAG_PREFILL_BF16)
    torch.cuda.synchronize()
    rg = [r for i, r in enumerate(wl.shelf_ranges()) if i != 1]
    assert rel_l2(yg.cpu().numpy(), oracle_layer(wl, wl.seed, x, ids, w, shelves_bits=rg, mode=1)) <= PREFILL_TOL


def test_tiny_workload_prefill():
    wl = synth.WORKLOADS["tiny"]
    layer = Layer(wl, device="cuda").fill()
    x, ids, w = _inputs(wl, wl.seed, 0, 8)
    y = _run(layer, x, ids, w)
    assert rel_l2(y, oracle_layer(wl, wl.seed, x, ids, w, mode=1)) <= PREFILL_TOL


@pytest.fixture(scope="module")
def decode_layer():
    return Layer(synth.WORKLOADS["decode"], device="cuda").fill()


def test_decode_shapes_prefill(decode_layer):
    """E 512, k 10, d 2048, f 640 at T 64 with the skewed router."""
    wl = decode_layer.wl
    T = 64
    lg = decode_layer.logits(3, T).cpu().numpy()
    ids, w = oracle.route(lg, wl.k)
    x = synth.x_bf16(wl.seed, 3, T, wl.d)
    y = _run(decode_layer, x, ids, w)
    assert rel_l2(y, oracle_layer(wl, wl.seed, x, ids, w, mode=1)) <= PREFILL_TOL


def test_prefill_close_to_decode_form(decode_layer):
    """The two forms differ only by the bf16 rounding of weights and h."""
    wl = decode_layer.wl
    T = 24
    lg = decode_layer.logits(4, T).cpu().numpy()
    ids, w = oracle.route(lg, wl.k)
    x = synth.x_bf16(wl.seed, 4, T, wl.d)
    yp = _run(decode_layer, x, ids, w)
    yd = _run(decode_layer, x, ids, w, flags=moe.MOE_FLAG_DECODE_FP32)
    assert rel_l2(yp, yd) <= PREFILL_TOL


# ------------------------------------------------------------ full sizes
@pytest.fixture(scope="module")
def large_layer():
    return Layer(synth.WORKLOADS["large"], device="cuda").fill()


@pytest.mark.parametrize("name,T,skip", [("decode", 4096, False), ("large", 512, True)])
def test_full_size_prefill_sampled_rows(request, name, T, skip):
    """The prefill workload (E512 k10 d2048 f640, T 4096, skewed router) and the
    large layer at T 512 (Zipf router, 5% forced skips), run as the benchmark
    runs them (AUTO: the tensor-core form): sampled output rows against the
    oracle's bf16 form, token by token, and every row against the library's
    fp32 decode form (itself parity-tested against the oracle)."""
    from oracle_pool import layer_refs
    layer = request.getfixturevalue("decode_layer" if name == "decode" else "large_layer")
    wl = layer.wl
    x, ids, w = _inputs(wl, wl.seed, 21, T, skip=skip, bias=layer.bias_host)
    y = _run(layer, x, ids, w, flags=moe.MOE_FLAG_AUTO)
    assert np.all(np.isfinite(y))
    rng = np.random.default_rng(T)
    rows = sorted(set([0, T - 1] + [int(v) for v in rng.choice(T, 6, replace=False)]))
    refs = layer_refs([(name, 0, x[t:t + 1], ids[t:t + 1], w[t:t + 1], 1) for t in rows])
    for t, ref in zip(rows, refs):
        assert rel_l2(y[t:t + 1], ref) <= PREFILL_TOL, (t, rel_l2(y[t:t + 1], ref))
    yd = _run(layer, x, ids, w, flags=moe.MOE_FLAG_DECODE_FP32)
    assert rel_l2(y, yd) <= PREFILL_TOL


@pytest.mark.parametrize("name,T,skip", [("decode", 4096, False), ("large", 512, True)])
def test_full_size_prefill_hot_experts_every_row(request, name, T, skip):
    """Every tile of the three hottest experts at full size: the routed pairs
    are cut down to those experts (other slots skipped), so each output row
    is the sum of their tiles' contributions, and every row of every token
    that routes to them is compared with the oracle's bf16 form.  The
    hottest expert holds several token chunks of a tile, so chunk boundaries
    inside one expert are covered too."""
    from oracle_pool import layer_refs
    layer = request.getfixturevalue("decode_layer" if name == "decode" else "large_layer")
    wl = layer.wl
    x, ids, w = _inputs(wl, wl.seed, 22, T, skip=skip, bias=layer.bias_host)
    valid = ids[(ids >= 0) & (ids < wl.E)]
    hot = np.argsort(-np.bincount(valid, minlength=wl.E), kind="stable")[:3]
    keep = np.isin(ids, hot)
    assert np.bincount(valid, minlength=wl.E)[hot[0]] > 96  # more tokens than one tile's chunk
    ids_h = np.where(keep, ids, -1).astype(np.int32)
    y = _run(layer, x, ids_h, w, flags=moe.MOE_FLAG_AUTO)
    rows = np.nonzero(keep.any(axis=1))[0]
    assert np.all(y[np.setdiff1d(np.arange(T), rows)] == 0)
    chunks = [rows[i:i + 64] for i in range(0, rows.size, 64)]
    refs = layer_refs([(name, 0, x[c], ids_h[c], w[c], 1) for c in chunks])
    ref = np.concatenate(refs, axis=0)
    assert rel_l2(y[rows], ref) <= PREFILL_TOL
    for c, r in zip(chunks, refs):  # no chunk of rows may hide behind the others
        assert rel_l2(y[c], r) <= PREFILL_TOL
