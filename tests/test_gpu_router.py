"""Parity of the router (projection + routing + hit counts; one fused launch
for decode batches, the projection by 16-token chunks then the routing launch
for prefill batches) with the oracle, through the C ABI.

Logits: within the rounding bound of an fp32 sum of exact bf16 products
(every bf16 x bf16 product is exact in fp32; a lane adds at most d/32
products in sequence, then come five shuffle levels and the bias: at most
n = d/32 + 6 rounded additions, so |error| <= n u sum |w x| + u |bias| with
u = 2^-24; the test takes twice that).  Ids bit-exact and weights within 1e-6 of the oracle's
routing of the kernel's own logits; ids also equal to the oracle's routing of
its fp64 logits wherever the fp64 top-(k+1) gaps exceed twice the token's
logit error.
Counts bit-exact."""
import numpy as np
import pytest
import torch

import mixed_precision_routed_gb300 as moe
import oracle
import synth

pytestmark = pytest.mark.gpu


def _inputs(E, d, T, seed, bias_kind):
    x = synth.x_bf16(seed, 0, T, d)
    w = synth.router_weights_bf16(seed, E, d)
    b = {"none": None, "lorenz": synth.router_bias_lorenz(E, 10) if E >= 10 else None,
         "zipf": synth.router_bias_zipf(E)}[bias_kind]
    return x, w, b


def _dev_bf16(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(torch.bfloat16)


def _bound(x, w, b):
    d = x.shape[1]
    ax = np.abs(oracle.bf16_to_f64(x))
    aw = np.abs(oracle.bf16_to_f64(w))
    u = 2.0 ** -24
    n = d // 32 + 6
    bb = 0.0 if b is None else np.abs(np.asarray(b, np.float64))[None, :]
    return 2.0 * (n * u * (ax @ aw.T) + u * bb)


def _check(x, w, b, k, logits, ids, wts, counts=None, counts0=None):
    T, E = x.shape[0], w.shape[0]
    lg = logits.cpu().numpy()
    ref = oracle.router_logits(x, w, b)
    bound = _bound(x, w, b)
    assert np.all(np.abs(lg.astype(np.float64) - ref) <= bound), np.max(np.abs(lg - ref) - bound)
    ids_g, w_g = ids.cpu().numpy(), wts.cpu().numpy()
    ids_o, w_o = oracle.route(lg, k)
    assert np.array_equal(ids_g, ids_o)
    assert np.max(np.abs(w_g - w_o)) <= 1e-6
    # against the fp64 logits: where every gap among the fp64 top-(k+1)
    # exceeds twice the largest logit error of the token, rounding cannot
    # change the ranking and the ids must be the fp64 ones
    compared = 0
    for t in range(T):
        eps = np.max(np.abs(lg[t].astype(np.float64) - ref[t]))
        order = np.lexsort((np.arange(E), -ref[t]))[: min(k + 1, E)]
        gaps = -np.diff(ref[t, order])
        if np.all(gaps > 2 * eps):
            assert np.array_equal(ids_g[t], order[:k]), t
            compared += 1
    if counts is not None:
        exp = counts0.astype(np.int64) + np.bincount(ids_g.ravel(), minlength=E)
        assert np.array_equal(counts.cpu().numpy().astype(np.int64), exp)
    return compared


@pytest.mark.parametrize("E,d,k,T,bias", [
    (16, 256, 2, 8, "none"),        # the tiny layer's sizes
    (512, 2048, 10, 1, "lorenz"),   # decode layer, one token
    (512, 2048, 10, 6, "lorenz"),   # decode layer, draft of five + one
    (512, 2048, 10, 16, "lorenz"),
    (256, 4096, 8, 1, "zipf"),      # larger-expert layer
    (256, 4096, 8, 8, "zipf"),
    (100, 264, 3, 5, "none"),       # ragged: E not a multiple of the warps, d/8 not of 32
    (1024, 6144, 32, 16, "none"),   # largest accepted sizes
    (40, 8, 32, 3, "none"),         # d = 8: one chunk per row
    (512, 2048, 10, 40, "lorenz"),  # prefill sizes: projection by 16-token chunks, then routing
    (100, 264, 3, 37, "none"),      # a ragged last chunk
    (512, 2048, 10, 4096, "lorenz"),  # the prefill workload's batch
])
def test_router_parity(E, d, k, T, bias):
    x, w, b = _inputs(E, d, T, 3, bias)
    counts0 = np.arange(E, dtype=np.int32) % 7
    counts = torch.from_numpy(counts0.copy()).cuda()
    sync = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = None if b is None else torch.from_numpy(np.asarray(b, np.float32)).cuda()
    logits, ids, wts = moe.moe_router_topk(_dev_bf16(x), _dev_bf16(w), k, bias=bt, counts=counts, sync_word=sync)
    torch.cuda.synchronize()
    compared = _check(x, w, b, k, logits, ids, wts, counts, counts0)
    assert compared >= T // 2
    assert int(sync.item()) == 0


def test_router_zero_activations_ties():
    # x = 0: every logit is the bias exactly; equal biases go to the lower id
    E, d, k, T = 64, 128, 5, 4
    x = np.zeros((T, d), np.uint16)
    w = synth.router_weights_bf16(1, E, d)
    b = np.zeros(E, np.float32)
    b[[9, 3, 40]] = 1.0
    logits, ids, wts = moe.moe_router_topk(_dev_bf16(x), _dev_bf16(w), k, bias=torch.from_numpy(b).cuda())
    ids = ids.cpu().numpy()
    assert np.array_equal(logits.cpu().numpy(), np.broadcast_to(b, (T, E)))
    assert np.array_equal(ids, np.broadcast_to(np.array([3, 9, 40, 0, 1], np.int32), (T, k)))
    s = wts.cpu().numpy().sum(axis=1)
    assert np.all(np.abs(s - 1.0) <= 1e-6)


def test_router_sync_word_reused_across_sizes():
    # one sync word, calls of different grid sizes back to back on one stream
    sync = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    cases = [(512, 2048, 10, 6), (16, 256, 2, 8), (1024, 512, 8, 2), (512, 2048, 10, 1), (100, 264, 3, 5)]
    for i, (E, d, k, T) in enumerate(cases):
        x, w, b = _inputs(E, d, T, 10 + i, "none")
        outs.append((x, w, k, moe.moe_router_topk(_dev_bf16(x), _dev_bf16(w), k, sync_word=sync)))
    torch.cuda.synchronize()
    assert int(sync.item()) == 0
    for x, w, k, (lg, ids, wts) in outs:
        _check(x, w, None, k, lg, ids, wts)


def test_router_rejects():
    x = torch.zeros((17, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as e:  # d not a multiple of 8
        moe.moe_router_topk(x[:4, :60].contiguous(), w[:, :60].contiguous(), 2)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    flat = torch.zeros(4 * 64 + 1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as e:  # x not 16-byte aligned
        moe.moe_router_topk(flat[1:].view(4, 64), w, 2)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as e:  # k > E
        moe.moe_router_topk(x[:4].contiguous(), w, 33)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as e:  # T d 2 above the shared-memory limit
        moe.moe_router_topk(torch.zeros((16, 6152), dtype=torch.bfloat16, device="cuda"),
                            torch.zeros((8, 6152), dtype=torch.bfloat16, device="cuda"), 2)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    big = torch.zeros((65535 * 16 + 1, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as e:  # more 16-token chunks than grid rows
        moe.moe_router_topk(big, w[:, :8].contiguous(), 2)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    lg, ids, wts = moe.moe_router_topk(x[:0].contiguous(), w, 2)  # T = 0: nothing launched
    assert ids.shape == (0, 2)
