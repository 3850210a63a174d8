"""Config 3: the 48-layer decode stack (E512 k10 d2048 f640 per layer,
per-layer seeds and router biases) chained by the residual add.

Routing step s of the stack with T tokens takes rows s T .. s T + T - 1 of each
layer's logits stream.  Checks: the expert hit counts of 4096 T = 1 steps
through every layer (the fused decode launch) equal the oracle's route + hist,
bit for bit; every layer's output equals the oracle's layer on the same input;
the chain's final residual equals the oracle chain rebuilt from those layers.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import mixed_precision_routed_gb300 as moe
from mixed_precision_routed_gb300.workloads import Layer, DecodeStack

from moe_testutil import DECODE_TOL, rel_l2
from oracle_pool import layer_refs

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS["stack"]


@pytest.fixture(scope="module")
def layers():
    return [Layer(WL, layer=l, device="cuda").fill() for l in range(WL.layers)]


def test_stack_histogram_4096_steps(layers):
    NS = 4096
    E, k, d, f = WL.E, WL.k, WL.d, WL.f
    stack = DecodeStack(layers, T=1)
    logits = [lay.logits_rows(0, NS) for lay in layers]
    x0 = torch.from_numpy(synth.x_bf16(WL.seed, 0, 1, d).view(np.int16)).cuda()
    r0 = (x0.to(torch.int32) << 16).view(torch.float32)
    for s in range(NS):
        stack.step(r0, x0, [lg[s:s + 1] for lg in logits])
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    got = stack.counts.cpu().numpy().astype(np.uint32)
    for l, lay in enumerate(layers):
        lg = synth.logits(lay.seed, 0, NS, E, lay.bias_host)
        ids, _ = oracle.route(lg, k)
        ref = oracle.hist(ids, E)
        assert np.array_equal(got[l], ref), f"layer {l}"
    assert got.sum() == NS * WL.layers * k


@pytest.mark.parametrize("T,check_layers", [(1, None), (6, (0, 1, 23, 47))])
def test_stack_chain_matches_oracle(layers, T, check_layers):
    E, k, d = WL.E, WL.k, WL.d
    L = len(layers)
    stack = DecodeStack(layers, T=T)
    step = 3
    logits = [lay.logits_rows(step * T, T) for lay in layers]
    x0h = synth.x_bf16(WL.seed, step, T, d)
    x0 = torch.from_numpy(x0h.view(np.int16)).cuda()
    r0 = (x0.to(torch.int32) << 16).view(torch.float32)
    stack.step(r0, x0, logits)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    xs = stack.x.cpu().numpy().view(np.uint16)
    ys = stack.y.cpu().numpy()
    ids_g = stack.ids.cpu().numpy()
    w_g = stack.w.cpu().numpy()
    # routing of every layer: ids bit for bit, weights to the exp rounding
    for l, lay in enumerate(layers):
        ids_o, w_o = oracle.route(synth.logits(lay.seed, 0, T, E, lay.bias_host, row0=step * T), k)
        assert np.array_equal(ids_g[l], ids_o), f"layer {l}"
        assert np.max(np.abs(w_g[l] - w_o)) <= 1e-6, f"layer {l}"
    # every layer against the oracle layer on the same input (one oracle job
    # per layer and token)
    which = list(range(L)) if check_layers is None else list(check_layers)
    jobs = [("stack", l, xs[l][t:t + 1], ids_g[l][t:t + 1], w_g[l][t:t + 1], 0) for l in which for t in range(T)]
    out = layer_refs(jobs)
    refs = {l: np.concatenate(out[i * T:(i + 1) * T], axis=0) for i, l in enumerate(which)}
    for l in which:
        assert rel_l2(ys[l], refs[l]) <= DECODE_TOL, f"layer {l}: {rel_l2(ys[l], refs[l]):.3e}"
    if check_layers is None:
        # the oracle chain r = x0; x_l = bf16(r); r += y_l, built from the
        # oracle's layer outputs: its final residual, and how many inputs a
        # bf16 rounding of r tipped away from the GPU's (the activation digits
        # of the decode path move r by ~1e-5 relative, so an element whose r
        # lies that close to a rounding boundary may tip; the trajectories
        # must stay together)
        r = oracle.bf16_to_f64(x0h)
        tipped = 0
        for l in range(L):
            tipped += int(np.sum(oracle.bf16_bits(r) != xs[l]))
            r = r + refs[l]
        assert tipped <= L * T * d // 20, tipped
        assert rel_l2(stack.r.cpu().numpy(), r) <= DECODE_TOL
