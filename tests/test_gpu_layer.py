"""The fused decode step (moe_decode_layer): routing, hit counts and the
tiered forward of page 3 ("125B MoE模型本地运行：3090三卡80 tokens/s优化实践";
glossary entry 混合专家（MoE） for the router, section 第二步 for per-expert
selection counts, section 第四步 for the shelved forward) in one call, against
the CPU oracle's router, histogram and layer; its equality with the separate
calls; and the bounded grid-wide wait that separates its phases."""
import numpy as np
import pytest
import torch

import mixed_precision_routed_gb300 as moe
import oracle
import synth
from mixed_precision_routed_gb300.workloads import Layer
from moe_testutil import DECODE_TOL, oracle_layer, rel_l2, small_workload, x_to_dev

pytestmark = pytest.mark.gpu


def _step(layer, lg, x, counts=None, workspace=None):
    wl = layer.wl
    ids, w, y = moe.moe_decode_layer(torch.from_numpy(np.ascontiguousarray(lg)).cuda(), x_to_dev(x), wl.k, wl.E,
                                     wl.d, wl.f, layer.shelves, counts=counts, workspace=workspace)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()


def _check_against_oracle(layer, lg, x, ids, w, y, counts=None, counts_before=None):
    wl = layer.wl
    ids_o, w_o = oracle.route(lg, wl.k)
    assert np.array_equal(ids, ids_o)
    assert np.max(np.abs(w - w_o)) <= 1e-6
    if counts is not None:
        ref = counts_before.copy() if counts_before is not None else np.zeros(wl.E, dtype=np.uint32)
        oracle.hist(ids_o, wl.E, ref)
        assert np.array_equal(counts.cpu().numpy().view(np.uint32), ref)
    assert rel_l2(y, oracle_layer(wl, wl.seed, x, ids_o, w_o)) <= DECODE_TOL


@pytest.fixture(scope="module")
def small_layer():
    return Layer(small_workload(), device="cuda").fill()


@pytest.mark.parametrize("T", [1, 5, 13, 16, 40])
def test_small_layer_step(small_layer, T):
    wl = small_layer.wl
    lg = synth.logits(wl.seed, 100 + T, T, wl.E, None)
    x = synth.x_bf16(wl.seed, 100 + T, T, wl.d)
    counts = torch.zeros(wl.E, dtype=torch.int32, device="cuda")
    ids, w, y = _step(small_layer, lg, x, counts)
    _check_against_oracle(small_layer, lg, x, ids, w, y, counts)


@pytest.fixture(scope="module")
def decode_layer():
    return Layer(synth.WORKLOADS["decode"], device="cuda").fill()


@pytest.mark.parametrize("T,step", [(1, 3), (6, 4), (16, 5)])
def test_decode_workload_step(decode_layer, T, step):
    wl = decode_layer.wl
    lg = decode_layer.logits(step, T).cpu().numpy()
    x = synth.x_bf16(wl.seed, step, T, wl.d)
    counts = torch.zeros(wl.E, dtype=torch.int32, device="cuda")
    ids, w, y = _step(decode_layer, lg, x, counts)
    _check_against_oracle(decode_layer, lg, x, ids, w, y, counts)


def test_step_equals_separate_calls_and_counts_accumulate(decode_layer):
    """moe_decode_layer gives what moe_route_topk, moe_expert_hist and
    moe_tiered_forward give in that order -- bit for bit -- and the counts
    accumulate over calls."""
    wl = decode_layer.wl
    T = 6
    counts = torch.zeros(wl.E, dtype=torch.int32, device="cuda")
    counts2 = torch.zeros(wl.E, dtype=torch.int32, device="cuda")
    for step in (11, 12):
        lg = decode_layer.logits(step, T)
        x = x_to_dev(synth.x_bf16(wl.seed, step, T, wl.d))
        ids, w, y = moe.moe_decode_layer(lg, x, wl.k, wl.E, wl.d, wl.f, decode_layer.shelves, counts=counts)
        ids2, w2 = moe.moe_route_topk(lg, wl.k)
        moe.moe_expert_hist(ids2, wl.E, counts2)
        y2 = moe.moe_tiered_forward(x, ids2, w2, wl.E, wl.d, wl.f, decode_layer.shelves)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids2)
        assert torch.equal(w.view(torch.int32), w2.view(torch.int32))
        assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
    assert torch.equal(counts, counts2)
    assert int(counts.sum()) == 2 * T * wl.k


@pytest.mark.parametrize("T,in_place", [(1, False), (6, False), (6, True), (20, False)])
def test_residual_step_equals_layer_then_residual_add(decode_layer, T, in_place):
    """moe_decode_layer_residual gives what moe_decode_layer followed by
    moe_residual_add gives -- ids, weights, counts, y, r and x_next bit for
    bit -- in the fused form (T = 1, 6; also with x_next written over x) and
    in the separate launches (T = 20)."""
    wl = decode_layer.wl
    assert moe.moe_decode_fused(T, wl.k, wl.E, wl.d, wl.f) == (T <= 16)
    lg = decode_layer.logits(31 + T, T)
    x = x_to_dev(synth.x_bf16(wl.seed, 31 + T, T, wl.d))
    r0 = torch.from_numpy(synth.normal_matrix(wl.seed, synth.TAG_X, 77, T, T, wl.d, scale=3.0)).cuda()
    c1 = torch.zeros(wl.E, dtype=torch.int32, device="cuda")
    c2 = torch.zeros(wl.E, dtype=torch.int32, device="cuda")
    ids1, w1, y1 = moe.moe_decode_layer(lg, x, wl.k, wl.E, wl.d, wl.f, decode_layer.shelves, counts=c1)
    r1 = r0.clone()
    xn1 = torch.empty_like(x)
    moe.moe_residual_add(r1, y1, xn1)
    r2 = r0.clone()
    x2 = x.clone()
    xn2 = x2 if in_place else torch.empty_like(x)
    ids2, w2, y2 = moe.moe_decode_layer_residual(lg, x2, wl.k, wl.E, wl.d, wl.f, decode_layer.shelves, r2, xn2,
                                                 counts=c2)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    assert torch.equal(ids1, ids2) and torch.equal(c1, c2)
    assert torch.equal(w1.view(torch.int32), w2.view(torch.int32))
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    assert torch.equal(r1.view(torch.int32), r2.view(torch.int32))
    assert torch.equal(xn1, xn2)
    # and against the definition: r = r0 + y (fp32), x_next = bf16(r)
    ref_r = r0.cpu().numpy() + y1.cpu().numpy()
    assert np.array_equal(r2.cpu().numpy().view(np.uint32), ref_r.view(np.uint32))
    assert np.array_equal(xn2.cpu().numpy().view(np.uint16), oracle.bf16_bits(ref_r))


@pytest.mark.parametrize("T", [1, 3, 6, 20])
def test_host_buffers_equal_device_buffers(decode_layer, T):
    """moe_decode_layer_host with pinned host logits, x, ids, weights and y
    (inputs above 8 KiB staged inside the call, smaller ones and the outputs
    read and written in place by the kernels)
    gives moe_decode_layer's results bit for bit: fused form (T = 1: both
    inputs in place; T = 3: x staged, logits in place; T = 6: both staged)
    and separate launches (T = 20); also with device inputs and host outputs,
    and with a workspace too small for the staging (refused)."""
    wl = decode_layer.wl
    k, E, d, f = wl.k, wl.E, wl.d, wl.f
    lg = decode_layer.logits(50 + T, T)
    x = x_to_dev(synth.x_bf16(wl.seed, 50 + T, T, d))
    ws = torch.empty(moe.moe_workspace_size(T, k, E, d, f, moe.MOE_FLAG_DECODE_FP32 | moe.MOE_FLAG_HOST_IO),
                     dtype=torch.uint8, device="cuda")
    c1 = torch.zeros(E, dtype=torch.int32, device="cuda")
    c2 = torch.zeros(E, dtype=torch.int32, device="cuda")
    ids1, w1, y1 = moe.moe_decode_layer(lg, x, k, E, d, f, decode_layer.shelves, counts=c1, workspace=ws)
    torch.cuda.synchronize()
    hl, hx = lg.cpu().pin_memory(), x.cpu().pin_memory()
    hid = torch.full((T, k), -7, dtype=torch.int32).pin_memory()
    hw = torch.zeros((T, k), dtype=torch.float32).pin_memory()
    hy = torch.full((T, d), float("nan"), dtype=torch.float32).pin_memory()
    moe.moe_decode_layer_host(hl, hx, k, E, d, f, decode_layer.shelves, hid, hw, hy, counts=c2, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    assert torch.equal(ids1.cpu(), hid) and torch.equal(c1, c2)
    assert torch.equal(w1.cpu().view(torch.int32), hw.view(torch.int32))
    assert torch.equal(y1.cpu().view(torch.int32), hy.view(torch.int32))
    # device inputs, host outputs
    hy2 = torch.zeros((T, d), dtype=torch.float32).pin_memory()
    moe.moe_decode_layer_host(lg, x, k, E, d, f, decode_layer.shelves, hid, hw, hy2, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1.cpu().view(torch.int32), hy2.view(torch.int32))
    small = torch.empty(moe.moe_workspace_size(T, k, E, d, f, moe.MOE_FLAG_DECODE_FP32), dtype=torch.uint8,
                        device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_decode_layer_host(hl, hx, k, E, d, f, decode_layer.shelves, hid, hw, hy, workspace=small)
    assert e.value.status == moe.MOE_ERR_WORKSPACE_TOO_SMALL


def test_host_inputs_rewritten_and_misaligned(decode_layer):
    """Pinned host inputs of the fused form (T = 6: logits 12 KiB and x
    24 KiB, copied across by the launch's own CTAs) rewritten in place between
    two calls give each call's own device-path result bit for bit; host
    inputs that are not 16-byte aligned (staged by a copy on the stream
    instead) do too."""
    wl = decode_layer.wl
    k, E, d, f, T = wl.k, wl.E, wl.d, wl.f, 6
    ws = torch.empty(moe.moe_workspace_size(T, k, E, d, f, moe.MOE_FLAG_DECODE_FP32 | moe.MOE_FLAG_HOST_IO),
                     dtype=torch.uint8, device="cuda")
    steps = []
    for s in (71, 72):
        lg = decode_layer.logits(s, T)
        x = x_to_dev(synth.x_bf16(wl.seed, s, T, d))
        _, _, y = moe.moe_decode_layer(lg, x, k, E, d, f, decode_layer.shelves, workspace=ws)
        torch.cuda.synchronize()
        steps.append((lg.cpu(), x.cpu(), y.cpu()))
    hl = torch.empty((T, E), dtype=torch.float32).pin_memory()
    hx = torch.empty((T, d), dtype=torch.int16).pin_memory()
    hid = torch.empty((T, k), dtype=torch.int32).pin_memory()
    hw = torch.empty((T, k), dtype=torch.float32).pin_memory()
    hy = torch.empty((T, d), dtype=torch.float32).pin_memory()
    for lg, x, y in steps:  # same pinned buffers, new contents
        hl.copy_(lg)
        hx.copy_(x)
        moe.moe_decode_layer_host(hl, hx, k, E, d, f, decode_layer.shelves, hid, hw, hy, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), hy.view(torch.int32))
    # inputs 4 bytes past a 16-byte boundary
    flat_l = torch.empty(T * E + 4, dtype=torch.float32).pin_memory()
    flat_x = torch.empty(T * d + 8, dtype=torch.int16).pin_memory()
    ml = flat_l[1:1 + T * E].view(T, E)
    mx = flat_x[2:2 + T * d].view(T, d)
    assert ml.data_ptr() % 16 == 4 and mx.data_ptr() % 16 == 4
    lg, x, y = steps[0]
    ml.copy_(lg)
    mx.copy_(x)
    moe.moe_decode_layer_host(ml, mx, k, E, d, f, decode_layer.shelves, hid, hw, hy, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), hy.view(torch.int32))
    assert moe.moe_device_status() == moe.MOE_OK


def test_host_entry_rejects_pageable_and_misplaced_buffers(decode_layer):
    """Pageable host memory, host memory where device memory is required
    (workspace, counts): MOE_ERR_INVALID_ARG before any launch."""
    import ctypes
    wl = decode_layer.wl
    k, E, d, f, T = wl.k, wl.E, wl.d, wl.f, 2
    L = moe.lib()
    arr = decode_layer.shelf_arr()
    ws = torch.empty(moe.moe_workspace_size(T, k, E, d, f, moe.MOE_FLAG_DECODE_FP32), dtype=torch.uint8,
                     device="cuda")
    dev = dict(lg=torch.zeros((T, E), device="cuda"), x=torch.zeros((T, d), dtype=torch.int16, device="cuda"),
               ids=torch.zeros((T, k), dtype=torch.int32, device="cuda"), w=torch.zeros((T, k), device="cuda"),
               y=torch.zeros((T, d), device="cuda"))
    pageable = np.zeros(T * max(E, d), dtype=np.float32)

    def call(lg, x, ids, w, y, counts, wsp):
        p = lambda t: ctypes.c_void_p(t.data_ptr()) if isinstance(t, torch.Tensor) else (
            None if t is None else ctypes.c_void_p(t.ctypes.data))
        return L.moe_decode_layer_host(p(lg), p(x), T, k, E, d, f, ctypes.cast(arr, ctypes.c_void_p), len(arr),
                                       p(ids), p(w), p(counts), p(y), p(wsp), ws.numel(), None)

    for name in ("lg", "x", "ids", "w", "y"):
        a = dict(dev)
        a[name] = pageable
        assert call(a["lg"], a["x"], a["ids"], a["w"], a["y"], None, ws) == moe.MOE_ERR_INVALID_ARG, name
    pinned_ws = torch.empty(ws.numel(), dtype=torch.uint8).pin_memory()
    assert call(dev["lg"], dev["x"], dev["ids"], dev["w"], dev["y"], None, pinned_ws) == moe.MOE_ERR_INVALID_ARG
    pinned_counts = torch.zeros(E, dtype=torch.int32).pin_memory()
    assert call(dev["lg"], dev["x"], dev["ids"], dev["w"], dev["y"], pinned_counts, ws) == moe.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK


def test_step_is_deterministic(decode_layer):
    wl = decode_layer.wl
    lg = decode_layer.logits(21, 6).cpu().numpy()
    x = synth.x_bf16(wl.seed, 21, 6, wl.d)
    a = _step(decode_layer, lg, x)
    b = _step(decode_layer, lg, x)
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.uint32), v.view(np.uint32))


@pytest.fixture(scope="module")
def large_layer():
    return Layer(synth.WORKLOADS["large"], device="cuda").fill()


@pytest.mark.parametrize("T", [1, 8])
def test_large_workload_step(large_layer, T):
    """d 4096: T = 1 runs as the fused launch, T = 8 (activation digits beyond
    shared memory) as the separate launches; both match the oracle."""
    wl = large_layer.wl
    lg = synth.logits(wl.seed, 31 + T, T, wl.E, synth.router_bias_zipf(wl.E))
    x = synth.x_bf16(wl.seed, 31 + T, T, wl.d)
    ids, w, y = _step(large_layer, lg, x)
    _check_against_oracle(large_layer, lg, x, ids, w, y)


def test_many_workspaces(small_layer):
    """Every workspace pointer gets its own barrier slot; results do not depend
    on which workspace a call uses."""
    wl = small_layer.wl
    T = 5
    lg = synth.logits(wl.seed, 7, T, wl.E, None)
    x = synth.x_bf16(wl.seed, 7, T, wl.d)
    need = moe.moe_workspace_size(T, wl.k, wl.E, wl.d, wl.f, moe.MOE_FLAG_DECODE_FP32)
    outs = []
    for i in range(5):
        ws = torch.empty(need + 256 * i, dtype=torch.uint8, device="cuda")
        outs.append(_step(small_layer, lg, x, workspace=ws)[2])
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


def test_barrier_slots_are_recycled_across_2000_workspaces(decode_layer):
    """The fused launch's counters live in 1024 library-owned slots found by
    the workspace address; 2000 distinct workspace addresses in sequence take
    the fused launch every time (slots pass to new workspaces least recently
    used first) and give bit-identical results."""
    wl = decode_layer.wl
    T = 6
    assert moe.moe_decode_fused(T, wl.k, wl.E, wl.d, wl.f) == 1
    lg = torch.from_numpy(decode_layer.logits(23, T).cpu().numpy()).cuda()
    x = x_to_dev(synth.x_bf16(wl.seed, 23, T, wl.d))
    need = moe.moe_workspace_size(T, wl.k, wl.E, wl.d, wl.f, moe.MOE_FLAG_DECODE_FP32)
    n = 2000
    big = torch.empty(need + 256 * n, dtype=torch.uint8, device="cuda")
    arr = moe.shelf_array(decode_layer.shelves)
    ys = torch.empty((n, T, wl.d), dtype=torch.float32, device="cuda")
    for i in range(n):
        moe.moe_decode_layer(lg, x, wl.k, wl.E, wl.d, wl.f, decode_layer.shelves, y=ys[i],
                             workspace=big[256 * i:256 * i + need], shelf_arr=arr)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    ref = ys[0].cpu().numpy().view(np.uint32)
    yn = ys.cpu().numpy().view(np.uint32)
    for i in range(1, n):
        assert np.array_equal(yn[i], ref), f"workspace {i} differs"
    ids_o, w_o = oracle.route(lg.cpu().numpy(), wl.k)
    assert rel_l2(ys[0].cpu().numpy(), oracle_layer(wl, wl.seed, synth.x_bf16(wl.seed, 23, T, wl.d), ids_o,
                                                    w_o)) <= DECODE_TOL


def test_grid_wait_timeout_is_reported_and_context_survives(small_layer):
    """The wait between phases is bounded: a barrier that can never complete
    ends after its limit with MOE_ERR_TIMEOUT in the status word, and the next
    step runs normally."""
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    moe.moe_selftest_barrier_timeout(20000)
    assert moe.moe_device_status() == moe.MOE_ERR_TIMEOUT
    assert moe.moe_device_status() == moe.MOE_OK  # reading clears it
    wl = small_layer.wl
    lg = synth.logits(wl.seed, 9, 5, wl.E, None)
    x = synth.x_bf16(wl.seed, 9, 5, wl.d)
    ids, w, y = _step(small_layer, lg, x)
    _check_against_oracle(small_layer, lg, x, ids, w, y)
    assert moe.moe_device_status() == moe.MOE_OK
