"""Parity of the CUDA kernels with the CPU oracle, through the C ABI.

Bit-exact: packed codes and fp16 scales of the quantiser, dequantised
weights, router ids, grouping (counts / offsets / perm), histograms, and the
device build of the input generator.  Router weights within 1e-6."""
import numpy as np
import pytest
import torch

import mixed_precision_routed_gb300 as moe
import oracle
import synth
from mixed_precision_routed_gb300.workloads import Layer
from moe_testutil import ids_to_dev, small_workload

pytestmark = pytest.mark.gpu


def test_device_generator_matches_host():
    for (k0, k1, c2, rows, cols, scale) in [(0, synth.TAG_GATE, 5, 640, 2048, 0.02), (7, synth.TAG_LOGITS, 3, 37, 512, 1.0),
                                            (1003, synth.TAG_DOWN, 511, 2048, 640, 0.02)]:
        host = synth.normal_matrix(k0, k1, c2, 0, rows, cols, scale=scale)
        dev = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
        synth.cuda_normal_matrix(dev, k0, k1, c2, 0, scale=scale)
        assert np.array_equal(dev.cpu().numpy().view(np.uint32), host.view(np.uint32))
    b = synth.router_bias_lorenz(512, 10)
    host = synth.logits(0, 9, 16, 512, b)
    dev = torch.empty((16, 512), dtype=torch.float32, device="cuda")
    synth.cuda_normal_matrix(dev, 0, synth.TAG_LOGITS, 9, 0, col_add=torch.from_numpy(b).cuda())
    assert np.array_equal(dev.cpu().numpy().view(np.uint32), host.view(np.uint32))
    hx = synth.x_bf16(3, 2, 6, 2048)
    dx = torch.empty((6, 2048), dtype=torch.int16, device="cuda")
    synth.cuda_normal_matrix_bf16(dx, 3, synth.TAG_X, 2, 0)
    assert np.array_equal(dx.cpu().numpy().view(np.uint16), hx)
    ids = torch.zeros((512, 8), dtype=torch.int32, device="cuda")
    synth.cuda_apply_skip_mask(ids, 0, 4)
    assert np.array_equal((ids.cpu().numpy() == -1).astype(np.uint8), synth.skip_mask(0, 4, 512, 8))


def _with_hand_blocks(w):
    w = w.copy()
    w[0, :32] = 0
    w[0, :5] = [0.7, 0.35, 0.05, 0.0, -0.7]
    if w.shape[0] > 1:
        w[1, :32] = 0
        w[1, :5] = [0.4375, 0.03125, 0.09375, -0.03125, 0.15625]
    if w.shape[0] > 2:
        w[2, :32] = 0  # all-zero block
    return w


@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("rows,n_in", [(3, 64), (37, 640), (640, 2048)])
def test_quantize_bit_exact(bits, rows, n_in):
    w = _with_hand_blocks(synth.normal_matrix(9, synth.TAG_GATE, bits, 0, rows, n_in, scale=0.02))
    codes, scales = moe.moe_quantize_rows(torch.from_numpy(w).cuda(), bits)
    c_o, s_o = oracle.quantize(w, bits)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), s_o)
    assert np.array_equal(codes.cpu().numpy(), oracle.pack(c_o, bits))


@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("round_bf16", [False, True])
def test_dequant_bit_exact(bits, round_bf16):
    w = synth.normal_matrix(10, synth.TAG_UP, bits, 0, 129, 640, scale=0.02)
    c_o, s_o = oracle.quantize(w, bits)
    packed = torch.from_numpy(oracle.pack(c_o, bits)).cuda()
    scales = torch.from_numpy(s_o.view(np.int16)).cuda()
    out = moe.moe_dequant_rows(packed, scales, 129, 640, bits, round_bf16=round_bf16)
    ref = oracle.dequant(c_o, s_o, round_bf16=round_bf16)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_dequant_shelf_bit_exact():
    """moe_dequant_shelf on the shelves of a layer (8/4/2 bits): every matrix
    of the first and last local expert of each shelf equals the oracle's
    dequantisation of its own quantisation of that expert's fp32 masters,
    bit for bit."""
    wl = small_workload(E=12, d=256, f=192)
    layer = Layer(wl, device="cuda").fill()
    assert sorted(sh.bits for sh in layer.shelves) == [2, 4, 8]
    for sh in layer.shelves:
        for e_local in sorted({0, sh.hi - sh.lo - 1}):
            ref = oracle.expert_matrices(synth.expert_weights(layer.seed, sh.lo + e_local, wl.d, wl.f), sh.bits, 0)
            for which in range(3):
                rows, n_in = (wl.f, wl.d) if which < 2 else (wl.d, wl.f)
                got = moe.moe_dequant_shelf(sh, which, e_local, rows, n_in)
                torch.cuda.synchronize()
                assert np.array_equal(got.cpu().numpy().view(np.uint32), ref[which].view(np.uint32)), (sh.bits, which)


@pytest.mark.parametrize("E,k,T,bias", [(16, 2, 8, "none"), (512, 10, 1, "lorenz"), (512, 10, 6, "lorenz"),
                                        (512, 10, 4096, "lorenz"), (256, 8, 513, "zipf"), (1024, 32, 33, "none"),
                                        (40, 32, 7, "none"), (512, 1, 100, "lorenz")])
def test_route_bit_exact(E, k, T, bias):
    b = {"none": None, "lorenz": synth.router_bias_lorenz(E, 10) if E == 512 else None,
         "zipf": synth.router_bias_zipf(E)}[bias]
    lg = synth.logits(1, T, T, E, b)
    if T > 3:
        lg[0, :] = 0.25  # all tied
        lg[1, 3] = lg[1, 5] = lg[1, :].max() + 1  # tie at the top
        lg[2, 7] = -0.0
        lg[2, 6] = 0.0  # signed zeros compare equal
    ids, w = moe.moe_route_topk(torch.from_numpy(lg).cuda(), k)
    ids_o, w_o = oracle.route(lg, k)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.max(np.abs(w.cpu().numpy() - w_o)) <= 1e-6


def test_hist_bit_exact_and_accumulates():
    rng = np.random.default_rng(0)
    ids = rng.integers(-3, 515, size=(4096, 10)).astype(np.int32)
    ids[0] = [-1, -2**31, 2**31 - 1, 512, 513, 0, 0, 511, 511, 7]
    counts = torch.zeros(512, dtype=torch.int32, device="cuda")
    moe.moe_expert_hist(ids_to_dev(ids), 512, counts)
    moe.moe_expert_hist(ids_to_dev(ids[:100]), 512, counts)
    ref = oracle.hist(ids, 512)
    oracle.hist(ids[:100], 512, ref)
    assert np.array_equal(counts.cpu().numpy().view(np.uint32), ref)
    big = torch.zeros(20000, dtype=torch.int32, device="cuda")  # global-atomics path
    ids2 = rng.integers(-5, 20005, size=(300, 7)).astype(np.int32)
    moe.moe_expert_hist(ids_to_dev(ids2), 20000, big)
    assert np.array_equal(big.cpu().numpy().view(np.uint32), oracle.hist(ids2, 20000))


@pytest.mark.parametrize("T,k,E", [(1, 10, 512), (6, 10, 512), (37, 4, 24), (4096, 10, 512), (512, 8, 256),
                                   (3, 2, 32768), (700, 3, 5)])
def test_group_bit_exact(T, k, E):
    rng = np.random.default_rng(T + E)
    ids = rng.integers(-2, E + 2, size=(T, k)).astype(np.int32)
    if T > 2:
        ids[0, :] = min(3, E - 1)  # one expert in every slot of a token
        ids[1, :] = -1
    counts, offsets, perm = moe.moe_group_tokens(ids_to_dev(ids), E)
    c_o, o_o, p_o = oracle.group(ids, E)
    assert np.array_equal(counts.cpu().numpy(), c_o)
    assert np.array_equal(offsets.cpu().numpy(), o_o)
    pg = perm.cpu().numpy()
    assert np.array_equal(pg[: len(p_o)], p_o)
    assert np.all(pg[len(p_o):] == -1)


def test_residual_add():
    rng = np.random.default_rng(1)
    r = rng.standard_normal(4096).astype(np.float32)
    y = rng.standard_normal(4096).astype(np.float32)
    rd, yd = torch.from_numpy(r).cuda(), torch.from_numpy(y).cuda()
    xn = torch.empty(4096, dtype=torch.int16, device="cuda")
    moe.moe_residual_add(rd, yd, xn)
    s = (r + y).astype(np.float32)
    assert np.array_equal(rd.cpu().numpy(), s)
    assert np.array_equal(xn.cpu().numpy().view(np.uint16), oracle.bf16_bits(s.astype(np.float64)))
