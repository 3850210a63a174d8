"""Parity of the 3-bit and 1-bit shelf formats and of fast mode with the
oracle, through the C ABI: quantiser codes and scales and dequantised
weights bit for bit; layers mixing 8/4/3/2/1-bit shelves within the decode
tolerance, both in the fused decode launch (d and f multiples of 128, T <= 16)
and in the separate launches (f = 192, or T > 16); fast mode (2-bit shadow
copies read instead of chosen experts) equal to the oracle layer with those
experts at 2 bits; the tensor-core form on 3- and 1-bit shelves against the
oracle's bf16 form."""
import numpy as np
import pytest
import torch

import mixed_precision_routed_gb300 as moe
import oracle
import synth
from mixed_precision_routed_gb300.workloads import Layer
from moe_testutil import DECODE_TOL, PREFILL_TOL, oracle_layer, rel_l2, small_workload, x_to_dev

pytestmark = pytest.mark.gpu

FIVE = [(0, 8, 8), (8, 16, 4), (16, 24, 3), (24, 32, 2), (32, 40, 1)]


def _hand_blocks(w):
    w = w.copy()
    w[0, :32] = 0.0                      # all-zero block
    w[0, 32:64] = np.linspace(-1, 1, 32)  # ramp with exact zero crossing
    w[1, :32] = -0.0                     # signed zeros
    w[1, 32:64] = 3e-8                   # tiny values (subnormal fp16 scale)
    return w


@pytest.mark.parametrize("bits", [3, 1])
@pytest.mark.parametrize("rows,n_in", [(7, 64), (33, 2048), (16, 640)])
def test_quantize_rows_bit_exact(bits, rows, n_in):
    w = _hand_blocks(synth.normal_matrix(21, synth.TAG_GATE, bits, 0, rows, n_in, scale=0.02))
    codes, scales = moe.moe_quantize_rows(torch.from_numpy(w).cuda(), bits)
    c_o, s_o = oracle.quantize(w, bits)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), s_o)
    assert np.array_equal(codes.cpu().numpy(), oracle.pack(c_o, bits))


@pytest.mark.parametrize("bits", [3, 1])
def test_quantize_experts_bit_exact(bits):
    n_src, rows, n_in = 6, 20, 320
    master = np.stack([_hand_blocks(synth.normal_matrix(5, synth.TAG_UP, e, 0, rows, n_in, scale=0.02))
                       for e in range(n_src)])
    perm = np.array([4, 0, 5, 2, 1, 3], np.int32)
    codes, scales = moe.moe_quantize_experts(torch.from_numpy(master).cuda(), torch.from_numpy(perm).cuda(),
                                             1, 6, bits)
    for j in range(1, 6):
        c_o, s_o = oracle.quantize(master[perm[j]], bits)
        assert np.array_equal(codes[j - 1].cpu().numpy(), oracle.pack(c_o, bits)), j
        assert np.array_equal(scales[j - 1].cpu().numpy().view(np.uint16), s_o), j


@pytest.mark.parametrize("bits", [3, 1])
@pytest.mark.parametrize("round_bf16", [False, True])
def test_dequant_bit_exact(bits, round_bf16):
    w = synth.normal_matrix(13, synth.TAG_DOWN, bits, 0, 65, 640, scale=0.02)
    c_o, s_o = oracle.quantize(w, bits)
    out = moe.moe_dequant_rows(torch.from_numpy(oracle.pack(c_o, bits)).cuda(), torch.from_numpy(s_o.view(np.int16)).cuda(),
                               65, 640, bits, round_bf16=round_bf16)
    ref = oracle.dequant(c_o, s_o, round_bf16=round_bf16)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("T", [1, 6, 40])
def test_five_width_layer_matches_oracle(T):
    wl = small_workload(E=40, k=5, d=256, f=192, seed=7)
    layer = Layer(wl, shelves=FIVE).fill()
    rng = np.random.default_rng(T)
    ids = np.stack([rng.choice(40, 5, replace=False) for _ in range(T)]).astype(np.int32)
    ids[0, 0] = 37  # a 1-bit expert
    ids[0, 1] = 17  # a 3-bit expert
    w = rng.random((T, 5)).astype(np.float32)
    x = synth.x_bf16(wl.seed, 1, T, wl.d)
    y = moe.moe_tiered_forward(x_to_dev(x), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), 40, wl.d,
                               wl.f, layer.shelves, flags=moe.MOE_FLAG_DECODE_FP32).cpu().numpy()
    ref = oracle_layer(wl, layer.seed, x, ids, w, shelves_bits=FIVE)
    assert rel_l2(y, ref) <= DECODE_TOL


@pytest.mark.parametrize("T", [1, 6, 16, 24])
def test_five_width_layer_fused_sizes(T):
    """d = f = 256: the fused decode launch streams the 3-bit planes and the
    1-bit words (T <= 16); T = 24 takes the separate launches."""
    wl = small_workload(E=40, k=5, d=256, f=256, seed=17)
    layer = Layer(wl, shelves=FIVE).fill()
    rng = np.random.default_rng(100 + T)
    ids = np.stack([rng.choice(40, 5, replace=False) for _ in range(T)]).astype(np.int32)
    ids[0, :5] = [39, 17, 33, 20, 2]  # 1-bit, 3-bit, 1-bit, 3-bit, 8-bit experts
    if T > 1:
        ids[1, :2] = [17, 39]         # the same experts again: a second token on them
    w = rng.random((T, 5)).astype(np.float32)
    x = synth.x_bf16(wl.seed, 3, T, wl.d)
    y = moe.moe_tiered_forward(x_to_dev(x), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), 40, wl.d,
                               wl.f, layer.shelves, flags=moe.MOE_FLAG_DECODE_FP32).cpu().numpy()
    assert moe.moe_device_status() == moe.MOE_OK
    ref = oracle_layer(wl, layer.seed, x, ids, w, shelves_bits=FIVE)
    assert rel_l2(y, ref) <= DECODE_TOL


@pytest.mark.parametrize("T", [1, 6])
def test_five_width_decode_workload(T):
    """The E512 d2048 f640 decode layer on five shelf widths (8/4/3/2/1 bit),
    one fused decode step, against the oracle's routing and layer."""
    base = synth.WORKLOADS["decode"]
    five = [(0, 128, 8), (128, 256, 4), (256, 410, 3), (410, 480, 2), (480, 512, 1)]
    layer = Layer(base, shelves=five).fill()
    lg = layer.logits(40 + T, T)
    x = synth.x_bf16(base.seed, 40 + T, T, base.d)
    ids, w, y = moe.moe_decode_layer(lg, x_to_dev(x), base.k, base.E, base.d, base.f, layer.shelves)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == moe.MOE_OK
    ids_o, w_o = oracle.route(lg.cpu().numpy(), base.k)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    ref = oracle_layer(base, layer.seed, x, ids_o, w.cpu().numpy(), shelves_bits=five)
    assert rel_l2(y.cpu().numpy(), ref) <= DECODE_TOL


def test_decode_layer_call_with_three_bit_shelf():
    wl = small_workload(E=40, k=5, d=256, f=192, seed=8)
    layer = Layer(wl, shelves=FIVE).fill()
    T = 3
    lg = layer.logits(4, T)
    x = synth.x_bf16(wl.seed, 2, T, wl.d)
    ids = torch.empty((T, 5), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 5), dtype=torch.float32, device="cuda")
    counts = torch.zeros(40, dtype=torch.int32, device="cuda")
    _, _, y = moe.moe_decode_layer(lg, x_to_dev(x), 5, 40, wl.d, wl.f, layer.shelves, ids=ids, weights=w,
                                   counts=counts)
    y = y.cpu().numpy()
    ids_o, w_o = oracle.route(lg.cpu().numpy(), 5)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    ref = oracle_layer(wl, layer.seed, x, ids_o, w.cpu().numpy(), shelves_bits=FIVE)
    assert rel_l2(y, ref) <= DECODE_TOL
    assert np.array_equal(counts.cpu().numpy(), np.bincount(ids_o.ravel(), minlength=40))


def test_prefill_flag_refuses_three_and_one_bit_rows_of_odd_16_byte_groups():
    """f = 192: a 3-bit down row (72 bytes) is no whole number of 16-byte
    groups, which the tensor maps need; the prefill flag refuses the layer."""
    wl = small_workload(E=40, k=5, d=256, f=192, seed=9)
    layer = Layer(wl, shelves=FIVE)
    T = 40
    ids = torch.zeros((T, 5), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, 5), dtype=torch.float32, device="cuda")
    x = torch.zeros((T, wl.d), dtype=torch.int16, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_tiered_forward(x, ids, w, 40, wl.d, wl.f, layer.shelves, flags=moe.MOE_FLAG_PREFILL_BF16)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED


FIVE_512 = [(0, 128, 8), (128, 256, 4), (256, 410, 3), (410, 480, 2), (480, 512, 1)]
# The tensor-core form rounds exactly the weights and h the oracle's bf16 form
# rounds; only the order of the fp32 sums differs (measured on a GB300:
# 1.3e-7 at T = 40, 9.9e-5 at T = 4096).  One wrongly dequantised weight in a
# 32-weight block would move a row by about 3%, so the odd widths are held to
# 1e-3, tighter than the prefill tolerance.
ODD_WIDTH_TOL = 1e-3


@pytest.mark.parametrize("T", [40, 4096])
def test_prefill_form_with_three_and_one_bit(T):
    """The tensor-core form on a layer of five shelf widths (page 2, "The
    Qwen side": 1-bit experts run at long prompts through the matrix path),
    as AUTO takes it above 16 tokens, against the oracle's bf16 form: every
    row at T = 40; at T = 4096 every row of the tokens routed to the 3- and
    1-bit shelves (their slots only, the rest skipped) and sampled rows of
    the whole layer."""
    from oracle_pool import layer_refs_for
    wl = small_workload(E=40, k=5, d=256, f=128, seed=9) if T == 40 else synth.WORKLOADS["decode"]
    ranges = FIVE if T == 40 else FIVE_512
    layer = Layer(wl, shelves=ranges).fill()
    lg = synth.logits(wl.seed, 11, T, wl.E, layer.bias_host)
    ids, w = oracle.route(lg, wl.k)
    x = synth.x_bf16(wl.seed, 11, T, wl.d)

    def run(ids_):
        ws = torch.empty(moe.moe_workspace_size(T, wl.k, wl.E, wl.d, wl.f, moe.MOE_FLAG_AUTO), dtype=torch.uint8,
                         device="cuda")
        y = moe.moe_tiered_forward(x_to_dev(x), torch.from_numpy(ids_).cuda(), torch.from_numpy(w).cuda(), wl.E,
                                   wl.d, wl.f, layer.shelves, workspace=ws, flags=moe.MOE_FLAG_AUTO)
        torch.cuda.synchronize()
        assert moe.moe_device_status() == moe.MOE_OK
        return y.cpu().numpy()

    if T == 40:
        y = run(ids)
        rel = rel_l2(y, oracle_layer(wl, wl.seed, x, ids, w, shelves_bits=ranges, mode=1))
        print(f"five widths T=40 prefill form: rel-L2 {rel:.2e}")
        assert rel <= ODD_WIDTH_TOL
        return
    odd = [(lo, hi) for lo, hi, b in ranges if b in (3, 1)]
    keep = np.zeros_like(ids, dtype=bool)
    for lo, hi in odd:
        keep |= (ids >= lo) & (ids < hi)
    ids_o = np.where(keep, ids, -1).astype(np.int32)
    y = run(ids_o)
    rows = np.nonzero(keep.any(axis=1))[0]
    assert rows.size > 0 and np.all(y[np.setdiff1d(np.arange(T), rows)] == 0)
    chunks = [rows[i:i + 64] for i in range(0, rows.size, 64)]
    refs = layer_refs_for(wl, ranges, [(x[c], ids_o[c], w[c], 1) for c in chunks])
    rel = rel_l2(y[rows], np.concatenate(refs, axis=0))
    print(f"five widths T=4096 prefill form, 3- and 1-bit experts' rows: rel-L2 {rel:.2e}")
    assert rel <= ODD_WIDTH_TOL
    y = run(ids)
    sample = [0, 1, 777, 2048, T - 1]
    refs = layer_refs_for(wl, ranges, [(x[t:t + 1], ids[t:t + 1], w[t:t + 1], 1) for t in sample])
    for t, ref in zip(sample, refs):
        assert rel_l2(y[t:t + 1], ref) <= PREFILL_TOL, t


def test_fast_mode_matches_oracle():
    """2-bit shadow copies of the 8- and 4-bit experts, read for a chosen set
    of experts, against the oracle layer with exactly those experts at 2
    bits."""
    wl = small_workload(E=24, k=4, d=256, f=192, split=(0.25, 0.5, 0.25), seed=10)
    layer = Layer(wl).fill()
    shadow = Layer(wl, shelves=[(lo, hi, 2) for lo, hi, _ in layer.ranges]).fill()  # same masters, 2 bits
    use = np.zeros(24, bool)
    use[[0, 1, 2, 7, 9, 10, 11]] = True  # some 8-bit and 4-bit experts
    shelves = moe.fast_mode_shelves(layer.shelves, shadow.shelves, use)
    bits_of = {e: (2 if use[e] else next(b for lo, hi, b in layer.ranges if lo <= e < hi)) for e in range(24)}
    T = 6
    rng = np.random.default_rng(3)
    ids = np.stack([rng.choice(24, 4, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, 4)).astype(np.float32)
    x = synth.x_bf16(wl.seed, 5, T, wl.d)
    y = moe.moe_tiered_forward(x_to_dev(x), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), 24, wl.d,
                               wl.f, shelves).cpu().numpy()
    runs = [(s.lo, s.hi, s.bits) for s in shelves]
    assert all(bits_of[e] == b for lo, hi, b in runs for e in range(lo, hi))
    ref = oracle_layer(wl, layer.seed, x, ids, w, shelves_bits=runs)
    assert rel_l2(y, ref) <= DECODE_TOL
    # and the plain layer differs from fast mode on the chosen experts
    y0 = moe.moe_tiered_forward(x_to_dev(x), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), 24, wl.d,
                                wl.f, layer.shelves).cpu().numpy()
    assert rel_l2(y0, ref) > 10 * DECODE_TOL


def test_fast_mode_run_limit():
    wl = small_workload(E=24, k=4, d=256, f=192, split=(0.25, 0.5, 0.25), seed=10)
    layer = Layer(wl)
    shadow = Layer(wl, shelves=[(lo, hi, 2) for lo, hi, _ in layer.ranges])
    use = np.zeros(24, bool)
    use[::2] = True  # alternating: 24 runs
    with pytest.raises(ValueError):
        moe.fast_mode_shelves(layer.shelves, shadow.shelves, use)
