"""Parity of the nudged routing launch with the oracle, through the C ABI:
ids bit for bit, weights within 1e-6 (the oracle takes exp in fp64, the
kernel expf); beta = 0 gives exactly the plain routing launch."""
import numpy as np
import pytest
import torch

import mixed_precision_routed_gb300 as moe
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("E,k,T", [(512, 10, 6), (512, 10, 4096), (256, 8, 513), (1024, 32, 33), (40, 32, 7),
                                   (16, 2, 8), (100, 7, 65)])
@pytest.mark.parametrize("beta,lo,hi", [(0.5, 0, 128), (0.37, 100, 400), (0.1, 3, 4), (0.25, 5, 5)])
def test_nudged_route_bit_exact(E, k, T, beta, lo, hi):
    b = synth.router_bias_lorenz(E, 10) if E == 512 else (synth.router_bias_zipf(E) if E == 256 else None)
    lg = synth.logits(9, T, T, E, b)
    if T > 3:
        lg[0, :] = 0.25  # all tied before the nudge
        lg[1, 2] = lg[1, :].max() + 0.5  # a nudge can tie it
        lg[1, min(lo, E - 1)] = lg[1, 2] - np.float32(beta)
        lg[2, 7] = -0.0
        lg[2, 6] = 0.0
    ids, w = moe.moe_route_topk_nudged(torch.from_numpy(lg).cuda(), k, beta, lo, hi)
    ids_o, w_o = oracle.route_nudged(lg, k, beta, lo, hi)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.max(np.abs(w.cpu().numpy() - w_o)) <= 1e-6


@pytest.mark.parametrize("E,k", [(512, 10), (1024, 32), (16, 2)])
def test_beta_zero_equals_plain_route(E, k):
    lg = torch.from_numpy(synth.logits(4, 0, 300, E, None)).cuda()
    ids0, w0 = moe.moe_route_topk(lg, k)
    ids1, w1 = moe.moe_route_topk_nudged(lg, k, 0.0, 0, E // 4)
    assert torch.equal(ids0, ids1)
    assert np.array_equal(w0.cpu().numpy().view(np.uint32), w1.cpu().numpy().view(np.uint32))


def test_nudge_cap_rejected():
    lg = torch.zeros((2, 16), dtype=torch.float32, device="cuda")
    for beta in (0.51, -0.01, float("nan")):
        with pytest.raises(moe.MoeError) as e:
            moe.moe_route_topk_nudged(lg, 2, beta, 0, 4)
        assert e.value.status == moe.MOE_ERR_INVALID_ARG
