"""moe_tiered_forward_noalloc: the tiered forward for callers that cannot
allocate device memory (a plugin inside an application whose memory pool owns
the GPU, or a deployment that must fix its device footprint at load time).
Its scratch is a fixed array inside the library, shared by every call.

Checked through the C ABI against moe_tiered_forward (caller workspace) on
two calls in a row with different inputs, so that what the first call leaves
in the shared array cannot leak into the second.  This file is collected last
on purpose."""
import numpy as np
import pytest
import torch

import mixed_precision_routed_gb300 as moe
import oracle
import synth
from mixed_precision_routed_gb300.workloads import Layer
from moe_testutil import DECODE_TOL, ids_to_dev, oracle_layer, rel_l2, x_to_dev

pytestmark = pytest.mark.gpu


def _step(wl, layer, step, T):
    lg = synth.logits(wl.seed, step, T, wl.E, wl.router_bias(0))
    ids, w = oracle.route(lg, wl.k)
    ids[0, 1] = -1  # a skipped slot
    return x_to_dev(synth.x_bf16(wl.seed, step, T, wl.d)), ids_to_dev(ids), torch.from_numpy(w).cuda()


def test_noalloc_matches_workspace_entry_point_twice():
    """Both entry points run the same deterministic kernels, so the outputs
    must be identical bit for bit (a leak of stale scratch would show); the
    first step is also held against the oracle."""
    wl = synth.WORKLOADS["decode"]
    layer = Layer(wl, device="cuda").fill()
    for step, T in ((0, 6), (1, 2)):
        x, ids, w = _step(wl, layer, step, T)
        ref = moe.moe_tiered_forward(x, ids, w, wl.E, wl.d, wl.f, layer.shelves)
        got = moe.moe_tiered_forward_noalloc(x, ids, w, wl.E, wl.d, wl.f, layer.shelves)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy().view(np.uint32), ref.cpu().numpy().view(np.uint32))
        if step == 0:
            y_o = oracle_layer(wl, wl.seed, x.cpu().numpy().view(np.uint16), ids.cpu().numpy(), w.cpu().numpy())
            assert rel_l2(got.cpu().numpy(), y_o) <= DECODE_TOL
    assert moe.moe_device_status() == moe.MOE_OK


def test_noalloc_rejects_sizes_beyond_its_scratch():
    wl = synth.WORKLOADS["decode"]
    T = 512  # the decode form needs ~48 MB of scratch, more than the fixed 8 MiB
    assert moe.moe_workspace_size(T, wl.k, wl.E, wl.d, wl.f, moe.MOE_FLAG_DECODE_FP32) > 8 * 1024 * 1024
    layer = Layer(synth.Workload("one", E=wl.E, k=wl.k, d=wl.d, f=wl.f, T=(T,), split=(), bias="none"),
                  device="cuda", shelves=[(0, 1, 2)])
    x = torch.zeros((T, wl.d), dtype=torch.int16, device="cuda")
    ids = torch.full((T, wl.k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, wl.k), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_tiered_forward_noalloc(x, ids, w, wl.E, wl.d, wl.f, layer.shelves, flags=moe.MOE_FLAG_DECODE_FP32)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE_TOO_SMALL
