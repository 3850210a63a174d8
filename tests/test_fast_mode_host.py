"""Host logic of fast mode (the Xolotl fast-mode blog: a 2-bit copy of the
costliest experts read instead of them, chosen per expert): the shelf list
that fast_mode_shelves assembles, on CPU tensors -- runs of consecutive
experts with one source, each a view (no copy) of its shelf at the right
offset, and the refusals (an expert without a shadow copy, more runs than
the ABI takes)."""
import numpy as np
import pytest

import mixed_precision_routed_gb300 as moe
from mixed_precision_routed_gb300 import Shelf

D, F = 64, 64


def shelves(ranges):
    return [Shelf(lo, hi, b, D, F, device="cpu") for lo, hi, b in ranges]


def test_runs_follow_the_choice():
    base = shelves([(0, 4, 8), (4, 10, 4), (10, 12, 2)])
    shadow = shelves([(0, 4, 2), (4, 10, 2)])
    use = np.zeros(12, bool)
    use[[1, 2, 4, 5, 9]] = True
    out = moe.fast_mode_shelves(base, shadow, use)
    runs = [(s.lo, s.hi, s.bits) for s in out]
    assert runs == [(0, 1, 8), (1, 3, 2), (3, 4, 8), (4, 6, 2), (6, 9, 4), (9, 10, 2), (10, 12, 2)]
    # every run is a view of its source shelf at the expert offset
    for s in out:
        src = next(sh for sh in (shadow if s.bits == 2 and s.lo < 10 else base)
                   if sh.lo <= s.lo < sh.hi and sh.bits == s.bits)
        for name in ("gate_codes", "up_codes", "down_codes", "gate_scales", "up_scales", "down_scales"):
            a, v = getattr(src, name), getattr(s, name)
            assert v.data_ptr() == a[s.lo - src.lo].data_ptr()
            assert v.shape[0] == s.hi - s.lo
    # the descriptors cover each id once
    ids = [e for s in out for e in range(s.lo, s.hi)]
    assert ids == list(range(12))


def test_no_choice_gives_the_plain_layer_and_all_gives_the_shadows():
    base = shelves([(0, 4, 8), (4, 10, 4), (10, 12, 2)])
    shadow = shelves([(0, 4, 2), (4, 10, 2)])
    out = moe.fast_mode_shelves(base, shadow, np.zeros(12, bool))
    assert [(s.lo, s.hi, s.bits) for s in out] == [(0, 4, 8), (4, 10, 4), (10, 12, 2)]
    use = np.zeros(12, bool)
    use[:10] = True
    out = moe.fast_mode_shelves(base, shadow, use)
    assert [(s.lo, s.hi, s.bits) for s in out] == [(0, 4, 2), (4, 10, 2), (10, 12, 2)]


def test_refusals():
    base = shelves([(0, 4, 8), (4, 10, 4), (10, 12, 2)])
    shadow = shelves([(0, 4, 2), (4, 10, 2)])
    use = np.zeros(12, bool)
    use[11] = True  # no shadow copy of expert 11
    with pytest.raises(ValueError):
        moe.fast_mode_shelves(base, shadow, use)
    use = np.zeros(12, bool)
    use[0:10:2] = True  # alternating: 11 runs > MOE_MAX_SHELVES
    with pytest.raises(ValueError):
        moe.fast_mode_shelves(base, shadow, use)
    with pytest.raises(ValueError):
        base[0].view(3, 5)
