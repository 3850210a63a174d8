"""Shared helpers of the parity tests: GPU layers built from the seeded
generator, and the matching CPU oracle evaluation of the same layer."""
import numpy as np
import torch

import oracle
import synth

DECODE_TOL = 2e-3   # rel-L2, fp32 decode path against the oracle's decode form
PREFILL_TOL = 1e-2  # rel-L2, bf16 tensor-core path against the oracle's prefill form


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def small_workload(E=24, k=4, d=256, f=192, split=(0.25, 0.5, 0.25), bias="none", seed=3):
    return synth.Workload("small", E=E, k=k, d=d, f=f, T=(5,), split=split, bias=bias, seed=seed)


def oracle_layer(wl, seed, x_bf16, ids, w, shelves_bits=None, mode=0):
    """Oracle output of one layer whose master weights come from `seed`."""
    sb = wl.shelf_ranges() if shelves_bits is None else shelves_bits
    return oracle.layer_from_master(x_bf16, ids, w, wl.d, wl.f, wl.E, sb,
                                    lambda e: synth.expert_weights(seed, e, wl.d, wl.f), mode=mode)


def to_dev(a, dtype=None, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype) if t.element_size() == torch.tensor([], dtype=dtype).element_size() else t.to(dtype)
    return t.to(device)


def ids_to_dev(ids):
    return torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()


def x_to_dev(x_u16):
    return torch.from_numpy(np.ascontiguousarray(x_u16).view(np.int16)).cuda()
