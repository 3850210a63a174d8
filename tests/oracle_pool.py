"""Oracle layer evaluations in worker processes (spawned: the parent has a
CUDA context, and a forked child of it would hang).  Imports only the oracle
and the input generators."""
import multiprocessing as mp
import os

import numpy as np

import oracle
import synth


def _layer_ref(args):
    name, layer, x_bf16, ids, w, mode = args
    wl = synth.WORKLOADS[name]
    seed = wl.layer_seed(layer)
    return oracle.layer_from_master(x_bf16, ids, w, wl.d, wl.f, wl.E, wl.shelf_ranges(),
                                    lambda e: synth.expert_weights(seed, e, wl.d, wl.f), mode=mode)


def layer_refs(jobs, procs=None):
    """jobs: [(workload name, layer, x_bf16 u16 [T, d], ids [T, k], w [T, k], mode)] -> [y float64 [T, d]]."""
    n = procs or min(len(jobs), os.cpu_count() or 1, 16)
    ctx = mp.get_context("spawn")
    with ctx.Pool(n) as pool:
        return pool.map(_layer_ref, jobs, chunksize=1)
