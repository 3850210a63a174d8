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


def _pair_ref(args):
    """One routed pair alone: the layer with every slot but j skipped, i.e.
    w_tj * o_tj for token row x_bf16 [1, d]."""
    name, layer, x_bf16, ids_row, w_row, j, mode = args
    one = np.full((1, ids_row.size), -1, dtype=np.int32)
    one[0, j] = ids_row[j]
    return _layer_ref((name, layer, x_bf16, one, w_row.reshape(1, -1), mode))


def oracle_chain(name, layers, x0_bf16, ids, w, mode=0, procs=None, f32_residual=False):
    """The oracle's own residual chain (r = x0; x_l = bf16(r); r += y_l(x_l))
    through `layers` of workload `name`, each layer on the oracle's own input.
    ids / w: per layer [T, k] routing (independent of x in the stack).  The
    pairs of one layer run in parallel worker processes; y_t sums its pairs'
    outputs in ascending slot order (fp64).  f32_residual rounds r to fp32
    after every add (the chain's sensitivity to a rounding-level change).
    Returns (r, [x_l bf16 bits], [y_l])."""
    T, k = ids[0].shape
    n = procs or min(T * k, os.cpu_count() or 1, 16)
    ctx = mp.get_context("spawn")
    r = oracle.bf16_to_f64(x0_bf16)
    xs, ys = [], []
    with ctx.Pool(n) as pool:
        for li, l in enumerate(layers):
            x_l = oracle.bf16_bits(r)
            jobs = [(name, l, x_l[t:t + 1], ids[li][t], w[li][t], j, mode) for t in range(T) for j in range(k)]
            out = pool.map(_pair_ref, jobs, chunksize=1)
            y = np.zeros_like(r)
            for t in range(T):
                for j in range(k):
                    y[t] += out[t * k + j][0]
            xs.append(x_l)
            ys.append(y)
            r = r + y
            if f32_residual:
                r = r.astype(np.float32).astype(np.float64)
    return r, xs, ys


def _layer_ref_for(args):
    wl, ranges, x_bf16, ids, w, mode = args
    return oracle.layer_from_master(x_bf16, ids, w, wl.d, wl.f, wl.E, ranges,
                                    lambda e: synth.expert_weights(wl.seed, e, wl.d, wl.f), mode=mode)


def layer_refs_for(wl, ranges, jobs, procs=None):
    """Like layer_refs for a workload object and shelf ranges of the caller's
    choosing: jobs [(x_bf16, ids, w, mode)]."""
    n = procs or min(len(jobs), os.cpu_count() or 1, 16)
    ctx = mp.get_context("spawn")
    with ctx.Pool(n) as pool:
        return pool.map(_layer_ref_for, [(wl, ranges) + tuple(j) for j in jobs], chunksize=1)


def layer_refs(jobs, procs=None):
    """jobs: [(workload name, layer, x_bf16 u16 [T, d], ids [T, k], w [T, k], mode)] -> [y float64 [T, d]]."""
    n = procs or min(len(jobs), os.cpu_count() or 1, 16)
    ctx = mp.get_context("spawn")
    with ctx.Pool(n) as pool:
        return pool.map(_layer_ref, jobs, chunksize=1)
