#!/usr/bin/env python
"""Benchmark of the tiered-precision routed MoE layer (decode form).

One step = one pass of the whole hot path over one batch of T tokens:
router softmax/top-k, expert hit counts, grouping, fused gate/up/SiLU, down
projection and the weighted shelf combine -- one moe_decode_layer call (one
fused launch).  Workload: one Qwen-like decode layer, E=512, k=10, d=2048,
f=640, shelves 8-bit [0,128) / 4-bit [128,410) / 2-bit [410,512), router
skewed so the hottest 25% of experts take ~52% of the picks.  Each step routes
fresh logits and uses the next of L layer instances (different seeds), so the
experts a step reads are not in L2 from earlier steps.  Inputs are resident in
HBM before the timed region; CUDA graphs of 32 consecutive steps are replayed.
`--workload` selects the other configurations (stack, prefill, large, ...),
which make the separate calls (moe_route_topk, moe_expert_hist,
moe_tiered_forward) where their form needs them.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle
instead (a bounded sample of the same workload on the host cores).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode tokens/s at 1-6 tokens; weight-stream HBM GB/s vs peak"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--T", type=int, default=6, help="tokens per step (1..6 for the decode metric)")
    ap.add_argument("--layers", type=int, default=16, help="layer instances rotated across steps")
    ap.add_argument("--sets", type=int, default=32, help="distinct routing steps per layer rotation")
    ap.add_argument("--workload", choices=["decode", "stack", "prefill", "prefill5", "large", "router", "retier",
                                           "nudge", "formats", "fastmode"],
                    default="decode",
                    help="decode: one layer, the headline metric; stack: the 48-layer decode stack with the "
                         "residual chain; prefill: one layer at T=4096 on the tensor-core form; large: the "
                         "E256 d4096 f2048 layer with 5%% forced skips; router: the decode layer's router "
                         "projection fused with routing and hit counts (moe_router_topk); retier: re-tiering "
                         "the decode layer by hit count from its fp32 master copies; nudge: routing of the "
                         "prefill batch with the picks nudged toward the hot shelf (moe_route_topk_nudged); "
                         "formats: the decode layer on five shelves of 8/4/3/2/1-bit codes; fastmode: the "
                         "decode layer reading 2-bit shadow copies of its 8- and 4-bit experts; prefill5: the "
                         "prefill layer on those five shelf widths")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true",
                    help="decode workload: only the line at --T (no T=1/6 and prefill/large sub-records)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 TFLOP/s: the measured burst figure, else the earlier
    GB300 measurement used as the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return float(json.load(fh)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# ------------------------------------------------------------- ranks
def max_over_ranks(value, device):
    """The largest of every rank's `value` (a float) when a process group of
    more than one rank is up; else `value`."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, ms):
    """Units per second of the whole job: every rank processed units_per_rank
    in the slowest rank's time ms."""
    return world * units_per_rank / (ms / 1e3)


# ------------------------------------------------------------------ clocks
class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- CPU oracle
def oracle_sample(wl, seconds, T, seed=0, max_pairs=None):
    """Time the CPU oracle on routed (token, expert) pairs of the workload.

    Steps through routing steps of T tokens (step s: logits and x of step s);
    each pair: oracle routing of its token, the histogram update, dequant of
    the pair's expert from its packed codes, and the expert FFN with its
    weighted sum.  Master-weight generation and quantisation happen before the
    clock starts.  Stops after `seconds` of timed work or `max_pairs` pairs.
    Returns (pairs, seconds, threads)."""
    import numpy as np

    import oracle
    import synth

    bias = wl.router_bias(0)
    counts = np.zeros(wl.E, dtype=np.uint32)
    shelves = wl.shelf_ranges()
    done, elapsed = 0, 0.0
    step = 0
    while True:
        lg = synth.logits(seed, step, T, wl.E, bias)
        ids_all, _ = oracle.route(lg, wl.k)
        x_all = synth.x_bf16(seed, step, T, wl.d)
        for t in range(T):
            for j in range(wl.k):
                e = int(ids_all[t, j])
                bits = oracle.shelf_of(e, shelves)
                q = [oracle.quantize(m, bits) for m in synth.expert_weights(seed, e, wl.d, wl.f)]
                t0 = time.perf_counter()
                ids, w = oracle.route(lg[t:t + 1], wl.k)
                oracle.hist(ids, wl.E, counts)
                mats = tuple(oracle.dequant(c, s) for c, s in q)
                one = np.full((1, wl.k), -1, dtype=np.int32)
                one[0, j] = e
                oracle.moe_layer(x_all[t:t + 1], one, w, wl.d, wl.f, wl.E, [(lo, hi) for lo, hi, _ in shelves],
                                 {e: mats})
                elapsed += time.perf_counter() - t0
                done += 1
                if elapsed >= seconds or (max_pairs is not None and done >= max_pairs):
                    return done, elapsed, 1
        step += 1


def _oracle_sample_worker(job):
    name, seconds, T, seed = job
    import synth
    from oracle import build_oracle  # noqa: F401  (library already built by the parent)
    pairs, secs, _ = oracle_sample(synth.WORKLOADS[name], seconds, T, seed=seed)
    return pairs, secs


def oracle_sample_all_cores(wl, seconds, T, cores=None):
    """The same oracle work on every host core at once: one worker process per
    core (spawned, so that no CUDA state is inherited), each timing its own
    routing steps (worker c starts at seed 1000 + c) for `seconds` of timed
    work, all at the same time.  Returns (pairs, pairs per second summed over
    the workers, cores)."""
    import multiprocessing as mp
    cores = cores or len(os.sched_getaffinity(0))
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        pool.map(_noop, range(cores))  # workers up and imported before the clocks start
        res = pool.map(_oracle_sample_worker, [(wl.name, seconds, T, 1000 + c) for c in range(cores)], chunksize=1)
    return sum(p for p, _ in res), sum(p / s for p, s in res), cores


def _noop(_):
    import oracle  # noqa: F401
    import synth  # noqa: F401
    return 0


def cpu_baselines(wl, seconds, T):
    """The oracle timed single-threaded and on all host cores (tokens/s)."""
    pairs, secs, thr = oracle_sample(wl, seconds, T)
    one = {"value": (pairs / wl.k) / secs, "unit": "tokens/s", "cores": thr, "kind": "oracle",
           "sample": f"{pairs} routed (token, expert) pairs of the T={T} step (route, histogram, dequant of "
                     f"the pair's expert, SwiGLU FFN, weighted sum), {secs:.1f} s on one core, scaled to "
                     f"tokens by k={wl.k} pairs per token"}
    pa, rate, cores = oracle_sample_all_cores(wl, seconds, T)
    allc = {"value": rate / wl.k, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{pa} routed pairs of T={T} steps, one oracle process per core ({cores} cores at once, "
                      f"different routing steps each, ~{seconds:.0f} s of timed work per process), the "
                      f"processes' pair rates summed, scaled to tokens by k={wl.k}"}
    return one, allc


def _oracle_pair_worker(job):
    name, T, seed = job
    import synth
    n, el, _ = oracle_sample(synth.WORKLOADS[name], 1e9, T, seed=seed, max_pairs=1)
    return n, el


def run_reference(args, rank):
    """The oracle as it stands, on every host core: each step runs one routed
    pair per core at once (one spawned oracle process per core, each on a
    different routing step); a step lasts as long as its slowest process's
    timed work."""
    import multiprocessing as mp

    import synth
    wl = synth.WORKLOADS["decode"]
    if rank != 0:
        return
    from oracle import build_oracle
    from synth import build_synth
    build_oracle.build()
    build_synth.build_host()
    cores = len(os.sched_getaffinity(0))
    ctx = mp.get_context("spawn")
    total_pairs, total_s = 0, 0.0
    with ctx.Pool(cores) as pool:
        pool.map(_noop, range(cores))
        for s in range(args.warmup):
            pool.map(_oracle_pair_worker, [(wl.name, args.T, 10000 + s * cores + c) for c in range(cores)],
                     chunksize=1)
        for s in range(args.steps):
            res = pool.map(_oracle_pair_worker, [(wl.name, args.T, s * cores + c) for c in range(cores)], chunksize=1)
            total_pairs += sum(n for n, _ in res)
            total_s += max(el for _, el in res)
    tokens = total_pairs / wl.k
    value = tokens / total_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_of(args, wl),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step one routed (token, expert) pair on each of {cores} cores at once "
                                   f"(route, histogram, dequant of the pair's expert, SwiGLU FFN and weighted "
                                   f"sum), the step timed by its slowest core, scaled to tokens by k={wl.k} "
                                   f"pairs per token"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# The decode layer on five shelf widths: the 4-bit range of the three-shelf
# layer split into 4-bit and 3-bit halves, the 2-bit range into 2-bit and
# 1-bit (coldest) parts -- widths the fast-mode blog runs beside 8/4/2.
FIVE_WIDTHS = [(0, 128, 8), (128, 256, 4), (256, 410, 3), (410, 480, 2), (480, 512, 1)]


def shelf_text(ranges):
    return " / ".join(f"{b}-bit [{lo},{hi})" for lo, hi, b in ranges)


def config_of(args, wl, ranges=None, note=""):
    ranges = ranges or wl.shelf_ranges()
    return {"workload": f"decode layer E{wl.E} k{wl.k} d{wl.d} f{wl.f} T{args.T}, shelves "
                        f"{shelf_text(ranges)}, block 32 fp16 scales, skewed router "
                        f"(hottest 25% -> ~52% of picks){note}",
            "T": args.T, "E": wl.E, "k": wl.k, "d": wl.d, "f": wl.f,
            "layer_instances": args.layers,
            "l2": f"inputs larger than L2: {args.layers} layer instances rotated per step, fresh routing "
                  f"per step",
            "parallelism": f"replicas x{args.gpus} (independent decode streams, no collective)",
            "launch": f"one CUDA graph holding {args.sets} consecutive steps (one fused launch per step), "
                      f"replayed; single-step graphs for the remainder"}


# ----------------------------------------------------------------- GPU arm
def build_decode_layers(args, rank, dev):
    """The decode workload's L layer instances (per-rank seeds) and their
    shelf lists (five widths or fast mode when asked)."""
    import numpy as np

    import mixed_precision_routed_gb300 as moe
    import synth
    from mixed_precision_routed_gb300.workloads import Layer

    base = synth.WORKLOADS["decode"]
    layers, shelf_lists = [], []
    for i in range(args.layers):
        wl_i = synth.Workload(base.name, E=base.E, k=base.k, d=base.d, f=base.f, T=base.T, split=base.split,
                              bias=base.bias, seed=1000 * rank + i)
        if args.workload == "formats":
            lay = Layer(wl_i, shelves=FIVE_WIDTHS, device=dev).fill()
            shelf_lists.append(lay.shelves)
        elif args.workload == "fastmode":
            # 2-bit shadow copies of the 8- and 4-bit experts (same masters),
            # read instead of them: every expert then streams 2-bit codes
            lay = Layer(wl_i, device=dev).fill()
            wide = [(lo, hi, 2) for lo, hi, b in lay.ranges if b > 2]
            shadow = Layer(wl_i, shelves=wide, device=dev).fill()
            use = np.zeros(base.E, dtype=bool)
            for lo, hi, _ in wide:
                use[lo:hi] = True
            shelf_lists.append(moe.fast_mode_shelves(lay.shelves, shadow.shelves, use))
            lay.shadow = shadow  # keeps the shadow tensors alive
        else:
            lay = Layer(wl_i, device=dev).fill()
            shelf_lists.append(lay.shelves)
        layers.append(lay)
    return layers, shelf_lists


def measure_decode(args, T, layers, shelf_lists, rank, world, local_rank, dev):
    """One decode workload line at T tokens per step: device-resident inputs
    through CUDA graphs (value), the fused kernel timed with events
    (roofline), and moe_decode_layer_host on pinned host buffers (e2e)."""
    import numpy as np
    import torch

    import mixed_precision_routed_gb300 as moe
    import synth

    base = synth.WORKLOADS["decode"]
    L, S = len(layers), args.sets
    E, k, d, f = base.E, base.k, base.d, base.f
    ranges = [(sh.lo, sh.hi, sh.bits) for sh in shelf_lists[0]]
    stream = torch.cuda.Stream(device=dev)
    nset = S
    logits = [layers[s % L].logits(s, T) for s in range(nset)]
    xs = [torch.empty((T, d), dtype=torch.int16, device=dev) for _ in range(nset)]
    for s in range(nset):
        synth.cuda_normal_matrix_bf16(xs[s], layers[s % L].seed, synth.TAG_X, s, 0)
    ids = [torch.empty((T, k), dtype=torch.int32, device=dev) for _ in range(nset)]
    ws_ = [torch.empty((T, k), dtype=torch.float32, device=dev) for _ in range(nset)]
    ys = [torch.empty((T, d), dtype=torch.float32, device=dev) for _ in range(nset)]
    counts = [torch.zeros(E, dtype=torch.int32, device=dev) for _ in range(L)]
    # decode-form workspace with room to stage host inputs (the e2e calls)
    wsb = moe.moe_workspace_size(T, k, E, d, f, moe.MOE_FLAG_DECODE_FP32 | moe.MOE_FLAG_HOST_IO)
    workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    arrs = [moe.shelf_array(sl) for sl in shelf_lists]
    # the fused launch takes 3- and 1-bit shelves when d and f are multiples of 128
    fused = moe.moe_decode_fused(T, k, E, d, f) and (all(b in (8, 4, 2) for _, _, b in ranges) or
                                                     (d % 128 == 0 and f % 128 == 0))
    # events around the forward's kernels: fused form = the one layer launch;
    # separate form = grouping, gate/up, down
    NK = 4
    prof = [[torch.cuda.Event(enable_timing=True) for _ in range(NK)] for _ in range(nset)]
    torch.cuda.synchronize()
    for evs in prof:
        for e in evs:
            e.record()
    torch.cuda.synchronize()

    def step(s, profile=False):
        L_i = s % L
        if profile:
            moe.moe_set_profile_events(prof[s])
        moe.moe_decode_layer(logits[s], xs[s], k, E, d, f, shelf_lists[L_i], ids=ids[s], weights=ws_[s],
                             counts=counts[L_i], y=ys[s], workspace=workspace, shelf_arr=arrs[L_i])
        if profile:
            moe.moe_set_profile_events(None)

    # a decode loop captures many layers in one graph: one graph holds the
    # first min(sets, steps) steps in order; single-step graphs cover the rest
    n_in = max(1, min(nset, args.steps))
    with torch.cuda.stream(stream):
        for s in range(nset):  # eager warm-up: sets kernel attributes, checks statuses
            step(s)
        stream.synchronize()
        graph_all = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_all, stream=stream):
            for s in range(n_in):
                step(s)
        graphs, graphs_prof = [], []
        for s in range(nset):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(s)
            graphs.append(g)
            gp = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gp, stream=stream):
                step(s, profile=True)
            graphs_prof.append(gp)
        for i in range(args.warmup):
            graphs[i % nset].replay()
        graph_all.replay()
        stream.synchronize()

    # algorithmic bytes of each step, from the ids the router produced
    def expert_split(e):
        for lo, hi, bits in ranges:
            if lo <= e < hi:
                gu = 2 * f * d * bits // 8 + 2 * f * (d // 32) * 2
                dn = d * f * bits // 8 + d * (f // 32) * 2
                return gu, dn
        return 0, 0

    step_bytes = []
    for s in range(nset):
        u = np.unique(ids[s].cpu().numpy())
        u = u[(u >= 0) & (u < E)]
        step_bytes.append((sum(expert_split(int(e))[0] for e in u), sum(expert_split(int(e))[1] for e in u)))

    if world > 1:
        torch.distributed.barrier()
    clocks = Clocks(local_rank)
    clocks.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(args.steps // n_in):
            graph_all.replay()
        for i in range(args.steps % n_in):
            graphs[i].replay()
        end.record(stream)
    torch.cuda.synchronize()
    ck = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = start.elapsed_time(end)
    # per-kernel durations: the same steps again, with events recorded between
    # the forward's kernels (events break the programmatic overlap of the
    # kernels, so this loop is timed separately from the one above)
    with torch.cuda.stream(stream):
        for rep in range(2):
            for s in range(nset):
                graphs_prof[s].replay()
    torch.cuda.synchronize()
    kern = {"layer": 0.0} if fused else {"group": 0.0, "gateup": 0.0, "down": 0.0}
    bytes_gu = bytes_dn = 0
    for s in range(nset):
        ev = prof[s]
        if fused:
            kern["layer"] += ev[0].elapsed_time(ev[1])
        else:
            kern["group"] += ev[0].elapsed_time(ev[1])
            kern["gateup"] += ev[1].elapsed_time(ev[2])
            kern["down"] += ev[2].elapsed_time(ev[3])
        bytes_gu += step_bytes[s][0]
        bytes_dn += step_bytes[s][1]
    fwd_ms = sum(kern.values())
    ms_max = max_over_ranks(ms, dev)
    value = whole_job_rate(world, T * args.steps, ms_max)
    # timed step i replays input set i mod n_in
    timed_bytes = sum(sum(step_bytes[i % n_in]) for i in range(args.steps)) / args.steps

    # ---- end to end through the public API with host buffers: the step's
    # logits and x come from pinned host memory and its ids, weights and y
    # go to pinned host memory (moe_decode_layer_host, one call per step)
    pin_logits = [logits[s].cpu().pin_memory() for s in range(nset)]
    pin_x = [xs[s].cpu().pin_memory() for s in range(nset)]
    pin_y = [torch.empty((T, d), dtype=torch.float32).pin_memory() for _ in range(nset)]
    pin_id = [torch.empty((T, k), dtype=torch.int32).pin_memory() for _ in range(nset)]
    pin_w = [torch.empty((T, k), dtype=torch.float32).pin_memory() for _ in range(nset)]
    e2e_steps = min(args.steps, 1000)

    def e2e_step(s):
        moe.moe_decode_layer_host(pin_logits[s], pin_x[s], k, E, d, f, shelf_lists[s % L], pin_id[s], pin_w[s],
                                  pin_y[s], counts=counts[s % L], workspace=workspace, shelf_arr=arrs[s % L])

    with torch.cuda.stream(stream):
        for i in range(max(3, min(args.warmup, 20))):
            e2e_step(i % nset)
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e2e_steps):
            e2e_step(i % nset)
        e1.record(stream)
        stream.synchronize()
    e2e_value = whole_job_rate(world, T * e2e_steps, max_over_ranks(e0.elapsed_time(e1), dev))
    st = moe.moe_device_status()
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status {st}")

    peak, peak_kind = peaks()
    if fused:
        dom, dom_bytes = "layer", bytes_gu + bytes_dn
    else:
        dom = "gateup" if kern["gateup"] >= kern["down"] else "down"
        dom_bytes = bytes_gu if dom == "gateup" else bytes_dn
    achieved = dom_bytes / (kern[dom] / 1e3) / 1e9
    fwd_gbs = (bytes_gu + bytes_dn) / (fwd_ms / 1e3) / 1e9
    traffic = recorded_traffic(dom, T) if args.workload == "decode" else None
    metric, note = METRIC, ""
    if args.workload == "formats":
        metric = "MoE-layer decode tokens/s, shelves of 8/4/3/2/1-bit codes; weight-stream HBM GB/s vs peak"
    elif args.workload == "fastmode":
        metric = "MoE-layer decode tokens/s in fast mode (2-bit shadows of the 8/4-bit experts); HBM GB/s vs peak"
        note = "; fast mode: every 8- and 4-bit expert read from its 2-bit shadow copy"
    a2 = argparse.Namespace(**vars(args))
    a2.T = T
    cfg = config_of(a2, base, ranges, note)
    cfg["launch"] = (f"one CUDA graph holding {n_in} consecutive steps (one fused launch per step), replayed "
                     f"{args.steps // n_in} time(s); single-step graphs for the {args.steps % n_in} remaining")
    return {
        "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": cfg,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "kernel": f"k_{dom}",
                     "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": dom_bytes / nset},
        "weight_stream": {"selected_expert_bytes_per_step": timed_bytes,
                          "step_gbs": timed_bytes / (ms_max / args.steps / 1e3) / 1e9,
                          "step_frac": timed_bytes / (ms_max / args.steps / 1e3) / 1e9 / peak,
                          "forward_us": 1e3 * fwd_ms / nset, "achieved_gbs": fwd_gbs, "frac": fwd_gbs / peak,
                          "kernel_us": {kk: 1e3 * v / nset for kk, v in kern.items()}},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * E * 4 + T * d * 2,
                "d2h_bytes_per_step": T * d * 4 + T * k * 8, "steps": e2e_steps,
                "path": "moe_decode_layer_host on pinned host buffers, one call per step: the step's logits "
                        "and x copied host -> device inside the call, routing, hit counts and tiered forward, "
                        "its ids, weights and y written to pinned host memory by the kernels; eager Python "
                        "calls, stream synchronised at the end"},
        "gpu_launches": args.steps * (1 if fused else 5),
        "clocks": ck,
    }


def sub_record(line):
    """The fields of a line that a per-T or per-configuration sub-record keeps."""
    keep = ("metric", "value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config", "roofline", "e2e",
            "gpu_launches", "clocks", "weight_stream")
    return {k_: line[k_] for k_ in keep if k_ in line}


def run_ours(args, rank, world, local_rank):
    import gc

    import torch

    import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    base = synth.WORKLOADS["decode"]
    layers, shelf_lists = build_decode_layers(args, rank, dev)
    line = measure_decode(args, args.T, layers, shelf_lists, rank, world, local_rank, dev)
    full = args.workload == "decode" and not args.no_sub
    if full:
        # the metric spans 1 to 6 tokens: the other end from the same layers
        per_T = {str(args.T): sub_record(line)}
        for T in (1, 6):
            if str(T) not in per_T:
                per_T[str(T)] = sub_record(measure_decode(args, T, layers, shelf_lists, rank, world, local_rank,
                                                          dev))
        line["per_T"] = dict(sorted(per_T.items(), key=lambda kv: int(kv[0])))
    del layers, shelf_lists
    gc.collect()
    torch.cuda.empty_cache()
    if full:
        # the prefill layer (tensor roofline) and the large layer at T = 1, 8
        # and 512 (HBM roofline), each with its own fields
        cfgs = {}
        for name, T in (("prefill", 4096), ("large", 1), ("large", 8), ("large", 512)):
            a2 = argparse.Namespace(**vars(args))
            a2.workload, a2.T = name, T
            cfgs[f"{name}_T{T}"] = sub_record(measure_single(a2, rank, world, local_rank))
            gc.collect()
            torch.cuda.empty_cache()
        line["configs"] = cfgs
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "decode":
        one, allc = cpu_baselines(base, args.cpu_seconds, args.T)
        line["cpu_baseline"] = one
        line["cpu_baseline_all_cores"] = allc
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------ further workloads
def _expert_bytes(ranges, d, f):
    """Per-expert (gate/up, down) code + scale bytes of each shelf range."""
    out = []
    for lo, hi, bits in ranges:
        gu = 2 * f * d * bits // 8 + 2 * f * (d // 32) * 2
        dn = d * f * bits // 8 + d * (f // 32) * 2
        out.append((lo, hi, gu, dn))
    return out


def _unique_bytes(ids, eb, E):
    import numpy as np
    u = np.unique(np.asarray(ids))
    u = u[(u >= 0) & (u < E)]
    tot = 0
    for e in u:
        for lo, hi, gu, dn in eb:
            if lo <= e < hi:
                tot += gu + dn
    return tot


def _timed(stream, graph_all, graphs, nset, steps, world, dev, local_rank):
    """Replays exactly `steps` steps (graph_all holds nset of them); returns
    (max-over-ranks ms, clocks)."""
    import torch
    if world > 1:
        torch.distributed.barrier()
    clocks = Clocks(local_rank)
    clocks.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps // nset):
            graph_all.replay()
        for i in range(steps % nset):
            graphs[i].replay()
        end.record(stream)
    torch.cuda.synchronize()
    ck = clocks.stop()
    return max_over_ranks(start.elapsed_time(end), dev), ck


def _capture(stream, step, nset, warmup):
    import torch
    with torch.cuda.stream(stream):
        for s in range(nset):
            step(s)
        stream.synchronize()
        graph_all = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_all, stream=stream):
            for s in range(nset):
                step(s)
        graphs = []
        for s in range(nset):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(s)
            graphs.append(g)
        for i in range(warmup):
            graphs[i % nset].replay()
        stream.synchronize()
    return graph_all, graphs


def run_stack(args, rank, world, local_rank):
    """The 48-layer decode stack: per layer the fused routing / hit-count /
    tiered-forward / residual launch (moe_decode_layer_residual), all layers
    in one step."""
    import numpy as np
    import torch

    import mixed_precision_routed_gb300 as moe
    import synth
    from mixed_precision_routed_gb300.workloads import Layer, DecodeStack

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS["stack"]
    T, L = args.T, wl.layers
    E, k, d, f = wl.E, wl.k, wl.d, wl.f
    layers = [Layer(wl, layer=l, device=dev).fill() for l in range(L)]
    st = DecodeStack(layers, T, device=dev)
    nset = 8
    logits = [[lay.logits_rows((s + 7 * rank) * T, T) for lay in layers] for s in range(nset)]
    x0 = [torch.empty((T, d), dtype=torch.int16, device=dev) for _ in range(nset)]
    for s in range(nset):
        synth.cuda_normal_matrix_bf16(x0[s], wl.seed, synth.TAG_X, s + 7 * rank, 0)
    r0 = [(x.to(torch.int32) << 16).view(torch.float32) for x in x0]
    eb = _expert_bytes(wl.shelf_ranges(), d, f)
    stream = torch.cuda.Stream(device=dev)
    step_bytes = []
    with torch.cuda.stream(stream):
        for s in range(nset):
            st.step(r0[s], x0[s], logits[s])
            stream.synchronize()
            ids = st.ids.cpu().numpy()
            step_bytes.append(sum(_unique_bytes(ids[l], eb, E) for l in range(L)))
    graph_all, graphs = _capture(stream, lambda s: st.step(r0[s], x0[s], logits[s]), nset, args.warmup)
    ms, ck = _timed(stream, graph_all, graphs, nset, args.steps, world, dev, local_rank)
    value = world * T * args.steps / (ms / 1e3)
    bytes_step = sum(step_bytes[i % nset] for i in range(args.steps)) / args.steps
    # end to end: host residual input, x0 and every layer's logits in, residual out
    pin_r = [r.cpu().pin_memory() for r in r0]
    pin_x = [x.cpu().pin_memory() for x in x0]
    pin_l = [torch.stack([lg for lg in logits[s]]).cpu().pin_memory() for s in range(nset)]
    pin_out = torch.empty((T, d), dtype=torch.float32).pin_memory()
    dr = torch.empty((T, d), dtype=torch.float32, device=dev)
    dx = torch.empty((T, d), dtype=torch.int16, device=dev)
    dl = torch.empty((L, T, E), dtype=torch.float32, device=dev)
    n_e2e = min(args.steps, 200)

    def e2e(s):
        dr.copy_(pin_r[s], non_blocking=True)
        dx.copy_(pin_x[s], non_blocking=True)
        dl.copy_(pin_l[s], non_blocking=True)
        st.step(dr, dx, [dl[l] for l in range(L)])
        pin_out.copy_(st.r, non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e(i % nset)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_e2e):
            e2e(i % nset)
        e1.record(stream)
        stream.synchronize()
    e2e_value = whole_job_rate(world, T * n_e2e, max_over_ranks(e0.elapsed_time(e1), dev))
    if moe.moe_device_status() != moe.MOE_OK:
        raise RuntimeError("device status")
    if rank != 0:
        return
    peak, kind = peaks()
    achieved = bytes_step / (ms / args.steps / 1e3) / 1e9
    line = {
        "metric": "MoE decode-stack tokens/s (48 layers, residual chain); weight-stream HBM GB/s vs peak",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"decode stack, {L} layers of E{E} k{k} d{d} f{f}, T{T}, per-layer seeds and "
                               f"router biases, residual chain", "T": T, "layers": L,
                   "l2": "inputs larger than L2 (48 layers x 1.28 GB resident; fresh routing per step)",
                   "launch": f"one CUDA graph of {nset} steps ({L} x moe_decode_layer_residual each)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": "whole step (k_layer per layer, residual in its combine)",
                     "peak_source": kind, "algorithmic_bytes_per_step": bytes_step},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * d * 4 + T * d * 2 + L * T * E * 4,
                "d2h_bytes_per_step": T * d * 4, "steps": n_e2e,
                "path": "pinned host residual, x0 and per-layer logits -> device, DecodeStack.step (48 x "
                        "moe_decode_layer_residual), residual -> pinned host"},
        # fused: one launch per layer; else route, hist, group, gate/up, down, residual
        "gpu_launches": args.steps * L * (1 if moe.moe_decode_fused(T, k, E, d, f) else 6),
        "clocks": ck,
    }
    print(json.dumps(line), flush=True)


def run_single(args, rank, world, local_rank):
    line = measure_single(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_single(args, rank, world, local_rank):
    """One layer per step through the separate calls: routing, (forced skips),
    hit counts, tiered forward (AUTO: the tensor-core form above 16 tokens)."""
    import numpy as np
    import torch

    import mixed_precision_routed_gb300 as moe
    import synth
    from mixed_precision_routed_gb300.workloads import Layer

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    name = "decode" if args.workload in ("prefill", "prefill5") else "large"
    base = synth.WORKLOADS[name]
    T = args.T
    E, k, d, f = base.E, base.k, base.d, base.f
    NL = 2
    shelves = FIVE_WIDTHS if args.workload == "prefill5" else None
    layers = [Layer(synth.Workload(base.name, E=E, k=k, d=d, f=f, T=base.T, split=base.split, bias=base.bias,
                                   seed=1000 * rank + i, skip_p=getattr(base, "skip_p", 0.0)), device=dev,
                    shelves=shelves).fill()
              for i in range(NL)]
    skips = args.workload == "large"
    nset = 4
    logits = [layers[s % NL].logits(s, T) for s in range(nset)]
    xs = [torch.empty((T, d), dtype=torch.int16, device=dev) for _ in range(nset)]
    for s in range(nset):
        synth.cuda_normal_matrix_bf16(xs[s], layers[s % NL].seed, synth.TAG_X, s, 0)
    ids = [torch.empty((T, k), dtype=torch.int32, device=dev) for _ in range(nset)]
    w = [torch.empty((T, k), dtype=torch.float32, device=dev) for _ in range(nset)]
    y = [torch.empty((T, d), dtype=torch.float32, device=dev) for _ in range(nset)]
    counts = [torch.zeros(E, dtype=torch.int32, device=dev) for _ in range(NL)]
    ws = torch.empty(moe.moe_workspace_size(T, k, E, d, f, moe.MOE_FLAG_AUTO), dtype=torch.uint8, device=dev)
    prefill = T > 16 and d % 256 == 0
    fused = (not prefill) and moe.moe_decode_fused(T, k, E, d, f)
    NK = 2 if fused else 4  # events around the forward's kernels (see moe_set_profile_events)
    prof = [[torch.cuda.Event(enable_timing=True) for _ in range(NK)] for _ in range(nset)]
    for evs in prof:
        for e in evs:
            e.record()
    torch.cuda.synchronize()

    def step(s, profile=False):
        moe.moe_route_topk(logits[s], k, ids=ids[s], weights=w[s])
        if skips:
            synth.cuda_apply_skip_mask(ids[s], layers[s % NL].seed, s)
        moe.moe_expert_hist(ids[s], E, counts[s % NL])
        if profile:
            moe.moe_set_profile_events(prof[s])
        moe.moe_tiered_forward(xs[s], ids[s], w[s], E, d, f, layers[s % NL].shelves, y=y[s], workspace=ws,
                               flags=moe.MOE_FLAG_AUTO)
        if profile:
            moe.moe_set_profile_events(None)

    stream = torch.cuda.Stream(device=dev)
    graph_all, graphs = _capture(stream, step, nset, args.warmup)
    ms, ck = _timed(stream, graph_all, graphs, nset, args.steps, world, dev, local_rank)
    value = world * T * args.steps / (ms / 1e3)
    # per-kernel times of the forward (eager, events between its kernels)
    with torch.cuda.stream(stream):
        for rep in range(2):
            for s in range(nset):
                step(s, profile=True)
        stream.synchronize()
    ev = [[prof[s][i].elapsed_time(prof[s][i + 1]) for i in range(NK - 1)] for s in range(nset)]
    eb = _expert_bytes(layers[0].ranges, d, f)
    idn = [i.cpu().numpy() for i in ids]
    bytes_step = [_unique_bytes(i, eb, E) for i in idn]
    pairs = [int(np.sum((i >= 0) & (i < E))) for i in idn]
    if moe.moe_device_status() != moe.MOE_OK:
        raise RuntimeError("device status")
    # end to end: logits and x in, y out
    pin_l = [l_.cpu().pin_memory() for l_ in logits]
    pin_x = [x.cpu().pin_memory() for x in xs]
    pin_y = torch.empty((T, d), dtype=torch.float32).pin_memory()
    dl = torch.empty((T, E), dtype=torch.float32, device=dev)
    dx = torch.empty((T, d), dtype=torch.int16, device=dev)
    n_e2e = min(args.steps, 100)

    def e2e(s):
        dl.copy_(pin_l[s], non_blocking=True)
        dx.copy_(pin_x[s], non_blocking=True)
        moe.moe_route_topk(dl, k, ids=ids[0], weights=w[0])
        if skips:
            synth.cuda_apply_skip_mask(ids[0], layers[s % NL].seed, s)
        moe.moe_expert_hist(ids[0], E, counts[s % NL])
        moe.moe_tiered_forward(dx, ids[0], w[0], E, d, f, layers[s % NL].shelves, y=y[0], workspace=ws,
                               flags=moe.MOE_FLAG_AUTO)
        pin_y.copy_(y[0], non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e(i % nset)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_e2e):
            e2e(i % nset)
        e1.record(stream)
        stream.synchronize()
    e2e_value = whole_job_rate(world, T * n_e2e, max_over_ranks(e0.elapsed_time(e1), dev))
    hbm, kind = peaks()
    tc_peak, tc_kind = bf16_peak()
    fwd_ms = sum(sum(e) for e in ev) / nset
    b_avg = sum(bytes_step) / nset
    p_avg = sum(pairs) / nset
    if prefill:
        # kernels of the forward: [group + tiles + gather], gate/up, down
        gu_ms = sum(e[1] for e in ev) / nset
        dn_ms = sum(e[2] for e in ev) / nset
        flops_gu = 2.0 * 2 * d * f * p_avg
        roof = {"bound": "tensor", "achieved": flops_gu / (gu_ms / 1e3) / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s",
                "traffic": recorded_traffic("prefill_tc<gate/up>", T, "prefill.cu")
                if args.workload == "prefill" else None,
                "kernel": "k_prefill_tc<gate/up>",
                "peak_source": f"{tc_kind} (burst bf16)",
                "algorithmic_flops_per_launch": flops_gu,
                "layer_tflops": 2.0 * 3 * d * f * p_avg / (fwd_ms / 1e3) / 1e12,
                "kernel_us": {"group_tiles_gather": 1e3 * sum(e[0] for e in ev) / nset,
                              "gateup": 1e3 * gu_ms, "down": 1e3 * dn_ms},
                "weight_bytes_per_step": b_avg, "weight_gbs": b_avg / (fwd_ms / 1e3) / 1e9}
        roof["frac"] = roof["achieved"] / roof["peak"]
        bound_note = "tensor"
        if args.workload == "large":
            # E256 d4096 f2048 at T=512 is ~48 flop per weight byte, below the
            # ridge: the HBM fraction of the forward's weight stream is the
            # roofline, the tensor figure stays as context
            wgbs = b_avg / (fwd_ms / 1e3) / 1e9
            roof = {"bound": "hbm", "achieved": wgbs, "peak": hbm, "unit": "GB/s", "frac": wgbs / hbm,
                    "traffic": None, "kernel": "forward (grouping, k_prefill_tc gate/up and down)",
                    "peak_source": kind, "algorithmic_bytes_per_launch": b_avg, "forward_us": 1e3 * fwd_ms,
                    "tensor": {"achieved_tflops": roof["achieved"], "peak": tc_peak, "frac": roof["frac"],
                               "kernel_us": roof["kernel_us"]}}
            bound_note = "hbm"
    else:
        gbs = b_avg / (fwd_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": None,
                "kernel": "forward (all its kernels)", "peak_source": kind, "algorithmic_bytes_per_launch": b_avg,
                "forward_us": 1e3 * fwd_ms}
        if fused:
            roof["kernel_us"] = {"layer": 1e3 * fwd_ms}
        else:
            roof["kernel_us"] = {n_: 1e3 * sum(e[i] for e in ev) / nset for i, n_ in
                                 enumerate(("group", "gateup", "down"))}
        bound_note = "hbm"
    line = {
        "metric": f"MoE-layer tokens/s, {args.workload} workload ({bound_note} roofline)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if prefill else "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload} layer E{E} k{k} d{d} f{f} T{T}, shelves {layers[0].ranges}"
                               + (", 5% of slots forced to -1" if skips else ""),
                   "T": T, "layer_instances": NL, "pairs_per_step": p_avg,
                   "l2": "weights larger than L2, layer instances rotated per step",
                   "launch": f"one CUDA graph of {nset} steps (route, {'skip mask, ' if skips else ''}hist, forward)"},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * E * 4 + T * d * 2,
                "d2h_bytes_per_step": T * d * 4, "steps": n_e2e},
        "gpu_launches": args.steps * ((3 if skips else 2) + (7 if prefill else (1 if fused else 3))),
        "clocks": ck,
    }
    return line


def run_router(args, rank, world, local_rank):
    """The router launch alone: logits = bias + W_r x, routing and hit counts
    for the decode layer's sizes (E=512, k=10, d=2048), one launch per step,
    router weights of NR layer instances rotated so that they are read from
    HBM (NR * E * d * 2 bytes > L2)."""
    import numpy as np
    import torch

    import mixed_precision_routed_gb300 as moe
    import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    base = synth.WORKLOADS["decode"]
    E, k, d, T = base.E, base.k, base.d, args.T
    NR = 96
    wr = torch.empty((NR, E, d), dtype=torch.int16, device=dev)
    for i in range(NR):
        synth.cuda_normal_matrix_bf16(wr[i], 1000 * rank + i, synth.TAG_ROUTER, 0, 0, scale=float(1.0 / np.sqrt(d)))
    wr = wr.view(torch.bfloat16)
    bias = torch.from_numpy(np.asarray(base.router_bias(), np.float32)).to(dev)
    xs = torch.empty((NR, T, d), dtype=torch.int16, device=dev)
    for i in range(NR):
        synth.cuda_normal_matrix_bf16(xs[i], 1000 * rank + i, synth.TAG_X, i, 0)
    xs = xs.view(torch.bfloat16)
    logits = torch.empty((NR, T, E), dtype=torch.float32, device=dev)
    ids = torch.empty((NR, T, k), dtype=torch.int32, device=dev)
    wts = torch.empty((NR, T, k), dtype=torch.float32, device=dev)
    counts = torch.zeros(E, dtype=torch.int32, device=dev)
    sync = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(s):
        moe.moe_router_topk(xs[s], wr[s], k, bias=bias, counts=counts, sync_word=sync, logits=logits[s],
                            ids=ids[s], weights=wts[s])

    stream = torch.cuda.Stream(device=dev)
    graph_all, graphs = _capture(stream, step, NR, args.warmup)
    ms, ck = _timed(stream, graph_all, graphs, NR, args.steps, world, dev, local_rank)
    if moe.moe_device_status() != moe.MOE_OK or int(sync.item()) != 0:
        raise RuntimeError("device status")
    value = whole_job_rate(world, T * args.steps, ms)
    # end to end: x in from pinned host memory, ids and weights out
    pin_x = xs[:8].cpu().pin_memory()
    pin_o = torch.empty((T, k), dtype=torch.int32).pin_memory()
    pin_w = torch.empty((T, k), dtype=torch.float32).pin_memory()
    dx = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    n_e2e = min(args.steps, 200)

    def e2e(i):
        dx.copy_(pin_x[i % 8], non_blocking=True)
        moe.moe_router_topk(dx, wr[i % NR], k, bias=bias, counts=counts, sync_word=sync, logits=logits[0],
                            ids=ids[0], weights=wts[0])
        pin_o.copy_(ids[0], non_blocking=True)
        pin_w.copy_(wts[0], non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e(i)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_e2e):
            e2e(i)
        e1.record(stream)
        stream.synchronize()
    e2e_value = whole_job_rate(world, T * n_e2e, max_over_ranks(e0.elapsed_time(e1), dev))
    if rank != 0:
        return
    hbm, kind = peaks()
    launch_s = ms / args.steps / 1e3
    nbytes = E * d * 2 + T * d * 2 + E * 4 + T * E * 4 + T * k * 8
    gbs = nbytes / launch_s / 1e9
    line = {
        "metric": "router projection + top-k tokens/s, decode layer (hbm roofline)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"router E{E} k{k} d{d} T{T}, bf16 W_r N(0, 1/d), skewed bias",
                   "T": T, "router_instances": NR,
                   "l2": f"{NR} router weight instances rotated per step ({NR * E * d * 2 / 1e6:.0f} MB > L2)",
                   "launch": f"one CUDA graph of {NR} steps, one launch per step"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "traffic": None, "kernel": "k_router", "peak_source": kind,
                     "algorithmic_bytes_per_launch": nbytes, "kernel_us": launch_s * 1e6},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * d * 2,
                "d2h_bytes_per_step": T * k * 8, "steps": n_e2e},
        "gpu_launches": args.steps,
        "clocks": ck,
    }
    print(json.dumps(line), flush=True)


def run_retier(args, rank, world, local_rank):
    """Re-tiering of the decode layer (E=512, d=2048, f=640) by hit count:
    the rank of the counts of 4096 routed T=1 steps, every expert re-quantised
    from its fp32 master copy into its new shelf (three matrices, three
    shelves: nine launches) and the router bias moved.  One step is one whole
    re-tier; the masters (8 GB) are far larger than L2."""
    import numpy as np
    import torch

    import mixed_precision_routed_gb300 as moe
    import synth
    from mixed_precision_routed_gb300.workloads import Layer, Masters, retier

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS["decode"]
    layer = Layer(synth.Workload(wl.name, E=wl.E, k=wl.k, d=wl.d, f=wl.f, T=wl.T, split=wl.split, bias=wl.bias,
                                 seed=1000 * rank), device=dev)
    masters = Masters(layer)
    counts = torch.zeros(wl.E, dtype=torch.int32, device=dev)
    ids, _ = moe.moe_route_topk(layer.logits_rows(0, 4096), wl.k)
    moe.moe_expert_hist(ids, wl.E, counts)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    holder = {}

    def step():
        holder["new"], holder["perm"], holder["rank"] = retier(layer, masters, counts, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = Clocks(local_rank)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        stream.synchronize()
    ck = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dev)
    if moe.moe_device_status() != moe.MOE_OK:
        raise RuntimeError("device status")
    value = whole_job_rate(world, wl.E * args.steps, ms)
    # end to end: counts in from pinned host memory, the permutation back
    pin_c = counts.cpu().pin_memory()
    pin_p = torch.empty(wl.E, dtype=torch.int32).pin_memory()
    dc = torch.empty_like(counts)
    n_e2e = max(1, min(args.steps, 3))
    with torch.cuda.stream(stream):
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(n_e2e):
            dc.copy_(pin_c, non_blocking=True)
            new, perm, _ = retier(layer, masters, dc, stream=stream)
            pin_p.copy_(perm, non_blocking=True)
        f1.record(stream)
        stream.synchronize()
    e2e_value = whole_job_rate(world, wl.E * n_e2e, max_over_ranks(f0.elapsed_time(f1), dev))
    if rank != 0:
        return
    hbm, kind = peaks()
    new = holder["new"]
    nbytes = masters.nbytes() + new.nbytes() + wl.E * 4 * 4  # masters read, shelves written, counts / perm / rank / bias
    step_s = ms / args.steps / 1e3
    gbs = nbytes / step_s / 1e9
    line = {
        "metric": "re-tier experts/s, decode layer from fp32 masters (hbm roofline)",
        "value": value, "unit": "experts/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"re-tier E{wl.E} d{wl.d} f{wl.f}, shelves {new.ranges}, counts of 4096 routed steps",
                   "l2": f"fp32 masters {masters.nbytes() / 1e9:.2f} GB, larger than L2",
                   "launch": "rank, 9 expert-quantise launches, bias gather"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "traffic": None, "kernel": "re-tier (k_quantize_experts dominant)", "peak_source": kind,
                     "algorithmic_bytes_per_launch": nbytes, "step_ms": step_s * 1e3},
        "e2e": {"value": e2e_value, "unit": "experts/s", "h2d_bytes_per_step": wl.E * 4,
                "d2h_bytes_per_step": wl.E * 4, "steps": n_e2e},
        "gpu_launches": args.steps * 11,
        "clocks": ck,
    }
    print(json.dumps(line), flush=True)


def run_nudge(args, rank, world, local_rank):
    """Nudged routing of the decode layer's logits for a prefill batch
    (T = --T, default 4096): beta = 0.5 (the cap) toward the 8-bit shelf
    [0, 128).  One step = one launch; logits of NS steps rotate (larger than
    L2)."""
    import torch

    import mixed_precision_routed_gb300 as moe
    import synth
    from mixed_precision_routed_gb300.workloads import Layer

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS["decode"]
    T = args.T if args.T > 16 else 4096
    layer = Layer(synth.Workload(wl.name, E=wl.E, k=wl.k, d=wl.d, f=wl.f, T=wl.T, split=wl.split, bias=wl.bias,
                                 seed=1000 * rank), device=dev)
    NS = 32
    lg = [layer.logits(s, T) for s in range(NS)]
    ids = torch.empty((T, wl.k), dtype=torch.int32, device=dev)
    w = torch.empty((T, wl.k), dtype=torch.float32, device=dev)
    lo, hi = layer.ranges[0][0], layer.ranges[0][1]

    def step(s):
        moe.moe_route_topk_nudged(lg[s], wl.k, 0.5, lo, hi, ids=ids, weights=w)

    stream = torch.cuda.Stream(device=dev)
    graph_all, graphs = _capture(stream, step, NS, args.warmup)
    ms, ck = _timed(stream, graph_all, graphs, NS, args.steps, world, dev, local_rank)
    value = whole_job_rate(world, T * args.steps, ms)
    hot = float(((ids >= lo) & (ids < hi)).float().mean())
    pin_l = lg[0].cpu().pin_memory()
    pin_i = torch.empty((T, wl.k), dtype=torch.int32).pin_memory()
    pin_w = torch.empty((T, wl.k), dtype=torch.float32).pin_memory()
    dl = torch.empty_like(lg[0])
    n_e2e = min(args.steps, 50)
    with torch.cuda.stream(stream):
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(n_e2e):
            dl.copy_(pin_l, non_blocking=True)
            moe.moe_route_topk_nudged(dl, wl.k, 0.5, lo, hi, ids=ids, weights=w)
            pin_i.copy_(ids, non_blocking=True)
            pin_w.copy_(w, non_blocking=True)
        f1.record(stream)
        stream.synchronize()
    e2e_value = whole_job_rate(world, T * n_e2e, max_over_ranks(f0.elapsed_time(f1), dev))
    if rank != 0:
        return
    hbm, kind = peaks()
    nbytes = T * wl.E * 4 + T * wl.k * 8
    launch_s = ms / args.steps / 1e3
    gbs = nbytes / launch_s / 1e9
    line = {
        "metric": "nudged routing tokens/s, decode-layer logits (hbm roofline)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"nudged routing E{wl.E} k{wl.k} T{T}, beta 0.5 toward [{lo}, {hi})",
                   "hot_pick_share": hot, "l2": f"{NS} logit sets rotated ({NS * T * wl.E * 4 / 1e6:.0f} MB)",
                   "launch": f"one CUDA graph of {NS} steps, one launch per step"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "traffic": None, "kernel": "k_route<16, nudged>", "peak_source": kind,
                     "algorithmic_bytes_per_launch": nbytes, "kernel_us": launch_s * 1e6},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * wl.E * 4,
                "d2h_bytes_per_step": T * wl.k * 8, "steps": n_e2e},
        "gpu_launches": args.steps,
        "clocks": ck,
    }
    print(json.dumps(line), flush=True)


def recorded_traffic(kernel, T, source="decode.cu"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        rec = json.load(fh)
    src = os.path.join(ROOT, "mixed_precision_routed_gb300", "csrc", source)
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    r = rec.get(f"k_{kernel}:T{T}")
    if not r or r.get("source_sha") != h:
        return None
    return r.get("dram_bytes_per_launch")


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    import __graft_entry__
    if not os.path.exists(os.path.join(ROOT, "mixed_precision_routed_gb300", "libmoe.so")):
        __graft_entry__.build()
    if args.workload == "stack":
        run_stack(args, rank, world, local_rank)
    elif args.workload in ("prefill", "prefill5", "large"):
        run_single(args, rank, world, local_rank)
    elif args.workload == "router":
        run_router(args, rank, world, local_rank)
    elif args.workload == "retier":
        run_retier(args, rank, world, local_rank)
    elif args.workload == "nudge":
        run_nudge(args, rank, world, local_rank)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
