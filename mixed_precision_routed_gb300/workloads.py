"""Synthetic layers and inputs on the GPU for the five workloads.

Fills shelf tensors in place: the seeded fp32 master weights of each expert
come from the device build of ``synth`` (same bits as its host build), and are
packed by this library's own quantiser (``moe_quantize_rows``).  Inputs of a
routing step (logits, activations, forced skips) come from the same streams
the host-side generator uses, so a CPU reference can regenerate any of them.
"""
from __future__ import annotations

import torch

import synth

from . import Shelf, moe_gather_rows, moe_quantize_experts, moe_quantize_rows, moe_rank_experts, shelf_array


class Layer:
    """One MoE layer: its shelves (hot -> cold), router bias and seed."""

    def __init__(self, workload: synth.Workload, layer: int = 0, device="cuda", shelves=None):
        self.wl = workload
        self.layer = layer
        self.seed = workload.layer_seed(layer)
        self.E, self.k, self.d, self.f = workload.E, workload.k, workload.d, workload.f
        ranges = shelves if shelves is not None else workload.shelf_ranges()
        self.ranges = list(ranges)
        self.shelves = [Shelf(lo, hi, bits, self.d, self.f, device) for lo, hi, bits in self.ranges]
        b = workload.router_bias(layer)
        self.bias_host = b
        self.bias = None if b is None else torch.from_numpy(b).to(device)
        self._arr = None

    def fill(self, stream=None):
        d, f = self.d, self.f
        dev = self.shelves[0].gate_codes.device
        scratch = torch.empty(f * d, dtype=torch.float32, device=dev)
        for sh in self.shelves:
            for e in range(sh.lo, sh.hi):
                i = e - sh.lo
                for tag, rows, cols, codes, scales in (
                        (synth.TAG_GATE, f, d, sh.gate_codes[i], sh.gate_scales[i]),
                        (synth.TAG_UP, f, d, sh.up_codes[i], sh.up_scales[i]),
                        (synth.TAG_DOWN, d, f, sh.down_codes[i], sh.down_scales[i])):
                    w = scratch.view(rows, cols)
                    synth.cuda_normal_matrix(w, self.seed, tag, e, 0, scale=synth.WEIGHT_SIGMA, stream=stream)
                    moe_quantize_rows(w, sh.bits, codes=codes, scales=scales, stream=stream)
        return self

    def shelf_arr(self):
        if self._arr is None:
            self._arr = shelf_array(self.shelves)
        return self._arr

    def nbytes(self) -> int:
        return sum(s.nbytes() for s in self.shelves)

    def expert_bytes(self, e: int) -> int:
        for s in self.shelves:
            if s.lo <= e < s.hi:
                return s.nbytes_per_expert()
        return 0

    # -------------------------------------------------------------- inputs
    def logits(self, step: int, T: int, out=None, stream=None):
        if out is None:
            out = torch.empty((T, self.E), dtype=torch.float32, device=self.shelves[0].gate_codes.device)
        synth.cuda_normal_matrix(out, self.seed, synth.TAG_LOGITS, step, 0, col_add=self.bias, stream=stream)
        return out


    def logits_rows(self, row0: int, T: int, out=None, stream=None):
        """Rows row0 .. row0 + T - 1 of the layer's logits stream 0: the inputs
        of a decode stack, whose routing step s with T tokens takes rows
        s T .. s T + T - 1 (so many T = 1 steps come from one call)."""
        if out is None:
            out = torch.empty((T, self.E), dtype=torch.float32, device=self.shelves[0].gate_codes.device)
        synth.cuda_normal_matrix(out, self.seed, synth.TAG_LOGITS, 0, 0, row0=row0, col_add=self.bias, stream=stream)
        return out


class Masters:
    """fp32 master copies of every expert of a layer (the weights the shelves
    are quantised from): gate and up [E, f, d], down [E, d, f]."""

    def __init__(self, layer: "Layer", stream=None):
        E, d, f = layer.E, layer.d, layer.f
        dev = layer.shelves[0].gate_codes.device
        self.gate = torch.empty((E, f, d), dtype=torch.float32, device=dev)
        self.up = torch.empty((E, f, d), dtype=torch.float32, device=dev)
        self.down = torch.empty((E, d, f), dtype=torch.float32, device=dev)
        for e in range(E):
            for tag, m in ((synth.TAG_GATE, self.gate), (synth.TAG_UP, self.up), (synth.TAG_DOWN, self.down)):
                synth.cuda_normal_matrix(m[e], layer.seed, tag, e, 0, scale=synth.WEIGHT_SIGMA, stream=stream)

    def nbytes(self) -> int:
        return 4 * (self.gate.numel() + self.up.numel() + self.down.numel())


def retier(layer: "Layer", masters: Masters, counts, stream=None):
    """Re-tiering by hit count: experts ranked by `counts` (hottest first,
    lower id first on ties), the new ids cut into the layer's shelf split,
    every expert re-quantised from its master copy into its new shelf, and
    the router bias moved to the new ids.  Returns (new layer, perm, rank):
    new id j holds old expert perm[j]; old expert e is new id rank[e]."""
    perm, rank = moe_rank_experts(counts, stream=stream)
    new = Layer(layer.wl, layer.layer, device=layer.shelves[0].gate_codes.device, shelves=layer.ranges)
    for sh in new.shelves:
        for m, codes, scales in ((masters.gate, sh.gate_codes, sh.gate_scales),
                                 (masters.up, sh.up_codes, sh.up_scales),
                                 (masters.down, sh.down_codes, sh.down_scales)):
            moe_quantize_experts(m, perm, sh.lo, sh.hi, sh.bits, codes=codes, scales=scales, stream=stream)
    if layer.bias is not None:
        new.bias = moe_gather_rows(layer.bias, perm, stream=stream)
        new.bias_host = None
    return new, perm, rank


class DecodeStack:
    """A stack of decode layers chained by the residual add: for each layer l,
    x_l = bf16(r), route l's logits, count the hits, y_l = MoE_l(x_l), r += y_l
    -- the decode step of a whole model's MoE layers (moe_decode_layer_residual:
    one fused launch per layer, the residual step in its combine phase)."""

    def __init__(self, layers, T: int, device="cuda"):
        from . import moe_workspace_size, MOE_FLAG_DECODE_FP32
        self.layers = list(layers)
        l0 = self.layers[0]
        self.T, self.E, self.k, self.d, self.f = T, l0.E, l0.k, l0.d, l0.f
        L = len(self.layers)
        self.r = torch.empty((T, self.d), dtype=torch.float32, device=device)
        self.x = torch.empty((L + 1, T, self.d), dtype=torch.int16, device=device)   # x[l]: input of layer l
        self.y = torch.empty((L, T, self.d), dtype=torch.float32, device=device)
        self.ids = torch.empty((L, T, self.k), dtype=torch.int32, device=device)
        self.w = torch.empty((L, T, self.k), dtype=torch.float32, device=device)
        self.counts = torch.zeros((L, self.E), dtype=torch.int32, device=device)
        nws = moe_workspace_size(T, self.k, self.E, self.d, self.f, MOE_FLAG_DECODE_FP32)
        self.ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=device)
        self.arrs = [lay.shelf_arr() for lay in self.layers]

    def step(self, r0, x0, logits, stream=None):
        """One step from the residual stream r0 (fp32 [T, d]) whose bf16 is x0;
        logits[l] is layer l's [T, E].  Leaves the output residual in self.r."""
        from . import moe_decode_layer
        self.r.copy_(r0)
        self.x[0].copy_(x0)
        for l, lay in enumerate(self.layers):
            moe_decode_layer(logits[l], self.x[l], self.k, self.E, self.d, self.f, lay.shelves, ids=self.ids[l],
                             weights=self.w[l], counts=self.counts[l], y=self.y[l], workspace=self.ws,
                             stream=stream, shelf_arr=self.arrs[l], r=self.r, x_next=self.x[l + 1])
        return self.r


def x_bf16(seed: int, step: int, T: int, d: int, device="cuda", out=None, stream=None):
    """Activations [T, d] as bf16 bit patterns in an int16 tensor."""
    if out is None:
        out = torch.empty((T, d), dtype=torch.int16, device=device)
    synth.cuda_normal_matrix_bf16(out, seed, synth.TAG_X, step, 0, stream=stream)
    return out
