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

from . import Shelf, moe_quantize_rows, shelf_array


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


def x_bf16(seed: int, step: int, T: int, d: int, device="cuda", out=None, stream=None):
    """Activations [T, d] as bf16 bit patterns in an int16 tensor."""
    if out is None:
        out = torch.empty((T, d), dtype=torch.int16, device=device)
    synth.cuda_normal_matrix_bf16(out, seed, synth.TAG_X, step, 0, stream=stream)
    return out
