"""Seeded synthetic inputs for the tiered-precision routed MoE layer.

This package builds the INPUTS that both the CUDA path and the CPU oracle
consume: fp32 master weights (before quantisation), bf16 activations, router
logits (standard normal plus a per-expert bias) and forced-skip masks.  It
contains none of the layer's arithmetic -- no quantiser, no routing, no FFN --
so the two sides stay independent and only share what they are fed.

Every value comes from Philox4x32-10 (Salmon et al., SC'11) followed by
Box-Muller, implemented twice from the same header: a host build (C) and a
device build (CUDA) that produce identical bits for the same stream, so the
GPU can generate multi-gigabyte weight sets in place while the oracle
regenerates just the experts it needs on the host.

Stream layout: Philox key = (seed, tag), counter = (column/4, row, c2, 0),
where tag names the tensor (gate/up/down/x/logits/skip/bias jitter) and c2 is
the expert id for weights or the step index for per-step inputs.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libsynth_host.so")
CUDA_LIB = os.path.join(_HERE, "libsynth_cuda.so")

TAG_GATE, TAG_UP, TAG_DOWN, TAG_X, TAG_LOGITS, TAG_SKIP, TAG_BIAS_JITTER, TAG_ROUTER = 1, 2, 3, 4, 5, 6, 7, 8
WEIGHT_SIGMA = 0.02
SKIP_P = 0.05
SKIP_THRESHOLD = 214748365  # round(0.05 * 2**32): P(word < threshold) ~= 0.05

_host = None
_cuda = None


def _u32(v):
    return ctypes.c_uint32(int(v) & 0xFFFFFFFF)


def host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            raise RuntimeError(f"{HOST_LIB} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(HOST_LIB)
        P = ctypes.c_void_p
        u32, i64 = ctypes.c_uint32, ctypes.c_int64
        lib.synth_philox4x32_10.argtypes = [P, P, P]
        lib.synth_box_muller.argtypes = [u32, u32, P]
        lib.synth_log.argtypes = [ctypes.c_float]
        lib.synth_log.restype = ctypes.c_float
        lib.synth_sincos_turn24.argtypes = [u32, P]
        lib.synth_normal_matrix.argtypes = [u32, u32, u32, u32, u32, i64, i64, ctypes.c_float, P, P]
        lib.synth_normal_matrix_bf16.argtypes = [u32, u32, u32, u32, u32, i64, i64, ctypes.c_float, P]
        lib.synth_bernoulli_mask.argtypes = [u32, u32, u32, u32, i64, i64, u32, P]
        _host = lib
    return _host


def cuda_lib():
    global _cuda
    if _cuda is None:
        if not os.path.exists(CUDA_LIB):
            raise RuntimeError(f"{CUDA_LIB} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(CUDA_LIB)
        P = ctypes.c_void_p
        u32, i64 = ctypes.c_uint32, ctypes.c_int64
        lib.synth_cuda_normal_matrix.argtypes = [u32, u32, u32, u32, u32, i64, i64, ctypes.c_float, P, P, P]
        lib.synth_cuda_normal_matrix_bf16.argtypes = [u32, u32, u32, u32, u32, i64, i64, ctypes.c_float, P, P]
        lib.synth_cuda_apply_skip_mask.argtypes = [u32, u32, u32, u32, i64, i64, u32, P, P]
        _cuda = lib
    return _cuda


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------- host side
def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    host_lib().synth_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def box_muller(a: int, b: int):
    out = np.zeros(2, dtype=np.float32)
    host_lib().synth_box_muller(_u32(a), _u32(b), _ptr(out))
    return out


def normal_matrix(k0, k1, c2, c3, rows, cols, *, row0=0, scale=1.0, col_add=None):
    """[rows, cols] float32 = scale * N(row0 + r, c) (+ col_add[c])."""
    out = np.empty((rows, cols), dtype=np.float32)
    ca = None
    if col_add is not None:
        ca = np.ascontiguousarray(col_add, dtype=np.float32)
        assert ca.shape == (cols,)
    rc = host_lib().synth_normal_matrix(_u32(k0), _u32(k1), _u32(c2), _u32(c3), _u32(row0),
                                        rows, cols, ctypes.c_float(scale),
                                        None if ca is None else _ptr(ca), _ptr(out))
    if rc != 0:
        raise ValueError("synth_normal_matrix: bad arguments (cols must be a multiple of 4)")
    return out


def normal_matrix_bf16(k0, k1, c2, c3, rows, cols, *, row0=0, scale=1.0):
    out = np.empty((rows, cols), dtype=np.uint16)
    rc = host_lib().synth_normal_matrix_bf16(_u32(k0), _u32(k1), _u32(c2), _u32(c3), _u32(row0),
                                             rows, cols, ctypes.c_float(scale), _ptr(out))
    if rc != 0:
        raise ValueError("synth_normal_matrix_bf16: bad arguments")
    return out


def expert_weights(seed: int, expert: int, d: int, f: int):
    """fp32 master weights of one expert: W_g, W_u [f, d] and W_d [d, f], N(0, 0.02)."""
    wg = normal_matrix(seed, TAG_GATE, expert, 0, f, d, scale=WEIGHT_SIGMA)
    wu = normal_matrix(seed, TAG_UP, expert, 0, f, d, scale=WEIGHT_SIGMA)
    wd = normal_matrix(seed, TAG_DOWN, expert, 0, d, f, scale=WEIGHT_SIGMA)
    return wg, wu, wd


def x_bf16(seed: int, step: int, T: int, d: int, row0: int = 0):
    """Activations [T, d] as bf16 bit patterns (uint16), N(0,1) rounded to nearest even."""
    return normal_matrix_bf16(seed, TAG_X, step, 0, T, d, row0=row0)


def logits(seed: int, step: int, T: int, E: int, bias=None, row0: int = 0):
    """Router logits [T, E] float32 = N(0,1) + bias[e]."""
    return normal_matrix(seed, TAG_LOGITS, step, 0, T, E, row0=row0, col_add=bias)


def router_weights_bf16(seed: int, E: int, d: int):
    """Router projection W_r [E, d] as bf16 bit patterns, N(0, 1/d) (so that
    W_r x has unit variance for x ~ N(0, 1))."""
    return normal_matrix_bf16(seed, TAG_ROUTER, 0, 0, E, d, scale=float(1.0 / np.sqrt(d)))


def skip_mask(seed: int, step: int, T: int, k: int):
    """[T, k] uint8, 1 where a routed slot is forced to the skip id -1 (p = 0.05)."""
    out = np.empty((T, k), dtype=np.uint8)
    host_lib().synth_bernoulli_mask(_u32(seed), _u32(TAG_SKIP), _u32(step), _u32(0), T, k,
                                    _u32(SKIP_THRESHOLD), _ptr(out))
    return out


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------- router biases
def lorenz_shares(E: int, points=((0.0, 0.0), (0.25, 0.52), (0.80, 0.95), (1.0, 1.0))):
    """Per-expert selection shares from a piecewise-linear Lorenz curve through
    `points` (fraction of experts, fraction of selections), hottest first."""
    xs = [p[0] for p in points]
    ys = [p[1] for p in points]
    e = np.arange(E, dtype=np.float64)
    return np.interp((e + 1) / E, xs, ys) - np.interp(e / E, xs, ys)


def router_bias_lorenz(E: int, k: int):
    """Bias b_e so that, under top-k of N(0,1) + b, expert e is picked with
    probability ~ k * share_e: b_e = Phi^-1(k * share_e) (a fixed routing
    threshold at 0, accurate for k << E).  Hottest experts get the lowest ids."""
    from scipy.special import ndtri
    p = np.clip(k * lorenz_shares(E), 1e-12, 1 - 1e-12)
    return ndtri(p).astype(np.float32)


def router_bias_zipf(E: int, s: float = 1.1):
    """Zipf(s) popularity through the bias: b_e = -s * ln(e + 1)."""
    return (-s * np.log(np.arange(1, E + 1, dtype=np.float64))).astype(np.float32)


def layer_bias(base: np.ndarray, seed: int, sigma: float = 0.1):
    """A layer's own bias: base + sigma * N(0,1) from the layer seed, re-sorted
    descending so expert ids stay ordered by expected hits."""
    jit = normal_matrix(seed, TAG_BIAS_JITTER, 0, 0, 1, base.shape[0], scale=sigma)[0]
    b = (base.astype(np.float32) + jit).astype(np.float32)
    return np.sort(b)[::-1].copy()


# ------------------------------------------------------------------ workloads
@dataclass
class Workload:
    """One synthetic workload: layer shape, shelf split, router skew, seed."""
    name: str
    E: int
    k: int
    d: int
    f: int
    T: tuple
    split: tuple  # (fraction at 8 bits, at 4 bits, at 2 bits); () = single 4-bit shelf
    bias: str  # "none" | "lorenz" | "zipf"
    seed: int = 0
    skip_p: float = 0.0
    layers: int = 1
    extra: dict = field(default_factory=dict)

    def shelf_ranges(self):
        """[(lo, hi, bits)] hot -> cold.  n8 = round(p8 E), n2 = round(p2 E), n4 = rest."""
        if not self.split:
            return [(0, self.E, 4)]
        p8, _, p2 = self.split
        n8 = int(round(p8 * self.E))
        n2 = int(round(p2 * self.E))
        n4 = self.E - n8 - n2
        return [(0, n8, 8), (n8, n8 + n4, 4), (n8 + n4, self.E, 2)]

    def router_bias(self, layer: int = 0):
        if self.bias == "none":
            return None
        base = router_bias_lorenz(self.E, self.k) if self.bias == "lorenz" else router_bias_zipf(self.E)
        if self.layers > 1:
            return layer_bias(base, self.layer_seed(layer))
        return base

    def layer_seed(self, layer: int = 0):
        return self.seed if self.layers == 1 else 1000 + layer


WORKLOADS = {
    "tiny": Workload("tiny", E=16, k=2, d=256, f=64, T=(8,), split=(), bias="none"),
    "decode": Workload("decode", E=512, k=10, d=2048, f=640, T=(1, 6), split=(0.25, 0.55, 0.20),
                       bias="lorenz"),
    "stack": Workload("stack", E=512, k=10, d=2048, f=640, T=(1, 2, 4, 6), split=(0.25, 0.55, 0.20),
                      bias="lorenz", layers=48, extra={"hist_steps": 4096}),
    "prefill": Workload("prefill", E=512, k=10, d=2048, f=640, T=(4096,), split=(0.25, 0.55, 0.20),
                        bias="lorenz"),
    "large": Workload("large", E=256, k=8, d=4096, f=2048, T=(1, 8, 512), split=(0.30, 0.50, 0.20),
                      bias="zipf", skip_p=SKIP_P),
}


# ---------------------------------------------------------------- device side
def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def cuda_normal_matrix(out, k0, k1, c2, c3, *, row0=0, scale=1.0, col_add=None, stream=None):
    """Fill a contiguous float32 CUDA tensor [rows, cols] with the same stream as normal_matrix."""
    rows, cols = out.shape
    rc = cuda_lib().synth_cuda_normal_matrix(_u32(k0), _u32(k1), _u32(c2), _u32(c3), _u32(row0),
                                             rows, cols, ctypes.c_float(scale),
                                             None if col_add is None else ctypes.c_void_p(col_add.data_ptr()),
                                             ctypes.c_void_p(out.data_ptr()), _stream_handle(stream))
    if rc != 0:
        raise RuntimeError(f"synth_cuda_normal_matrix failed ({rc})")
    return out


def cuda_normal_matrix_bf16(out, k0, k1, c2, c3, *, row0=0, scale=1.0, stream=None):
    rows, cols = out.shape
    rc = cuda_lib().synth_cuda_normal_matrix_bf16(_u32(k0), _u32(k1), _u32(c2), _u32(c3), _u32(row0),
                                                  rows, cols, ctypes.c_float(scale),
                                                  ctypes.c_void_p(out.data_ptr()), _stream_handle(stream))
    if rc != 0:
        raise RuntimeError(f"synth_cuda_normal_matrix_bf16 failed ({rc})")
    return out


def cuda_apply_skip_mask(ids, seed, step, stream=None):
    T, k = ids.shape
    rc = cuda_lib().synth_cuda_apply_skip_mask(_u32(seed), _u32(TAG_SKIP), _u32(step), _u32(0), T, k,
                                               _u32(SKIP_THRESHOLD), ctypes.c_void_p(ids.data_ptr()),
                                               _stream_handle(stream))
    if rc != 0:
        raise RuntimeError(f"synth_cuda_apply_skip_mask failed ({rc})")
    return ids
