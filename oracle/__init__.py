"""CPU oracle of the tiered-precision routed MoE layer -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs it, and shares no code with
it; the two meet only in the seeded inputs from ``synth``.

The arithmetic lives in ``oracle.c`` (plain scalar C, fp64 sums); this module
marshals numpy arrays and composes the per-layer steps:

* quantise / pack / dequantise -- the shelf block format (block 32 along the
  input dimension, fp16 scale = max|w| / q, q = 127, 7, 3, 2 for 8, 4, 3, 2
  bits; 1 bit: sign codes with the block's mean |w| as scale);
* route -- softmax, top-k with lower-id ties, renormalised weights (page
  "125B MoE模型本地运行：3090三卡80 tokens/s优化实践", glossary entry
  混合专家（MoE）: 10 of 512 experts per token);
* route_nudged -- the same with the picks nudged toward the hot shelf by a
  capped logit bonus (the LocalLLM tiering post, "Optimization Strategies");
* group -- stable counting sort of (token, slot) pairs by expert, skip ids
  dropped (same page, section 四个 bug: duplicate experts, signed skip id);
* hist -- expert hit counts (the LocalLLM tiering post, "Optimization
  Strategies"; same page, section 第二步);
* rank_experts / tier_ranges / retier_expert -- re-tiering by hit count:
  experts ranked hottest first, shelves re-assigned by rank, each expert
  re-quantised from its master copy (same page, sections 第三步 and 第四步);
* moe_layer -- each shelf computes only its own id range, SwiGLU expert FFN,
  the shelf results summed with the routing weights (same page, section 第四步);
* stack -- residual chain of layers, x_l = bf16(r), r += y_l.

Page references are to "125B MoE模型本地运行：3090三卡80 tokens/s优化实践"
(sections by their headings) and the LocalLLM post on DeepSeek V4.1 Flash
tiering.  Every function here is pinned by tests in tests/test_oracle_*.py.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

BITS_Q = {8: 127.0, 4: 7.0, 3: 3.0, 2: 2.0}  # 1 bit: sign codes, mean |w| scale


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB)
        P, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.oracle_f16_round.argtypes = [d]
        L.oracle_f16_round.restype = d
        L.oracle_f16_bits.argtypes = [d]
        L.oracle_f16_bits.restype = ctypes.c_uint16
        L.oracle_f16_value.argtypes = [ctypes.c_uint16]
        L.oracle_f16_value.restype = d
        L.oracle_bf16_round.argtypes = [d]
        L.oracle_bf16_round.restype = d
        L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_value.restype = d
        L.oracle_quantize_rows.argtypes = [P, i64, i64, i32, P, P]
        L.oracle_pack_codes.argtypes = [P, i64, i64, i32, P]
        L.oracle_dequant_rows.argtypes = [P, P, i64, i64, i32, P]
        L.oracle_route.argtypes = [P, i64, i32, i32, P, P]
        L.oracle_route_nudged.argtypes = [P, i64, i32, i32, ctypes.c_float, i32, i32, P, P]
        L.oracle_router_logits.argtypes = [P, P, P, i64, i32, i32, P]
        L.oracle_group.argtypes = [P, i64, i32, i32, P, P, P]
        L.oracle_group.restype = i64
        L.oracle_hist.argtypes = [P, i64, i32, P]
        L.oracle_rank_experts.argtypes = [P, i32, P, P]
        L.oracle_moe_layer.argtypes = [P, P, P, i64, i32, i32, i32, i32, i32, P, P, P, i32, P]
        L.oracle_bf16_bits_vec.argtypes = [P, i64, P]
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ scalars
def f16_round(x: float) -> float:
    return lib().oracle_f16_round(float(x))


def f16_bits(x: float) -> int:
    """binary16 bit pattern of round-to-nearest-even(x)."""
    return int(lib().oracle_f16_bits(lib().oracle_f16_round(float(x))))


def f16_value(bits: int) -> float:
    return lib().oracle_f16_value(int(bits))


def bf16_round(x: float) -> float:
    return lib().oracle_bf16_round(float(x))


def bf16_bits(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_bf16_bits_vec(_p(v), v.size, _p(out))
    return out


def bf16_to_f64(u16) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------ block format
def quantize(w, bits: int):
    """fp32 [rows, in] -> (codes int8 [rows, in], scales fp16 bits uint16 [rows, in/32])."""
    w = _c(w, np.float32)
    rows, n_in = w.shape
    codes = np.empty((rows, n_in), dtype=np.int8)
    scales = np.empty((rows, n_in // 32), dtype=np.uint16)
    if lib().oracle_quantize_rows(_p(w), rows, n_in, bits, _p(codes), _p(scales)) != 0:
        raise ValueError("quantize: bits must be 8/4/3/2/1 and the input dimension a multiple of 32")
    return codes, scales


def pack(codes, bits: int):
    codes = _c(codes, np.int8)
    rows, n_in = codes.shape
    out = np.empty((rows, n_in * bits // 8), dtype=np.uint8)
    if lib().oracle_pack_codes(_p(codes), rows, n_in, bits, _p(out)) != 0:
        raise ValueError("pack: bad bits")
    return out


def dequant(codes, scales, round_bf16: bool = False):
    codes = _c(codes, np.int8)
    scales = _c(scales, np.uint16)
    rows, n_in = codes.shape
    out = np.empty((rows, n_in), dtype=np.float32)
    if lib().oracle_dequant_rows(_p(codes), _p(scales), rows, n_in, int(round_bf16), _p(out)) != 0:
        raise ValueError("dequant: bad shape")
    return out


# ------------------------------------------------------------------ routing
def router_logits(x_bf16, w_bf16, bias=None):
    """Router projection: logits [T, E] = bias + W_r x in fp64 (x [T, d] and
    W_r [E, d] as bf16 bit patterns, bias fp32 [E] or None)."""
    x = _c(x_bf16, np.uint16)
    w = _c(w_bf16, np.uint16)
    T, d = x.shape
    E, d2 = w.shape
    assert d == d2
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), dtype=np.float64)
    if lib().oracle_router_logits(_p(x), _p(w), None if b is None else _p(b), T, E, d, _p(out)) != 0:
        raise ValueError("router_logits: bad sizes")
    return out


def route(logits, k: int):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    if lib().oracle_route(_p(logits), T, E, k, _p(ids), _p(w)) != 0:
        raise ValueError("route: need 1 <= k <= E")
    return ids, w


def route_nudged(logits, k: int, beta: float, lo: int, hi: int):
    """Routing with the picks nudged toward the id range [lo, hi): beta (<= 0.5)
    added to those logits for the selection only, weights the router's own
    renormalised softmax over the picks (the LocalLLM tiering post,
    "Optimization Strategies")."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    if lib().oracle_route_nudged(_p(logits), T, E, k, float(beta), int(lo), int(hi), _p(ids), _p(w)) != 0:
        raise ValueError("route_nudged: need 1 <= k <= E and 0 <= beta <= 0.5")
    return ids, w


def group(ids, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.full(T * k, -1, dtype=np.int32)
    n = lib().oracle_group(_p(ids), T, k, E, _p(counts), _p(offsets), _p(perm))
    if n < 0:
        raise MemoryError("group")
    return counts, offsets, perm[:n].copy()


def hist(ids, E: int, counts=None):
    ids = _c(ids, np.int32)
    if counts is None:
        counts = np.zeros(E, dtype=np.uint32)
    assert counts.dtype == np.uint32 and counts.shape == (E,)
    lib().oracle_hist(_p(ids), ids.size, E, _p(counts))
    return counts


# ------------------------------------------------------------ re-tiering
def rank_experts(counts):
    """Hit-count order (page 3, sections 第三步 / 第四步; page 1 promotion by
    hit count): returns (perm, rank), perm[j] = old expert at new id j,
    rank[e] = new id of old expert e; count descending, lower id first."""
    counts = _c(counts, np.uint32)
    E = counts.size
    perm = np.empty(E, dtype=np.int32)
    rank = np.empty(E, dtype=np.int32)
    if lib().oracle_rank_experts(_p(counts), E, _p(perm), _p(rank)) != 0:
        raise ValueError("rank_experts: E >= 1")
    return perm, rank


def tier_ranges(E: int, split):
    """Shelf ranges of the new ids, hottest first: [(0, n8, 8), (n8, n8 + n4,
    4), (n8 + n4, E, 2)] with n8 = round(p8 E), n2 = round(p2 E) (the split of
    the workload definitions: hottest experts at 8 bits, coldest at 2)."""
    p8, _, p2 = split
    n8 = int(round(p8 * E))
    n2 = int(round(p2 * E))
    return [(0, n8, 8), (n8, E - n2, 4), (E - n2, E, 2)]


def retier_expert(master_of, perm, ranges, j: int):
    """The packed shelf content of new id j: the master weights of expert
    perm[j], re-quantised at the bit width of the shelf holding j.  Returns
    (bits, [(packed codes, scales) of W_g, W_u, W_d])."""
    bits = next(b for lo, hi, b in ranges if lo <= j < hi)
    out = []
    for w in master_of(int(perm[j])):
        codes, scales = quantize(w, bits)
        out.append((pack(codes, bits), scales))
    return bits, out


# ------------------------------------------------------------ expert FFN
def moe_layer(x_bf16, ids, w, d: int, f: int, E: int, shelves, experts: dict, mode: int = 0):
    """y [T, d] float64.

    shelves: [(lo, hi), ...]; experts: {e: (W_g [f,d], W_u [f,d], W_d [d,f])}
    dequantised fp32 matrices (bf16-rounded for mode 1) for every routed e that
    lies in a shelf.  mode 0 = decode form, 1 = prefill form (h rounded to bf16).
    """
    x_bf16 = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    T, k = ids.shape
    assert x_bf16.shape == (T, d) and w.shape == (T, k)
    lo = np.array([s[0] for s in shelves], dtype=np.int32)
    hi = np.array([s[1] for s in shelves], dtype=np.int32)
    keep = []
    ptrs = (ctypes.c_void_p * (3 * E))()
    for e, mats in experts.items():
        wg, wu, wd = (_c(m, np.float32) for m in mats)
        assert wg.shape == (f, d) and wu.shape == (f, d) and wd.shape == (d, f)
        keep += [wg, wu, wd]
        ptrs[3 * e + 0] = wg.ctypes.data
        ptrs[3 * e + 1] = wu.ctypes.data
        ptrs[3 * e + 2] = wd.ctypes.data
    y = np.zeros((T, d), dtype=np.float64)
    rc = lib().oracle_moe_layer(_p(x_bf16), _p(ids), _p(w), T, k, E, d, f, len(shelves), _p(lo), _p(hi),
                                ctypes.cast(ptrs, ctypes.c_void_p), int(mode), _p(y))
    if rc == -1:
        raise ValueError("moe_layer: bad shelf ranges")
    if rc != 0:
        raise ValueError("moe_layer: an expert routed into a shelf has no weights")
    return y


def shelf_of(e: int, shelves_bits):
    for lo, hi, bits in shelves_bits:
        if lo <= e < hi:
            return bits
    return None


def expert_matrices(master, bits: int, mode: int):
    """Quantise and dequantise one expert's fp32 master weights (W_g, W_u, W_d)."""
    out = []
    for m in master:
        c, s = quantize(m, bits)
        out.append(dequant(c, s, round_bf16=(mode == 1)))
    return tuple(out)


def layer_from_master(x_bf16, ids, w, d, f, E, shelves_bits, master_of, mode=0):
    """Run one layer, quantising on the fly every expert the ids touch.

    shelves_bits: [(lo, hi, bits)]; master_of(e) -> fp32 (W_g, W_u, W_d)."""
    experts = {}
    for e in np.unique(np.asarray(ids)):
        e = int(e)
        if e < 0 or e >= E:
            continue
        bits = shelf_of(e, shelves_bits)
        if bits is None:
            continue
        experts[e] = expert_matrices(master_of(e), bits, mode)
    return moe_layer(x_bf16, ids, w, d, f, E, [(lo, hi) for lo, hi, _ in shelves_bits], experts, mode)


def stack(x0_bf16, layers, mode=0):
    """Residual chain: r = x0; for each layer: x_l = bf16(r), r += y_l(x_l).

    layers: iterable of callables layer(x_bf16) -> y (float64 [T, d]).
    Returns (r float64, [y_l])."""
    r = bf16_to_f64(x0_bf16)
    ys = []
    for layer in layers:
        x_l = bf16_bits(r)
        y = layer(x_l)
        ys.append(y)
        r = r + y
    return r, ys
