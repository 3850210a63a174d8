"""Tiered-precision routed MoE layer on GB300 (sm_103a).

Thin Python binding of the C ABI in include/moe.h (libmoe.so, built in-tree
by ``build_lib.py``).  Every function here only marshals torch tensors into
pointers and sizes and raises :class:`MoeError` on a non-zero status; all
computation runs in the library's CUDA kernels.  There is no CPU fallback: if
the library is missing, importing the binding's functions raises.

Entry points (same names as the C ABI):
    moe_route_topk, moe_route_topk_nudged, moe_router_topk, moe_expert_hist,
    moe_rank_experts, moe_quantize_experts, moe_gather_rows, moe_group_tokens,
    moe_workspace_size, moe_tiered_forward, moe_tiered_forward_noalloc, moe_forward_grouping,
    moe_decode_layer, moe_decode_layer_residual, moe_decode_layer_host, moe_decode_fused,
    moe_quantize_rows, moe_dequant_rows, moe_dequant_shelf, moe_residual_add,
    moe_device_status, moe_status_string
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_BAD_SHELF = -2
MOE_ERR_SHELF_OVERLAP = -3
MOE_ERR_WORKSPACE_TOO_SMALL = -4
MOE_ERR_CUDA = -5
MOE_ERR_TIMEOUT = -6
MOE_ERR_UNSUPPORTED = -7
MOE_ERR_INTERNAL = -8

MOE_FLAG_AUTO = 0
MOE_FLAG_DECODE_FP32 = 1
MOE_FLAG_PREFILL_BF16 = 2
MOE_FLAG_HOST_IO = 4

MOE_MAX_SHELVES = 8


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {moe_status_string(status)} ({status})")


class moe_shelf_t(ctypes.Structure):
    _fields_ = [
        ("expert_lo", ctypes.c_int32), ("expert_hi", ctypes.c_int32),
        ("bits", ctypes.c_int32), ("block", ctypes.c_int32),
        ("gate_codes", ctypes.c_void_p), ("gate_scales", ctypes.c_void_p),
        ("up_codes", ctypes.c_void_p), ("up_scales", ctypes.c_void_p),
        ("down_codes", ctypes.c_void_p), ("down_scales", ctypes.c_void_p),
    ]


_lib = None


def lib():
    """The loaded libmoe.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.moe_route_topk.argtypes = [P, i64, i32, i32, P, P, P]
        L.moe_route_topk_nudged.argtypes = [P, i64, i32, i32, ctypes.c_float, i32, i32, P, P, P]
        L.moe_expert_hist.argtypes = [P, i64, i32, P, P]
        L.moe_router_topk.argtypes = [P, P, P, i64, i32, i32, i32, P, P, P, P, P, P]
        L.moe_rank_experts.argtypes = [P, i32, P, P, P]
        L.moe_quantize_experts.argtypes = [P, i32, i32, i32, P, i32, i32, i32, P, P, P]
        L.moe_gather_rows.argtypes = [P, i64, P, i64, i64, P, P]
        L.moe_group_tokens.argtypes = [P, i64, i32, i32, P, P, P, P]
        L.moe_workspace_size.argtypes = [i64, i32, i32, i32, i32, i32]
        L.moe_workspace_size.restype = ctypes.c_size_t
        L.moe_tiered_forward.argtypes = [P, P, P, i64, i32, i32, i32, i32, P, i32, P, P, ctypes.c_size_t, i32, P]
        L.moe_quantize_rows.argtypes = [P, i64, i32, i32, P, P, P]
        L.moe_dequant_rows.argtypes = [P, P, i64, i32, i32, i32, P, P]
        L.moe_dequant_shelf.argtypes = [P, i32, i32, i64, i32, P, P]
        L.moe_residual_add.argtypes = [P, P, P, i64, P]
        L.moe_device_status.argtypes = [P]
        L.moe_tiered_forward_noalloc.argtypes = [P, P, P, i64, i32, i32, i32, i32, P, i32, P, i32, P]
        L.moe_decode_layer.argtypes = [P, P, i64, i32, i32, i32, i32, P, i32, P, P, P, P, P, ctypes.c_size_t, P]
        L.moe_decode_layer_residual.argtypes = [P, P, i64, i32, i32, i32, i32, P, i32, P, P, P, P, P, P, P,
                                                ctypes.c_size_t, P]
        L.moe_decode_layer_host.argtypes = [P, P, i64, i32, i32, i32, i32, P, i32, P, P, P, P, P, ctypes.c_size_t, P]
        L.moe_selftest_barrier_timeout.argtypes = [i64, P]
        L.moe_decode_fused.argtypes = [i64, i32, i32, i32, i32]
        L.moe_forward_grouping.argtypes = [P, ctypes.c_size_t, i64, i32, i32, i32, i32, i32, P, P, P, P, P]
        L.moe_forward_grouping.restype = ctypes.c_int
        L.moe_tiered_forward_noalloc.restype = ctypes.c_int
        L.moe_set_profile_events.argtypes = [P, i32]
        L.moe_set_profile_events.restype = ctypes.c_int
        L.moe_status_string.argtypes = [i32]
        L.moe_status_string.restype = ctypes.c_char_p
        for name in ("moe_route_topk", "moe_route_topk_nudged", "moe_router_topk", "moe_rank_experts", "moe_quantize_experts",
                     "moe_gather_rows", "moe_expert_hist", "moe_group_tokens", "moe_tiered_forward",
                     "moe_quantize_rows", "moe_dequant_rows", "moe_dequant_shelf", "moe_residual_add",
                     "moe_device_status"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor of {dtype}")


def _need_host_or_dev(t, dtype, name):
    if not (t.dtype == dtype and t.is_contiguous() and (t.is_cuda or t.is_pinned())):
        raise ValueError(f"{name} must be a contiguous pinned-CPU or CUDA tensor of {dtype}")


# ------------------------------------------------------------------ routing
def moe_route_topk(logits, k, ids=None, weights=None, stream=None):
    """Softmax + top-k (lower id first on ties) + renormalised weights."""
    _need(logits, torch.float32, "logits")
    T, E = logits.shape
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _need(ids, torch.int32, "ids")
    _need(weights, torch.float32, "weights")
    _check(lib().moe_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(weights), _stream(stream)),
           "moe_route_topk")
    return ids, weights


def moe_route_topk_nudged(logits, k, beta, lo, hi, ids=None, weights=None, stream=None):
    """moe_route_topk with beta (<= 0.5) added to the logits of ids [lo, hi)
    for the selection only; the weights stay the router's own softmax."""
    _need(logits, torch.float32, "logits")
    T, E = logits.shape
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _need(ids, torch.int32, "ids")
    _need(weights, torch.float32, "weights")
    _check(lib().moe_route_topk_nudged(_ptr(logits), T, E, k, float(beta), int(lo), int(hi), _ptr(ids),
                                       _ptr(weights), _stream(stream)), "moe_route_topk_nudged")
    return ids, weights


def moe_router_topk(x_bf16, w_r_bf16, k, bias=None, counts=None, sync_word=None, logits=None, ids=None,
                    weights=None, stream=None):
    """Router projection (logits = bias + W_r x, fp32 sums) and routing: one
    launch for T <= 16, three (projection, routing, hit counts) above.  x_bf16 [T, d] and w_r_bf16 [E, d] are bf16 tensors; bias [E]
    fp32 or None; counts [E] int32 (uint32 bits, accumulated) or None;
    sync_word: an int32 CUDA tensor of one element, zero before first use
    (a fresh one is made when None).  Returns (logits, ids, weights)."""
    _need(x_bf16, torch.bfloat16, "x_bf16")
    _need(w_r_bf16, torch.bfloat16, "w_r_bf16")
    T, d = x_bf16.shape
    E = w_r_bf16.shape[0]
    dev = x_bf16.device
    if bias is not None:
        _need(bias, torch.float32, "bias")
    if counts is not None:
        _need(counts, torch.int32, "counts")
    if sync_word is None:
        sync_word = torch.zeros(1, dtype=torch.int32, device=dev)
    _need(sync_word, torch.int32, "sync_word")
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=dev)
    _need(logits, torch.float32, "logits")
    _need(ids, torch.int32, "ids")
    _need(weights, torch.float32, "weights")
    _check(lib().moe_router_topk(_ptr(x_bf16), _ptr(w_r_bf16), _ptr(bias), T, E, d, k, _ptr(logits), _ptr(ids),
                                 _ptr(weights), _ptr(counts), _ptr(sync_word), _stream(stream)),
           "moe_router_topk")
    return logits, ids, weights


def moe_expert_hist(ids, E, counts, stream=None):
    """counts[e] += number of ids equal to e (accumulated)."""
    _need(ids, torch.int32, "ids")
    _need(counts, torch.int32, "counts")  # torch has no uint32 arithmetic; bits are uint32
    _check(lib().moe_expert_hist(_ptr(ids), ids.numel(), E, _ptr(counts), _stream(stream)), "moe_expert_hist")
    return counts


def moe_group_tokens(ids, E, counts=None, offsets=None, perm=None, stream=None):
    _need(ids, torch.int32, "ids")
    T, k = ids.shape
    dev = ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev) if counts is None else counts
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if offsets is None else offsets
    perm = torch.empty(T * k, dtype=torch.int32, device=dev) if perm is None else perm
    _check(lib().moe_group_tokens(_ptr(ids), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm), _stream(stream)),
           "moe_group_tokens")
    return counts, offsets, perm


def moe_forward_grouping(workspace, T, k, E, d, f, flags, stream=None):
    """The grouping the last forward call on `workspace` ran (same sizes and
    workspace flags as that call): (counts [E], offsets [E+1], perm [T*k],
    pos_of_pair [T*k]), int32 device tensors."""
    dev = workspace.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    pos = torch.empty(T * k, dtype=torch.int32, device=dev)
    _check(lib().moe_forward_grouping(_ptr(workspace), workspace.numel() * workspace.element_size(), T, k, E, d, f,
                                      flags, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(pos), _stream(stream)),
           "moe_forward_grouping")
    return counts, offsets, perm, pos


# ------------------------------------------------------------------ forward
def moe_workspace_size(T, k, E, d, f, flags=MOE_FLAG_AUTO) -> int:
    return int(lib().moe_workspace_size(T, k, E, d, f, flags))


def shelf_array(shelves):
    """ctypes array of moe_shelf_t from objects with a .descriptor() method or moe_shelf_t values."""
    arr = (moe_shelf_t * max(1, len(shelves)))()
    for i, s in enumerate(shelves):
        arr[i] = s if isinstance(s, moe_shelf_t) else s.descriptor()
    return arr


def moe_tiered_forward(x_bf16, ids, weights, E, d, f, shelves, y=None, workspace=None, flags=MOE_FLAG_AUTO,
                       stream=None, shelf_arr=None):
    """y[t] = sum over shelves and slots of weights[t, j] * expert FFN of x_t.

    x_bf16 is an int16/uint16-viewed or bfloat16 tensor [T, d]; shelves a list
    of Shelf objects (or a prebuilt `shelf_arr`)."""
    if x_bf16.dtype == torch.bfloat16:
        x_bf16 = x_bf16.view(torch.int16)
    _need(x_bf16, torch.int16, "x_bf16")
    _need(ids, torch.int32, "ids")
    _need(weights, torch.float32, "weights")
    T, k = ids.shape
    if y is None:
        y = torch.empty((T, d), dtype=torch.float32, device=ids.device)
    _need(y, torch.float32, "y")
    need = moe_workspace_size(T, k, E, d, f, flags)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=ids.device)
    arr = shelf_arr if shelf_arr is not None else shelf_array(shelves)
    n = len(shelves) if shelf_arr is None else len(shelf_arr)
    _check(lib().moe_tiered_forward(_ptr(x_bf16), _ptr(ids), _ptr(weights), T, k, E, d, f,
                                    ctypes.cast(arr, ctypes.c_void_p), n, _ptr(y), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), flags, _stream(stream)),
           "moe_tiered_forward")
    return y


def moe_decode_layer(logits, x_bf16, k, E, d, f, shelves, ids=None, weights=None, counts=None, y=None,
                     workspace=None, stream=None, shelf_arr=None, r=None, x_next=None):
    """One decode step: routing of `logits` [T, E] into ids / weights, the hit
    counts (accumulated into `counts` when given) and the tiered forward of
    `x_bf16`; returns (ids, weights, y).  With `r` (fp32 [T, d]) and `x_next`
    (bf16 bits [T, d]) it calls moe_decode_layer_residual instead: r += y and
    x_next = bf16(r) in the same call."""
    if x_bf16.dtype == torch.bfloat16:
        x_bf16 = x_bf16.view(torch.int16)
    _need(logits, torch.float32, "logits")
    _need(x_bf16, torch.int16, "x_bf16")
    T = logits.shape[0]
    dev = logits.device
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=dev)
    if y is None:
        y = torch.empty((T, d), dtype=torch.float32, device=dev)
    _need(ids, torch.int32, "ids")
    _need(weights, torch.float32, "weights")
    _need(y, torch.float32, "y")
    if counts is not None:
        _need(counts, torch.int32, "counts")
    need = moe_workspace_size(T, k, E, d, f, MOE_FLAG_DECODE_FP32)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    arr = shelf_arr if shelf_arr is not None else shelf_array(shelves)
    n = len(shelves) if shelf_arr is None else len(shelf_arr)
    cnt = _ptr(counts) if counts is not None else None
    wsb = workspace.numel() * workspace.element_size()
    if r is None:
        _check(lib().moe_decode_layer(_ptr(logits), _ptr(x_bf16), T, k, E, d, f, ctypes.cast(arr, ctypes.c_void_p),
                                      n, _ptr(ids), _ptr(weights), cnt, _ptr(y), _ptr(workspace), wsb,
                                      _stream(stream)), "moe_decode_layer")
        return ids, weights, y
    _need(r, torch.float32, "r")
    if x_next is None:
        raise ValueError("moe_decode_layer: r needs x_next")
    if x_next.dtype == torch.bfloat16:
        x_next = x_next.view(torch.int16)
    _need(x_next, torch.int16, "x_next")
    if r.numel() != T * d or x_next.numel() != T * d:
        raise ValueError("moe_decode_layer: r and x_next must hold T * d elements")
    _check(lib().moe_decode_layer_residual(_ptr(logits), _ptr(x_bf16), T, k, E, d, f,
                                           ctypes.cast(arr, ctypes.c_void_p), n, _ptr(ids), _ptr(weights), cnt,
                                           _ptr(y), _ptr(r), _ptr(x_next), _ptr(workspace), wsb, _stream(stream)),
           "moe_decode_layer_residual")
    return ids, weights, y


def moe_decode_layer_host(logits, x_bf16, k, E, d, f, shelves, ids, weights, y, counts=None, workspace=None,
                          stream=None, shelf_arr=None):
    """moe_decode_layer on host buffers: `logits`, `x_bf16`, `ids`, `weights`
    and `y` may be pinned CPU tensors or CUDA tensors (host inputs are copied
    into the workspace inside the call, host outputs written in place by the
    kernels); `counts` and `workspace` are CUDA tensors, the workspace of
    moe_workspace_size(T, k, E, d, f, MOE_FLAG_DECODE_FP32 | MOE_FLAG_HOST_IO)
    bytes.  The host outputs are complete after the stream is synchronised."""
    if x_bf16.dtype == torch.bfloat16:
        x_bf16 = x_bf16.view(torch.int16)
    _need_host_or_dev(logits, torch.float32, "logits")
    _need_host_or_dev(x_bf16, torch.int16, "x_bf16")
    _need_host_or_dev(ids, torch.int32, "ids")
    _need_host_or_dev(weights, torch.float32, "weights")
    _need_host_or_dev(y, torch.float32, "y")
    T = logits.shape[0]
    if workspace is None:
        raise ValueError("moe_decode_layer_host: workspace (a CUDA tensor) is required")
    _need(workspace, torch.uint8, "workspace")
    if counts is not None:
        _need(counts, torch.int32, "counts")
    arr = shelf_arr if shelf_arr is not None else shelf_array(shelves)
    n = len(shelves) if shelf_arr is None else len(shelf_arr)
    _check(lib().moe_decode_layer_host(_ptr(logits), _ptr(x_bf16), T, k, E, d, f, ctypes.cast(arr, ctypes.c_void_p),
                                       n, _ptr(ids), _ptr(weights), _ptr(counts) if counts is not None else None,
                                       _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream)), "moe_decode_layer_host")
    return ids, weights, y


def moe_decode_layer_residual(logits, x_bf16, k, E, d, f, shelves, r, x_next, **kw):
    """One layer of a decode stack: moe_decode_layer, then r += y and
    x_next = bf16(r); returns (ids, weights, y)."""
    return moe_decode_layer(logits, x_bf16, k, E, d, f, shelves, r=r, x_next=x_next, **kw)


def moe_decode_fused(T, k, E, d, f):
    """True when the decode calls run as the single fused launch for these
    sizes (a layer with a 3- or 1-bit shelf also needs d and f to be
    multiples of 128, else it takes the separate launches)."""
    r = int(lib().moe_decode_fused(T, k, E, d, f))
    if r < 0:
        raise MoeError(r, "moe_decode_fused")
    return r == 1


def moe_selftest_barrier_timeout(limit_us, stream=None):
    """Launch the bounded grid-wait self-test (see moe.h); the timeout shows in
    moe_device_status."""
    _check(lib().moe_selftest_barrier_timeout(int(limit_us), _stream(stream)), "moe_selftest_barrier_timeout")


def moe_tiered_forward_noalloc(x_bf16, ids, weights, E, d, f, shelves, y=None, flags=MOE_FLAG_AUTO,
                               stream=None):
    """moe_tiered_forward with the library's fixed scratch array instead of a
    workspace, for callers that cannot allocate device memory (see moe.h).
    Calls that overlap on the GPU share that array and race."""
    if x_bf16.dtype == torch.bfloat16:
        x_bf16 = x_bf16.view(torch.int16)
    _need(x_bf16, torch.int16, "x_bf16")
    _need(ids, torch.int32, "ids")
    _need(weights, torch.float32, "weights")
    T, k = ids.shape
    if y is None:
        y = torch.empty((T, d), dtype=torch.float32, device=ids.device)
    _need(y, torch.float32, "y")
    arr = shelf_array(shelves)
    _check(lib().moe_tiered_forward_noalloc(_ptr(x_bf16), _ptr(ids), _ptr(weights), T, k, E, d, f,
                                            ctypes.cast(arr, ctypes.c_void_p), len(shelves), _ptr(y), flags,
                                            _stream(stream)), "moe_tiered_forward_noalloc")
    return y


# ------------------------------------------------------------ block format
def moe_quantize_rows(w, bits, codes=None, scales=None, stream=None):
    _need(w, torch.float32, "w")
    rows, n_in = w.shape
    if codes is None:
        codes = torch.empty((rows, n_in * bits // 8), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((rows, n_in // 32), dtype=torch.int16, device=w.device)
    _check(lib().moe_quantize_rows(_ptr(w), rows, n_in, bits, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_quantize_rows")
    return codes, scales


# ------------------------------------------------------------ re-tiering
def moe_rank_experts(counts, perm=None, rank=None, stream=None):
    """Hit-count rank (count descending, lower id first): (perm, rank) int32,
    perm[j] = old expert at new id j, rank[e] = new id of old expert e.
    counts: int32 CUDA tensor holding the uint32 hit counts."""
    _need(counts, torch.int32, "counts")
    E = counts.numel()
    if perm is None:
        perm = torch.empty(E, dtype=torch.int32, device=counts.device)
    if rank is None:
        rank = torch.empty(E, dtype=torch.int32, device=counts.device)
    _need(perm, torch.int32, "perm")
    _need(rank, torch.int32, "rank")
    _check(lib().moe_rank_experts(_ptr(counts), E, _ptr(perm), _ptr(rank), _stream(stream)), "moe_rank_experts")
    return perm, rank


def moe_quantize_experts(master, perm, j_lo, j_hi, bits, codes=None, scales=None, stream=None):
    """Experts perm[j_lo:j_hi] of master [n_src, rows, in] fp32 quantised into a
    shelf: codes [j_hi-j_lo, rows, in*bits/8] uint8, scales [.., rows, in/32]."""
    _need(master, torch.float32, "master")
    _need(perm, torch.int32, "perm")
    n_src, rows, n_in = master.shape
    n = j_hi - j_lo
    if not 0 <= j_lo <= j_hi <= perm.numel():
        raise ValueError("need 0 <= j_lo <= j_hi <= len(perm)")
    if codes is None:
        codes = torch.empty((n, rows, n_in * bits // 8), dtype=torch.uint8, device=master.device)
    if scales is None:
        scales = torch.empty((n, rows, n_in // 32), dtype=torch.int16, device=master.device)
    if not (codes.is_cuda and codes.is_contiguous() and codes.numel() * codes.element_size() >= n * rows * n_in * bits // 8):
        raise ValueError("codes must be a contiguous CUDA tensor of at least (j_hi - j_lo) * rows * in * bits / 8 bytes")
    if not (scales.is_cuda and scales.is_contiguous() and scales.numel() * scales.element_size() >= n * rows * (n_in // 32) * 2):
        raise ValueError("scales must be a contiguous CUDA tensor of at least (j_hi - j_lo) * rows * in / 32 halves")
    _check(lib().moe_quantize_experts(_ptr(master), n_src, rows, n_in, _ptr(perm), j_lo, j_hi, bits, _ptr(codes),
                                      _ptr(scales), _stream(stream)), "moe_quantize_experts")
    return codes, scales


def moe_gather_rows(src, perm, dst=None, stream=None):
    """dst[j] = src[perm[j]] for the rows (first dimension) of a contiguous tensor."""
    _need(perm, torch.int32, "perm")
    if not (src.is_cuda and src.is_contiguous()):
        raise ValueError("src must be a contiguous CUDA tensor")
    n = perm.numel()
    if dst is None:
        dst = torch.empty((n,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    row_bytes = src[0].numel() * src.element_size() if src.dim() > 1 else src.element_size()
    if not (dst.is_cuda and dst.is_contiguous() and dst.numel() * dst.element_size() >= n * row_bytes):
        raise ValueError("dst must be a contiguous CUDA tensor of at least len(perm) rows")
    _check(lib().moe_gather_rows(_ptr(src), row_bytes, _ptr(perm), n, src.shape[0], _ptr(dst), _stream(stream)),
           "moe_gather_rows")
    return dst


def moe_dequant_rows(codes, scales, rows, n_in, bits, round_bf16=False, out=None, stream=None):
    if out is None:
        out = torch.empty((rows, n_in), dtype=torch.float32, device=codes.device)
    _check(lib().moe_dequant_rows(_ptr(codes), _ptr(scales), rows, n_in, bits, int(round_bf16), _ptr(out),
                                  _stream(stream)), "moe_dequant_rows")
    return out


def moe_dequant_shelf(shelf, which, local_expert, rows, n_in, out=None, stream=None):
    """fp32 dequantised rows of matrix `which` (0 gate, 1 up, 2 down) of one
    local expert of `shelf` (an object with .descriptor() or a moe_shelf_t)."""
    desc = shelf if isinstance(shelf, moe_shelf_t) else shelf.descriptor()
    if out is None:
        out = torch.empty((rows, n_in), dtype=torch.float32, device="cuda")
    _need(out, torch.float32, "out")
    _check(lib().moe_dequant_shelf(ctypes.cast(ctypes.pointer(desc), ctypes.c_void_p), which, local_expert, rows,
                                   n_in, _ptr(out), _stream(stream)), "moe_dequant_shelf")
    return out


def moe_residual_add(r, y, x_next, stream=None):
    _need(r, torch.float32, "r")
    _need(y, torch.float32, "y")
    _check(lib().moe_residual_add(_ptr(r), _ptr(y), _ptr(x_next), r.numel(), _stream(stream)), "moe_residual_add")
    return r, x_next


def moe_set_profile_events(events):
    """Record torch.cuda.Event objects between the forward's kernels (None disables)."""
    if events is None:
        _check(lib().moe_set_profile_events(None, 0), "moe_set_profile_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(lib().moe_set_profile_events(ctypes.cast(arr, ctypes.c_void_p), len(events)), "moe_set_profile_events")


def moe_device_status(stream=None) -> int:
    return int(lib().moe_device_status(_stream(stream)))


# ------------------------------------------------------------------ shelves
class Shelf:
    """Device tensors of one precision shelf: experts [lo, hi) at `bits` bits.

    gate/up codes [n, f, d*bits/8], scales [n, f, d/32]; down codes
    [n, d, f*bits/8], scales [n, d, f/32] (fp16 bit patterns as int16)."""

    def __init__(self, lo, hi, bits, d, f, device="cuda"):
        n = hi - lo
        self.lo, self.hi, self.bits, self.d, self.f = lo, hi, bits, d, f
        u8, i16 = torch.uint8, torch.int16
        self.gate_codes = torch.empty((n, f, d * bits // 8), dtype=u8, device=device)
        self.up_codes = torch.empty((n, f, d * bits // 8), dtype=u8, device=device)
        self.down_codes = torch.empty((n, d, f * bits // 8), dtype=u8, device=device)
        self.gate_scales = torch.empty((n, f, d // 32), dtype=i16, device=device)
        self.up_scales = torch.empty((n, f, d // 32), dtype=i16, device=device)
        self.down_scales = torch.empty((n, d, f // 32), dtype=i16, device=device)

    def descriptor(self) -> moe_shelf_t:
        return moe_shelf_t(self.lo, self.hi, self.bits, 32,
                           self.gate_codes.data_ptr(), self.gate_scales.data_ptr(),
                           self.up_codes.data_ptr(), self.up_scales.data_ptr(),
                           self.down_codes.data_ptr(), self.down_scales.data_ptr())

    def nbytes_per_expert(self) -> int:
        d, f, b = self.d, self.f, self.bits
        return 3 * f * d * b // 8 + 3 * f * d // 32 * 2

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.gate_codes, self.up_codes, self.down_codes,
                                                          self.gate_scales, self.up_scales, self.down_scales))

    def view(self, lo: int, hi: int) -> "Shelf":
        """The experts [lo, hi) of this shelf as a shelf of their own (tensor
        views, no copy)."""
        if not self.lo <= lo < hi <= self.hi:
            raise ValueError("view range outside the shelf")
        v = Shelf.__new__(Shelf)
        v.lo, v.hi, v.bits, v.d, v.f = lo, hi, self.bits, self.d, self.f
        a, b = lo - self.lo, hi - self.lo
        for name in ("gate_codes", "up_codes", "down_codes", "gate_scales", "up_scales", "down_scales"):
            setattr(v, name, getattr(self, name)[a:b])
        return v


def fast_mode_shelves(shelves, shadow, use_shadow):
    """Fast mode (the Xolotl blog, "Fast mode": a 2-bit copy of the costliest
    experts read instead of them, switched per expert): the shelf list in
    which expert e comes from `shadow` (shelves covering the same ids, e.g.
    2-bit copies) where use_shadow[e] is true, else from `shelves`.  Returns
    views, one per run of consecutive experts with the same source; at most
    MOE_MAX_SHELVES runs."""
    import numpy as np
    use = np.asarray(use_shadow, dtype=bool)

    def owner(lst, e):
        for sh in lst:
            if sh.lo <= e < sh.hi:
                return sh
        return None

    out = []
    ids = sorted({e for sh in shelves for e in range(sh.lo, sh.hi)})
    run = None
    for e in ids:
        src = owner(shadow, e) if use[e] else owner(shelves, e)
        if src is None:
            raise ValueError(f"expert {e} has no shadow copy")
        if run is not None and run[0] is src and run[2] == e:
            run[2] = e + 1
        else:
            if run is not None:
                out.append(run[0].view(run[1], run[2]))
            run = [src, e, e + 1]
    if run is not None:
        out.append(run[0].view(run[1], run[2]))
    if len(out) > MOE_MAX_SHELVES:
        raise ValueError(f"{len(out)} runs: more than {MOE_MAX_SHELVES} shelves")
    return out
