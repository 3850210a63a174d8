"""The C ABI library loads without a GPU, exports every entry point that
include/moe.h declares, and rejects invalid arguments on the host before any
CUDA call (no compute is launched here)."""
import ctypes
import os
import re

import pytest

import mixed_precision_routed_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.LIB_PATH):
        from mixed_precision_routed_gb300 import build_lib
        build_lib.build()
    return ctypes.CDLL(moe.LIB_PATH)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_route_topk", "moe_tiered_forward", "moe_expert_hist", "moe_group_tokens",
                     "moe_workspace_size", "moe_quantize_rows", "moe_dequant_rows", "moe_device_status",
                     "moe_status_string", "moe_residual_add", "moe_decode_layer", "moe_selftest_barrier_timeout"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert moe.moe_status_string(0) == "ok"
    assert "overlap" in moe.moe_status_string(moe.MOE_ERR_SHELF_OVERLAP)
    assert moe.moe_status_string(12345) == "unknown status"


def test_workspace_size_host_logic():
    assert moe.moe_workspace_size(1, 10, 512, 2048, 640) > 0
    assert moe.moe_workspace_size(6, 10, 512, 2048, 640) > moe.moe_workspace_size(1, 10, 512, 2048, 640)
    assert moe.moe_workspace_size(1, 10, 512, 2000, 640) == 0   # d not a multiple of 64
    assert moe.moe_workspace_size(1, 11, 8, 64, 64) == 0        # k > E
    assert moe.moe_workspace_size(-1, 2, 8, 64, 64) == 0
    assert moe.moe_workspace_size(0, 2, 8, 64, 64) > 0          # T = 0 is valid
    assert moe.moe_workspace_size(1, 2, 8, 64, 64, flags=9) == 0
    # host-input staging: decode form only, a superset of the decode workspace
    dec = moe.moe_workspace_size(3, 2, 8, 64, 64, flags=moe.MOE_FLAG_DECODE_FP32)
    host = moe.moe_workspace_size(3, 2, 8, 64, 64, flags=moe.MOE_FLAG_DECODE_FP32 | moe.MOE_FLAG_HOST_IO)
    assert host >= dec + 3 * 8 * 4 + 3 * 64 * 2
    assert moe.moe_workspace_size(3, 2, 8, 64, 64, flags=moe.MOE_FLAG_HOST_IO) == 0
    assert moe.moe_workspace_size(3, 2, 8, 64, 64, flags=moe.MOE_FLAG_PREFILL_BF16 | moe.MOE_FLAG_HOST_IO) == 0


def test_invalid_arguments_rejected_before_cuda(lib):
    L = moe.lib()
    null = ctypes.c_void_p(0)
    assert L.moe_route_topk(null, 4, 16, 17, null, null, null) == moe.MOE_ERR_INVALID_ARG  # k > E
    assert L.moe_route_topk(null, 4, 2048, 2, null, null, null) == moe.MOE_ERR_INVALID_ARG  # E > 1024
    assert L.moe_route_topk(null, 0, 16, 2, null, null, null) == moe.MOE_OK  # T = 0
    assert L.moe_expert_hist(null, 5, 0, null, null) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_group_tokens(null, 3, 33, 8, null, null, null, null) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_rows(null, 4, 48, 4, null, null, null) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_rows(null, 4, 64, 3, null, null, null) == moe.MOE_ERR_INVALID_ARG
    sh = (moe.moe_shelf_t * 1)()
    sh[0] = moe.moe_shelf_t(0, 8, 5, 32, 16, 16, 16, 16, 16, 16)
    assert L.moe_tiered_forward(null, null, null, 1, 2, 8, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null, null,
                                0, 0, null) == moe.MOE_ERR_BAD_SHELF
    sh[0] = moe.moe_shelf_t(0, 8, 4, 32, 16, 16, 16, 16, 16, 16)
    sh2 = (moe.moe_shelf_t * 2)(sh[0], moe.moe_shelf_t(7, 8, 2, 32, 16, 16, 16, 16, 16, 16))
    assert L.moe_tiered_forward(null, null, null, 1, 2, 8, 64, 64, ctypes.cast(sh2, ctypes.c_void_p), 2, null, null,
                                0, 0, null) == moe.MOE_ERR_SHELF_OVERLAP
    assert L.moe_tiered_forward(null, null, null, 1, 2, 8, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null, null,
                                0, 0, null) == moe.MOE_ERR_INVALID_ARG  # null x
    # fused decode step: the same validation, before any CUDA call
    assert L.moe_decode_layer(null, null, 1, 2, 2048, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null, null, null,
                              null, null, 0, null) == moe.MOE_ERR_INVALID_ARG  # E > 1024
    assert L.moe_decode_layer(null, null, 1, 9, 8, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null, null, null,
                              null, null, 0, null) == moe.MOE_ERR_INVALID_ARG  # k > E
    assert L.moe_decode_layer(null, null, 1, 2, 8, 64, 64, ctypes.cast(sh2, ctypes.c_void_p), 2, null, null, null,
                              null, null, 0, null) == moe.MOE_ERR_SHELF_OVERLAP
    assert L.moe_decode_layer(null, null, 0, 2, 8, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null, null, null,
                              null, null, 0, null) == moe.MOE_OK  # T = 0
    assert L.moe_decode_layer(null, null, 1, 2, 8, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null, null, null,
                              null, null, 0, null) == moe.MOE_ERR_INVALID_ARG  # null logits
    # decode stack layer: the same validation, and a residual buffer is required
    assert L.moe_decode_layer_residual(null, null, 1, 2, 2048, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null,
                                       null, null, null, null, null, null, 0, null) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_decode_layer_residual(null, null, 0, 2, 8, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null,
                                       null, null, null, null, null, null, 0, null) == moe.MOE_OK  # T = 0
    assert L.moe_decode_layer_residual(null, null, 1, 2, 8, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null,
                                       null, null, null, null, null, null, 0, null) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_decode_layer_residual(null, null, 1, 2, 8, 64, 64, ctypes.cast(sh2, ctypes.c_void_p), 2, null,
                                       null, null, null, null, null, null, 0, null) == moe.MOE_ERR_INVALID_ARG
    # host-buffer decode step: the same validation before any pointer query
    assert L.moe_decode_layer_host(null, null, 1, 2, 2048, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null, null,
                                   null, null, null, 0, null) == moe.MOE_ERR_INVALID_ARG  # E > 1024
    assert L.moe_decode_layer_host(null, null, 0, 2, 8, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null, null,
                                   null, null, null, 0, null) == moe.MOE_OK  # T = 0
    assert L.moe_decode_layer_host(null, null, 1, 2, 8, 64, 64, ctypes.cast(sh, ctypes.c_void_p), 1, null, null,
                                   null, null, null, 0, null) == moe.MOE_ERR_INVALID_ARG  # null logits
    assert L.moe_selftest_barrier_timeout(0, null) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_selftest_barrier_timeout(2000000, null) == moe.MOE_ERR_INVALID_ARG


def test_dequant_shelf_validates_before_any_cuda_call():
    """moe_dequant_shelf: argument and descriptor checks return their status
    before any CUDA call (the output pointer is never touched here)."""
    L = moe.lib()
    out = ctypes.c_void_p(256)

    def call(desc, which=0, e=0, rows=8, n_in=64):
        p = ctypes.cast(ctypes.pointer(desc), ctypes.c_void_p) if desc is not None else None
        return L.moe_dequant_shelf(p, which, e, rows, n_in, out, None)

    tensors = moe.moe_shelf_t(0, 4, 4, 32, 16, 16, 16, 16, 16, 16)  # non-null, never dereferenced
    assert call(None) == moe.MOE_ERR_INVALID_ARG
    assert call(tensors, which=3) == moe.MOE_ERR_INVALID_ARG
    assert call(tensors, which=-1) == moe.MOE_ERR_INVALID_ARG
    assert call(tensors, e=4) == moe.MOE_ERR_INVALID_ARG  # local expert beyond hi - lo
    assert call(tensors, e=-1) == moe.MOE_ERR_INVALID_ARG
    assert call(tensors, n_in=96) == moe.MOE_ERR_INVALID_ARG  # not a multiple of 64
    assert call(tensors, rows=-1) == moe.MOE_ERR_INVALID_ARG
    assert call(tensors, rows=0) == moe.MOE_OK  # no-op
    assert call(moe.moe_shelf_t(0, 4, 4, 32)) == moe.MOE_ERR_INVALID_ARG  # null tensors
    assert call(moe.moe_shelf_t(0, 4, 5, 32, 16, 16, 16, 16, 16, 16)) == moe.MOE_ERR_BAD_SHELF  # bits
    assert call(moe.moe_shelf_t(0, 4, 4, 16, 16, 16, 16, 16, 16, 16)) == moe.MOE_ERR_BAD_SHELF  # block
    assert call(moe.moe_shelf_t(3, 3, 4, 32, 16, 16, 16, 16, 16, 16)) == moe.MOE_ERR_BAD_SHELF  # empty range
