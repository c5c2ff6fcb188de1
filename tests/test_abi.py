"""The C-ABI library without a GPU: it builds, loads, exports every entry
point include/moe.h declares, and rejects bad arguments on the host before
touching the device."""
import ctypes
import os
import re

import pytest

import bit_moe_expert_routing_gb300 as moe
from bit_moe_expert_routing_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return moe.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_entry_points():
    syms = declared_symbols()
    assert "moe_layer_forward" in syms and "moe_route" in syms and len(syms) >= 10


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in moe.SIGNATURES, f"binding lacks {name}"


def _weights(D=256, E=16, k=2, I=128, ptr=0x1000):
    q = moe.moe_qmatrix(ptr, ptr, ptr)
    return moe.moe_weights(D, E, k, I, ptr, None, q, q, q, q, q, q)


def test_workspace_size_and_shape_checks(lib):
    w = _weights()
    assert moe.moe_workspace_size(w, 16) > 0
    assert moe.moe_workspace_size(w, 0) > 0
    assert moe.moe_workspace_size(w, -1) == 0
    for bad in (dict(D=100), dict(I=96), dict(k=0), dict(k=17), dict(E=2000, k=2), dict(k=33, E=64)):
        assert moe.moe_workspace_size(_weights(**bad), 4) == 0, bad
    # grows with T
    assert moe.moe_workspace_size(w, 4096) > moe.moe_workspace_size(w, 16)


def test_host_side_validation_needs_no_gpu(lib):
    w = _weights()
    ws = 0x100000
    n = moe.moe_workspace_size(w, 4)
    # workspace too small, misaligned or missing: rejected before any CUDA call
    assert moe.moe_layer_forward(w, 0x2000, 4, 0x3000, ws, n - 1, None) == moe.MOE_ERR_WORKSPACE
    assert moe.moe_layer_forward(w, 0x2000, 4, 0x3000, ws + 16, n, None) == moe.MOE_ERR_WORKSPACE
    assert moe.moe_layer_forward(w, 0x2000, 4, 0x3000, None, n, None) == moe.MOE_ERR_WORKSPACE
    # bad shapes and pointers
    assert moe.moe_layer_forward(_weights(D=100), 0x2000, 4, 0x3000, ws, n, None) == moe.MOE_ERR_SHAPE
    assert moe.moe_layer_forward(w, 0x2000, -1, 0x3000, ws, n, None) == moe.MOE_ERR_ARG
    assert moe.moe_layer_forward(w, None, 4, 0x3000, ws, n, None) == moe.MOE_ERR_ARG
    assert moe.moe_layer_forward(w, 0x2000, 4, 0x2000, ws, n, None) == moe.MOE_ERR_ARG  # y aliases x
    assert moe.moe_layer_forward(w, 0x2001, 4, 0x3000, ws, n, None) == moe.MOE_ERR_ARG  # unaligned x
    nullw = _weights(ptr=0)
    assert moe.moe_layer_forward(nullw, 0x2000, 4, 0x3000, ws, n, None) == moe.MOE_ERR_ARG
    # T = 0 is a no-op
    assert moe.moe_layer_forward(w, 0x2000, 0, 0x3000, ws, moe.moe_workspace_size(w, 0), None) == moe.MOE_OK
    assert moe.moe_last_launch_count() == 0


def test_static_entry_point_host_checks(lib):
    # the allocation-free entry point validates on the host like the others,
    # and an empty call is a no-op that needs no device
    w = _weights()
    assert moe.moe_layer_forward_static(w, 0x2000, 0, 0x3000, None) == moe.MOE_OK
    assert moe.moe_last_launch_count() == 0
    assert moe.moe_layer_forward_static(w, None, 0, None, None) == moe.MOE_OK
    assert moe.moe_layer_forward_static(w, None, 4, 0x3000, None) == moe.MOE_ERR_ARG
    assert moe.moe_layer_forward_static(w, 0x2000, 4, None, None) == moe.MOE_ERR_ARG
    assert moe.moe_layer_forward_static(w, 0x2000, 4, 0x2000, None) == moe.MOE_ERR_ARG  # y aliases x
    assert moe.moe_layer_forward_static(w, 0x2000, -1, 0x3000, None) == moe.MOE_ERR_ARG
    assert moe.moe_layer_forward_static(_weights(D=100), 0x2000, 4, 0x3000, None) == moe.MOE_ERR_SHAPE
    assert moe.moe_layer_forward_static(_weights(ptr=0), 0x2000, 0, 0x3000, None) == moe.MOE_ERR_ARG
    assert lib.moe_layer_forward_static(None, 0x2000, 4, 0x3000, None) == moe.MOE_ERR_ARG


def test_expanded_entry_point_host_checks(lib):
    # the unfused form's buffer size and its host-side argument checks
    w = _weights(D=256, E=16, k=2, I=128)
    nb = moe.moe_expanded_weights_bytes(w)
    assert nb == (3 * 16 + 3) * 128 * 256 * 2  # E x (gate, up, down) + the shared expert's three, bf16
    assert moe.moe_expanded_weights_bytes(_weights(D=100)) == 0
    ws, wsn = 1 << 30, moe.moe_workspace_size(w, 4)
    wb = 1 << 34
    assert moe.moe_layer_forward_expanded(w, 0x2000, 4, 0x3000, ws, wsn, None, nb, None) == moe.MOE_ERR_ARG
    assert moe.moe_layer_forward_expanded(w, 0x2000, 4, 0x3000, ws, wsn, wb + 16, nb, None) == moe.MOE_ERR_ARG
    assert moe.moe_layer_forward_expanded(w, 0x2000, 4, 0x3000, ws, wsn, wb, nb - 1, None) == moe.MOE_ERR_ARG
    assert moe.moe_layer_forward_expanded(w, 0x2000, -1, 0x3000, ws, wsn, wb, nb, None) == moe.MOE_ERR_ARG
    assert moe.moe_layer_forward_expanded(_weights(D=100), 0x2000, 4, 0x3000, ws, wsn, wb, nb, None) == \
        moe.MOE_ERR_SHAPE
    # an empty call is a no-op
    assert moe.moe_layer_forward_expanded(w, None, 0, None, ws, wsn, None, 0, None) == moe.MOE_OK


def test_workspace_view_layout(lib):
    w = _weights(D=256, E=16, k=2, I=128)
    T = 37
    n = moe.moe_workspace_size(w, T)
    v = moe.moe_route_view()
    base = 1 << 30
    assert moe.moe_workspace_view(w, T, base, n, v) == moe.MOE_OK
    assert v.T == T and v.block_m in (128, 256)
    ptrs = [v.logits, v.topk_idx, v.topk_w, v.count, v.off, v.perm, v.inv, v.blocks, v.n_blocks, v.h, v.y_acc]
    assert all(p % 256 == 0 for p in ptrs)
    assert all(base < p < base + n for p in ptrs)
    assert ptrs == sorted(ptrs)
    assert v.y_acc + T * 256 * 4 <= base + n
    assert v.max_blocks >= (T * 2) // 128 + min(16, T * 2) + 1


def test_options(lib):
    old = moe.moe_get_option(moe.MOE_OPT_GEMV_MAX_ROWS)
    assert moe.moe_set_option(moe.MOE_OPT_GEMV_MAX_ROWS, 3) == moe.MOE_OK
    assert moe.moe_get_option(moe.MOE_OPT_GEMV_MAX_ROWS) == 3
    assert moe.moe_set_option(moe.MOE_OPT_GEMV_MAX_ROWS, 99) == moe.MOE_ERR_ARG
    assert moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, 3) == moe.MOE_ERR_ARG
    assert moe.moe_set_option(12345, 0) == moe.MOE_ERR_ARG
    assert moe.moe_get_option(12345) == -1
    moe.moe_set_option(moe.MOE_OPT_GEMV_MAX_ROWS, old)


def test_block_m_option(lib):
    old = moe.moe_get_option(moe.MOE_OPT_BLOCK_M)
    for bad in (8, 17, 200, -16):
        assert moe.moe_set_option(moe.MOE_OPT_BLOCK_M, bad) == moe.MOE_ERR_ARG, bad
    w = _weights()
    n0 = moe.moe_workspace_size(w, 300)
    for good in (0, 16, 64, 192):
        assert moe.moe_set_option(moe.MOE_OPT_BLOCK_M, good) == moe.MOE_OK
        assert moe.moe_get_option(moe.MOE_OPT_BLOCK_M) == good
        # the workspace is sized for the smallest block, whatever the option
        assert moe.moe_workspace_size(w, 300) == n0
    moe.moe_set_option(moe.MOE_OPT_BLOCK_M, old)


def test_chunk_option_bounds_the_workspace(lib):
    old = moe.moe_get_option(moe.MOE_OPT_CHUNK_TOKENS)
    assert old == 8192  # the default
    for bad in (-1, (1 << 20) + 1):
        assert moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, bad) == moe.MOE_ERR_ARG, bad
    w = _weights()
    try:
        assert moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, 1000) == moe.MOE_OK
        assert moe.moe_get_option(moe.MOE_OPT_CHUNK_TOKENS) == 1000
        # one pass's tables: the size stops growing at the chunk size
        n1000 = moe.moe_workspace_size(w, 1000)
        assert moe.moe_workspace_size(w, 999) < n1000
        assert moe.moe_workspace_size(w, 1001) == n1000 == moe.moe_workspace_size(w, 50000)
        assert moe.moe_host_staging_size(w, 50000) == moe.moe_host_staging_size(w, 1000)
        # chunking off: the size keeps growing with T
        assert moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, 0) == moe.MOE_OK
        assert moe.moe_workspace_size(w, 50000) > 40 * n1000
        assert moe.moe_host_staging_size(w, 50000) > moe.moe_host_staging_size(w, 1000)
        # a workspace one byte short of one pass is still rejected before anything runs
        assert moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, 1000) == moe.MOE_OK
        ws = 1 << 30
        assert moe.moe_layer_forward(w, 0x2000, 5000, 0x9000000, ws, n1000 - 1, None) == moe.MOE_ERR_WORKSPACE
        assert moe.moe_last_launch_count() == 0
    finally:
        moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, old)


def test_host_sync_routing_option(lib):
    assert moe.moe_get_option(moe.MOE_OPT_HOST_SYNC_ROUTING) == 0  # off by default
    for bad in (-1, 2):
        assert moe.moe_set_option(moe.MOE_OPT_HOST_SYNC_ROUTING, bad) == moe.MOE_ERR_ARG
    assert moe.moe_set_option(moe.MOE_OPT_HOST_SYNC_ROUTING, 1) == moe.MOE_OK
    assert moe.moe_get_option(moe.MOE_OPT_HOST_SYNC_ROUTING) == 1
    assert moe.moe_set_option(moe.MOE_OPT_HOST_SYNC_ROUTING, 0) == moe.MOE_OK


def test_status_strings(lib):
    for s in range(7):
        assert moe.moe_status_string(s)
    assert moe.moe_status_string(999) == "unknown status"


def test_product_path_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(moe, "_lib", None)
    monkeypatch.setattr(moe, "LIB_PATH", "/nonexistent/libmoe.so")
    with pytest.raises(RuntimeError):
        moe.lib()


def test_static_pass_size_of_the_d2048_layer(lib):
    # The allocation-free entry point runs passes of the largest token count
    # whose workspace fits MOE_STATIC_SCRATCH_BYTES; include/moe.h quotes that
    # count for the D=2048, E=256, k=8, I=512 layer.
    w = _weights(D=2048, E=256, k=8, I=512)
    lim = 8 << 20
    assert moe.moe_workspace_size(w, 369) <= lim < moe.moe_workspace_size(w, 370)
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    assert "I=512 layer, 369 tokens" in text


def test_row_switch_default_matches_the_header(lib):
    # include/moe.h documents the measured default of MOE_OPT_GEMV_MAX_ROWS
    assert moe.moe_get_option(moe.MOE_OPT_GEMV_MAX_ROWS) == 4
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    assert "T <= this runs the decode GEMV path (0..8; default 4" in text
