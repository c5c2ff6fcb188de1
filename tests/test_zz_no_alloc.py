"""The allocation-free entry point, moe_layer_forward_static().

It serves callers that cannot allocate device memory: loops that forbid
cudaMalloc after start-up, and hosts that give plug-ins only their input and
output buffers. It must give the same
layer output as the regular entry point (within the tests' tolerance), also
on a second call in a row (the shared scratch keeps the previous call's
contents), and for token counts whose scratch would not fit in one pass.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import bit_moe_expert_routing_gb300 as moe
from bit_moe_expert_routing_gb300 import build, synth

from gpu_util import bf16_to_np, check_output, x_to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    moe.lib()
    moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_AUTO)
    moe.moe_set_option(moe.MOE_OPT_GEMM_IMPL, moe.GEMM_TENSOR_CORE)


def _static_pass_tokens(w):
    # the largest token count whose workspace fits the static array: the
    # size of the entry point's passes (the workspace grows with T)
    lim = moe_static_bytes()
    lo, hi = 0, 1 << 16  # size(lo) fits (or lo = 0), size(hi) does not
    assert moe.moe_workspace_size(w, hi) > lim
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if moe.moe_workspace_size(w, mid) <= lim:
            lo = mid
        else:
            hi = mid
    return lo


def _static_forward(dl, x):
    y = torch.empty_like(x)
    st = moe.moe_layer_forward_static(dl.w, x.data_ptr(), x.shape[0], y.data_ptr(), None)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    return y


@pytest.mark.parametrize("name,T", [("tiny", 16), ("tiny", 3), ("sweep", 8), ("sweep", 2)])
def test_static_scratch_matches_workspace_entry_point(name, T):
    layer, x_bits = synth.make_config(name, T)
    dl = moe.DeviceLayer(layer)
    x = x_to_device(x_bits)
    ref = bf16_to_np(dl.forward(x))
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row share the scratch
        y = bf16_to_np(_static_forward(dl, x))
        torch.cuda.synchronize()
        check_output(y, ref, f"static scratch {name} T={T}")
    assert np.isfinite(y).all()


def test_static_scratch_runs_large_token_counts_in_passes():
    # 1000 tokens of the D=2048 layer need more scratch than the array holds
    # (one pass fits 369 tokens), so the call runs consecutive passes of the
    # largest count that fits; the output is the regular entry point's.
    layer, x_bits = synth.make_config("prefill512", 1000)
    dl = moe.DeviceLayer(layer)
    n = _static_pass_tokens(dl.w)
    assert 1 < n < 500
    assert moe.moe_workspace_size(dl.w, 1000) > moe_static_bytes()
    x = x_to_device(x_bits)
    ref = bf16_to_np(dl.forward(x))
    torch.cuda.synchronize()
    y = bf16_to_np(_static_forward(dl, x))
    static_launches = moe.moe_last_launch_count()
    torch.cuda.synchronize()
    check_output(y, ref, "static scratch, 1000 tokens in passes")
    assert np.isfinite(y).all()
    assert moe.moe_get_device_status_static(None) == moe.MOE_OK
    # the launch count covers every pass: the same passes through the
    # workspace entry point (chunks of n tokens) launch as many kernels
    old = moe.moe_get_option(moe.MOE_OPT_CHUNK_TOKENS)
    try:
        assert moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, n) == moe.MOE_OK
        dl.forward(x)
        assert moe.moe_last_launch_count() == static_launches
    finally:
        moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, old)
    torch.cuda.synchronize()


def test_static_status_keeps_an_earlier_pass_error():
    # n + 2 tokens run as an n-token grouped-GEMM pass (n the largest count
    # that fits the array) and a 2-token GEMV pass. The test hook makes the
    # tensor-core epilogue of the first pass give up a bounded wait
    # (MOE_ERR_DEVICE_TIMEOUT); the second pass has no such wait, and must not
    # wipe the first pass's error. The next call starts afresh and is correct.
    layer, _ = synth.make_config("prefill512", 1)
    dl = moe.DeviceLayer(layer)
    n = _static_pass_tokens(dl.w)
    _, x_bits = synth.make_config("prefill512", n + 2)
    x = x_to_device(x_bits)
    old_rows = moe.moe_get_option(moe.MOE_OPT_GEMV_MAX_ROWS)
    assert moe.moe_set_option(moe.MOE_OPT_GEMV_MAX_ROWS, 4) == moe.MOE_OK  # the 2-token pass takes the GEMV path
    assert moe.moe_set_option(moe.MOE_OPT_TEST_WAIT_CYCLES, 20000) == moe.MOE_OK
    try:
        _static_forward(dl, x)
        st = moe.moe_get_device_status_static(None)
    finally:
        moe.moe_set_option(moe.MOE_OPT_TEST_WAIT_CYCLES, 0)
        moe.moe_set_option(moe.MOE_OPT_GEMV_MAX_ROWS, old_rows)
    assert st == moe.MOE_ERR_DEVICE_TIMEOUT, moe.moe_status_string(st)
    assert moe.moe_get_device_status_static(None) == moe.MOE_OK  # read and cleared
    ref = bf16_to_np(dl.forward(x))
    y = bf16_to_np(_static_forward(dl, x))
    torch.cuda.synchronize()
    assert moe.moe_get_device_status_static(None) == moe.MOE_OK
    check_output(y, ref, "static scratch after a recorded timeout")


def test_static_empty_call_is_a_noop():
    layer, x_bits = synth.make_config("tiny", 4)
    dl = moe.DeviceLayer(layer)
    assert moe.moe_layer_forward_static(dl.w, None, 0, None, None) == moe.MOE_OK
    assert moe.moe_last_launch_count() == 0


def moe_static_bytes():
    return 8 << 20
