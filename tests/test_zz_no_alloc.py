"""The allocation-free entry point, moe_layer_forward_static().

It serves callers that cannot allocate device memory: code running while a
CUDA graph is captured, loops that forbid cudaMalloc after start-up, and hosts
that give plug-ins only their input and output buffers. It must give the same
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
    # (one pass fits 451), so the call runs consecutive passes of the largest
    # count that fits; the output is the regular entry point's.
    layer, x_bits = synth.make_config("prefill512", 1000)
    dl = moe.DeviceLayer(layer)
    assert moe.moe_workspace_size(dl.w, 1000) > moe_static_bytes()
    x = x_to_device(x_bits)
    ref = bf16_to_np(dl.forward(x))
    torch.cuda.synchronize()
    y = bf16_to_np(_static_forward(dl, x))
    torch.cuda.synchronize()
    check_output(y, ref, "static scratch, 1000 tokens in passes")
    assert np.isfinite(y).all()


def moe_static_bytes():
    return 8 << 20
