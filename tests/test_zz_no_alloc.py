"""The allocation-free entry point, moe_layer_forward_static().

It serves callers that cannot allocate device memory: code running while a
CUDA graph is captured, loops that forbid cudaMalloc after start-up, and hosts
that give plug-ins only their input and output buffers. It must give the same
layer output as the regular entry point (within the tests' tolerance), also
on a second call in a row (the shared scratch keeps the previous call's
contents), and it must refuse token counts whose scratch would not fit.

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


def test_static_scratch_rejects_too_many_tokens():
    layer, _ = synth.make_config("tiny")
    dl = moe.DeviceLayer(layer)
    T = 1
    while moe.moe_workspace_size(dl.w, T) <= moe_static_bytes():
        T *= 2
    x = torch.zeros((T, layer.D), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    st = moe.moe_layer_forward_static(dl.w, x.data_ptr(), T, y.data_ptr(), None)
    assert st == moe.MOE_ERR_WORKSPACE


def moe_static_bytes():
    return 8 << 20
