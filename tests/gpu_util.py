"""Helpers shared by the GPU parity tests (not a test module)."""
from __future__ import annotations

import functools

import numpy as np

from bit_moe_expert_routing_gb300 import synth

# Output tolerance of the layer (bf16 I/O, fp32 accumulation):
# max |y - y_ref| <= 2e-2 * max |y_ref| and sum |y - y_ref| / sum |y_ref| <= 5e-3.
MAX_ABS_REL = 2e-2
MEAN_REL = 5e-3
# Renormalised routing weights: fp32 exp and division against fp64.
WEIGHT_ATOL = 1e-6


def bf16_to_np(t) -> np.ndarray:
    """torch bf16 tensor -> float64 numpy."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def x_to_device(x_bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).cuda()


def check_output(y: np.ndarray, y_ref: np.ndarray, what: str = "") -> dict:
    d = np.abs(y - y_ref)
    m = dict(max_abs=float(d.max()), max_ref=float(np.abs(y_ref).max()),
             mean_rel=float(d.sum() / np.abs(y_ref).sum()))
    assert m["max_abs"] <= MAX_ABS_REL * m["max_ref"], (what, m)
    assert m["mean_rel"] <= MEAN_REL, (what, m)
    return m


@functools.lru_cache(maxsize=8)
def config(name: str, T: int | None = None):
    """(layer, x) of a named workload; cached because the large layers take seconds."""
    return synth.make_config(name, T)


def rne_bf16(v: np.ndarray) -> np.ndarray:
    """fp64 values (exact in fp32) rounded to bf16, as float64."""
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(v.astype(np.float32))).astype(np.float64)
