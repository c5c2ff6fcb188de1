"""Seeded synthetic MoE layers and activations.

This module only draws random numbers. It holds none of the layer's
arithmetic (no dequantisation, routing, SwiGLU or combine), so both the CUDA
path and the CPU oracle can be fed from it without sharing any of the method.

Generator: a counter-based splitmix64. Value ``i`` of stream ``(seed, tid)`` is
``mix(key(seed, tid) + (i + 1) * 0x9E3779B97F4A7C15)``, where ``mix`` is the
splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014). Uniforms take the top 53 bits. Normals use the
Box-Muller transform on two consecutive counter values, in fp64, then round.

Value distributions follow the workload statement of the layer (the
Qwen3.6-35B-A3B expert shape of "Optimizing on-device inference for Apple
Silicon", section "Dequantise weights during matrix multiplication"):

* x ~ N(0, 1), rounded to bf16 (round to nearest even);
* router weight W_r ~ N(0, 1/D) in fp32;
* 4-bit codes uniform in 0..15, eight per uint32 word, code j of a word at
  bits 4j..4j+3 (element 8m+j of the row);
* one bf16 scale per group of 64 weights, scale = bf16(U(0.5, 1.5) / (8 sqrt(D))),
  and bias = -8 * scale (exact: a power-of-two multiple);
* optional skewed routing: an additive router bias that is the log of a
  Zipf(s) pmf over a seeded permutation of the experts,
  bias[pi(r)] = -s * ln(r) for rank r = 1..E.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream ids, one per tensor. Shared-expert tensors are offset by 100.
TID_X = 1
TID_ROUTER_W = 2
TID_ZIPF_PERM = 3
TID_CODES = {"gate": 10, "up": 12, "down": 14}
TID_SCALES = {"gate": 11, "up": 13, "down": 15}
TID_SHARED = 100


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser, in place on a uint64 array."""
    t = np.empty_like(z)
    np.right_shift(z, np.uint64(30), out=t)
    z ^= t
    z *= _M1
    np.right_shift(z, np.uint64(27), out=t)
    z ^= t
    z *= _M2
    np.right_shift(z, np.uint64(31), out=t)
    z ^= t
    return z


def _key(seed: int, tid: int) -> np.uint64:
    s = np.array([(seed * 0x100000001B3 + tid * 0x9E3779B1 + 0x632BE59BD9B4E019) & 0xFFFFFFFFFFFFFFFF],
                 dtype=np.uint64)
    return _mix(s)[0]


def u64_stream(seed: int, tid: int, n: int, start: int = 0) -> np.ndarray:
    """Values start..start+n-1 of the splitmix64 stream (seed, tid)."""
    with np.errstate(over="ignore"):
        z = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z *= _GOLDEN
        z += _key(seed, tid)
        return _mix(z)


def uniform(seed: int, tid: int, n: int) -> np.ndarray:
    """n doubles in [0, 1) from the top 53 bits."""
    return (u64_stream(seed, tid, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, tid: int, n: int) -> np.ndarray:
    """n standard normals (Box-Muller, the cosine branch) in fp64."""
    z = u64_stream(seed, tid, 2 * n).reshape(n, 2)
    u1 = ((z[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (z[:, 1] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class QMatrix:
    """One packed 4-bit matrix family [n_exp, rows, K]: codes [n_exp, rows, K/8] uint32,
    scales and biases [n_exp, rows, K/64] as bf16 bit patterns (uint16)."""
    codes: np.ndarray
    scales: np.ndarray
    biases: np.ndarray

    @property
    def nbytes(self) -> int:
        return self.codes.nbytes + self.scales.nbytes + self.biases.nbytes


@dataclasses.dataclass
class Layer:
    D: int
    E: int
    k: int
    I: int
    router_w: np.ndarray            # fp32 [E, D]
    router_bias: np.ndarray | None  # fp32 [E] or None
    gate: QMatrix                   # [E, I, D]
    up: QMatrix                     # [E, I, D]
    down: QMatrix                   # [E, D, I]
    s_gate: QMatrix                 # [1, I, D]
    s_up: QMatrix                   # [1, I, D]
    s_down: QMatrix                 # [1, D, I]
    seed: int = 0

    def expert_bytes(self) -> int:
        """Packed bytes of one routed expert (its three matrices)."""
        return (self.gate.nbytes + self.up.nbytes + self.down.nbytes) // self.E


def qmatrix(seed: int, which: str, n_exp: int, rows: int, K: int, D: int, shared: bool = False,
            scale_mult: float = 1.0) -> QMatrix:
    assert K % 64 == 0
    off = TID_SHARED if shared else 0
    n_words = n_exp * rows * K // 8
    w64 = u64_stream(seed, TID_CODES[which] + off, (n_words + 1) // 2)
    codes = w64.view(np.uint32)[:n_words].reshape(n_exp, rows, K // 8).copy()
    n_groups = n_exp * rows * (K // 64)
    u = uniform(seed, TID_SCALES[which] + off, n_groups)
    s32 = ((0.5 + u) / (8.0 * math.sqrt(D)) * scale_mult).astype(np.float32)
    scales = f32_to_bf16_bits(s32)
    biases = f32_to_bf16_bits(-8.0 * bf16_bits_to_f32(scales))  # exact: -8 * bf16 is a bf16
    return QMatrix(codes, scales.reshape(n_exp, rows, K // 64), biases.reshape(n_exp, rows, K // 64))


def zipf_router_bias(seed: int, E: int, s: float) -> np.ndarray:
    """bias[pi(r)] = -s * ln(r), r = 1..E, pi a seeded permutation of the experts."""
    keys = u64_stream(seed, TID_ZIPF_PERM, E)
    pi = np.argsort(keys, kind="stable")
    bias = np.empty(E, dtype=np.float64)
    bias[pi] = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    return bias.astype(np.float32)


def make_layer(seed: int, D: int, E: int, k: int, I: int, zipf_s: float | None = None) -> Layer:
    assert D % 64 == 0 and I % 64 == 0 and 1 <= k <= E
    wr = (normal(seed, TID_ROUTER_W, E * D) / math.sqrt(D)).astype(np.float32).reshape(E, D)
    rb = zipf_router_bias(seed, E, zipf_s) if zipf_s is not None else None
    return Layer(
        D=D, E=E, k=k, I=I, router_w=wr, router_bias=rb,
        gate=qmatrix(seed, "gate", E, I, D, D),
        up=qmatrix(seed, "up", E, I, D, D),
        down=qmatrix(seed, "down", E, D, I, D),
        s_gate=qmatrix(seed, "gate", 1, I, D, D, shared=True),
        s_up=qmatrix(seed, "up", 1, I, D, D, shared=True),
        s_down=qmatrix(seed, "down", 1, D, I, D, shared=True),
        seed=seed,
    )


def make_x(seed: int, T: int, D: int, row0: int = 0) -> np.ndarray:
    """Activations x[T, D] ~ N(0,1) as bf16 bit patterns; rows row0..row0+T-1 of the seed's stream."""
    n = normal(seed, TID_X, (row0 + T) * D)[row0 * D:]
    return f32_to_bf16_bits(n.astype(np.float32)).reshape(T, D)


# The five workloads. The decode-shape layer is D=2048, E=256, top-8 + 1 shared, I=512.
CONFIGS = {
    "tiny":    dict(seed=0, T=16,   D=256,  E=16,  k=2, I=128, zipf_s=None),
    "decode":  dict(seed=1, T=1,    D=2048, E=256, k=8, I=512, zipf_s=None),
    "prefill512": dict(seed=2, T=512, D=2048, E=256, k=8, I=512, zipf_s=None),
    "prefill4096_zipf": dict(seed=3, T=4096, D=2048, E=256, k=8, I=512, zipf_s=1.1),
    "sweep":   dict(seed=4, T=8,    D=2048, E=256, k=8, I=512, zipf_s=None),  # T in {2,3,4,5,8}
}
SWEEP_T = (2, 3, 4, 5, 8)


def make_config(name: str, T: int | None = None) -> tuple[Layer, np.ndarray]:
    c = CONFIGS[name]
    layer = make_layer(c["seed"], c["D"], c["E"], c["k"], c["I"], c["zipf_s"])
    x = make_x(c["seed"], c["T"] if T is None else T, c["D"])
    return layer, x
