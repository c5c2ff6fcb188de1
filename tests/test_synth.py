"""The seeded input generator: determinism and the workload statistics it must produce."""
import math

import numpy as np
import pytest

from bit_moe_expert_routing_gb300 import synth


def test_splitmix64_reference_values():
    # splitmix64 from state 0: the first outputs of the published generator
    # (Steele, Lea, Flood 2014; also Vigna's reference C code) are
    # 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F.
    z = np.arange(1, 4, dtype=np.uint64) * synth._GOLDEN
    out = synth._mix(z)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_streams_deterministic_and_independent():
    a = synth.u64_stream(3, 10, 1000)
    assert np.array_equal(a, synth.u64_stream(3, 10, 1000))
    assert np.array_equal(a[500:], synth.u64_stream(3, 10, 500, start=500))
    assert not np.array_equal(a, synth.u64_stream(3, 11, 1000))
    assert not np.array_equal(a, synth.u64_stream(4, 10, 1000))


def test_distributions():
    n = synth.normal(1, 1, 200_000)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1) < 0.01
    L = synth.make_layer(0, 256, 16, 2, 128)
    codes = (L.gate.codes[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & 15
    assert set(np.unique(codes)) == set(range(16))
    s = synth.bf16_bits_to_f32(L.gate.scales).astype(np.float64)
    b = synth.bf16_bits_to_f32(L.gate.biases).astype(np.float64)
    lo, hi = 0.5 / (8 * math.sqrt(256)), 1.5 / (8 * math.sqrt(256))
    assert s.min() >= lo * (1 - 2 ** -8) and s.max() <= hi * (1 + 2 ** -8)
    assert np.array_equal(b, -8 * s)
    assert abs(L.router_w.std() * math.sqrt(256) - 1) < 0.05  # 4096 samples


def test_bf16_rounding_is_nearest_even():
    v = np.array([1.0, 1.00390625, 1.01171875, -2.0 ** -130, 3.0e38], np.float32)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties to even -> 1 + 2^-6
    out = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(v))
    assert out[0] == 1.0 and out[1] == 1.0 and out[2] == 1.015625
    assert out[3] == np.float32(-2.0 ** -130) or out[3] < 0


@pytest.mark.slow
def test_zipf_routing_is_skewed():
    from oracle import oracle as O
    L, x = synth.make_config("prefill4096_zipf")
    _, idx, _ = O.route(O.OracleLayer(L), x)
    counts = np.bincount(idx.reshape(-1), minlength=L.E)
    assert counts.max() > 1000 and counts.min() == 0
