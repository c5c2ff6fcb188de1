"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test ties one part of the oracle to hand-worked values, a closed form, an
invariant, a special case that reduces to a library routine (numpy sort,
torch fp64 matmul / silu) or a brute-force twin, so that a dropped term, a
wrong sign or index, or a transposed operand fails at least one of them.
"""
import copy
import os

import numpy as np
import pytest
import torch

from bit_moe_expert_routing_gb300 import synth
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _row_qmat(words, scales, biases):
    """A one-expert matrix from explicit rows: words [rows, K/8], scales/biases [rows, K/64]."""
    w = np.asarray(words, np.uint32)
    return synth.QMatrix(w[None].copy(), np.asarray(scales, np.uint16)[None].copy(),
                         np.asarray(biases, np.uint16)[None].copy())


def _golden_dequant():
    rows = []
    with open(os.path.join(GOLDEN, "dequant_vectors.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, word, s, b, exact, rne = [p.strip() for p in line.split("|")]
            rows.append((name, int(word, 16), int(s, 16), int(b, 16),
                         [float(v) for v in exact.split()], [float(v) for v in rne.split()]))
    return rows


@pytest.mark.parametrize("vec", _golden_dequant(), ids=lambda v: v[0])
def test_dequant_hand_vectors(vec):
    name, word, s, b, exact, rne = vec
    m = _row_qmat([[word] * 8], [[s]], [[b]])
    w = O.dequant(m, 0, 1, 64)[0]
    assert np.array_equal(w, np.tile(exact, 8)), name
    # the bf16 operand value: one round-to-nearest-even of the exact value
    w_bf16 = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(w.astype(np.float32)))
    assert np.array_equal(w_bf16.astype(np.float64), np.tile(rne, 8)), name


def test_dequant_group_and_row_indexing():
    # row 0: q=1 everywhere, group 0 (s=1, b=0) -> 1, group 1 (s=2, b=0.5) -> 2.5
    # row 1: q=2 everywhere, group 0 (s=0.25, b=-1) -> -0.5, group 1 (s=4, b=1) -> 9
    bf = lambda v: int(synth.f32_to_bf16_bits(np.array([v], np.float32))[0])
    m = _row_qmat([[0x11111111] * 16, [0x22222222] * 16],
                  [[bf(1.0), bf(2.0)], [bf(0.25), bf(4.0)]],
                  [[bf(0.0), bf(0.5)], [bf(-1.0), bf(1.0)]])
    w = O.dequant(m, 0, 2, 128)
    assert np.array_equal(w[0], np.r_[np.full(64, 1.0), np.full(64, 2.5)])
    assert np.array_equal(w[1], np.r_[np.full(64, -0.5), np.full(64, 9.0)])


def test_dequant_second_expert_offset():
    L = synth.make_layer(5, 128, 3, 1, 64)
    # expert 2, row 7 of the gate matrix, read straight from the packed arrays
    w = O.dequant(L.gate, 2, 64, 128)[7]
    words = L.gate.codes[2, 7]
    q = np.array([(int(words[kk // 8]) >> (4 * (kk % 8))) & 15 for kk in range(128)], np.float64)
    s = synth.bf16_bits_to_f32(L.gate.scales[2, 7]).astype(np.float64)
    b = synth.bf16_bits_to_f32(L.gate.biases[2, 7]).astype(np.float64)
    assert np.array_equal(w, q * np.repeat(s, 64) + np.repeat(b, 64))


def _small_layer(seed=7, D=128, E=8, k=2, I=64, zipf=None):
    return synth.make_layer(seed, D, E, k, I, zipf)


def test_router_uniform_when_logits_equal():
    # k = E and W_r = 0: every logit is 0, the softmax is exactly 1/E for every
    # expert, renormalising over all E changes nothing, ties go to lower index.
    L = _small_layer(E=16, k=16)
    L.router_w = np.zeros_like(L.router_w)
    x = synth.make_x(1, 5, L.D)
    _, idx, w = O.route(O.OracleLayer(L), x)
    assert np.array_equal(idx, np.tile(np.arange(16), (5, 1)))
    assert np.array_equal(w, np.full((5, 16), 1.0 / 16))


def test_router_exact_integer_logits():
    # Small integers make every fp32 product and partial sum exact, so the
    # logits must equal the exact integer dot products (plus the bias).
    rng = np.random.default_rng(3)
    L = _small_layer(D=256, E=12, k=3)
    xi = rng.integers(-3, 4, size=(6, L.D))
    wi = rng.integers(-4, 5, size=(L.E, L.D))
    bi = rng.integers(-8, 9, size=L.E)
    L.router_w = wi.astype(np.float32)
    L.router_bias = bi.astype(np.float32)
    x = synth.f32_to_bf16_bits(xi.astype(np.float32))
    logits, idx, _ = O.route(O.OracleLayer(L), x)
    assert np.array_equal(logits.astype(np.int64), xi @ wi.T + bi)


def test_router_order_closed_form():
    # Reading R3 fixes the fp32 order: 32 partial sums, partial l taking the
    # elements 32c+l in order c = 0, 1, ... with an FMA, then the pairwise tree
    # l += l+16, l += l+8, ..., l += l+1. With x = 1 and D = 256 (8 terms per
    # partial), worked by hand:
    #   row A = [2^24 at d=0, -2^24 at d=32, 1 elsewhere]: partial 0 cancels
    #     to 0 after two terms and collects 6 ones; the tree then adds exact
    #     small integers: 6 + 31*8 = 254. (One chain in index order loses the
    #     31 ones before d=32 to round-to-even at 2^24 and gives 223.)
    #   row B = [2^24 at d=0, -2^24 at d=1, 1 elsewhere]: partial 0 stays 2^24
    #     (its 7 ones are lost), partial 1 is -2^24 + 7 exactly, the others 8;
    #     the tree levels give 2^24+8, 2^24+24, 2^24+56, 2^24+120 on lane 0 and
    #     -2^24+15, +31, +63, +127 on lane 1, then 247. (One chain gives 254.)
    L = _small_layer(D=256, E=8, k=2)
    big = np.float32(2.0 ** 24)
    w = np.zeros((L.E, L.D), np.float32)
    w[0, :] = 1.0
    w[0, 0], w[0, 32] = big, -big
    w[1, :] = 1.0
    w[1, 0], w[1, 1] = big, -big
    L.router_w = w
    L.router_bias = np.zeros(L.E, np.float32)
    x = synth.f32_to_bf16_bits(np.ones((3, L.D), np.float32))
    logits, _, _ = O.route(O.OracleLayer(L), x)
    assert np.all(logits[:, 0] == 254.0)
    assert np.all(logits[:, 1] == 247.0)
    assert np.all(logits[:, 2:] == 0.0)


def test_router_close_to_fp64_dot():
    L = _small_layer(D=512, E=32, k=4)
    x = synth.make_x(2, 9, L.D)
    logits, _, _ = O.route(O.OracleLayer(L), x)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    ref = xf @ L.router_w.astype(np.float64).T
    mag = np.abs(xf) @ np.abs(L.router_w.astype(np.float64)).T
    assert np.all(np.abs(logits - ref) <= 1e-6 * mag + 1e-30)


def test_topk_order_ties_and_weights():
    L = _small_layer(D=128, E=16, k=4)
    # experts 3 and 9, and 5 and 6, get identical router rows -> identical logits
    L.router_w[9] = L.router_w[3]
    L.router_w[6] = L.router_w[5]
    x = synth.make_x(4, 40, L.D)
    logits, idx, w = O.route(O.OracleLayer(L), x)
    for t in range(x.shape[0]):
        order = np.argsort(-logits[t].astype(np.float64), kind="stable")[:L.k]
        assert np.array_equal(idx[t], order)
        p = torch.softmax(torch.tensor(logits[t], dtype=torch.float64), 0).numpy()
        assert np.allclose(w[t], p[order] / p[order].sum(), rtol=0, atol=1e-15)
        assert abs(w[t].sum() - 1.0) < 1e-15
    assert np.array_equal(logits[:, 9], logits[:, 3])
    both = [(3 in idx[t] and 9 in idx[t]) for t in range(x.shape[0])]
    for t in range(x.shape[0]):
        if both[t]:
            j3, j9 = list(idx[t]).index(3), list(idx[t]).index(9)
            assert j3 < j9


def test_topk_non_finite_and_signed_zero_logits_hand_worked():
    # The pages give no rule for non-finite logits. The reading: a NaN logit
    # ranks (and weighs) as -inf, -0 equals +0, and equal values go to the
    # lower index. Worked by hand for logits [NaN, 1, -0, +0, -inf, 2]:
    #   order 5 (2), 1 (1), 2 (-0) before 3 (+0), then 0 (NaN = -inf) before
    #   4 (-inf); weights exp(l - 2) over the kept: 1, e^-1, e^-2, e^-2, 0, 0.
    lg = np.array([np.nan, 1.0, -0.0, 0.0, -np.inf, 2.0], np.float32)
    assert np.signbit(lg[2]) and not np.signbit(lg[3])
    e1, e2 = np.exp(-1.0), np.exp(-2.0)
    for k, order, num in ((6, [5, 1, 2, 3, 0, 4], [1.0, e1, e2, e2, 0.0, 0.0]),
                          (4, [5, 1, 2, 3], [1.0, e1, e2, e2]),
                          (1, [5], [1.0])):
        idx, w = O.topk(lg, k)
        assert list(idx) == order, k
        want = np.array(num) / sum(num)
        assert np.allclose(w, want, rtol=0, atol=1e-15), (k, w, want)
    # +0 listed before -0 keeps index order as well: the sign is no tie-break
    idx, _ = O.topk(np.array([0.0, -0.0, -1.0], np.float32), 2)
    assert list(idx) == [0, 1]


def _check_tables(idx, E, BM, tb):
    T, k = idx.shape
    A = T * k
    flat = idx.reshape(-1)
    assert np.array_equal(tb["count"], np.bincount(flat, minlength=E))
    assert tb["count"].sum() == A
    assert tb["off"][0] == 0 and tb["off"][-1] == A and np.all(np.diff(tb["off"]) >= 0)
    # stable counting sort by expert == the scatter with ascending assignment index
    assert np.array_equal(tb["perm"], np.argsort(flat, kind="stable"))
    assert np.array_equal(tb["inv"][tb["perm"]], np.arange(A))
    # block map: blocks tile every segment in order, each at most BM rows
    covered = []
    for g, first, rows in tb["blocks"]:
        assert 1 <= rows <= BM
        if g < E:
            assert tb["off"][g] <= first and first + rows <= tb["off"][g + 1]
        else:
            assert g == E and A <= first and first + rows <= A + T
        covered.extend(range(first, first + rows))
    assert covered == list(range(A + T))
    gs = tb["blocks"][:, 0]
    assert np.all(np.diff(gs) >= 0)
    for g in range(E + 1):
        r = tb["blocks"][gs == g, 2]
        if len(r):
            assert np.all(r[:-1] == BM)


@pytest.mark.parametrize("BM", [1, 4, 128])
def test_route_tables(BM):
    L = _small_layer(D=128, E=16, k=4)
    x = synth.make_x(8, 37, L.D)
    _, idx, _ = O.route(O.OracleLayer(L), x)
    tb = O.route_tables(idx, L.E, BM)
    _check_tables(idx, L.E, BM, tb)
    for t in range(x.shape[0]):
        assert len(set(idx[t])) == L.k


def test_route_tables_empty():
    tb = O.route_tables(np.zeros((0, 4), np.int32), 8, 128)
    assert tb["count"].sum() == 0 and len(tb["perm"]) == 0 and len(tb["blocks"]) == 0


def _torch_ffn(L, which, e, x):
    """Dense SwiGLU expert with torch fp64 matmul on oracle-dequantised weights."""
    if which == "shared":
        g, u, d, e = L.s_gate, L.s_up, L.s_down, 0
    else:
        g, u, d = L.gate, L.up, L.down
    wg = torch.tensor(O.dequant(g, e, L.I, L.D))
    wu = torch.tensor(O.dequant(u, e, L.I, L.D))
    wd = torch.tensor(O.dequant(d, e, L.D, L.I))
    xt = torch.tensor(synth.bf16_bits_to_f32(x).astype(np.float64))
    h = torch.nn.functional.silu(xt @ wg.T) * (xt @ wu.T)
    return (h @ wd.T).numpy(), h.numpy()


def test_single_expert_reduces_to_dense_swiglu():
    # E = 1, k = 1: the layer is two dense SwiGLU FFNs with weight 1 each.
    L = _small_layer(D=192, E=1, k=1, I=128)
    x = synth.make_x(11, 7, L.D)
    y = O.forward(O.OracleLayer(L), x)
    y0, h0 = _torch_ffn(L, "routed", 0, x)
    ys, hs = _torch_ffn(L, "shared", 0, x)
    assert np.allclose(y, y0 + ys, rtol=1e-12, atol=1e-12)
    ol = O.OracleLayer(L)
    for t in range(3):
        assert np.allclose(O.expert_h(ol, 0, x[t]), h0[t], rtol=1e-12, atol=1e-14)
        assert np.allclose(O.expert_h(ol, -1, x[t]), hs[t], rtol=1e-12, atol=1e-14)


def test_uniform_routing_reduces_to_mean_of_experts():
    # k = E with W_r = 0: every expert weighs exactly 1/E.
    L = _small_layer(D=128, E=4, k=4, I=64)
    L.router_w = np.zeros_like(L.router_w)
    x = synth.make_x(12, 5, L.D)
    y = O.forward(O.OracleLayer(L), x)
    ref = _torch_ffn(L, "shared", 0, x)[0]
    for e in range(L.E):
        ref = ref + 0.25 * _torch_ffn(L, "routed", e, x)[0]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_all_zero_weights_give_zero_output():
    L = _small_layer(D=128, E=8, k=2, I=64)
    for m in (L.gate, L.up, L.down, L.s_gate, L.s_up, L.s_down):
        m.codes[:] = 0x88888888
        m.biases[:] = synth.f32_to_bf16_bits(-8.0 * synth.bf16_bits_to_f32(m.scales))
    x = synth.make_x(13, 4, L.D)
    assert np.array_equal(O.forward(O.OracleLayer(L), x), np.zeros((4, L.D)))


def test_shared_down_linearity():
    # Doubling the shared expert's down scales and biases doubles its term:
    # y(2x) - y(1x) equals the shared expert's output alone.
    L = _small_layer(D=128, E=8, k=2, I=64)
    x = synth.make_x(14, 6, L.D)
    y1 = O.forward(O.OracleLayer(L), x)
    L2 = copy.deepcopy(L)
    for arr in (L2.s_down.scales, L2.s_down.biases):
        arr[:] = synth.f32_to_bf16_bits(2.0 * synth.bf16_bits_to_f32(arr))
    y2 = O.forward(O.OracleLayer(L2), x)
    ys = _torch_ffn(L, "shared", 0, x)[0]
    assert np.allclose(y2 - y1, ys, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("cfg", [dict(D=256, E=16, k=2, I=128, T=16, seed=0),
                                 dict(D=512, E=32, k=8, I=128, T=8, seed=21)])
def test_sparse_equals_dense_masked(cfg):
    T = cfg.pop("T")
    seed = cfg.pop("seed")
    L = synth.make_layer(seed, **cfg)
    x = synth.make_x(seed, T, L.D)
    ol = O.OracleLayer(L)
    y = O.forward(ol, x)
    yd = O.forward_dense_masked(ol, x)
    assert np.allclose(y, yd, rtol=1e-12, atol=1e-12 * np.abs(yd).max())


def test_token_subset_matches_full():
    L, x = synth.make_config("tiny")
    ol = O.OracleLayer(L)
    y = O.forward(ol, x)
    sel = np.array([15, 0, 7])
    assert np.array_equal(O.forward(ol, x, tokens=sel, n_threads=2), y[sel])
