"""CUDA path vs the CPU oracle, through the C ABI, on the five workloads and
edge cases. Routing tables and logits must be bit-exact; the layer output must
be within the tolerance of gpu_util.check_output."""
import ctypes
import functools

import numpy as np
import pytest

import bit_moe_expert_routing_gb300 as moe
from bit_moe_expert_routing_gb300 import build, synth
from oracle import oracle as O

from gpu_util import WEIGHT_ATOL, bf16_to_np, check_output, config, rne_bf16, x_to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    moe.lib()
    yield
    moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_AUTO)
    moe.moe_set_option(moe.MOE_OPT_GEMM_IMPL, moe.GEMM_TENSOR_CORE)


_dev_layers = {}


def dev_layer(name, layer):
    key = (name, id(layer))
    if key not in _dev_layers:
        _dev_layers[key] = moe.DeviceLayer(layer)
    return _dev_layers[key]


def run_forward(dl, x_bits, path=moe.PATH_AUTO, impl=moe.GEMM_TENSOR_CORE):
    assert moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, path) == moe.MOE_OK
    assert moe.moe_set_option(moe.MOE_OPT_GEMM_IMPL, impl) == moe.MOE_OK
    x = x_to_device(x_bits)
    ws = dl.workspace(x.shape[0])
    y = dl.forward(x, workspace=ws)
    torch.cuda.synchronize()
    st = moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), None)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    return bf16_to_np(y), ws


# --- dequantisation ------------------------------------------------------------------------

def test_debug_dequant_matches_rounded_oracle():
    layer, _ = config("tiny")
    dl = dev_layer("tiny", layer)
    for m, qm, rows, K in ((layer.gate, dl.w.gate, layer.I, layer.D), (layer.down, dl.w.down, layer.D, layer.I)):
        for e in (0, 3, layer.E - 1):
            out = torch.empty(rows * K, dtype=torch.int16, device="cuda")
            assert moe.moe_debug_dequant(qm, e, rows, K, out.data_ptr(), None) == moe.MOE_OK
            torch.cuda.synchronize()
            got = synth.bf16_bits_to_f32(out.cpu().numpy().view(np.uint16)).astype(np.float64)
            want = rne_bf16(O.dequant(m, e, rows, K)).reshape(-1)
            assert np.array_equal(got, want)


def test_debug_dequant_golden_vectors():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "dequant_vectors.txt")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        name, word, s, b, exact, rne = [p.strip() for p in line.split("|")]
        codes = torch.tensor([int(word, 16)] * 8, dtype=torch.int64).to(torch.int32).cuda()
        sc = torch.tensor([int(s, 16)], dtype=torch.int32).to(torch.int16).cuda()
        bi = torch.tensor([int(b, 16)], dtype=torch.int32).to(torch.int16).cuda()
        qm = moe.moe_qmatrix(codes.data_ptr(), sc.data_ptr(), bi.data_ptr())
        out = torch.empty(64, dtype=torch.int16, device="cuda")
        assert moe.moe_debug_dequant(qm, 0, 1, 64, out.data_ptr(), None) == moe.MOE_OK
        torch.cuda.synchronize()
        got = synth.bf16_bits_to_f32(out.cpu().numpy().view(np.uint16))
        assert np.array_equal(got, np.tile(np.array([float(v) for v in rne.split()], np.float32), 8)), name


# --- routing: bit-exact --------------------------------------------------------------------

def check_logits(got, want):
    """Logits bit for bit; a NaN only has to be a NaN on both sides (the
    payload bits of a NaN that an fma propagates differ between the CPU and
    the GPU, and the rank of a NaN does not depend on them)."""
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan), "NaN logits differ"
    assert np.array_equal(got.view(np.uint32)[~nan], want.view(np.uint32)[~nan]), "router logits differ in bits"


def check_routing(layer, x_bits, name):
    dl = dev_layer(name, layer)
    x = x_to_device(x_bits)
    T = x.shape[0]
    ws = dl.workspace(T)
    v = dl.route(x, ws)
    torch.cuda.synchronize()
    ol = O.OracleLayer(layer)
    logits, idx, w = O.route(ol, x_bits)
    tb = O.route_tables(idx, layer.E, v.block_m)
    g = lambda p, shape, dt: moe.ws_tensor(ws, p, shape, dt).cpu().numpy()
    A = T * layer.k
    check_logits(g(v.logits, (T, layer.E), torch.float32), logits)
    assert np.array_equal(g(v.topk_idx, (T, layer.k), torch.int32), idx)
    assert np.abs(g(v.topk_w, (T, layer.k), torch.float32) - w).max() <= WEIGHT_ATOL
    assert np.array_equal(g(v.count, (layer.E,), torch.int32), tb["count"])
    assert np.array_equal(g(v.off, (layer.E + 1,), torch.int32), tb["off"])
    assert np.array_equal(g(v.perm, (A,), torch.int32), tb["perm"])
    assert np.array_equal(g(v.inv, (A,), torch.int32), tb["inv"])
    nb = int(g(v.n_blocks, (1,), torch.int32)[0])
    assert nb == len(tb["blocks"])
    assert np.array_equal(g(v.blocks, (v.max_blocks, 3), torch.int32)[:nb], tb["blocks"])
    assert moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), None) == moe.MOE_OK
    return tb


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill512", "prefill4096_zipf", "sweep"])
def test_routing_bit_exact(name):
    layer, x = config(name)
    tb = check_routing(layer, x, name)
    if name == "prefill4096_zipf":
        assert tb["count"].max() > 1000 and (tb["count"] == 0).any()


@pytest.mark.parametrize("T", [1, 2, 3, 63, 64, 65, 200])
def test_routing_ragged_token_counts(T):
    layer = synth.make_layer(31, 256, 16, 4, 128)
    check_routing(layer, synth.make_x(31, T, 256), f"ragged{T}")


def test_routing_ties_go_to_lower_index():
    layer = synth.make_layer(32, 256, 16, 4, 128)
    layer.router_w[9] = layer.router_w[3]
    layer.router_w[12] = layer.router_w[2]
    layer.router_w[15] = layer.router_w[2]
    x = synth.make_x(32, 96, 256)
    check_routing(layer, x, "ties")


def _special_logit_layer(k):
    """A 16-expert layer whose router yields every kind of logit the ordering
    rule covers: expert 2 NaN (one NaN weight), 7 -inf (bias), 5 and 11 +0
    (zero rows); expert 9's row is -2^-140 everywhere, so a token whose x is
    2^-12 everywhere gets the logit -0 from it (each product rounds to -0),
    and a token whose x is -2^-12 gets +0. The other rows carry a bias of -3,
    so the zero-valued logits lead the top-k."""
    layer = synth.make_layer(36, 256, 16, k, 128)
    layer.router_w[2, 7] = np.nan
    layer.router_w[5, :] = 0.0
    layer.router_w[11, :] = 0.0
    layer.router_w[9, :] = -np.float32(2.0 ** -140)
    bias = np.full(16, -3.0, np.float32)
    bias[[5, 9, 11]] = -0.0  # -0 + -0 keeps the sign; +0 + -0 is +0
    bias[7] = -np.inf
    layer.router_bias = bias
    return layer


def _special_logit_tokens(T):
    x = synth.make_x(36, T, 256)
    x[0] = synth.f32_to_bf16_bits(np.full(256, 2.0 ** -12, np.float32))
    x[1] = synth.f32_to_bf16_bits(np.full(256, -(2.0 ** -12), np.float32))
    return x


@pytest.mark.parametrize("T", [3, 70])
@pytest.mark.parametrize("k", [6, 16])
def test_routing_non_finite_and_signed_zero_logits(k, T):
    # NaN ranks as -inf, -0 equals +0, and equal values go to the lower
    # expert index, on the small-T and the larger-T routing kernels; with
    # k = E every expert is kept, so NaN and -inf take the last two slots in
    # index order with weight 0.
    layer = _special_logit_layer(k)
    x = _special_logit_tokens(T)
    logits, idx, _ = O.route(O.OracleLayer(layer), x)
    assert np.signbit(logits[0, 9]) and logits[0, 9] == 0 and not np.signbit(logits[1, 9])
    assert np.isnan(logits[:, 2]).all() and np.isneginf(logits[:, 7]).all()
    assert list(idx[0, :3]) == [5, 9, 11]
    if k == 16:
        assert list(idx[0, -2:]) == [2, 7]
    check_routing(layer, x, f"special{k}_{T}")


@pytest.mark.parametrize("path", [moe.PATH_GEMV, moe.PATH_GEMM], ids=["gemv", "gemm"])
@pytest.mark.parametrize("T", [1, 3])
def test_layer_with_non_finite_and_signed_zero_logits(path, T):
    # every expert kept (k = E): the NaN and -inf experts carry weight 0, so
    # the layer output stays finite and matches the oracle
    layer = _special_logit_layer(16)
    x = _special_logit_tokens(max(T, 2))[:T]
    dl = moe.DeviceLayer(layer)
    y, ws = run_forward(dl, x, path)
    assert np.isfinite(y).all()
    ol = O.OracleLayer(layer)
    check_output(y, O.forward(ol, x), f"special logits T={T}")
    # the top-k the forward itself wrote into its workspace
    _, idx, w = O.route(ol, x)
    v = dl.view(T, ws)
    assert np.array_equal(moe.ws_tensor(ws, v.topk_idx, (T, 16), torch.int32).cpu().numpy(), idx)
    assert np.abs(moe.ws_tensor(ws, v.topk_w, (T, 16), torch.float32).cpu().numpy() - w).max() <= WEIGHT_ATOL


@pytest.mark.parametrize("T", [3, 16, 70])
def test_routing_logit_order_matches_the_canonical_tree(T):
    # Rows whose fp32 logit depends on the summation order (the tree gives
    # 254 and 247, one sequential chain 223 and 254): the kernels for small T
    # and for larger T both follow the oracle's order bit for bit.
    layer = synth.make_layer(34, 256, 16, 4, 128)
    big = np.float32(2.0 ** 24)
    layer.router_w[0, :] = 1.0
    layer.router_w[0, 0], layer.router_w[0, 32] = big, -big
    layer.router_w[5, :] = 1.0
    layer.router_w[5, 0], layer.router_w[5, 1] = big, -big
    x = synth.f32_to_bf16_bits(np.ones((T, 256), np.float32))
    check_routing(layer, x, f"order{T}")


@pytest.mark.parametrize("bm", [16, 48, 192])
def test_routing_block_size_option(bm):
    layer = synth.make_layer(35, 256, 16, 4, 128)
    assert moe.moe_set_option(moe.MOE_OPT_BLOCK_M, bm) == moe.MOE_OK
    try:
        tb = check_routing(layer, synth.make_x(35, 200, 256), f"bm{bm}")
        assert tb["blocks"][:, 2].max() <= bm
    finally:
        moe.moe_set_option(moe.MOE_OPT_BLOCK_M, 0)


@pytest.mark.parametrize("impl", [moe.GEMM_TENSOR_CORE, moe.GEMM_TENSOR_CORE_SMEM, moe.GEMM_CUDA_CORE],
                         ids=["tc", "tc_smem", "simt"])
def test_layer_small_blocks(impl):
    # 16- and 48-row blocks: many partly filled tiles on every GEMM path
    layer, x = config("prefill512")
    for bm in (16, 48):
        assert moe.moe_set_option(moe.MOE_OPT_BLOCK_M, bm) == moe.MOE_OK
        try:
            y, ws = run_forward(dev_layer("prefill512", layer), x, moe.PATH_GEMM, impl)
        finally:
            moe.moe_set_option(moe.MOE_OPT_BLOCK_M, 0)
        toks = np.arange(0, x.shape[0], 7)
        check_output(y[toks], O.forward(O.OracleLayer(layer), x, tokens=toks), f"prefill512 bm={bm} impl={impl}")


def test_routing_all_equal_logits():
    layer = synth.make_layer(33, 128, 8, 8, 64)
    layer.router_w[:] = 0
    check_routing(layer, synth.make_x(33, 5, 128), "equal")


# --- the layer -----------------------------------------------------------------------------

PATHS = [("gemm_tc", moe.PATH_GEMM, moe.GEMM_TENSOR_CORE), ("gemm_simt", moe.PATH_GEMM, moe.GEMM_CUDA_CORE),
         ("gemv", moe.PATH_GEMV, moe.GEMM_TENSOR_CORE)]


@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 16])
def test_layer_tiny(path, T):
    layer, x = config("tiny")
    x = x[:T]
    _, p, impl = path
    if p == moe.PATH_GEMV and T > 8:
        pytest.skip("the GEMV path takes at most 8 rows")
    y, _ = run_forward(dev_layer("tiny", layer), x, p, impl)
    check_output(y, O.forward(O.OracleLayer(layer), x), f"tiny T={T} {path[0]}")


@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
def test_layer_decode(path):
    layer, x = config("decode")
    y, _ = run_forward(dev_layer("decode", layer), x, path[1], path[2])
    check_output(y, O.forward(O.OracleLayer(layer), x), f"decode {path[0]}")


@pytest.mark.parametrize("fused", [0, 1], ids=["separate", "fused"])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_layer_decode_fused_and_separate(fused, T):
    # a few rows on the GEMV path: the one-launch cooperative kernels (one
    # token: router, grid barrier, top-k, gate/up and down per 32-row item,
    # combine; 2..8 rows: a second grid barrier before down) and the separate
    # routing + GEMV kernels, all against the oracle, with the routing tables
    # each leaves in its workspace
    layer, x = config("sweep") if T > 1 else config("decode")
    x = x[:T]
    name = "sweep" if T > 1 else "decode"
    assert moe.moe_set_option(moe.MOE_OPT_DECODE_FUSED, fused) == moe.MOE_OK
    try:
        dl = dev_layer(name, layer)
        ws = dl.workspace(T)
        ws.fill_(0x5A)  # no table may come from an earlier call
        assert moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_GEMV) == moe.MOE_OK
        y = bf16_to_np(dl.forward(x_to_device(x), workspace=ws))
        launches = moe.moe_last_launch_count()
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), None) == moe.MOE_OK
    finally:
        moe.moe_set_option(moe.MOE_OPT_DECODE_FUSED, 1)
    ol = O.OracleLayer(layer)
    check_output(y, O.forward(ol, x), f"T={T} fused={fused}")
    assert launches == (1 if fused else 4)
    v = dl.view(T, ws)
    g = lambda p_, shape, dt: moe.ws_tensor(ws, p_, shape, dt).cpu().numpy()
    logits, idx, w = O.route(ol, x)
    tb = O.route_tables(idx, layer.E, v.block_m)
    A = T * layer.k
    check_logits(g(v.logits, (T, layer.E), torch.float32), logits)
    assert np.array_equal(g(v.topk_idx, (T, layer.k), torch.int32), idx)
    assert np.abs(g(v.topk_w, (T, layer.k), torch.float32) - w).max() <= WEIGHT_ATOL
    assert np.array_equal(g(v.count, (layer.E,), torch.int32), tb["count"])
    assert np.array_equal(g(v.off, (layer.E + 1,), torch.int32), tb["off"])
    assert np.array_equal(g(v.perm, (A,), torch.int32), tb["perm"])
    assert np.array_equal(g(v.inv, (A,), torch.int32), tb["inv"])
    nb = int(g(v.n_blocks, (1,), torch.int32)[0])
    assert nb == len(tb["blocks"])
    assert np.array_equal(g(v.blocks, (v.max_blocks, 3), torch.int32)[:nb], tb["blocks"])


@pytest.mark.parametrize("name", ["decode", "tiny"])
def test_one_token_kernel_h_and_repeated_calls(name):
    # The one-token kernel leaves h slot-major: row j < k for the token's j-th
    # expert, row k for the shared expert, each the oracle's SwiGLU
    # intermediate. Its combine adds fp32 partials in arrival order, so
    # repeated calls agree up to the summation order, and each matches the
    # oracle.
    layer, x = config(name)
    x = x[:1]
    dl = dev_layer(name, layer)
    ol = O.OracleLayer(layer)
    k = layer.k
    ys = []
    for _ in range(4):
        y, ws = run_forward(dl, x, moe.PATH_GEMV)
        assert moe.moe_last_launch_count() == 1
        ys.append(y)
    v = dl.view(1, ws)
    h = bf16_to_np(moe.ws_tensor(ws, v.h, (k + 1, layer.I), torch.bfloat16))
    idx = moe.ws_tensor(ws, v.topk_idx, (1, k), torch.int32).cpu().numpy()
    ref = np.stack([O.expert_h(ol, int(idx[0, j]), x[0]) for j in range(k)] + [O.expert_h(ol, -1, x[0])])
    check_output(h, ref, f"{name}: one-token h")
    want = O.forward(ol, x)
    for y in ys:
        check_output(y, want, f"{name}: one-token y")
        assert np.allclose(y, ys[0], rtol=2 ** -7, atol=1e-6)


@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
@pytest.mark.parametrize("T", synth.SWEEP_T)
def test_layer_crossover_sweep(path, T):
    layer, x = config("sweep")
    x = x[:T]
    y, _ = run_forward(dev_layer("sweep", layer), x, path[1], path[2])
    check_output(y, O.forward(O.OracleLayer(layer), x), f"sweep T={T} {path[0]}")


@pytest.mark.parametrize("impl", [moe.GEMM_TENSOR_CORE, moe.GEMM_CUDA_CORE], ids=["tc", "simt"])
def test_layer_prefill512_all_tokens(impl):
    layer, x = config("prefill512")
    y, _ = run_forward(dev_layer("prefill512", layer), x, moe.PATH_GEMM, impl)
    check_output(y, O.forward(O.OracleLayer(layer), x), "prefill512")


@pytest.mark.parametrize("chunk,extra", [(200, 0), (256, 3)], ids=["3-passes", "ragged-gemv-tail"])
def test_layer_chunked_prefill(chunk, extra):
    # Prompt chunking: 512 (+3) tokens in passes of `chunk` tokens reusing one
    # workspace sized for a single pass. Passes 200, 200, 112; or 256, 256, 3,
    # whose last pass takes the decode GEMV path. Each token's output matches
    # the oracle, and the one-pass output up to the combine's summation order.
    layer, x = config("prefill512")
    if extra:
        x = np.concatenate([x, x[:extra]])
    T = x.shape[0]
    dl = dev_layer("prefill512", layer)
    y_one, _ = run_forward(dl, x)
    old = moe.moe_get_option(moe.MOE_OPT_CHUNK_TOKENS)
    old_rows = moe.moe_get_option(moe.MOE_OPT_GEMV_MAX_ROWS)
    try:
        assert moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, chunk) == moe.MOE_OK
        assert moe.moe_set_option(moe.MOE_OPT_GEMV_MAX_ROWS, 4) == moe.MOE_OK  # the 3-token tail takes the GEMV path
        assert moe.moe_workspace_size(dl.w, T) == moe.moe_workspace_size(dl.w, chunk)
        y, _ = run_forward(dl, x)
        launches = moe.moe_last_launch_count()
    finally:
        moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, old)
        moe.moe_set_option(moe.MOE_OPT_GEMV_MAX_ROWS, old_rows)
    assert launches > 8  # more than one pass ran
    # rows that took the same (GEMM) path in both runs agree up to summation
    # order; a GEMV tail pass rounds differently (fp32 weights) and is held to
    # the oracle only
    same = T - extra
    assert np.allclose(y[:same], y_one[:same], rtol=2 ** -7, atol=1e-6)
    check_output(y, O.forward(O.OracleLayer(layer), x), f"chunked prefill, {chunk}-token passes")


@pytest.mark.parametrize("path", [moe.PATH_GEMV, moe.PATH_GEMM], ids=["gemv", "gemm"])
def test_layer_host_synchronised_routing(path):
    # the host round trip after routing changes nothing in the result
    layer, x = config("prefill512")
    x = x[:3] if path == moe.PATH_GEMV else x
    dl = dev_layer("prefill512", layer)
    y_ref, _ = run_forward(dl, x, path)
    assert moe.moe_set_option(moe.MOE_OPT_HOST_SYNC_ROUTING, 1) == moe.MOE_OK
    try:
        y, _ = run_forward(dl, x, path)
    finally:
        moe.moe_set_option(moe.MOE_OPT_HOST_SYNC_ROUTING, 0)
    assert np.allclose(y, y_ref, rtol=2 ** -7, atol=1e-6)
    check_output(y, O.forward(O.OracleLayer(layer), x), "host-synchronised routing")


def _sample_tokens(idx, count, T):
    heavy = int(np.argmax(count))
    light = int(np.argmin(np.where(count > 0, count, 1 << 30)))
    on_heavy = np.where((idx == heavy).any(1))[0]
    on_light = np.where((idx == light).any(1))[0]
    pick = list(range(8)) + list(range(T - 8, T)) + list(on_heavy[:8]) + list(on_light[:4]) + \
        list(np.random.default_rng(0).choice(T, 12, replace=False))
    return np.array(sorted(set(int(t) for t in pick)), dtype=np.int32)


@functools.lru_cache(maxsize=1)
def _prefill4096_reference():
    """The oracle's output for all 4096 tokens of the Zipf-routed prefill
    workload (about 20 s on 16 host cores), shared by the tests below."""
    layer, x = config("prefill4096_zipf")
    return O.forward(O.OracleLayer(layer), x)


def test_layer_prefill4096_zipf_all_tokens():
    # the headline configuration in the launch configuration the benchmark
    # times (tensor-core path, 192-token blocks): every token of the output,
    # element by element, against the oracle
    layer, x = config("prefill4096_zipf")
    y, _ = run_forward(dev_layer("prefill4096_zipf", layer), x, moe.PATH_GEMM, moe.GEMM_TENSOR_CORE)
    assert np.isfinite(y).all()
    ref = _prefill4096_reference()
    check_output(y, ref, "prefill4096, all tokens")
    # and per token block of 256, so that one bad tile cannot hide in the mean
    for t0 in range(0, x.shape[0], 256):
        check_output(y[t0:t0 + 256], ref[t0:t0 + 256], f"prefill4096 tokens {t0}..{t0 + 255}")


def test_layer_prefill4096_zipf_repeated_calls():
    # An ordering race between the MMA issuer and the epilogue corrupted about
    # one down launch in four before it was fixed: repeated calls on the same
    # workspace must all match the oracle.
    layer, x = config("prefill4096_zipf")
    dl = dev_layer("prefill4096_zipf", layer)
    ref = _prefill4096_reference()
    moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_GEMM)
    moe.moe_set_option(moe.MOE_OPT_GEMM_IMPL, moe.GEMM_TENSOR_CORE)
    xd = x_to_device(x)
    ws = dl.workspace(x.shape[0])
    for i in range(8):
        y = bf16_to_np(dl.forward(xd, workspace=ws))
        assert moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), None) == moe.MOE_OK
        check_output(y, ref, f"prefill4096 call {i}")


@pytest.mark.parametrize("name,T", [("prefill512", 512), ("sweep", 3)])
def test_layer_graph_replay(name, T):
    # The layer captured in a CUDA graph (its prefill kernels are programmatic
    # dependent launches, captured as such) and replayed: every replay matches
    # the oracle, and the first equals a stream-launched call up to the fp32
    # order of the combine's atomic adds.
    layer, x = config(name)
    x = x[:T]
    dl = dev_layer(name, layer)
    moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_GEMM)
    moe.moe_set_option(moe.MOE_OPT_GEMM_IMPL, moe.GEMM_TENSOR_CORE)
    xd = x_to_device(x)
    ws = dl.workspace(T)
    y_stream = bf16_to_np(dl.forward(xd, workspace=ws))
    y = torch.empty_like(xd)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        dl.forward(xd, y=y, workspace=ws, stream=side)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        dl.forward(xd, y=y, workspace=ws, stream=side)
    ref = O.forward(O.OracleLayer(layer), x)
    for i in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), None) == moe.MOE_OK
        yn = bf16_to_np(y)
        check_output(yn, ref, f"graph replay {i} {name} T={T}")
        assert np.allclose(yn, y_stream, rtol=2 ** -7, atol=1e-6)


def test_layer_prefill4096_zipf_sampled_cuda_core():
    layer, x = config("prefill4096_zipf")
    y, _ = run_forward(dev_layer("prefill4096_zipf", layer), x, moe.PATH_GEMM, moe.GEMM_CUDA_CORE)
    ol = O.OracleLayer(layer)
    _, idx, _ = O.route(ol, x)
    toks = _sample_tokens(idx, np.bincount(idx.reshape(-1), minlength=layer.E), x.shape[0])
    check_output(y[toks], _prefill4096_reference()[toks], "prefill4096 sampled, CUDA cores")
    assert np.isfinite(y).all()


@pytest.mark.parametrize("name", ["tiny", "prefill512"])
def test_layer_expanded_weights_matches_fused(name):
    # The unfused form (a separate pass expands the selected experts' weights
    # to bf16, then the GEMMs read them) against the fused shared-memory
    # GEMM: the same weights rounded the same way, so h is identical bit for
    # bit (y differs only in the order of its fp32 atomic adds); the output
    # matches the oracle; and a selected expert's expanded matrices equal
    # moe_debug_dequant's.
    layer, x = config(name)
    dl = dev_layer(name, layer)
    T, k, I, D, E = x.shape[0], layer.k, layer.I, layer.D, layer.E
    y_fused, ws_f = run_forward(dl, x, moe.PATH_GEMM, moe.GEMM_TENSOR_CORE_SMEM)
    n_fused = moe.moe_last_launch_count()
    v = dl.view(T, ws_f)
    h_fused = moe.ws_tensor(ws_f, v.h, (T * k + T, I), torch.int16).clone()
    xd = x_to_device(x)
    ws = dl.workspace(T)
    nb = moe.moe_expanded_weights_bytes(dl.w)
    wbuf = torch.empty(nb, dtype=torch.uint8, device="cuda")
    y = torch.empty_like(xd)
    st = moe.moe_layer_forward_expanded(dl.w, xd.data_ptr(), T, y.data_ptr(), ws.data_ptr(), ws.numel(),
                                        wbuf.data_ptr(), nb, None)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), None) == moe.MOE_OK
    assert moe.moe_last_launch_count() == n_fused + 6  # the same kernels plus six expansion launches
    v = dl.view(T, ws)
    h = moe.ws_tensor(ws, v.h, (T * k + T, I), torch.int16)
    assert torch.equal(h, h_fused)
    yn = bf16_to_np(y)
    assert np.allclose(yn, y_fused, rtol=2 ** -7, atol=1e-6)
    check_output(yn, O.forward(O.OracleLayer(layer), x), f"expanded weights {name}")
    # one selected expert's matrices and the shared expert's down matrix
    idx = moe.ws_tensor(ws, v.topk_idx, (T, k), torch.int32).cpu().numpy()
    e = int(idx[0, 0])
    wb = wbuf.view(torch.int16)
    gu = I * D
    for m, ex, off, rows, K in ((dl.w.gate, e, e * gu, I, D), (dl.w.up, e, (E + e) * gu, I, D),
                                (dl.w.down, e, (2 * E + e) * gu, D, I), (dl.w.s_down, 0, (3 * E + 2) * gu, D, I)):
        want = torch.empty(rows * K, dtype=torch.int16, device="cuda")
        assert moe.moe_debug_dequant(m, ex, rows, K, want.data_ptr(), None) == moe.MOE_OK
        torch.cuda.synchronize()
        assert torch.equal(wb[off:off + rows * K], want)


def test_intermediate_h_matches_oracle():
    layer, x = config("tiny")
    dl = dev_layer("tiny", layer)
    ol = O.OracleLayer(layer)
    for p, impl in ((moe.PATH_GEMM, moe.GEMM_TENSOR_CORE), (moe.PATH_GEMM, moe.GEMM_CUDA_CORE),
                    (moe.PATH_GEMV, moe.GEMM_TENSOR_CORE)):
        xx = x[:8]
        _, ws = run_forward(dl, xx, p, impl)
        v = dl.view(xx.shape[0], ws)
        T, k = xx.shape[0], layer.k
        h = bf16_to_np(moe.ws_tensor(ws, v.h, (T * k + T, layer.I), torch.bfloat16))
        perm = moe.ws_tensor(ws, v.perm, (T * k,), torch.int32).cpu().numpy()
        idx = moe.ws_tensor(ws, v.topk_idx, (T, k), torch.int32).cpu().numpy()
        ref = np.stack([O.expert_h(ol, int(idx[a // k, a % k]), xx[a // k]) for a in perm] +
                       [O.expert_h(ol, -1, xx[t]) for t in range(T)])
        check_output(h, ref, f"h path={p} impl={impl}")


@pytest.mark.parametrize("shape", [dict(D=128, E=1, k=1, I=64), dict(D=192, E=8, k=8, I=128),
                                   dict(D=320, E=40, k=3, I=192), dict(D=1024, E=64, k=6, I=256)],
                         ids=["E1k1", "kE", "odd", "mid"])
@pytest.mark.parametrize("T", [1, 7, 130])
def test_layer_shapes(shape, T):
    layer = synth.make_layer(40, **shape)
    x = synth.make_x(40, T, shape["D"])
    dl = moe.DeviceLayer(layer)
    ref = O.forward(O.OracleLayer(layer), x)
    for p, impl in ((moe.PATH_GEMM, moe.GEMM_TENSOR_CORE), (moe.PATH_GEMM, moe.GEMM_CUDA_CORE),
                    (moe.PATH_GEMV, moe.GEMM_TENSOR_CORE)):
        if p == moe.PATH_GEMV and T > 8:
            continue
        y, _ = run_forward(dl, x, p, impl)
        check_output(y, ref, f"{shape} T={T} path={p} impl={impl}")


# Largest sizes the boundary accepts along each axis (E = 1024 with k = 32,
# D = 16384, I = 4096), E = 512, the largest the one-token fused kernel takes
# (16 logits per lane), and k = 30 on the fused kernel (more down slots than
# the 28 lanes that issue their copies in one pass). Where a path's limits exclude a shape, the call
# falls back to the path that takes it; every result is held to the oracle.
@pytest.mark.parametrize("shape", [dict(D=128, E=1024, k=32, I=128), dict(D=16384, E=4, k=2, I=128),
                                   dict(D=128, E=4, k=2, I=4096), dict(D=256, E=512, k=8, I=128),
                                   dict(D=128, E=64, k=30, I=128)],
                         ids=["E1024k32", "D16384", "I4096", "E512", "k30-fused"])
@pytest.mark.parametrize("T", [1, 7, 130])
def test_layer_max_shapes(shape, T):
    layer = synth.make_layer(41, **shape)
    x = synth.make_x(41, T, shape["D"])
    dl = moe.DeviceLayer(layer)
    ref = O.forward(O.OracleLayer(layer), x)
    for p in (moe.PATH_GEMM, moe.PATH_GEMV):
        if p == moe.PATH_GEMV and T > 8:
            continue
        y, ws = run_forward(dl, x, p)
        check_output(y, ref, f"{shape} T={T} path={p}")
        v = dl.view(T, ws)
        idx = moe.ws_tensor(ws, v.topk_idx, (T, layer.k), torch.int32).cpu().numpy()
        _, ridx, _ = O.route(O.OracleLayer(layer), x)
        assert np.array_equal(idx, ridx)


def test_long_k_gemm_is_stable_over_repeats():
    # 128 pipeline stages per gate/up tile (D = 16384). A dequantising warp
    # once reused the registers of a tensor-memory store for the next group
    # before the store had read them (tcgen05.st reads its sources
    # asynchronously), which corrupted a group now and then: scattered errors
    # in about half the runs. Ten runs on workspaces holding stale bytes must
    # all match the oracle.
    shape = dict(D=16384, E=4, k=2, I=128)
    layer = synth.make_layer(41, **shape)
    x = synth.make_x(41, 130, shape["D"])
    dl = moe.DeviceLayer(layer)
    ref = O.forward(O.OracleLayer(layer), x)
    assert moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_GEMM) == moe.MOE_OK
    assert moe.moe_set_option(moe.MOE_OPT_GEMM_IMPL, moe.GEMM_TENSOR_CORE) == moe.MOE_OK
    xd = x_to_device(x)
    for r in range(10):
        ws = dl.workspace(130)
        ws.fill_(0x3F)
        y = bf16_to_np(dl.forward(xd, workspace=ws))
        torch.cuda.synchronize()
        check_output(y, ref, f"long-K GEMM, repeat {r}")


def test_zero_tokens_is_noop():
    layer, _ = config("tiny")
    dl = dev_layer("tiny", layer)
    ws = dl.workspace(0)
    r = moe.moe_layer_forward(dl.w, 0, 0, 0, ws.data_ptr(), ws.numel(), None)
    assert r == moe.MOE_OK and moe.moe_last_launch_count() == 0


def test_workspace_too_small_rejected():
    layer, x = config("tiny")
    dl = dev_layer("tiny", layer)
    xd = x_to_device(x)
    y = torch.empty_like(xd)
    ws = dl.workspace(x.shape[0])
    r = moe.moe_layer_forward(dl.w, xd.data_ptr(), x.shape[0], y.data_ptr(), ws.data_ptr(), ws.numel() - 256,
                              None)
    assert r == moe.MOE_ERR_WORKSPACE


@pytest.mark.parametrize("path", [moe.PATH_GEMV, moe.PATH_GEMM], ids=["gemv", "gemm"])
def test_host_buffers_entry_point_matches_device_entry_point(path):
    layer, x = config("sweep")
    x = x[:5]
    dl = dev_layer("sweep", layer)
    y_dev, _ = run_forward(dl, x, path)
    ws = dl.workspace(5, host_staging=True)
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    r = moe.moe_layer_forward_host(dl.w, xh.data_ptr(), 5, yh.data_ptr(), ws.data_ptr(), ws.numel(), None)
    assert r == moe.MOE_OK
    y_host = synth.bf16_bits_to_f32(yh.numpy().view(np.uint16)).astype(np.float64)
    # both paths combine with fp32 atomic adds: equal up to the summation order
    assert np.allclose(y_host, y_dev, rtol=2 ** -7, atol=1e-6)
    check_output(y_host, O.forward(O.OracleLayer(layer), x), "host entry point")


@pytest.mark.parametrize("y_pinned", [True, False], ids=["y-written-directly", "y-staged"])
def test_host_entry_slices_its_input_copy(y_pinned):
    # 2100 tokens go in as slices of whole router waves (four at E = 256 on a
    # 152-SM GPU, the last one ragged) on the library's copy stream, and the
    # router runs on each slice as it lands. Page-locked y is written by the
    # layer's last kernel directly; pageable y is staged and copied back.
    # Logits, top-k and weights must equal the device entry point's bit for
    # bit; y agrees up to the fp32 combine's summation order.
    layer, x = config("prefill4096_zipf")
    x = x[:2100]
    T = x.shape[0]
    dl = dev_layer("prefill4096_zipf", layer)
    y_dev, ws_dev = run_forward(dl, x, moe.PATH_GEMM)
    ws = dl.workspace(T, host_staging=True)
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    yh = torch.empty_like(xh)
    if y_pinned:
        yh = yh.pin_memory()
    r = moe.moe_layer_forward_host(dl.w, xh.data_ptr(), T, yh.data_ptr(), ws.data_ptr(), ws.numel(), None)
    assert r == moe.MOE_OK
    assert moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), None) == moe.MOE_OK

    def tables(w_):
        v = moe.moe_route_view()
        assert moe.moe_workspace_view(dl.w, T, w_.data_ptr(), w_.numel(), v) == moe.MOE_OK
        g = lambda p, shape, dt: moe.ws_tensor(w_, p, shape, dt).cpu().numpy()
        return (g(v.logits, (T, layer.E), torch.float32).view(np.uint32),
                g(v.topk_idx, (T, layer.k), torch.int32),
                g(v.topk_w, (T, layer.k), torch.float32).view(np.uint32))

    for a, b, what in zip(tables(ws), tables(ws_dev), ("logits", "top-k", "weights")):
        assert np.array_equal(a, b), what
    y_host = synth.bf16_bits_to_f32(yh.numpy().view(np.uint16)).astype(np.float64)
    assert np.allclose(y_host, y_dev, rtol=2 ** -7, atol=1e-6)


def test_host_entry_chunked_passes_and_unaligned_y():
    # 1300 tokens in passes of 608 (608, 608, 84): each pass copies its x on
    # the library's copy stream once the previous pass is done with the
    # staging buffer, and reuses the slice events. y starts 2 bytes into a
    # page-locked buffer, so it is not 16-byte aligned: the layer writes it to
    # the staging buffer and copies it back. The output must match the device
    # entry point run with the same passes.
    layer, x = config("prefill4096_zipf")
    x = x[:1300]
    T = x.shape[0]
    dl = dev_layer("prefill4096_zipf", layer)
    old = moe.moe_get_option(moe.MOE_OPT_CHUNK_TOKENS)
    try:
        assert moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, 608) == moe.MOE_OK
        y_dev, _ = run_forward(dl, x, moe.PATH_GEMM)
        ws = dl.workspace(T, host_staging=True)
        xh = torch.from_numpy(x.view(np.int16)).pin_memory()
        buf = torch.empty(T * layer.D + 8, dtype=torch.int16).pin_memory()
        yh = buf[1:1 + T * layer.D]
        assert yh.data_ptr() % 16 == 2
        r = moe.moe_layer_forward_host(dl.w, xh.data_ptr(), T, yh.data_ptr(), ws.data_ptr(), ws.numel(), None)
        assert r == moe.MOE_OK
        assert moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), None) == moe.MOE_OK
    finally:
        moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, old)
    y_host = synth.bf16_bits_to_f32(yh.numpy().view(np.uint16).reshape(T, layer.D)).astype(np.float64)
    assert np.allclose(y_host, y_dev, rtol=2 ** -7, atol=1e-6)


def test_device_status_survives_later_passes():
    # 515 tokens in passes of 256, 256 and 3: the test hook makes the
    # grouped-GEMM passes record MOE_ERR_DEVICE_TIMEOUT, the 3-token GEMV pass
    # runs no such wait; its first kernel must not clear the call's status
    layer, x = config("prefill512")
    x = np.concatenate([x, x[:3]])
    dl = dev_layer("prefill512", layer)
    xd = x_to_device(x)
    ws = dl.workspace(x.shape[0])
    old = moe.moe_get_option(moe.MOE_OPT_CHUNK_TOKENS)
    old_rows = moe.moe_get_option(moe.MOE_OPT_GEMV_MAX_ROWS)
    try:
        assert moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, 256) == moe.MOE_OK
        assert moe.moe_set_option(moe.MOE_OPT_GEMV_MAX_ROWS, 4) == moe.MOE_OK  # the 3-token pass takes the GEMV path
        assert moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_AUTO) == moe.MOE_OK
        assert moe.moe_set_option(moe.MOE_OPT_TEST_WAIT_CYCLES, 20000) == moe.MOE_OK
        ws = dl.workspace(x.shape[0])
        dl.forward(xd, workspace=ws)
        assert moe.moe_set_option(moe.MOE_OPT_TEST_WAIT_CYCLES, 0) == moe.MOE_OK
        st = moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), None)
        assert st == moe.MOE_ERR_DEVICE_TIMEOUT, moe.moe_status_string(st)
        y, _ = run_forward(dl, x)  # a fresh call starts its status afresh
    finally:
        moe.moe_set_option(moe.MOE_OPT_TEST_WAIT_CYCLES, 0)
        moe.moe_set_option(moe.MOE_OPT_CHUNK_TOKENS, old)
        moe.moe_set_option(moe.MOE_OPT_GEMV_MAX_ROWS, old_rows)
    check_output(y, O.forward(O.OracleLayer(layer), x), "after a timeout in an earlier pass")


def test_gemv_paths_repeat():
    # The one-launch row kernel adds fp32 partials into the accumulator in
    # arrival order: repeated calls agree up to the summation order. The
    # separate GEMV kernels reduce in a fixed order: bit for bit.
    layer, x = config("sweep")
    dl = dev_layer("sweep", layer)
    a, _ = run_forward(dl, x[:3], moe.PATH_GEMV)
    b, _ = run_forward(dl, x[:3], moe.PATH_GEMV)
    assert np.allclose(a, b, rtol=2 ** -7, atol=1e-6)
    assert moe.moe_set_option(moe.MOE_OPT_DECODE_FUSED, 0) == moe.MOE_OK
    try:
        c, _ = run_forward(dl, x[:3], moe.PATH_GEMV)
        d, _ = run_forward(dl, x[:3], moe.PATH_GEMV)
    finally:
        moe.moe_set_option(moe.MOE_OPT_DECODE_FUSED, 1)
    assert np.array_equal(c, d)


def test_kernel_timing_and_launch_count():
    layer, x = config("tiny")
    dl = dev_layer("tiny", layer)
    moe.moe_kernel_times()
    assert moe.moe_set_option(moe.MOE_OPT_KERNEL_TIMING, 1) == moe.MOE_OK
    try:
        run_forward(dl, x, moe.PATH_GEMM, moe.GEMM_CUDA_CORE)
        n = moe.moe_last_launch_count()
        times = moe.moe_kernel_times()
    finally:
        moe.moe_set_option(moe.MOE_OPT_KERNEL_TIMING, 0)
    assert n == 5  # small-T router (also clears y_acc), routing, gate/up, down, cast
    assert sum(c for _, c in times.values()) == n
    assert all(ms >= 0 for ms, _ in times.values())
    assert ("router_logits" in times or "router_small" in times) and "gateup_simt" in times


def test_bounded_wait_expiry_reports_status_and_context_survives():
    """A wait that runs out (the test hook makes the tensor-core epilogue wait
    on a barrier nothing arrives on, for at most 20000 cycles) makes the kernel
    record MOE_ERR_DEVICE_TIMEOUT, drain its copies and MMAs and exit; the next
    call on the same context is correct."""
    layer, x = config("tiny")
    dl = dev_layer("tiny", layer)
    xd = x_to_device(x)
    ws = dl.workspace(x.shape[0])
    assert moe.moe_set_option(moe.MOE_OPT_FORCE_PATH, moe.PATH_GEMM) == moe.MOE_OK
    assert moe.moe_set_option(moe.MOE_OPT_GEMM_IMPL, moe.GEMM_TENSOR_CORE) == moe.MOE_OK
    assert moe.moe_set_option(moe.MOE_OPT_TEST_WAIT_CYCLES, 20000) == moe.MOE_OK
    try:
        dl.forward(xd, workspace=ws)
        st = moe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), None)
    finally:
        moe.moe_set_option(moe.MOE_OPT_TEST_WAIT_CYCLES, 0)
    assert st == moe.MOE_ERR_DEVICE_TIMEOUT
    y, _ = run_forward(dl, x, moe.PATH_GEMM, moe.GEMM_TENSOR_CORE)
    check_output(y, O.forward(O.OracleLayer(layer), x), "after a forced timeout")
