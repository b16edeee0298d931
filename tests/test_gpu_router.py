"""GPU parity of the router projection (logits = X W_r^T) through the C ABI.

The logits are checked against the fp64 oracle within the error bound of fp32
accumulation: |gpu - exact| <= n u sum_i |x_i w_i| (n = d additions, u = 2^-24),
written below with a margin.  The routing that moe_route_x derives from them is
then checked bit for bit against the oracle's routing of the same fp32 logits,
so the selection is decided in the same precision on both sides.
"""
import zlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import bit_moe_expert_gb300 as bm  # noqa: E402
from bit_moe_expert_gb300 import synth  # noqa: E402
from tests import gpu_util as G  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_expert_gb300 import build
    build.build()
    bm.lib()


def _draw(T, d, E, seed):
    rng = np.random.default_rng(seed)
    X = synth.f32_to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    Wr = synth.f32_to_bf16_bits((rng.standard_normal((E, d)) / np.sqrt(d)).astype(np.float32))
    return X, Wr


def _gpu_logits(X, Wr):
    Xd = torch.from_numpy(X.view(np.int16)).cuda()
    Wd = torch.from_numpy(Wr.view(np.int16)).cuda()
    lg = torch.full((X.shape[0], Wr.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
    bm.moe_router_logits(Xd, Wd, lg)
    torch.cuda.synchronize()
    return lg.cpu().numpy(), (Xd, Wd, lg)


def _assert_logits_close(got, X, Wr):
    ref = oracle.router_logits(X, Wr)
    absdot = np.abs(synth.bf16_bits_to_f32(X).astype(np.float64)) @ np.abs(
        synth.bf16_bits_to_f32(Wr).astype(np.float64)).T
    d = X.shape[1]
    bound = 2.0 * d * 2.0 ** -24 * absdot + 1e-30
    err = np.abs(got.astype(np.float64) - ref)
    assert np.isfinite(got).all()
    worst = (err / bound).max() if err.size else 0.0
    assert worst <= 1.0, f"logit error {worst:.3g} x the fp32 accumulation bound"


# (T, d, E): the decode token, the tiny layer, ragged experts and tokens on
# the three kernel shapes (up to 32 tokens a warp per router row; more tokens
# the tensor-core kernel when E is a multiple of 128 and d of 256, else the
# warp-MMA tiles of 32 x 64), the widest router and a full 1024-token chunk
CASES = [
    ("decode", 1, 2048, 256),
    ("decode4", 4, 2048, 256),
    ("tiny", 16, 256, 16),
    ("ragged_small", 5, 64, 33),
    ("eight", 8, 192, 24),
    ("nine", 9, 128, 16),
    ("ragged_large", 70, 512, 80),
    ("half_chunk", 100, 192, 48),
    ("wide", 33, 256, 1024),
    ("chunk", 1024, 2048, 256),
    ("canvas", 256, 2816, 128),
    # the tensor-core shape (more than 32 tokens, E a multiple of 128, d of
    # 256): a ragged last token tile over three router-row tiles, a K quarter
    # of one stage, two passes over the stage ring, and a long prompt
    ("tc_ragged", 65, 512, 384),
    ("tc_one_stage", 200, 256, 128),
    ("tc_two_rings", 300, 4096, 128),
    ("tc_long", 4096, 2048, 256),
]


@pytest.mark.parametrize("name,T,d,E", CASES, ids=[c[0] for c in CASES])
def test_router_logits_parity(name, T, d, E):
    X, Wr = _draw(T, d, E, seed=zlib.crc32(name.encode()))
    got, _ = _gpu_logits(X, Wr)
    _assert_logits_close(got, X, Wr)


@pytest.mark.parametrize("T,d,E,tc", [
    (1024, 2048, 256, True), (33, 256, 1024, True), (300, 4096, 128, True), (32, 2048, 256, False),
    (100, 192, 48, False), (64, 2048, 200, False),
])
def test_router_shape_choice(T, d, E, tc, monkeypatch):
    # MOE_ROUTER_TC=0 keeps the warp-MMA kernels.  On a shape the tensor-core
    # kernel takes, the two sum in different orders, so some of the fp32
    # logits differ in their last bits (identical logits would mean the
    # tensor-core kernel did not run); both agree with the oracle within the
    # accumulation bound.  On any other shape the switch changes nothing.
    X, Wr = _draw(T, d, E, seed=T + d + E)
    default, _ = _gpu_logits(X, Wr)
    monkeypatch.setenv("MOE_ROUTER_TC", "0")
    warp_mma, _ = _gpu_logits(X, Wr)
    _assert_logits_close(default, X, Wr)
    _assert_logits_close(warp_mma, X, Wr)
    assert (not np.array_equal(default.view(np.uint32), warp_mma.view(np.uint32))) == tc


def test_router_tc_tile_independence():
    # a token's logits do not depend on the other tokens of its tile or on the
    # tile it falls in (zero-filled rows past T multiply into nothing)
    X, Wr = _draw(200, 512, 256, seed=77)
    whole, _ = _gpu_logits(X, Wr)
    shifted, _ = _gpu_logits(np.ascontiguousarray(X[37:]), Wr)
    assert np.array_equal(whole[37:].view(np.uint32), shifted.view(np.uint32))


def test_router_logits_one_hot_tokens_are_exact():
    # a unit token's logits are one column of the router, with no rounding at all
    d, E = 256, 40
    _, Wr = _draw(1, d, E, seed=5)
    cols = [0, 1, 31, 32, 100, 255, 7, 64, 200]
    X = np.zeros((len(cols), d), np.uint16)
    for t, i in enumerate(cols):
        X[t, i] = 0x3F80
    got, _ = _gpu_logits(X, Wr)
    want = synth.bf16_bits_to_f32(Wr)[:, cols].T
    np.testing.assert_array_equal(got, want)


def test_router_tc_one_hot_tokens_are_exact():
    # the same on the tensor-core shape: unit tokens in every K quarter, every
    # 16-wide K slice of a stage and both halves of a 128-byte swizzled row
    # pick out single router columns, so a misplaced quarter, stage or slice
    # shows as a wrong column
    d, E = 1024, 256
    _, Wr = _draw(1, d, E, seed=6)
    cols = [0, 15, 16, 31, 32, 47, 48, 63, 64, 100, 255, 256, 300, 511, 512, 700, 767, 768, 1000, 1023]
    cols = cols + [(37 * j) % d for j in range(70 - len(cols))]
    X = np.zeros((len(cols), d), np.uint16)
    for t, i in enumerate(cols):
        X[t, i] = 0x3F80
    got, _ = _gpu_logits(X, Wr)
    want = synth.bf16_bits_to_f32(Wr)[:, cols].T
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("T", [1, 300, 1024])
def test_router_logits_deterministic(T):
    X, Wr = _draw(T, 1024, 256, seed=9)
    a, _ = _gpu_logits(X, Wr)
    b, _ = _gpu_logits(X, Wr)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("name,T,d,E,k,br", [
    ("decode", 1, 2048, 256, 8, 96),
    ("chunk", 1024, 2048, 256, 8, 96),
    ("small", 37, 128, 33, 5, 7),
], ids=["decode", "chunk", "small"])
def test_route_x_routes_its_own_logits(name, T, d, E, k, br):
    X, Wr = _draw(T, d, E, seed=zlib.crc32(name.encode()) + 1)
    Xd = torch.from_numpy(X.view(np.int16)).cuda()
    Wd = torch.from_numpy(Wr.view(np.int16)).cuda()
    lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
    r = bm.Routing.empty(T, E, k, br)
    ws = bm.workspace(bm.moe_route_workspace_bytes(T, E, k))
    bm.moe_route_x(Xd, Wd, k, br, r, ws, lg)
    torch.cuda.synchronize()
    assert bm.moe_check_status(ws) == 0
    got_lg = lg.cpu().numpy()
    _assert_logits_close(got_lg, X, Wr)
    alone, _ = _gpu_logits(X, Wr)
    assert np.array_equal(got_lg.view(np.uint32), alone.view(np.uint32))
    G.assert_routing_equal(G.routing_to_host(r), oracle.route(got_lg, k, br))


def test_router_zero_tokens_and_bad_arguments():
    X = torch.zeros((0, 128), dtype=torch.int16, device="cuda")
    W = torch.zeros((16, 128), dtype=torch.int16, device="cuda")
    lg = torch.zeros((0, 16), dtype=torch.float32, device="cuda")
    bm.moe_router_logits(X, W, lg)  # T = 0: nothing to do
    X1 = torch.zeros((1, 96), dtype=torch.int16, device="cuda")
    W1 = torch.zeros((16, 96), dtype=torch.int16, device="cuda")
    with pytest.raises(bm.MoeError) as ei:
        bm.moe_router_logits(X1, W1, torch.zeros((1, 16), dtype=torch.float32, device="cuda"))
    assert bm.STATUS_NAMES[ei.value.status] == "MOE_ERR_INVALID_ARG"  # d not a multiple of 64
    X2 = torch.zeros((1, 64), dtype=torch.int16, device="cuda")
    W2 = torch.zeros((1025, 64), dtype=torch.int16, device="cuda")
    with pytest.raises(bm.MoeError) as ei:
        bm.moe_router_logits(X2, W2, torch.zeros((1, 1025), dtype=torch.float32, device="cuda"))
    assert bm.STATUS_NAMES[ei.value.status] == "MOE_ERR_UNSUPPORTED"  # E above 1024


@pytest.mark.parametrize("name,kw,br", [
    ("T1_fused", dict(T=1, d=1024, E=64, k=8, I=256, I_shared=192), 32),
    ("T4_fused", dict(T=4, d=512, E=40, k=6, I=128, I_shared=64), 8),
    ("T40_gemm", dict(T=40, d=256, E=16, k=2, I=128, I_shared=128), 32),
], ids=["T1_fused", "T4_fused", "T40_gemm"])
def test_layer_x_from_hidden_state(name, kw, br):
    """moe_layer_x: the logits within the accumulation bound, the routing of those
    logits bit for bit, and Y within the layer tolerance of the oracle's layer on
    that routing."""
    cfg = synth.small_config(**kw)
    layer = synth.draw_layer(cfg)
    Wr = synth.f32_to_bf16_bits(
        (np.random.default_rng(zlib.crc32(name.encode())).standard_normal((cfg.E, cfg.d)) /
         np.sqrt(cfg.d)).astype(np.float32))
    dl = G.DeviceLayer.from_host(layer)
    Wd = torch.from_numpy(Wr.view(np.int16)).cuda()
    T = cfg.T
    lg = torch.empty((T, cfg.E), dtype=torch.float32, device="cuda")
    r = bm.Routing.empty(T, cfg.E, cfg.k, br)
    ws = bm.workspace(bm.moe_layer_workspace_bytes(T, cfg.d, cfg.I, cfg.E, cfg.k, cfg.I_shared))
    Y = torch.empty((T, cfg.d), dtype=torch.int16, device="cuda")
    bm.moe_layer_x(dl.X, Wd, dl.routed, dl.shared, cfg.k, br, lg, r, Y, ws)
    torch.cuda.synchronize()
    assert bm.moe_check_status(ws) == 0
    got_lg = lg.cpu().numpy()
    _assert_logits_close(got_lg, layer.X, Wr)
    ref = oracle.route(got_lg, cfg.k, br)
    G.assert_routing_equal(G.routing_to_host(r), ref)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, ref["ids"], ref["w"])
    G.assert_y_close(Y.cpu().numpy().view(np.uint16), Y64, name)
