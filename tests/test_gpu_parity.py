"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Routing (ids, weights, counts, offsets, permutation, block map) must match bit
for bit; Y must be within relative L2 5e-3 and elementwise 2e-2*max(1,|Y|).
Small cases run the oracle on every token; the full-size workloads run the
whole layer on the GPU in the launch configuration the benchmark uses and the
oracle on a sample of tokens (tokens are independent, so a sample is exact).
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


# ------------------------------------------------------------------ prepack

def test_prepack_is_exact_transpose():
    rng = np.random.default_rng(0)
    for (E, N, K) in [(3, 64, 128), (2, 704, 2816), (1, 2048, 512)]:
        s = rng.integers(0, 2**16, size=(E, N, K // 64), dtype=np.uint16)
        b = rng.integers(0, 2**16, size=(E, N, K // 64), dtype=np.uint16)
        sd = torch.from_numpy(s.view(np.int16)).cuda()
        bd = torch.from_numpy(b.view(np.int16)).cuda()
        sb = torch.empty((E, K // 64, N), dtype=torch.int32, device="cuda")
        bm.moe_prepack_scales(sd, bd, sb)
        got = sb.cpu().numpy().view(np.uint32)
        ref = (s.astype(np.uint32) | (b.astype(np.uint32) << 16)).transpose(0, 2, 1)
        np.testing.assert_array_equal(got, ref)


def test_prepack_codes_is_exact_reordering():
    rng = np.random.default_rng(1)
    for (E, N, K) in [(3, 64, 128), (2, 704, 2816), (1, 2048, 512)]:
        q = rng.integers(0, 2**32, size=(E, N, K // 8), dtype=np.uint32)
        qd = torch.from_numpy(q.view(np.int32)).cuda()
        qp = torch.empty((E, K // 64, N, 8), dtype=torch.int32, device="cuda")
        bm.moe_prepack_codes(qd, qp)
        got = qp.cpu().numpy().view(np.uint32)
        ref = _interleave_nibbles(q.reshape(E, N, K // 64, 8).transpose(0, 2, 1, 3))
        np.testing.assert_array_equal(got, ref)


def _interleave_nibbles(w):
    """The prepacked word order: column 2p of a word's eight in bits 4p,
    column 2p+1 in bits 4p+16."""
    out = np.zeros_like(w)
    for p in range(4):
        for h in range(2):
            k = 2 * p + h
            out |= ((w >> np.uint32(4 * k)) & np.uint32(0xF)) << np.uint32(4 * p + 16 * h)
    return out


def test_interleave_nibbles_helper():
    # column k of the word holds value k: the interleaved word reads, from the
    # low nibble up, columns 0 2 4 6 1 3 5 7
    w = np.array([0x76543210], dtype=np.uint32)
    assert int(_interleave_nibbles(w)[0]) == 0x75316420


# ------------------------------------------------------------------ routing

ROUTE_CASES = [
    ("tiny", dict(T=16, E=16, k=2), 16),
    ("decode", dict(T=1, E=256, k=8), 128),
    ("prefill512", dict(T=512, E=256, k=8), 128),
    ("canvas", dict(T=256, E=128, k=8), 128),
    ("ragged", dict(T=37, E=33, k=5), 7),
    ("k_equals_E", dict(T=20, E=16, k=16), 32),
    ("wide", dict(T=70, E=1024, k=32), 64),
    ("long", dict(T=4096, E=256, k=8), 128),
    ("empty", dict(T=0, E=64, k=4), 32),
    ("bm1", dict(T=9, E=8, k=3), 1),
]


@pytest.mark.parametrize("name,sz,bm_rows", ROUTE_CASES, ids=[c[0] for c in ROUTE_CASES])
def test_route_bit_exact(name, sz, bm_rows):
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    lg = rng.standard_normal((sz["T"], sz["E"])).astype(np.float32)
    r, _ = G.route_gpu(lg, sz["k"], bm_rows)
    ref = oracle.route(lg, sz["k"], bm_rows)
    G.assert_routing_equal(G.routing_to_host(r), ref)


def test_route_zipf_chunk_bit_exact():
    cfg = synth.CONFIGS["prefill4096"]
    for c in range(4):
        lg = synth.draw_logits(cfg, 4096, 0)[c * 1024:(c + 1) * 1024]
        r, _ = G.route_gpu(lg, cfg.k, 128)
        G.assert_routing_equal(G.routing_to_host(r), oracle.route(lg, cfg.k, 128))


def test_route_forced_ties_bit_exact():
    rng = np.random.default_rng(11)
    lg = rng.integers(-3, 4, size=(300, 64)).astype(np.float32)  # many equal logits
    lg[0] = 1.0
    lg[1, 5:] = -0.0
    lg[1, :5] = 0.0
    r, _ = G.route_gpu(lg, 8, 32)
    G.assert_routing_equal(G.routing_to_host(r), oracle.route(lg, 8, 32))


def test_route_repeated_calls_reuse_workspace():
    rng = np.random.default_rng(12)
    T, E, k = 200, 64, 4
    lg_dev = []
    r = bm.Routing.empty(T, E, k, 32)
    ws = bm.workspace(bm.moe_route_workspace_bytes(T, E, k))
    for it in range(3):
        lg = rng.standard_normal((T, E)).astype(np.float32)
        x = torch.from_numpy(lg).cuda()
        bm.moe_route(x, k, 32, r, ws)
        torch.cuda.synchronize()
        G.assert_routing_equal(G.routing_to_host(r), oracle.route(lg, k, 32))
        lg_dev.append(x)
    assert bm.moe_check_status(ws) == 0


def test_route_nonfinite_is_reported():
    lg = np.zeros((40, 16), np.float32)
    lg[33, 7] = np.nan
    r, ws = G.route_gpu(lg, 2, 16)
    assert bm.moe_check_status(ws) == 6
    assert bm.moe_check_status(ws) == 0  # cleared
    lg[33, 7] = np.inf
    r, ws = G.route_gpu(lg, 2, 16)
    assert bm.moe_check_status(ws) == 6


# ------------------------------------------------------------------ forward, small (all tokens)

SMALL = [
    ("tiny", dict()),
    ("tiny_no_shared", dict(I_shared=0)),
    ("ragged_I", dict(T=23, d=192, E=8, k=3, I=192, I_shared=320)),
    ("one_token", dict(T=1, d=256, E=32, k=8, I=128, I_shared=128)),
    ("k1_E1", dict(T=7, E=1, k=1, I=128, I_shared=0)),
    ("many_tokens", dict(T=300, d=128, E=4, k=2, I=64, I_shared=64)),
    ("skewed", dict(T=130, d=256, E=6, k=1, I=256, I_shared=0)),
    ("max_E_and_k", dict(T=40, d=128, E=1024, k=32, I=64, I_shared=64)),  # the largest E and k the library takes
]


@pytest.mark.parametrize("path", ["gemv", "gemm"])
@pytest.mark.parametrize("name,kw", SMALL, ids=[c[0] for c in SMALL])
def test_forward_small(name, kw, path):
    if path == "gemv":  # the decode kernel takes at most 4 tokens
        kw = dict(kw, T=min(kw.get("T", synth.small_config().T), 4))
    cfg = synth.small_config(**kw)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 96 if path == "gemm" else 32)
    rh = G.routing_to_host(r)
    Y = dl.forward(r, path)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, rh["ids"], rh["w"])
    G.assert_y_close(Y, Y64, f"{name}/{path}")


@pytest.mark.parametrize("block_rows,T,E", [(1, 200, 8), (16, 200, 8), (32, 200, 8), (50, 200, 8), (64, 200, 8),
                                             (96, 200, 8), (128, 200, 8), (128, 600, 4), (96, 600, 4)])
def test_forward_gemm_block_rows(block_rows, T, E):
    """Tiles of every height up to the 128-row maximum; with T = 600 over four
    experts each expert fills two 128-row tiles (or three of 96) and a ragged
    one, and the shared expert's 600 tokens make four full tiles and a tail."""
    cfg = synth.small_config(T=T, d=256, E=E, k=2, I=128, I_shared=128)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, block_rows)
    rh = G.routing_to_host(r)
    Y = dl.forward(r, "gemm")
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, rh["ids"], rh["w"])
    G.assert_y_close(Y, Y64, f"block_rows={block_rows}, T={T}, E={E}")


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_forward_decode_token_counts(T):
    """Every token count the decode kernel handles, on a layer shaped like the
    decode workload but with fewer experts; tokens share some experts."""
    cfg = synth.small_config(T=T, d=1024, E=12, k=8, I=256, I_shared=192)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 32)
    rh = G.routing_to_host(r)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, rh["ids"], rh["w"])
    G.assert_y_close(dl.forward(r, "gemv"), Y64, f"T={T}")


def test_forward_decode_rejects_more_than_4_tokens():
    cfg = synth.small_config(T=5, d=128, E=4, k=2, I=64, I_shared=0)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 32)
    with pytest.raises(bm.MoeError) as ei:
        dl.forward(r, "gemv")
    assert bm.STATUS_NAMES[ei.value.status] == "MOE_ERR_UNSUPPORTED"


def test_forward_gemm_rejects_routing_over_128_rows():
    """The tensor-core path holds at most 128 tokens per tile (moe_route's
    own limit); a routing struct that claims taller tiles is refused before
    any launch."""
    cfg = synth.small_config(T=40, d=128, E=4, k=2, I=64, I_shared=0)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 128)
    r.block_rows = 129
    with pytest.raises(bm.MoeError) as ei:
        dl.forward(r, "gemm")
    assert bm.STATUS_NAMES[ei.value.status] == "MOE_ERR_UNSUPPORTED"


@pytest.mark.parametrize("bits,expect", [(0x477F, 0), (0xC77F, 0), (0x4780, 2), (0xFF80, 2), (0x7FC0, 2)],
                         ids=["65280", "-65280", "65536", "-inf", "nan"])
def test_forward_gemm_x_range_check(bits, expect):
    """The tensor-core path converts X to fp16: a value outside the fp16 range
    (|x| > 65504; for bf16 input, anything above 65280 = 0x477F, and
    infinities and NaN) is recorded as MOE_ERR_UNSUPPORTED (2); the largest
    bf16 inside the range passes.  The planted value sits in a column whose
    quantisation group has zero scale and bias in every gate and up row, so
    the layer's other outputs stay finite and still match the oracle."""
    cfg = synth.small_config(T=64, d=256, E=8, k=2, I=128, I_shared=128)
    layer = synth.draw_layer(cfg)
    X = layer.X.copy()
    X[17, 101] = bits  # group 1 of the d = 256 input columns
    for ex in (layer.routed, layer.shared):
        for mat in ("gate", "up"):
            q, sc, bi = ex[mat]
            sc[..., 1] = 0
            bi[..., 1] = 0
    dl = G.DeviceLayer(X, layer.logits, layer.routed, layer.shared, bm.prepare_experts(layer.routed),
                       bm.prepare_experts(layer.shared))
    r, _ = G.route_gpu(layer.logits, cfg.k, 32)
    ws = bm.workspace(bm.moe_forward_workspace_bytes(cfg.T, cfg.d, cfg.I, cfg.E, cfg.k, cfg.I_shared))
    Y = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device="cuda")
    bm.moe_forward(dl.X, dl.routed, dl.shared, r, Y, ws)
    torch.cuda.synchronize()
    assert bm.STATUS_NAMES[bm.moe_check_status(ws)] == bm.STATUS_NAMES[expect]
    if expect == 0:
        rh = G.routing_to_host(r)
        Y64, _ = oracle.forward(X, layer.routed, layer.shared, rh["ids"], rh["w"])
        G.assert_y_close(Y.cpu().numpy().view(np.uint16), Y64, f"x = bf16 {bits:#06x}")


@pytest.mark.parametrize("path,T", [("gemv", 1), ("gemv", 4), ("gemm", 64)])
def test_forward_deterministic(path, T):
    cfg = synth.small_config(T=T, d=256, E=8, k=2, I=128, I_shared=128)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 64)
    first = dl.forward(r, path)
    for _ in range(3):
        np.testing.assert_array_equal(dl.forward(r, path), first)


def test_forward_zero_tokens():
    cfg = synth.small_config(T=0)
    layer = synth.draw_layer(cfg, T=0)
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 32)
    assert int(r.num_blocks.item()) == 0
    assert dl.forward(r, "gemm").size == 0


@pytest.mark.parametrize("path,T", [("gemv", 3), ("gemm", 40)])
def test_forward_code8_experts_give_shared_only(path, T):
    """All routed weights dequantise to exactly 0: Y is the shared expert alone."""
    cfg = synth.small_config(T=T)
    layer = synth.draw_layer(cfg)
    layer.routed = {m: (np.full_like(q, 0x88888888), s, b) for m, (q, s, b) in layer.routed.items()}
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 32)
    ids = np.zeros((cfg.T, cfg.k), np.int32)
    w = np.zeros((cfg.T, cfg.k), np.float32)
    Ysh, _ = oracle.forward(layer.X, layer.routed, layer.shared, ids, w)
    G.assert_y_close(dl.forward(r, path), Ysh, path)


# ------------------------------------------------------------------ full-size workloads, sampled tokens

FULL = ["decode", "prefill512", "prefill4096", "canvas"]


@pytest.mark.parametrize("name", FULL)
def test_forward_full_size_sampled(name):
    cfg = synth.CONFIGS[name]
    T = cfg.tokens_per_call
    dl = G.DeviceLayer.from_device_draw(cfg, 0, T)
    r, _ = G.route_gpu(dl.logits, cfg.k, 96)
    rh = G.routing_to_host(r)
    G.assert_routing_equal(rh, oracle.route(dl.logits, cfg.k, 96))
    Y = dl.forward(r)  # the path moe_forward picks for this T
    sample = sorted({0, T - 1, T // 2, T // 3, (2 * T) // 3, 1 % T, 7 % T, 123 % T})
    for t in sample:
        Y64, _ = oracle.forward(dl.X_host, dl.routed_host, dl.shared_host, rh["ids"], rh["w"], t, t + 1)
        G.assert_y_close(Y[t:t + 1], Y64, f"{name} token {t}")
    assert np.all(np.isfinite(synth.bf16_bits_to_f32(Y)))


@pytest.mark.parametrize("name", ["decode", "prefill512"])
def test_full_size_gemv_and_gemm_agree(name):
    """The two paths compute the same layer; on a full-size layer compare them
    everywhere against each other and on sampled tokens against the oracle."""
    cfg = synth.CONFIGS[name]
    T = min(cfg.tokens_per_call, 4)
    dl = G.DeviceLayer.from_device_draw(cfg, 1, T)
    r, _ = G.route_gpu(dl.logits, cfg.k, 96)
    rh = G.routing_to_host(r)
    Yv = dl.forward(r, "gemv")
    Ym = dl.forward(r, "gemm")
    Y64, _ = oracle.forward(dl.X_host, dl.routed_host, dl.shared_host, rh["ids"], rh["w"])
    G.assert_y_close(Yv, Y64, "gemv")
    G.assert_y_close(Ym, Y64, "gemm")


# ------------------------------------------------------------------ whole layer (moe_layer)

def _layer_gpu(layer, cfg, block_rows):
    dl = G.DeviceLayer.from_host(layer)
    T, E = cfg.T, cfg.E
    lg = torch.from_numpy(np.ascontiguousarray(layer.logits, dtype=np.float32)).cuda()
    r = bm.Routing.empty(T, E, cfg.k, block_rows)
    ws = bm.workspace(bm.moe_layer_workspace_bytes(T, cfg.d, cfg.I, E, cfg.k, cfg.I_shared))
    Y = torch.empty((T, cfg.d), dtype=torch.int16, device="cuda")
    bm.moe_layer(lg, dl.X, dl.routed, dl.shared, cfg.k, block_rows, r, Y, ws)
    torch.cuda.synchronize()
    return r, ws, Y.cpu().numpy().view(np.uint16)


LAYER_CASES = [
    ("T1_fused", dict(T=1, d=1024, E=64, k=8, I=256, I_shared=192), 32),
    ("T2_fused_no_shared", dict(T=2, d=512, E=32, k=4, I=128, I_shared=0), 8),
    ("T3_fused_shared_experts", dict(T=3, d=512, E=12, k=8, I=128, I_shared=128), 16),
    ("T4_fused", dict(T=4, d=768, E=40, k=6, I=192, I_shared=64), 1),
    ("T2_two_launches_E300", dict(T=2, d=256, E=300, k=4, I=64, I_shared=64), 16),
    ("T20_two_launches", dict(T=20, d=256, E=16, k=2, I=128, I_shared=128), 32),
]


@pytest.mark.parametrize("name,kw,br", LAYER_CASES, ids=[c[0] for c in LAYER_CASES])
def test_layer_matches_oracle(name, kw, br):
    """moe_layer: every routing output bit-exact, Y within tolerance, whether it
    runs as one launch (decode kernel routing its own tokens) or as two."""
    cfg = synth.small_config(**kw)
    layer = synth.draw_layer(cfg)
    r, ws, Y = _layer_gpu(layer, cfg, br)
    assert bm.moe_check_status(ws) == 0
    ref = oracle.route(layer.logits, cfg.k, br)
    G.assert_routing_equal(G.routing_to_host(r), ref)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, ref["ids"], ref["w"])
    G.assert_y_close(Y, Y64, name)


def test_layer_fused_forced_ties_and_nonfinite():
    cfg = synth.small_config(T=2, d=256, E=16, k=4, I=64, I_shared=64)
    layer = synth.draw_layer(cfg)
    layer.logits[0, :] = 0.5  # all equal: experts 0..3, weights 1/4
    layer.logits[1, 3] = -0.0
    layer.logits[1, 9] = 0.0
    r, ws, Y = _layer_gpu(layer, cfg, 4)
    assert bm.moe_check_status(ws) == 0
    ref = oracle.route(layer.logits, cfg.k, 4)
    G.assert_routing_equal(G.routing_to_host(r), ref)
    assert list(ref["ids"][0]) == [0, 1, 2, 3]
    layer.logits[1, 5] = np.nan
    r, ws, Y = _layer_gpu(layer, cfg, 4)
    assert bm.moe_check_status(ws) == 6


def test_layer_decode_full_size_and_deterministic():
    cfg = synth.CONFIGS["decode"]
    dl = G.DeviceLayer.from_device_draw(cfg, 2, 1)
    lg = torch.from_numpy(dl.logits).cuda()
    r = bm.Routing.empty(1, cfg.E, cfg.k, 96)
    ws = bm.workspace(bm.moe_layer_workspace_bytes(1, cfg.d, cfg.I, cfg.E, cfg.k, cfg.I_shared))
    outs = []
    for _ in range(3):
        Y = torch.empty((1, cfg.d), dtype=torch.int16, device="cuda")
        bm.moe_layer(lg, dl.X, dl.routed, dl.shared, cfg.k, 96, r, Y, ws)
        torch.cuda.synchronize()
        assert bm.moe_check_status(ws) == 0
        outs.append(Y.cpu().numpy().view(np.uint16))
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])
    ref = oracle.route(dl.logits, cfg.k, 96)
    G.assert_routing_equal(G.routing_to_host(r), ref)
    Y64, _ = oracle.forward(dl.X_host, dl.routed_host, dl.shared_host, ref["ids"], ref["w"])
    G.assert_y_close(outs[0], Y64, "decode layer")
