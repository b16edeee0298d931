"""GPU parity of the 2-bit experts: the prepacked layout bit for bit, and both
paths (decode kernel, tensor-core GEMM) against the oracle's layer on 2-bit
codes, with the routing and tolerance of the 4-bit tests."""
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


def _interleave_pairs2(w):
    """The prepacked 2-bit word order: column 2p of the word's sixteen in bits 2p,
    column 2p+1 in bits 2p+16."""
    out = np.zeros_like(w)
    for p in range(8):
        for h in range(2):
            k = 2 * p + h
            out |= ((w >> np.uint32(2 * k)) & np.uint32(3)) << np.uint32(2 * p + 16 * h)
    return out


def test_interleave_pairs2_helper():
    # column k of the word holds k mod 4: from the low bits up the interleaved word reads
    # the even columns 0 2 4 .. 14, then the odd ones
    w = np.array([sum((k % 4) << (2 * k) for k in range(16))], dtype=np.uint32)
    got = int(_interleave_pairs2(w)[0])
    assert [(got >> (2 * i)) & 3 for i in range(16)] == [(2 * i) % 4 for i in range(8)] + \
        [(2 * i + 1) % 4 for i in range(8)]


def test_prepack_codes_two_bit_is_exact_reordering():
    rng = np.random.default_rng(7)
    for (E, N, K) in [(3, 64, 128), (2, 704, 2816), (1, 2048, 512)]:
        q = rng.integers(0, 2**32, size=(E, N, K // 16), dtype=np.uint32)
        qd = torch.from_numpy(q.view(np.int32)).cuda()
        qp = torch.empty((E, K // 64, N, 4), dtype=torch.int32, device="cuda")
        bm.moe_prepack_codes(qd, qp, bits=2)
        got = qp.cpu().numpy().view(np.uint32)
        ref = _interleave_pairs2(q.reshape(E, N, K // 64, 4).transpose(0, 2, 1, 3))
        np.testing.assert_array_equal(got, ref)


SMALL2 = [
    ("tiny2", dict(bits=2)),
    ("ragged2", dict(T=23, d=192, E=8, k=3, I=192, I_shared=320, bits=2)),
    ("one_token2", dict(T=1, d=256, E=32, k=8, I=128, I_shared=128, bits=2)),
    ("many_tokens2", dict(T=300, d=128, E=4, k=2, I=64, I_shared=64, bits=2)),
]


@pytest.mark.parametrize("path", ["gemv", "gemm"])
@pytest.mark.parametrize("name,kw", SMALL2, ids=[c[0] for c in SMALL2])
def test_forward_two_bit(name, kw, path):
    if path == "gemv":  # the decode kernel takes at most 4 tokens
        kw = dict(kw, T=min(kw.get("T", synth.small_config().T), 4))
    cfg = synth.small_config(**kw)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    assert dl.routed.bits == 2
    r, _ = G.route_gpu(layer.logits, cfg.k, 96 if path == "gemm" else 32)
    rh = G.routing_to_host(r)
    Y = dl.forward(r, path)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, rh["ids"], rh["w"])
    G.assert_y_close(Y, Y64, f"{name}/{path}")


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_forward_two_bit_decode_token_counts(T):
    cfg = synth.small_config(T=T, d=1024, E=12, k=8, I=256, I_shared=192, bits=2)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 32)
    rh = G.routing_to_host(r)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, rh["ids"], rh["w"])
    G.assert_y_close(dl.forward(r, "gemv"), Y64, f"T={T}")


def test_two_bit_code_two_experts_give_shared_only():
    """Every code 2 with bias = -2 scale: the routed weights dequantise to exactly 0, and Y is the shared
    expert alone on both paths."""
    cfg = synth.small_config(T=3, d=256, E=8, k=2, I=128, I_shared=128, bits=2)
    layer = synth.draw_layer(cfg)
    layer.routed = {m: (np.full_like(q, 0xAAAAAAAA), s, b) for m, (q, s, b) in layer.routed.items()}
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 32)
    ids = np.zeros((cfg.T, cfg.k), np.int32)
    w = np.zeros((cfg.T, cfg.k), np.float32)
    Ysh, _ = oracle.forward(layer.X, layer.routed, layer.shared, ids, w)
    for path in ("gemv", "gemm"):
        G.assert_y_close(dl.forward(r, path), Ysh, f"code 2/{path}")


def test_layer_decode_two_bit_full_size():
    """The decode workload's dimensions with 2-bit codes through moe_layer (one launch), routing bit-exact,
    Y against the oracle; deterministic across calls."""
    cfg = synth.CONFIGS["decode2b"]
    dl = G.DeviceLayer.from_device_draw(cfg, 1, 1)
    assert dl.routed.bits == 2
    lg = torch.from_numpy(dl.logits).cuda()
    r = bm.Routing.empty(1, cfg.E, cfg.k, 96)
    ws = bm.workspace(bm.moe_layer_workspace_bytes(1, cfg.d, cfg.I, cfg.E, cfg.k, cfg.I_shared))
    outs = []
    for _ in range(2):
        Y = torch.empty((1, cfg.d), dtype=torch.int16, device="cuda")
        bm.moe_layer(lg, dl.X, dl.routed, dl.shared, cfg.k, 96, r, Y, ws)
        torch.cuda.synchronize()
        assert bm.moe_check_status(ws) == 0
        outs.append(Y.cpu().numpy().view(np.uint16))
    np.testing.assert_array_equal(outs[0], outs[1])
    ref = oracle.route(dl.logits, cfg.k, 96)
    G.assert_routing_equal(G.routing_to_host(r), ref)
    Y64, _ = oracle.forward(dl.X_host, dl.routed_host, dl.shared_host, ref["ids"], ref["w"])
    G.assert_y_close(outs[0], Y64, "decode 2-bit layer")


def test_gemm_two_bit_full_width_sampled():
    """The decode layer's dimensions with 2-bit codes on the tensor-core path at 96 tokens (every expert
    of the sample routed); the oracle checks a sample of tokens (tokens are independent)."""
    cfg = synth.CONFIGS["decode2b"]
    T = 96
    dl = G.DeviceLayer.from_device_draw(cfg, 2, T)
    r, _ = G.route_gpu(dl.logits, cfg.k, 96)
    rh = G.routing_to_host(r)
    Y = dl.forward(r, "gemm")
    rows = np.array([0, 1, 17, 50, 95])
    Y64, _ = oracle.forward(dl.X_host[rows], dl.routed_host, dl.shared_host, rh["ids"][rows], rh["w"][rows])
    G.assert_y_close(Y[rows], Y64, "gemm 2-bit")
