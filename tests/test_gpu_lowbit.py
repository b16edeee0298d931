"""GPU parity of the 2- and 3-bit experts: the prepacked layouts bit for bit,
and both paths (decode kernel, tensor-core GEMM) against the oracle's layer
on low-bit codes, with the routing and tolerance of the 4-bit tests."""
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


def _repack3(q):
    """The prepacked 3-bit layout from the row-major bit streams: per row and 64-column group, words
    0..3 hold the low two bits (column 16j+2p+h of word j at bits 2p+16h), words 4 and 5 the high bits
    (column 16j+2p+h at bit 16h + 8(j%2) + p of word 4 + j//2)."""
    E, N, W = q.shape
    K = W * 32 // 3
    bits = np.unpackbits(np.ascontiguousarray(q).astype("<u4").view(np.uint8).reshape(E, N, -1), axis=2,
                         bitorder="little").reshape(E, N, K, 3).astype(np.uint32)
    codes = bits[..., 0] | (bits[..., 1] << 1) | (bits[..., 2] << 2)
    c = codes.reshape(E, N, K // 64, 64).transpose(0, 2, 1, 3)      # [E][G][N][64]
    out = np.zeros(c.shape[:3] + (6,), np.uint32)
    for col in range(64):
        j, p, h = col // 16, (col % 16) // 2, col % 2
        out[..., j] |= (c[..., col] & 3) << np.uint32(2 * p + 16 * h)
        out[..., 4 + j // 2] |= (c[..., col] >> 2) << np.uint32(16 * h + 8 * (j % 2) + p)
    return out


def test_repack3_helper():
    # codes 0..7 cycling along the row: column c holds c % 8
    K = 64
    stream = 0
    for col in range(K):
        stream |= (col % 8) << (3 * col)
    q = np.array([[[(stream >> (32 * w)) & 0xFFFFFFFF for w in range(6)]]], dtype=np.uint32)
    got = _repack3(q)[0, 0, 0]
    for col in range(K):
        j, p, h = col // 16, (col % 16) // 2, col % 2
        lo = (int(got[j]) >> (2 * p + 16 * h)) & 3
        hi = (int(got[4 + j // 2]) >> (16 * h + 8 * (j % 2) + p)) & 1
        assert lo + 4 * hi == col % 8, col


def test_prepack_codes_three_bit_is_exact_reordering():
    rng = np.random.default_rng(8)
    for (E, N, K) in [(3, 64, 128), (2, 704, 2816), (1, 2048, 512)]:
        q = rng.integers(0, 2**32, size=(E, N, K * 3 // 32), dtype=np.uint32)
        qd = torch.from_numpy(q.view(np.int32)).cuda()
        qp = torch.empty((E, K // 64, N, 6), dtype=torch.int32, device="cuda")
        bm.moe_prepack_codes(qd, qp, bits=3)
        np.testing.assert_array_equal(qp.cpu().numpy().view(np.uint32), _repack3(q))


SMALL_LOWBIT = [
    ("tiny", dict()),
    ("ragged", dict(T=23, d=192, E=8, k=3, I=192, I_shared=320)),
    ("one_token", dict(T=1, d=256, E=32, k=8, I=128, I_shared=128)),
    ("many_tokens", dict(T=300, d=128, E=4, k=2, I=64, I_shared=64)),
]


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("path", ["gemv", "gemm"])
@pytest.mark.parametrize("name,kw", SMALL_LOWBIT, ids=[c[0] for c in SMALL_LOWBIT])
def test_forward_low_bit(name, kw, path, bits):
    if path == "gemv":  # the decode kernel takes at most 4 tokens
        kw = dict(kw, T=min(kw.get("T", synth.small_config().T), 4))
    cfg = synth.small_config(bits=bits, **kw)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    assert dl.routed.bits == bits
    r, _ = G.route_gpu(layer.logits, cfg.k, 96 if path == "gemm" else 32)
    rh = G.routing_to_host(r)
    Y = dl.forward(r, path)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, rh["ids"], rh["w"])
    G.assert_y_close(Y, Y64, f"{name}/{path}/{bits}-bit")


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_forward_low_bit_decode_token_counts(T, bits):
    cfg = synth.small_config(T=T, d=1024, E=12, k=8, I=256, I_shared=192, bits=bits)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 32)
    rh = G.routing_to_host(r)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, rh["ids"], rh["w"])
    G.assert_y_close(dl.forward(r, "gemv"), Y64, f"T={T}/{bits}-bit")


# every code 2^(b-1) as row-major words: 2-bit code 2 is 0b10 repeated; the 3-bit stream 001 repeated
# cycles through three words
_MID_CODE_WORDS = {2: np.array([0xAAAAAAAA], np.uint32),
                   3: np.array([0x24924924, 0x49249249, 0x92492492], np.uint32)}


@pytest.mark.parametrize("bits", [2, 3])
def test_low_bit_mid_code_experts_give_shared_only(bits):
    """Every code 2^(b-1) with bias = -2^(b-1) scale: the routed weights dequantise to exactly 0, and Y is
    the shared expert alone on both paths."""
    cfg = synth.small_config(T=3, d=256, E=8, k=2, I=128, I_shared=128, bits=bits)
    layer = synth.draw_layer(cfg)
    mid = _MID_CODE_WORDS[bits]
    layer.routed = {m: (np.broadcast_to(np.resize(mid, q.shape[-1]), q.shape).copy(), s, b)
                    for m, (q, s, b) in layer.routed.items()}
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 32)
    ids = np.zeros((cfg.T, cfg.k), np.int32)
    w = np.zeros((cfg.T, cfg.k), np.float32)
    Ysh, _ = oracle.forward(layer.X, layer.routed, layer.shared, ids, w)
    for path in ("gemv", "gemm"):
        G.assert_y_close(dl.forward(r, path), Ysh, f"mid code/{path}/{bits}-bit")


@pytest.mark.parametrize("name", ["decode2b", "decode3b"])
def test_layer_decode_low_bit_full_size(name):
    """The decode workload's dimensions with 2- or 3-bit codes through moe_layer (one launch), routing
    bit-exact, Y against the oracle; deterministic across calls."""
    cfg = synth.CONFIGS[name]
    dl = G.DeviceLayer.from_device_draw(cfg, 1, 1)
    assert dl.routed.bits == cfg.bits
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
    G.assert_y_close(outs[0], Y64, f"{name} layer")


@pytest.mark.parametrize("name", ["decode2b", "decode3b"])
def test_gemm_low_bit_full_width_sampled(name):
    """The decode layer's dimensions with 2- or 3-bit codes on the tensor-core path at 96 tokens; the
    oracle checks a sample of tokens (tokens are independent)."""
    cfg = synth.CONFIGS[name]
    T = 96
    dl = G.DeviceLayer.from_device_draw(cfg, 2, T)
    r, _ = G.route_gpu(dl.logits, cfg.k, 96)
    rh = G.routing_to_host(r)
    Y = dl.forward(r, "gemm")
    rows = np.array([0, 1, 17, 50, 95])
    Y64, _ = oracle.forward(dl.X_host[rows], dl.routed_host, dl.shared_host, rh["ids"][rows], rh["w"][rows])
    G.assert_y_close(Y[rows], Y64, f"gemm {name}")
