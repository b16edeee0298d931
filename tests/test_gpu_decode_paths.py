"""The one-token decode kernel reads its gate/up codes in one of two ways: straight
from global memory into the MMA fragment registers (every CTA has at most one
32-row item and d <= 2048; the default), or through the shared-memory stage
ring that TMA fills (MOE_DECODE_REG=0, and every call with more tokens).  The
arithmetic and its order are the same, so both give the same bits; the
register variant is also checked against the oracle."""
import contextlib
import os

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


@contextlib.contextmanager
def _ring_path():
    old = os.environ.get("MOE_DECODE_REG")
    os.environ["MOE_DECODE_REG"] = "0"
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("MOE_DECODE_REG", None)
        else:
            os.environ["MOE_DECODE_REG"] = old


def _layer_twice(dl, cfg):
    """moe_layer on one token with the register variant, then with the stage ring; Y bits and routing of each."""
    lg = torch.from_numpy(dl.logits).cuda()
    ws = bm.workspace(bm.moe_layer_workspace_bytes(1, cfg.d, cfg.I, cfg.E, cfg.k, cfg.I_shared))
    out = []
    for ring in (False, True):
        r = bm.Routing.empty(1, cfg.E, cfg.k, 32)
        Y = torch.empty((1, cfg.d), dtype=torch.int16, device="cuda")
        with _ring_path() if ring else contextlib.nullcontext():
            bm.moe_layer(lg, dl.X, dl.routed, dl.shared, cfg.k, 32, r, Y, ws)
        torch.cuda.synchronize()
        assert bm.moe_check_status(ws) == 0
        out.append((Y.cpu().numpy().view(np.uint16), G.routing_to_host(r)))
    return out


@pytest.mark.parametrize("name", ["decode", "decode3b", "decode2b"])
def test_register_and_ring_variants_agree_full_size(name):
    cfg = synth.CONFIGS[name]
    dl = G.DeviceLayer.from_device_draw(cfg, 3, 1)
    (y_reg, r_reg), (y_ring, r_ring) = _layer_twice(dl, cfg)
    np.testing.assert_array_equal(y_reg, y_ring)
    ref = oracle.route(dl.logits, cfg.k, 32)
    G.assert_routing_equal(r_reg, ref)
    G.assert_routing_equal(r_ring, ref)
    Y64, _ = oracle.forward(dl.X_host, dl.routed_host, dl.shared_host, ref["ids"], ref["w"])
    G.assert_y_close(y_reg, Y64, f"{name}, register variant")


SMALL = [
    # d = 256: one chunk of four groups, so half the warps have no group
    ("d256", dict(T=1, d=256, E=32, k=8, I=128, I_shared=128)),
    ("no_shared", dict(T=1, d=1024, E=16, k=4, I=192, I_shared=0)),
    # a shared expert wider than the routed ones
    ("wide_shared", dict(T=1, d=2048, E=8, k=2, I=64, I_shared=256)),
    ("k1_E1", dict(T=1, d=512, E=1, k=1, I=128, I_shared=64)),
    # the largest k: 2 + 32 x 2 items, still one per CTA
    ("k32", dict(T=1, d=512, E=64, k=32, I=64, I_shared=64)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[c[0] for c in SMALL])
def test_register_and_ring_variants_agree_small(name, kw):
    cfg = synth.small_config(**kw)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    (y_reg, r_reg), (y_ring, _) = _layer_twice(dl, cfg)
    np.testing.assert_array_equal(y_reg, y_ring)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, r_reg["ids"], r_reg["w"])
    G.assert_y_close(y_reg, Y64, f"{name}, register variant")


def test_register_variant_with_routing_from_memory():
    """moe_forward at one token (routing read from memory rather than computed in the kernel)."""
    cfg = synth.small_config(T=1, d=2048, E=64, k=8, I=512, I_shared=512)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    r, _ = G.route_gpu(layer.logits, cfg.k, 32)
    rh = G.routing_to_host(r)
    y_reg = dl.forward(r, "gemv")
    with _ring_path():
        y_ring = dl.forward(r, "gemv")
    np.testing.assert_array_equal(y_reg, y_ring)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, rh["ids"], rh["w"])
    G.assert_y_close(y_reg, Y64, "moe_forward, register variant")
