"""Failure detection on the GPU without a fault: a bounded device-side wait
that nothing completes gives up, records MOE_ERR_TIMEOUT in the workspace
status word, and leaves the context usable.

The decode kernel's CTAs meet once at a barrier over the grid (every h value
of the call written) with a bounded wait.  The test hook moe_debug_decode skips
one CTA's arrival and shortens the wait limit to about a millisecond, so every
CTA's wait runs out; nothing faults or traps.
"""
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

TIMEOUT = 5


def _layer(cfg, layer, ws, r, dl):
    lg = torch.from_numpy(np.ascontiguousarray(layer.logits, dtype=np.float32)).cuda()
    Y = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device="cuda")
    bm.moe_layer(lg, dl.X, dl.routed, dl.shared, cfg.k, 32, r, Y, ws)
    torch.cuda.synchronize()
    return Y.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("T,drop", [(1, 0), (1, 37), (3, 5)])
def test_decode_wait_runs_out_then_recovers(T, drop):
    cfg = synth.small_config(T=T, d=1024, E=64, k=8, I=256, I_shared=192)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    r = bm.Routing.empty(T, cfg.E, cfg.k, 32)
    ws = bm.workspace(bm.moe_layer_workspace_bytes(T, cfg.d, cfg.I, cfg.E, cfg.k, cfg.I_shared))
    ref = oracle.route(layer.logits, cfg.k, 32)
    Y64, _ = oracle.forward(layer.X, layer.routed, layer.shared, ref["ids"], ref["w"])

    Y = _layer(cfg, layer, ws, r, dl)  # a clean call first: the workspace is in use
    assert bm.moe_check_status(ws) == 0
    G.assert_y_close(Y, Y64, "before")
    bm.moe_debug_decode(2_000_000, drop)  # about 1 ms of SM clock per wait
    try:
        _layer(cfg, layer, ws, r, dl)
        assert bm.moe_check_status(ws) == TIMEOUT
    finally:
        bm.moe_debug_decode(0, -1)
    # the context still works; a re-zeroed workspace gives the right answer again
    ws.zero_()
    Y = _layer(cfg, layer, ws, r, dl)
    assert bm.moe_check_status(ws) == 0
    G.assert_y_close(Y, Y64, "after")
    G.assert_routing_equal(G.routing_to_host(r), ref)
