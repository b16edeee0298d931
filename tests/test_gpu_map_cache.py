"""The host-side caches of encoded tensor maps never serve a stale map: calls
that alternate between expert sets, and an expert set rewritten in place (same
addresses, new values), match the oracle on both paths.  The caches hold
addresses and shapes only, so new values at an old address must show up."""
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


def _layer_call(dl, k, path_T):
    """moe_layer on the layer's first path_T tokens; returns Y bits and the oracle's Y."""
    T = path_T
    lg = torch.from_numpy(np.ascontiguousarray(dl.logits[:T])).cuda()
    X = dl.X[:T].contiguous()
    d = X.shape[1]
    E, I = dl.routed.n_experts, dl.routed.I
    I_sh = dl.shared.I if dl.shared is not None else 0
    r = bm.Routing.empty(T, E, k, 32)
    ws = bm.workspace(bm.moe_layer_workspace_bytes(T, d, I, E, k, I_sh))
    Y = torch.empty((T, d), dtype=torch.int16, device="cuda")
    bm.moe_layer(lg, X, dl.routed, dl.shared, k, 32, r, Y, ws)
    torch.cuda.synchronize()
    assert bm.moe_check_status(ws) == 0
    ref = oracle.route(dl.logits[:T], k, 32)
    Y64, _ = oracle.forward(dl.X_host[:T], dl.routed_host, dl.shared_host, ref["ids"], ref["w"])
    return Y.cpu().numpy().view(np.uint16), Y64


@pytest.mark.parametrize("T", [1, 12])  # the decode kernel, the tensor-core path
def test_alternating_expert_sets(T):
    cfgs = [synth.small_config(T=12, d=256, E=8, k=2, I=128, I_shared=128, seed=s) for s in (31, 32)]
    layers = [G.DeviceLayer.from_host(synth.draw_layer(c)) for c in cfgs]
    for rep in range(2):
        for i, dl in enumerate(layers):
            y, ref = _layer_call(dl, 2, T)
            G.assert_y_close(y, ref, f"set {i}, pass {rep}")


@pytest.mark.parametrize("T", [1, 12])
def test_expert_set_rewritten_in_place(T):
    cfg = synth.small_config(T=12, d=256, E=8, k=2, I=128, I_shared=128, seed=33)
    layer = synth.draw_layer(cfg)
    dl = G.DeviceLayer.from_host(layer)
    y, ref = _layer_call(dl, 2, T)
    G.assert_y_close(y, ref, "before")
    # new weights written into the same device buffers (the prepacked layout of a fresh draw)
    fresh = synth.draw_layer(synth.small_config(T=12, d=256, E=8, k=2, I=128, I_shared=128, seed=34))
    new_routed = bm.prepare_experts(fresh.routed)
    new_shared = bm.prepare_experts(fresh.shared)
    for old, new in ((dl.routed, new_routed), (dl.shared, new_shared)):
        for m in ("gate", "up", "down"):
            getattr(old, m).q.copy_(getattr(new, m).q)
            getattr(old, m).sb.copy_(getattr(new, m).sb)
    torch.cuda.synchronize()
    dl.routed_host, dl.shared_host = fresh.routed, fresh.shared
    y2, ref2 = _layer_call(dl, 2, T)
    G.assert_y_close(y2, ref2, "after the rewrite")
    assert not np.allclose(ref, ref2), "the two draws should give different layers"
