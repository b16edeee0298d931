"""Helpers shared by the GPU tests: upload synthetic inputs, run the C ABI,
compare with the oracle.  The tolerance is the one the layer is specified with
(relative L2 error 5e-3; elementwise 2e-2 scaled by max(1, |Y|), because a bf16
output alone is off by up to half an ulp, 0.0625 at |Y| = 16)."""
import numpy as np
import torch

import bit_moe_expert_gb300 as bm
from bit_moe_expert_gb300 import synth

REL_L2 = 5e-3
ELEM = 2e-2


def route_gpu(logits_np, k, block_rows, device="cuda"):
    lg = torch.from_numpy(np.ascontiguousarray(logits_np, dtype=np.float32)).to(device)
    T, E = lg.shape
    r = bm.Routing.empty(T, E, k, block_rows, device)
    ws = bm.workspace(bm.moe_route_workspace_bytes(T, E, k), device)
    bm.moe_route(lg, k, block_rows, r, ws)
    torch.cuda.synchronize()
    return r, ws


def routing_to_host(r):
    nb = int(r.num_blocks.item())
    A = r.ids.numel()
    return dict(ids=r.ids.cpu().numpy(), w=r.w.cpu().numpy(), counts=r.counts.cpu().numpy(),
                offsets=r.offsets.cpu().numpy(), perm=r.perm.cpu().numpy()[:A], inv_perm=r.inv_perm.cpu().numpy()[:A],
                block_map=r.block_map.cpu().numpy()[:nb], num_blocks=nb)


def assert_routing_equal(got, ref):
    np.testing.assert_array_equal(got["ids"], ref["ids"])
    wg = got["w"].view(np.int32).astype(np.int64)
    wr = ref["w"].view(np.int32).astype(np.int64)
    if not np.array_equal(wg, wr):
        bad = np.argwhere(wg != wr)
        raise AssertionError(f"routing weights differ at {len(bad)} places, max {np.abs(wg - wr).max()} ulp, "
                             f"first {bad[:4].tolist()}")
    for key in ("counts", "offsets", "perm", "inv_perm", "block_map"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    assert got["num_blocks"] == ref["num_blocks"]


def y_errors(y_bits, ref64):
    y = synth.bf16_bits_to_f32(y_bits).astype(np.float64)
    diff = y - ref64
    rel_l2 = float(np.linalg.norm(diff) / max(np.linalg.norm(ref64), 1e-300))
    mixed = float(np.max(np.abs(diff) / np.maximum(1.0, np.abs(ref64)))) if diff.size else 0.0
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    return dict(rel_l2=rel_l2, mixed=mixed, max_abs=max_abs)


def assert_y_close(y_bits, ref64, what=""):
    e = y_errors(y_bits, ref64)
    assert np.all(np.isfinite(synth.bf16_bits_to_f32(y_bits))), f"{what}: non-finite output"
    assert e["rel_l2"] <= REL_L2 and e["mixed"] <= ELEM, f"{what}: {e}"
    return e


class DeviceLayer:
    """One layer's inputs on the device plus the host copies the oracle reads."""

    def __init__(self, X, logits, routed_host, shared_host, routed_dev, shared_dev):
        self.X_host, self.logits = X, logits
        self.routed_host, self.shared_host = routed_host, shared_host
        self.routed, self.shared = routed_dev, shared_dev
        self.X = torch.from_numpy(X.view(np.int16)).cuda()

    @staticmethod
    def from_host(layer):
        routed = bm.prepare_experts(layer.routed)
        shared = bm.prepare_experts(layer.shared) if layer.shared is not None else None
        return DeviceLayer(layer.X, layer.logits, layer.routed, layer.shared, routed, shared)

    @staticmethod
    def from_device_draw(cfg, layer_idx, T):
        """Large weights drawn on the device; host copies pulled back for the oracle."""
        dev = torch.device("cuda")
        rex = synth.draw_experts_torch(cfg, layer_idx, dev)
        sex = synth.draw_experts_torch(cfg, layer_idx, dev, E=1, I=cfg.I_shared, tag=20) if cfg.I_shared else None

        def host(ex):
            return {m: (q.cpu().numpy().view(np.uint32), s.cpu().numpy().view(np.uint16),
                        b.cpu().numpy().view(np.uint16)) for m, (q, s, b) in ex.items()}

        X = synth.draw_x(cfg, T, layer_idx)
        logits = synth.draw_logits(cfg, T, layer_idx)
        return DeviceLayer(X, logits, host(rex), host(sex) if sex else None, bm.prepare_experts(rex),
                           bm.prepare_experts(sex) if sex else None)

    def forward(self, r, path=None):
        import os
        T, d = self.X.shape
        k = r.ids.shape[1]
        E = self.routed.n_experts
        I_sh = self.shared.I if self.shared is not None else 0
        ws = bm.workspace(bm.moe_forward_workspace_bytes(T, d, self.routed.I, E, k, I_sh))
        Y = torch.empty((T, d), dtype=torch.int16, device="cuda")
        old = os.environ.get("MOE_PATH")
        try:
            if path:
                os.environ["MOE_PATH"] = path
            bm.moe_forward(self.X, self.routed, self.shared, r, Y, ws)
        finally:
            if path:
                if old is None:
                    os.environ.pop("MOE_PATH", None)
                else:
                    os.environ["MOE_PATH"] = old
        torch.cuda.synchronize()
        status = bm.moe_check_status(ws)
        assert status == 0, bm.moe_status_string(status)
        return Y.cpu().numpy().view(np.uint16)
