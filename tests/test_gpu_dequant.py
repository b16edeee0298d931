"""moe_dequant_experts: the expanded weights q * scale + bias of a prepacked
matrix, rounded once to fp16, against the oracle's fp64 dequantisation of the
checkpoint-layout codes rounded to fp16 -- bit for bit, for 4-, 3- and 2-bit
codes and a ragged number of rows."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import bit_moe_expert_gb300 as bm  # noqa: E402
from bit_moe_expert_gb300 import synth  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_expert_gb300 import build
    build.build()
    bm.lib()


@pytest.mark.parametrize("bits", [4, 3, 2])
def test_dequant_matches_oracle(bits):
    cfg = synth.small_config(T=4, d=192, E=3, k=2, I=64, I_shared=0, bits=bits)
    layer = synth.draw_layer(cfg)
    ex = bm.prepare_experts(layer.routed)
    for name in ("gate", "down"):
        q, s, b = layer.routed[name]
        E, N, G = s.shape
        W = torch.empty((E, N, G * 64), dtype=torch.int16, device="cuda")
        bm.moe_dequant_experts(getattr(ex, name), bits, W)
        got = W.cpu().numpy().view(np.uint16)
        for e in range(E):
            ref = oracle.dequant_matrix((q, s, b), e).astype(np.float16).view(np.uint16)
            np.testing.assert_array_equal(got[e], ref, err_msg=f"{bits}-bit {name} expert {e}")
