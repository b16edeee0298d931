"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: code hosted by a framework that owns all
device memory and forbids allocation once it has started, or code running while
a stream is captured into a CUDA graph.  moe_route_noalloc serves them by using
a scratch array compiled into the library instead of a caller-provided
workspace.  Its outputs must equal moe_route's bit for bit (routing is integer
bookkeeping plus weights rounded the same way), including when two calls follow
each other and share that scratch array.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import bit_moe_expert_gb300 as bm  # noqa: E402


def _route_with_workspace(lg, k, block_rows):
    T, E = lg.shape
    r = bm.Routing.empty(T, E, k, block_rows)
    ws = bm.workspace(bm.moe_route_workspace_bytes(T, E, k))
    bm.moe_route(lg, k, block_rows, r, ws)
    return r


def _host(r):
    nb = int(r.num_blocks.item())
    A = r.ids.numel()
    return dict(ids=r.ids.cpu().numpy(), w=r.w.cpu().numpy().view(np.int32), counts=r.counts.cpu().numpy(),
                offsets=r.offsets.cpu().numpy(), perm=r.perm.cpu().numpy()[:A],
                inv_perm=r.inv_perm.cpu().numpy()[:A], block_map=r.block_map.cpu().numpy()[:nb], num_blocks=nb)


def test_route_noalloc_equals_moe_route_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_expert_gb300 import build
    build.build()
    rng = np.random.default_rng(77)
    # two calls in a row on the shared scratch array, then the largest size it accepts
    cases = [(512, 256, 8, 128), (1000, 128, 8, 64), (8192, 256, 8, 128)]
    outs = []
    for T, E, k, block_rows in cases:
        lg = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).cuda()
        ref = _route_with_workspace(lg, k, block_rows)
        got = bm.Routing.empty(T, E, k, block_rows)
        bm.moe_route_noalloc(lg, k, block_rows, got)
        outs.append((ref, got))
    torch.cuda.synchronize()
    for (ref, got), (T, E, k, block_rows) in zip(outs, cases):
        a, b = _host(ref), _host(got)
        assert a["num_blocks"] == b["num_blocks"]
        for key in ("ids", "w", "counts", "offsets", "perm", "inv_perm", "block_map"):
            np.testing.assert_array_equal(b[key], a[key], err_msg=f"{key} T={T} E={E}")
        assert got.block_rows == block_rows


@pytest.mark.parametrize("mode", ["ticket", "gridsync"])
def test_route_noalloc_both_multi_chunk_modes(mode, monkeypatch):
    """At T = 8192 (256 chunks of 32 tokens) the routing kernel places the
    assignments either after a bounded barrier over the grid or in the last CTA
    to arrive (per-chunk bases in the scratch array); both must equal moe_route
    (in its default mode) bit for bit."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rng = np.random.default_rng(78)
    T, E, k, block_rows = 8192, 256, 8, 96
    lg = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).cuda()
    ref = _route_with_workspace(lg, k, block_rows)
    torch.cuda.synchronize()
    monkeypatch.setenv("MOE_ROUTE_MODE", mode)
    got = []
    for _ in range(2):
        r = bm.Routing.empty(T, E, k, block_rows)
        bm.moe_route_noalloc(lg, k, block_rows, r)
        got.append(r)
    torch.cuda.synchronize()
    assert bm.moe_route_noalloc_check_status() == 0
    a = _host(ref)
    for r in got:
        b = _host(r)
        assert a["num_blocks"] == b["num_blocks"]
        for key in ("ids", "w", "counts", "offsets", "perm", "inv_perm", "block_map"):
            np.testing.assert_array_equal(b[key], a[key], err_msg=f"{key} mode={mode}")


def test_route_noalloc_reports_device_errors():
    """A non-finite logit is recorded in the scratch array's status word, read
    (and cleared) by moe_route_noalloc_check_status; the next clean call
    reports nothing."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    T, E, k = 64, 256, 8
    lg = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    lg[5, 17] = float("nan")
    r = bm.Routing.empty(T, E, k, 32)
    assert bm.moe_route_noalloc_check_status() == 0
    bm.moe_route_noalloc(lg, k, 32, r)
    assert bm.moe_route_noalloc_check_status() == 6  # MOE_ERR_NONFINITE
    lg[5, 17] = 0.0
    bm.moe_route_noalloc(lg, k, 32, r)
    assert bm.moe_route_noalloc_check_status() == 0


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    T, E, k = 8193, 256, 8   # T*k = 65544 > 65536 assignments
    r = bm.Routing.empty(T, E, k, 128)
    lg = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    with pytest.raises(bm.MoeError) as e:
        bm.moe_route_noalloc(lg, k, 128, r)
    assert e.value.status == 2  # MOE_ERR_UNSUPPORTED
