"""GPU parity of the exact wide top-K (moe_topk_wide) through the C ABI: indices
and values bit for bit against the oracle's full sort of each row."""
import zlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import bit_moe_expert_gb300 as bm  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_expert_gb300 import build
    build.build()
    bm.lib()


def _gpu(lg, K):
    x = torch.from_numpy(np.ascontiguousarray(lg, dtype=np.float32)).cuda()
    T = lg.shape[0]
    vals = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    bm.moe_topk_wide(x, K, vals, idx)
    torch.cuda.synchronize()
    return vals.cpu().numpy(), idx.cpu().numpy()


def _check(lg, K, rows=None):
    vals, idx = _gpu(lg, K)
    sel = np.arange(lg.shape[0]) if rows is None else np.asarray(rows)
    rv, ri = oracle.topk_wide(lg[sel], K)
    np.testing.assert_array_equal(idx[sel], ri)
    np.testing.assert_array_equal(vals[sel].view(np.uint32), rv.view(np.uint32))


CASES = [  # (name, T, V, K): the canvas width and its sampler K, ragged widths (scalar loads when V % 4 != 0),
    # fewer chunks than K, K = V, K = 1
    ("canvas_rows", 16, 262144, 64),
    ("ragged", 3, 1000, 5),
    ("odd_width", 2, 1001, 64),
    ("fewer_chunks_than_K", 4, 300, 64),
    ("K_equals_V", 2, 64, 64),
    ("K1", 5, 262144, 1),
    ("mid", 7, 50000, 37),
]


@pytest.mark.parametrize("name,T,V,K", CASES, ids=[c[0] for c in CASES])
def test_topk_wide_random(name, T, V, K):
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    _check(rng.standard_normal((T, V)).astype(np.float32), K)


def test_topk_wide_full_canvas_sampled():
    # the benchmark's launch: 256 positions x 262,144 logits, K = 64; the oracle checks a sample of rows
    rng = np.random.default_rng(41)
    lg = rng.standard_normal((256, 262144)).astype(np.float32)
    _check(lg, 64, rows=[0, 1, 2, 63, 64, 127, 128, 147, 148, 200, 254, 255])


def test_topk_wide_heavy_ties():
    # 7 distinct values over 262,144 entries: every selected chunk's entries tie with theta,
    # so the candidate set is as large as it can be (K x 256)
    rng = np.random.default_rng(42)
    lg = rng.integers(-3, 4, size=(3, 262144)).astype(np.float32)
    _check(lg, 64)
    _check(np.zeros((2, 5000), np.float32), 64)


def test_topk_wide_candidate_counts_on_each_path():
    # integer values 0..10: every chunk's maximum is 10 and about 23 of its entries tie with it, so the 64
    # selected chunks give about 1,500 candidates (sorted in the buffer); 0..2 gives about 5,500 (more
    # than the buffer: the radix select over the candidates' keys); normal values give about K (ranked)
    rng = np.random.default_rng(45)
    _check(rng.integers(0, 11, size=(2, 262144)).astype(np.float32), 64)
    _check(rng.integers(0, 3, size=(2, 262144)).astype(np.float32), 64)
    _check(rng.integers(0, 11, size=(3, 70001)).astype(np.float32), 17)


def test_topk_wide_clustered_signed_zero_and_infinities():
    rng = np.random.default_rng(43)
    lg = rng.standard_normal((4, 20000)).astype(np.float32)
    lg[0, 512:768] += 50.0        # every top entry in one chunk
    lg[1, :] = -np.inf
    lg[1, 7] = 1.0
    lg[2, :] = np.where(rng.random(20000) < 0.5, -0.0, 0.0).astype(np.float32)
    lg[3, 100] = np.inf
    lg[3, 19999] = np.inf
    _check(lg, 64)


def test_topk_wide_deterministic_and_bad_arguments():
    rng = np.random.default_rng(44)
    lg = rng.standard_normal((9, 70000)).astype(np.float32)
    a = _gpu(lg, 64)
    b = _gpu(lg, 64)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[0].view(np.uint32), b[0].view(np.uint32))
    x = torch.zeros((1, 100), dtype=torch.float32, device="cuda")
    v = torch.zeros((1, 65), dtype=torch.float32, device="cuda")
    i = torch.zeros((1, 65), dtype=torch.int32, device="cuda")
    with pytest.raises(bm.MoeError) as ei:
        bm.moe_topk_wide(x, 65, v, i)
    assert bm.STATUS_NAMES[ei.value.status] == "MOE_ERR_UNSUPPORTED"
    with pytest.raises(bm.MoeError) as ei:
        bm.moe_topk_wide(torch.zeros((1, 10), dtype=torch.float32, device="cuda"), 20, v, i)
    assert bm.STATUS_NAMES[ei.value.status] == "MOE_ERR_INVALID_ARG"
    bm.moe_topk_wide(torch.zeros((0, 100), dtype=torch.float32, device="cuda"), 8, v, i)  # T = 0
