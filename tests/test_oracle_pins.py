"""Pins for the CPU oracle: checks against facts the pages print, closed forms,
invariants, special cases and independent brute force.  No GPU needed.

None of these re-types the oracle's own code: the dequantisation is checked on a
hand-worked example, routing against properties of a top-k selection and a
library softmax, and the layer against a dense NumPy brute force written in a
different shape (every expert on every token, then masked).
"""
import json
import math
import os

import numpy as np
import pytest

from bit_moe_expert_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_known_values(oracle):
    cases = {1.0: 0x3F80, -2.0: 0xC000, 0.5: 0x3F00, 0.0: 0x0000, 1.0 / 3.0: 0x3EAB,
             0.1: 0x3DCD, 3.0e38: 0x7F62, 65504.0: 0x4780}
    for x, bits in cases.items():
        assert oracle.double_to_bf16(x) == bits, x
    assert oracle.double_to_bf16(-0.0) == 0x8000
    # ties to even: 1 + 2^-8 is halfway between 1 (even) and 1 + 2^-7
    assert oracle.double_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert oracle.double_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # one rounding step, not two: just above the tie must round up even though
    # a detour through float32 would land exactly on the tie first
    assert oracle.double_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    # overflow
    assert oracle.double_to_bf16(4.0e38) == 0x7F80
    for bits in (0x3F80, 0xC2F7, 0x0001, 0x7F7F, 0x3A83):
        v = oracle.bf16_to_double(bits)
        assert oracle.double_to_bf16(v) == bits


def test_bf16_matches_torch_and_bit_trick(oracle):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(4000) * np.exp(rng.uniform(-20, 20, 4000))).astype(np.float32)
    ref_torch = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref_trick = synth.f32_to_bf16_bits(x)
    ours = np.array([oracle.double_to_bf16(float(v)) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(ours, ref_torch)
    np.testing.assert_array_equal(ours, ref_trick)


# ---------------------------------------------------------------- dequantisation

def _hand_example():
    g = _golden("dequant_example.json")
    words = np.array([int(h, 16) for h in g["words_hex"]], dtype=np.uint32).reshape(1, 1, -1)
    s = np.array([int(h, 16) for h in g["scale_bf16_hex"]], dtype=np.uint16).reshape(1, 1, -1)
    b = np.array([int(h, 16) for h in g["bias_bf16_hex"]], dtype=np.uint16).reshape(1, 1, -1)
    return g, (words, s, b)


def test_dequant_hand_worked_example(oracle):
    g, qsb = _hand_example()
    for k, v in g["expected"].items():
        assert oracle.dequant(qsb, 0, 0, int(k)) == v, k
    full = oracle.dequant_matrix(qsb, 0)
    assert full.shape == (1, g["K"])
    for k, v in g["expected"].items():
        assert full[0, int(k)] == v


def test_dequant_special_cases(oracle):
    rng = np.random.default_rng(1)
    q, s, b = synth.draw_qmat(rng, 2, 8, 128)
    # q = 0 gives the bias
    q0 = np.zeros_like(q)
    m = oracle.dequant_matrix((q0, s, b), 1)
    bias = synth.bf16_bits_to_f32(b[1]).astype(np.float64)
    np.testing.assert_array_equal(m, np.repeat(bias, 64, axis=1))
    # zero scale and bias gives exactly zero
    z = np.zeros_like(s)
    assert not np.any(oracle.dequant_matrix((q, z, z), 0))
    # every code 8 with bias = -8*scale gives exactly zero
    q8 = np.full_like(q, 0x88888888)
    assert not np.any(oracle.dequant_matrix((q8, s, b), 0))
    # code 15 gives 15*scale + bias = 7*scale when bias = -8*scale
    q15 = np.full_like(q, 0xFFFFFFFF)
    sc = synth.bf16_bits_to_f32(s[0]).astype(np.float64)
    np.testing.assert_array_equal(oracle.dequant_matrix((q15, s, b), 0), np.repeat(7.0 * sc, 64, axis=1))


def _numpy_dequant(qsb, e):
    """Independent vectorised dequantisation: each row's words unpacked into
    its bit stream (np.unpackbits, least significant bit first), then read
    `bits` bits per column; the code width follows from the shapes (K*bits/32
    words and K/64 groups per row)."""
    q, s, b = qsb
    bits = 32 * q.shape[-1] // (64 * s.shape[-1])
    N = q.shape[1]
    stream = np.unpackbits(np.ascontiguousarray(q[e]).astype("<u4").view(np.uint8).reshape(N, -1), axis=1,
                           bitorder="little")
    weights = (1 << np.arange(bits)).astype(np.float64)
    codes = stream.reshape(N, -1, bits).astype(np.float64) @ weights
    sc = np.repeat(synth.bf16_bits_to_f32(s[e]).astype(np.float64), 64, axis=1)
    bi = np.repeat(synth.bf16_bits_to_f32(b[e]).astype(np.float64), 64, axis=1)
    return codes * sc + bi


def test_dequant_matches_independent_numpy(oracle):
    rng = np.random.default_rng(2)
    for bits in (4, 3, 2):
        qsb = synth.draw_qmat(rng, 3, 16, 192, bits)
        for e in range(3):
            np.testing.assert_array_equal(oracle.dequant_matrix(qsb, e), _numpy_dequant(qsb, e))


def test_dequant_two_bit_hand_worked_example(oracle):
    # word 0xE4 = 0b11_10_01_00 holds codes 0, 1, 2, 3 for columns 0..3 (low bits first), then zeros;
    # the second word's top code (column 31) is 3; scale 0.25 and bias -0.5 give q / 4 - 1 / 2
    words = np.zeros((1, 1, 4), np.uint32)
    words[0, 0, 0] = 0xE4
    words[0, 0, 1] = 0xC0000000
    s = np.full((1, 1, 1), 0x3E80, np.uint16)   # 0.25
    b = np.full((1, 1, 1), 0xBF00, np.uint16)   # -0.5
    qsb = (words, s, b)
    want = {0: -0.5, 1: -0.25, 2: 0.0, 3: 0.25, 4: -0.5, 30: -0.5, 31: 0.25, 63: -0.5}
    for k, v in want.items():
        assert oracle.dequant(qsb, 0, 0, k) == v, k
    row = oracle.dequant_matrix(qsb, 0)[0]
    assert row.shape == (64,) and row[3] == 0.25 and row[31] == 0.25 and np.count_nonzero(row == 0.25) == 2


def test_dequant_two_bit_special_cases(oracle):
    rng = np.random.default_rng(3)
    q, s, b = synth.draw_qmat(rng, 2, 8, 128, bits=2)
    assert q.shape == (2, 8, 8)
    bias = synth.bf16_bits_to_f32(b[1]).astype(np.float64)
    np.testing.assert_array_equal(oracle.dequant_matrix((np.zeros_like(q), s, b), 1), np.repeat(bias, 64, axis=1))
    # every code 2 with bias = -2*scale gives exactly zero; code 3 gives the scale
    assert not np.any(oracle.dequant_matrix((np.full_like(q, 0xAAAAAAAA), s, b), 0))
    sc = synth.bf16_bits_to_f32(s[0]).astype(np.float64)
    np.testing.assert_array_equal(oracle.dequant_matrix((np.full_like(q, 0xFFFFFFFF), s, b), 0),
                                  np.repeat(sc, 64, axis=1))


def test_dequant_three_bit_hand_worked_example(oracle):
    # a row of 64 three-bit codes is 192 bits in 6 words, low bits first; code k starts at bit 3k, so
    # code 10 (bits 30..32) and code 21 (bits 63..65) straddle words.  Codes: 7 at column 0, 5 at
    # column 10, 6 at column 21, 3 at column 63, zero elsewhere; scale 0.25 and bias -1 give q / 4 - 1
    words = np.zeros((1, 1, 6), np.uint32)
    words[0, 0, 0] = 0x40000007   # bits 0..2 = 7; bit 30 = low bit of code 10
    words[0, 0, 1] = 0x00000001   # bit 32 = top bit of code 10 (5 = 0b101); bit 63 (low bit of code 21) = 0
    words[0, 0, 2] = 0x00000003   # bits 64, 65 = upper bits of code 21 (6 = 0b110)
    words[0, 0, 5] = 0x60000000   # bits 189, 190 = code 63 (3 = 0b011)
    s = np.full((1, 1, 1), 0x3E80, np.uint16)   # 0.25
    b = np.full((1, 1, 1), 0xBF80, np.uint16)   # -1.0
    qsb = (words, s, b)
    want = {0: 0.75, 1: -1.0, 9: -1.0, 10: 0.25, 11: -1.0, 20: -1.0, 21: 0.5, 22: -1.0, 62: -1.0, 63: -0.25}
    for k, v in want.items():
        assert oracle.dequant(qsb, 0, 0, k) == v, k
    row = oracle.dequant_matrix(qsb, 0)[0]
    assert row.shape == (64,) and np.count_nonzero(row != -1.0) == 4


def test_dequant_three_bit_special_cases(oracle):
    rng = np.random.default_rng(4)
    q, s, b = synth.draw_qmat(rng, 2, 8, 128, bits=3)
    assert q.shape == (2, 8, 12)
    bias = synth.bf16_bits_to_f32(b[1]).astype(np.float64)
    np.testing.assert_array_equal(oracle.dequant_matrix((np.zeros_like(q), s, b), 1), np.repeat(bias, 64, axis=1))
    # every code 4 (bit stream 001 repeated: the words cycle through 0x24924924, 0x49249249, 0x92492492)
    # with bias = -4*scale gives exactly zero; every code 7 gives 3*scale
    fours = np.tile(np.array([0x24924924, 0x49249249, 0x92492492], np.uint32), 4)
    assert not np.any(oracle.dequant_matrix((np.broadcast_to(fours, q.shape).copy(), s, b), 0))
    sc = synth.bf16_bits_to_f32(s[0]).astype(np.float64)
    np.testing.assert_array_equal(oracle.dequant_matrix((np.full_like(q, 0xFFFFFFFF), s, b), 0),
                                  np.repeat(3.0 * sc, 64, axis=1))


# ---------------------------------------------------------------- top-k routing

def _check_topk_properties(logits, ids, k):
    T, E = logits.shape
    for t in range(T):
        sel = list(ids[t])
        assert len(set(sel)) == k
        vals = logits[t, sel]
        # selection order: descending value, lower index first among equal values
        for a, b in zip(range(k - 1), range(1, k)):
            assert (vals[a] > vals[b]) or (vals[a] == vals[b] and sel[a] < sel[b])
        rest = np.setdiff1d(np.arange(E), sel)
        if rest.size:
            worst = vals.min()
            assert np.all(logits[t, rest] <= worst)
            # an unselected expert tied with the worst selected value must have a higher index
            tied = rest[logits[t, rest] == worst]
            assert np.all(tied > max(s for s in sel if logits[t, s] == worst))


# ---------------------------------------------------------------- router projection

def test_router_logits_one_hot_tokens_pick_router_columns(oracle):
    # a token that is the i-th unit vector scores expert e with Wr[e][i] exactly
    rng = np.random.default_rng(21)
    d, E = 64, 16
    Wr = synth.f32_to_bf16_bits(rng.standard_normal((E, d)).astype(np.float32))
    cols = [0, 5, 63, 17]
    X = np.zeros((len(cols), d), np.uint16)
    for t, i in enumerate(cols):
        X[t, i] = 0x3F80  # 1.0
    lg = oracle.router_logits(X, Wr)
    want = synth.bf16_bits_to_f32(Wr).astype(np.float64)[:, cols].T
    assert np.array_equal(lg, want)


def test_router_logits_exact_rational_brute_force(oracle):
    # small integers and halves: every product and partial sum is exact in fp64,
    # so the oracle must equal the exact rational dot products
    from fractions import Fraction
    rng = np.random.default_rng(22)
    T, d, E = 3, 32, 8
    xv = rng.integers(-8, 9, size=(T, d)) / 2.0
    wv = rng.integers(-16, 17, size=(E, d)) / 4.0
    X = synth.f32_to_bf16_bits(xv.astype(np.float32))
    Wr = synth.f32_to_bf16_bits(wv.astype(np.float32))
    lg = oracle.router_logits(X, Wr)
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(xv[t, i])) * Fraction(float(wv[e, i])) for i in range(d))
            assert Fraction(lg[t, e]) == exact, (t, e)


def test_router_logits_linear_and_transposed_roles(oracle):
    # scaling a token by 2 (exact in bf16) doubles its logits; swapping the roles of the
    # token block and the router (both d-wide) transposes the result
    rng = np.random.default_rng(23)
    d = 128
    A = synth.f32_to_bf16_bits(rng.standard_normal((6, d)).astype(np.float32))
    B = synth.f32_to_bf16_bits(rng.standard_normal((6, d)).astype(np.float32))
    lg = oracle.router_logits(A, B)
    A2 = synth.f32_to_bf16_bits(2.0 * synth.bf16_bits_to_f32(A))
    assert np.array_equal(oracle.router_logits(A2, B), 2.0 * lg)
    assert np.allclose(oracle.router_logits(B, A), lg.T, rtol=0, atol=1e-12)


def test_router_logits_scale_of_synthetic_router(oracle):
    # the synthetic router (N(0, 1/d) rows) gives logits of about unit variance on
    # N(0, 1) tokens, the scale of the logits the other workloads draw directly
    cfg = synth.CONFIGS["decode"]
    X = synth.draw_x(cfg, 16, 0)
    Wr = synth.draw_router(cfg, 0)
    lg = oracle.router_logits(X, Wr)
    assert lg.shape == (16, cfg.E)
    assert 0.8 < lg.std() < 1.25


# ---------------------------------------------------------------- wide top-K (the sampler's candidates)

def _stable_desc(row):
    # library stable sort on the negated values (-0.0 made +0.0 first): equal values keep index order
    r = np.where(row == 0.0, np.float32(0.0), row)
    return np.argsort(-r.astype(np.float64), kind="stable")


def test_topk_wide_matches_library_stable_sort(oracle):
    rng = np.random.default_rng(31)
    for (T, V, K) in [(3, 1000, 5), (2, 4096, 64), (1, 300, 300), (4, 257, 1)]:
        lg = rng.standard_normal((T, V)).astype(np.float32)
        vals, idx = oracle.topk_wide(lg, K)
        for t in range(T):
            want = _stable_desc(lg[t])[:K]
            assert np.array_equal(idx[t], want)
            assert np.array_equal(vals[t], lg[t][want])


def test_topk_wide_ties_and_signed_zero(oracle):
    lg = np.array([[1.0, 3.0, 3.0, -0.0, 0.0, 3.0, 2.0, 0.0]], np.float32)
    vals, idx = oracle.topk_wide(lg, 6)
    assert idx[0].tolist() == [1, 2, 5, 6, 0, 3]
    lg2 = np.zeros((1, 50), np.float32)
    _, idx2 = oracle.topk_wide(lg2, 7)
    assert idx2[0].tolist() == list(range(7))


def test_topk_wide_closed_form_ramp(oracle):
    V, K = 262144, 64
    lg = np.arange(V, dtype=np.float32)[None, :]  # exact in fp32 below 2^24
    vals, idx = oracle.topk_wide(lg, K)
    assert idx[0].tolist() == list(range(V - 1, V - 1 - K, -1))
    assert np.array_equal(vals[0], lg[0][idx[0]])


def _chunked_topk(row, K, chunk):
    """The two-stage selection: chunk maxima, the K chunks with the largest maxima, then the top K of their
    entries; the order is by (value, lower index), so every comparison is strict."""
    V = row.size
    keys = [(float(0.0 if v == 0 else v), -i) for i, v in enumerate(row)]
    nch = -(-V // chunk)
    cmax = [max(keys[c * chunk:(c + 1) * chunk]) for c in range(nch)]
    best = sorted(range(nch), key=lambda c: cmax[c], reverse=True)[:K]
    cand = [k for c in best for k in keys[c * chunk:(c + 1) * chunk]]
    return [-i for _, i in sorted(cand, reverse=True)[:K]]


def test_topk_wide_two_stage_selection_is_exact(oracle):
    # the pages' argument: a top-K entry has fewer than K chunk maxima above it, so
    # its chunk is among the K best chunks; checked on random rows, heavy ties and
    # clustered maxima (all large values in one chunk)
    rng = np.random.default_rng(32)
    rows = [rng.standard_normal(2048).astype(np.float32),
            rng.integers(-3, 4, size=2048).astype(np.float32),
            np.concatenate([rng.standard_normal(256) + 10, rng.standard_normal(1792)]).astype(np.float32),
            np.zeros(1000, np.float32)]
    for row in rows:
        for K in (1, 8, 64):
            _, idx = oracle.topk_wide(row[None, :], K)
            assert _chunked_topk(row, K, 64) == idx[0].tolist()


def test_topk_wide_rejects_nan(oracle):
    lg = np.zeros((1, 10), np.float32)
    lg[0, 3] = np.nan
    with pytest.raises(ValueError):
        oracle.topk_wide(lg, 2)


def test_topk_properties_random(oracle):
    rng = np.random.default_rng(3)
    for (T, E, k) in [(40, 16, 2), (25, 256, 8), (9, 128, 8), (7, 33, 5), (3, 5, 5)]:
        lg = rng.standard_normal((T, E)).astype(np.float32)
        ids, w = oracle.topk(lg, k)
        _check_topk_properties(lg, ids, k)
        # brute force by Python's sort
        for t in range(T):
            ref = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))[:k]
            assert list(ids[t]) == ref


def test_topk_forced_ties(oracle):
    rng = np.random.default_rng(4)
    lg = rng.integers(-2, 3, size=(64, 32)).astype(np.float32)  # heavy ties
    lg[0] = 0.0
    lg[1] = -1.0
    lg[1, ::2] = 1.0
    ids, w = oracle.topk(lg, 8)
    _check_topk_properties(lg, ids, 8)
    assert list(ids[0]) == list(range(8))
    assert list(ids[1]) == [0, 2, 4, 6, 8, 10, 12, 14]


def test_topk_equal_logits_uniform_weights(oracle):
    for k in (1, 2, 3, 8):
        lg = np.full((4, 16), 0.75, dtype=np.float32)
        ids, w = oracle.topk(lg, k)
        assert (ids == np.arange(k)).all()
        assert (w == np.float32(1.0 / k)).all()


def test_topk_weights_closed_forms(oracle):
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(6)
    lg = (rng.standard_normal((50, 64)) * 3).astype(np.float32)
    # k = E: the weights are the plain softmax over all experts, in selection order
    ids, w = oracle.topk(lg, 64)
    p = scipy_special.softmax(lg.astype(np.float64), axis=1)
    ref = np.take_along_axis(p, ids.astype(np.int64), axis=1).astype(np.float32)
    assert np.max(np.abs(w.view(np.int32) - ref.view(np.int32))) <= 1
    # k < E: softmax over E renormalised over the selected k (the configs' wording)
    ids, w = oracle.topk(lg, 8)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    ref = (sel / sel.sum(axis=1, keepdims=True)).astype(np.float32)
    assert np.max(np.abs(w.view(np.int32) - ref.view(np.int32))) <= 1
    # ratios follow exp(l_i - l_j); weights sum to one
    r = w[:, 1].astype(np.float64) / w[:, 0]
    l_sel = np.take_along_axis(lg, ids.astype(np.int64), axis=1).astype(np.float64)
    np.testing.assert_allclose(r, np.exp(l_sel[:, 1] - l_sel[:, 0]), rtol=3e-7)
    np.testing.assert_allclose(w.sum(axis=1, dtype=np.float64), 1.0, atol=8 * 2 ** -24)


def test_topk_rejects_nonfinite(oracle):
    lg = np.zeros((2, 8), np.float32)
    lg[1, 3] = np.nan
    with pytest.raises(ValueError):
        oracle.topk(lg, 2)
    lg[1, 3] = np.inf
    with pytest.raises(ValueError):
        oracle.topk(lg, 2)


# ---------------------------------------------------------------- routing layout

def _check_layout(ids, E, BM, r):
    T, k = ids.shape
    A = T * k
    flat = ids.reshape(-1)
    assert r["counts"].sum() == A
    np.testing.assert_array_equal(r["counts"], np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(r["offsets"], np.concatenate([[0], np.cumsum(r["counts"])]))
    perm, inv = r["perm"], r["inv_perm"]
    np.testing.assert_array_equal(np.sort(perm), np.arange(A))
    np.testing.assert_array_equal(inv[perm], np.arange(A))
    for e in range(E):
        seg = perm[r["offsets"][e]:r["offsets"][e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)  # stable: ascending assignment index
    bm = r["block_map"]
    assert r["num_blocks"] == int(np.sum(-(-r["counts"] // BM)))
    assert bm[:, 2].sum() == A
    assert np.all((bm[:, 2] >= 1) & (bm[:, 2] <= BM))
    # blocks tile each expert's segment in order
    pos = 0
    for e_, start, rows in bm:
        assert start == pos
        assert r["offsets"][e_] <= start and start + rows <= r["offsets"][e_ + 1]
        pos += rows
    assert pos == A


def test_route_layout_invariants(oracle):
    rng = np.random.default_rng(7)
    for (T, E, k, BM) in [(16, 16, 2, 16), (100, 256, 8, 32), (37, 8, 3, 4), (1, 256, 8, 128), (0, 4, 2, 8)]:
        lg = rng.standard_normal((T, E)).astype(np.float32)
        r = oracle.route(lg, k, BM)
        _check_layout(r["ids"], E, BM, r)


def test_route_layout_skewed_and_empty_experts(oracle):
    cfg = synth.CONFIGS["prefill4096"]
    lg = synth.draw_logits(cfg, 1024, 0)
    r = oracle.route(lg, cfg.k, 128)
    _check_layout(r["ids"], cfg.E, 128, r)
    assert (r["counts"] == 0).sum() > cfg.E // 2  # Zipf offsets leave most experts empty


def test_route_assignments_at_2k_tokens(oracle):
    fact = _golden("page_facts.json")["assignments_at_2k_tokens"]
    rng = np.random.default_rng(8)
    lg = rng.standard_normal((fact["tokens"], fact["E"])).astype(np.float32)
    r = oracle.route(lg, fact["k"], 32)
    assert r["counts"].sum() == fact["assignments"]
    assert r["counts"].mean() == fact["rows_per_expert_mean"]


# ---------------------------------------------------------------- format

def test_format_bytes_match_pages():
    facts = _golden("page_facts.json")
    # 4.5 bits per weight: 4-bit code + 16+16 bits per 64 weights
    assert synth.expert_bytes(512, 2048) * 8 / (512 * 2048) == 4.5
    assert synth.ffn_bytes(2048, 512) == 1_769_472
    c = facts["canvas_step_bytes"]
    step = c["E"] * c["layers"] * synth.ffn_bytes(c["d"], c["I"])
    assert step == 12_846_366_720  # 3,345,408 B per expert x 128 x 30
    assert abs(step / 1e9 - c["approx_GB"]) < 0.05
    ck = facts["checkpoint_size"]
    q4 = ck["params"] * 4.5 / 8 / 1e9
    bf16 = ck["params"] * 2 / 1e9
    assert abs(q4 - ck["q4_GB"]) / ck["q4_GB"] < 0.03
    assert bf16 == ck["bf16_GB"]


# ---------------------------------------------------------------- the layer

def _silu(v):
    return v / (1.0 + np.exp(-v))


def _dense_brute_force(layer, ids, w):
    """Every expert applied to every token, then masked by the routing and
    weighted; plus the shared expert.  NumPy float64, independent of the oracle."""
    X = synth.bf16_bits_to_f32(layer.X).astype(np.float64)
    T = X.shape[0]
    E = layer.routed["gate"][0].shape[0]
    d = X.shape[1]
    Y = np.zeros((T, d))
    for e in range(E):
        Wg = _numpy_dequant(layer.routed["gate"], e)
        Wu = _numpy_dequant(layer.routed["up"], e)
        Wd = _numpy_dequant(layer.routed["down"], e)
        Ye = (_silu(X @ Wg.T) * (X @ Wu.T)) @ Wd.T          # [T][d] for every token
        mask = np.where(ids == e, w.astype(np.float64), 0.0).sum(axis=1)  # routing weight or 0
        Y += mask[:, None] * Ye
    if layer.shared is not None:
        Wg = _numpy_dequant(layer.shared["gate"], 0)
        Wu = _numpy_dequant(layer.shared["up"], 0)
        Wd = _numpy_dequant(layer.shared["down"], 0)
        Y += (_silu(X @ Wg.T) * (X @ Wu.T)) @ Wd.T
    return Y


@pytest.mark.parametrize("kw", [dict(), dict(T=9, E=8, k=3, I=64, I_shared=0, d=128),
                                dict(T=5, E=4, k=4, I=64, I_shared=192, d=64),
                                dict(T=7, E=6, k=2, I=128, I_shared=64, d=128, bits=2),
                                dict(T=6, E=5, k=2, I=192, I_shared=64, d=128, bits=3)])
def test_forward_matches_dense_brute_force(oracle, kw):
    cfg = synth.small_config(**kw)
    layer = synth.draw_layer(cfg)
    ids, w = oracle.topk(layer.logits, cfg.k)
    Y64, Y16 = oracle.forward(layer.X, layer.routed, layer.shared, ids, w)
    ref = _dense_brute_force(layer, ids, w)
    np.testing.assert_allclose(Y64, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())
    # the bf16 copy is the fp64 result rounded once
    assert all(Y16.reshape(-1)[i] == oracle.double_to_bf16(Y64.reshape(-1)[i]) for i in range(0, Y64.size, 37))


def test_forward_token_subrange_equals_full(oracle):
    cfg = synth.small_config()
    layer = synth.draw_layer(cfg)
    ids, w = oracle.topk(layer.logits, cfg.k)
    full, _ = oracle.forward(layer.X, layer.routed, layer.shared, ids, w)
    part, _ = oracle.forward(layer.X, layer.routed, layer.shared, ids, w, 5, 11)
    np.testing.assert_array_equal(part, full[5:11])


def test_forward_single_expert_is_dense_swiglu_mlp(oracle):
    cfg = synth.small_config(E=1, k=1, I_shared=0, T=6)
    layer = synth.draw_layer(cfg)
    ids, w = oracle.topk(layer.logits, 1)
    assert (ids == 0).all() and (w == 1.0).all()
    Y64, _ = oracle.forward(layer.X, layer.routed, None, ids, w)
    X = synth.bf16_bits_to_f32(layer.X).astype(np.float64)
    Wg, Wu, Wd = (_numpy_dequant(layer.routed[m], 0) for m in ("gate", "up", "down"))
    # textbook SwiGLU MLP: (silu(x Wg^T) * (x Wu^T)) Wd^T
    np.testing.assert_allclose(Y64, (_silu(X @ Wg.T) * (X @ Wu.T)) @ Wd.T, rtol=1e-11, atol=1e-12)


def test_forward_one_hot_token_closed_form(oracle):
    cfg = synth.small_config(T=1, E=4, k=2, I=64, I_shared=64, d=128)
    layer = synth.draw_layer(cfg)
    m = 77
    X = np.zeros((1, cfg.d), np.uint16)
    X[0, m] = 0x3F80  # 1.0
    ids = np.array([[2, 0]], np.int32)
    w = np.array([[0.75, 0.25]], np.float32)
    Y64, _ = oracle.forward(X, layer.routed, layer.shared, ids, w)
    # with x = e_m: g_i = Wg[i][m], u_i = Wu[i][m], y_n = sum_i Wd[n][i] silu(g_i) u_i
    ref = np.zeros(cfg.d)
    for e, wt in [(2, 0.75), (0, 0.25)]:
        ex = layer.routed
        h = [_silu(oracle.dequant(ex["gate"], e, i, m)) * oracle.dequant(ex["up"], e, i, m) for i in range(cfg.I)]
        for n in range(cfg.d):
            ref[n] += wt * sum(oracle.dequant(ex["down"], e, n, i) * h[i] for i in range(cfg.I))
    sh = layer.shared
    h = [_silu(oracle.dequant(sh["gate"], 0, i, m)) * oracle.dequant(sh["up"], 0, i, m) for i in range(cfg.I_shared)]
    for n in range(cfg.d):
        ref[n] += sum(oracle.dequant(sh["down"], 0, n, i) * h[i] for i in range(cfg.I_shared))
    np.testing.assert_allclose(Y64[0], ref, rtol=1e-12, atol=1e-14)


def test_forward_zero_expert_contributes_nothing(oracle):
    cfg = synth.small_config()
    layer = synth.draw_layer(cfg)
    ids, w = oracle.topk(layer.logits, cfg.k)
    e0 = int(ids[0, 0])
    zeroed = {m: (q, s.copy(), b.copy()) for m, (q, s, b) in layer.routed.items()}
    for m in zeroed:
        zeroed[m][1][e0] = 0
        zeroed[m][2][e0] = 0
    w_masked = np.where(ids == e0, np.float32(0), w)
    Ya, _ = oracle.forward(layer.X, zeroed, layer.shared, ids, w)
    Yb, _ = oracle.forward(layer.X, layer.routed, layer.shared, ids, w_masked)
    np.testing.assert_array_equal(Ya, Yb)


def test_forward_code8_experts_leave_only_shared(oracle):
    cfg = synth.small_config()
    layer = synth.draw_layer(cfg)
    ids, w = oracle.topk(layer.logits, cfg.k)
    r8 = {m: (np.full_like(q, 0x88888888), s, b) for m, (q, s, b) in layer.routed.items()}
    Y, _ = oracle.forward(layer.X, r8, layer.shared, ids, w)
    Ys, _ = oracle.forward(layer.X, {m: (np.zeros_like(q), np.zeros_like(s), np.zeros_like(b))
                                     for m, (q, s, b) in layer.routed.items()}, layer.shared, ids, w)
    np.testing.assert_array_equal(Y, Ys)
    X = synth.bf16_bits_to_f32(layer.X).astype(np.float64)
    Wg, Wu, Wd = (_numpy_dequant(layer.shared[m], 0) for m in ("gate", "up", "down"))
    np.testing.assert_allclose(Y, (_silu(X @ Wg.T) * (X @ Wu.T)) @ Wd.T, rtol=1e-11, atol=1e-12)


def test_silu_closed_form_through_layer(oracle):
    # One routed expert with a single nonzero weight per matrix: the layer reduces
    # to y = wd * silu(wg * x) * (wu * x) at one output, checkable by hand.
    cfg = synth.small_config(T=1, E=1, k=1, I=64, I_shared=0, d=64)
    q = np.zeros((1, 64, 8), np.uint32)
    s = np.zeros((1, 64, 1), np.uint16)
    b = np.zeros((1, 64, 1), np.uint16)
    gate = (q.copy(), s.copy(), b.copy())
    up = (q.copy(), s.copy(), b.copy())
    down = (q.copy(), s.copy(), b.copy())
    gate[1][0, 5, 0] = 0x3F80   # scale 1.0 on row 5
    gate[0][0, 5, 0] = 0x2      # code 2 at column 0 -> Wg[5][0] = 2
    up[2][0, 5, 0] = 0xBF00     # bias -0.5 on row 5 -> Wu[5][k] = -0.5 for every k
    down[2][0, 9, 0] = 0x4040   # bias 3.0 on row 9 -> Wd[9][i] = 3 for every i
    X = np.zeros((1, 64), np.uint16)
    X[0, 0] = 0x3FC0            # x0 = 1.5
    ids = np.zeros((1, 1), np.int32)
    w = np.ones((1, 1), np.float32)
    Y, _ = oracle.forward(X, {"gate": gate, "up": up, "down": down}, None, ids, w)
    g = 2 * 1.5
    u = -0.5 * 1.5
    expect = 3.0 * (g / (1 + math.exp(-g))) * u
    assert Y[0, 9] == pytest.approx(expect, rel=1e-15)
    assert np.count_nonzero(Y) == 1
