"""ctypes wrapper over the C++ oracle (oracle/moe_oracle.cpp).

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and by
bench.py's CPU-baseline leg.  The product package never imports it.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

import numpy as np

from . import build as _build

_lib = None


class QMat(C.Structure):
    _fields_ = [("q", C.c_void_p), ("scale", C.c_void_p), ("bias", C.c_void_p), ("bits", C.c_int)]


def code_bits(qsb) -> int:
    """Bits per code of a packed matrix (q [E][N][K*bits/32], scale [E][N][K/64])."""
    words, groups = qsb[0].shape[-1], qsb[1].shape[-1]
    bits = 32 * words // (64 * groups)
    if bits not in (2, 3, 4) or 32 * words != bits * 64 * groups:
        raise ValueError("codes and group parameters disagree on K")
    return bits


class Experts(C.Structure):
    _fields_ = [("gate", QMat), ("up", QMat), ("down", QMat), ("n_experts", C.c_int)]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        L.oracle_bf16_to_double.restype = C.c_double
        L.oracle_bf16_to_double.argtypes = [C.c_uint16]
        L.oracle_double_to_bf16.restype = C.c_uint16
        L.oracle_double_to_bf16.argtypes = [C.c_double]
        L.oracle_dequant.restype = C.c_double
        L.oracle_dequant.argtypes = [C.POINTER(QMat), C.c_int, C.c_int, C.c_int, C.c_int, C.c_int]
        L.oracle_dequant_matrix.restype = None
        L.oracle_dequant_matrix.argtypes = [C.POINTER(QMat), C.c_int, C.c_int, C.c_int, C.c_void_p]
        L.oracle_router_logits.restype = None
        L.oracle_router_logits.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_void_p]
        L.oracle_topk_wide.restype = C.c_int
        L.oracle_topk_wide.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.oracle_topk.restype = C.c_int
        L.oracle_topk.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.oracle_route_layout.restype = C.c_int
        L.oracle_route_layout.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int] + [C.c_void_p] * 6
        L.oracle_expert_apply.restype = None
        L.oracle_expert_apply.argtypes = [C.c_void_p, C.c_int, C.c_int, C.POINTER(Experts), C.c_int, C.c_void_p]
        L.oracle_forward.restype = C.c_int
        L.oracle_forward.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int,
                                     C.POINTER(Experts), C.POINTER(Experts), C.c_int,
                                     C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class _Keep:
    """Keeps the numpy arrays behind a ctypes struct alive."""

    def __init__(self):
        self.arrays = []

    def qmat(self, qsb) -> QMat:
        q, s, b = (_c(qsb[0], np.uint32), _c(qsb[1], np.uint16), _c(qsb[2], np.uint16))
        self.arrays += [q, s, b]
        return QMat(_ptr(q), _ptr(s), _ptr(b), code_bits(qsb))

    def experts(self, ex: Optional[dict]) -> Optional[Experts]:
        if ex is None:
            return None
        E = ex["gate"][0].shape[0]
        return Experts(self.qmat(ex["gate"]), self.qmat(ex["up"]), self.qmat(ex["down"]), E)


def bf16_to_double(h: int) -> float:
    return lib().oracle_bf16_to_double(int(h))


def double_to_bf16(x: float) -> int:
    return int(lib().oracle_double_to_bf16(float(x)))


def dequant(qsb, e: int, n: int, k: int) -> float:
    keep = _Keep()
    m = keep.qmat(qsb)
    N, K = qsb[1].shape[1], qsb[1].shape[2] * 64
    return lib().oracle_dequant(C.byref(m), N, K, e, n, k)


def dequant_matrix(qsb, e: int) -> np.ndarray:
    keep = _Keep()
    m = keep.qmat(qsb)
    N, K = qsb[1].shape[1], qsb[1].shape[2] * 64
    out = np.empty((N, K), dtype=np.float64)
    lib().oracle_dequant_matrix(C.byref(m), N, K, e, _ptr(out))
    return out


def router_logits(X: np.ndarray, Wr: np.ndarray) -> np.ndarray:
    """fp64 logits [T][E] of bf16 X [T][d] (uint16 bit patterns) and bf16 Wr [E][d]."""
    X = _c(X, np.uint16)
    Wr = _c(Wr, np.uint16)
    T, d = X.shape
    E, d2 = Wr.shape
    if d != d2:
        raise ValueError("X and Wr disagree on d")
    out = np.empty((T, E), np.float64)
    lib().oracle_router_logits(_ptr(X), T, d, _ptr(Wr), E, _ptr(out))
    return out


def topk_wide(logits: np.ndarray, K: int):
    """values [T][K] fp32 and indices [T][K] int32 of each row's K largest entries (descending, lower index
    first among equal values)."""
    lg = _c(logits, np.float32)
    T, V = lg.shape
    vals = np.empty((T, K), np.float32)
    idx = np.empty((T, K), np.int32)
    if lib().oracle_topk_wide(_ptr(lg), T, V, K, _ptr(vals), _ptr(idx)) != 0:
        raise ValueError("oracle_topk_wide rejected its input")
    return vals, idx


def topk(logits: np.ndarray, k: int):
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    rc = lib().oracle_topk(_ptr(lg), T, E, k, _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError("oracle_topk rejected its input")
    return ids, w


def route_layout(ids: np.ndarray, E: int, block_rows: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    A = T * k
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(A, np.int32)
    inv = np.empty(A, np.int32)
    max_blocks = -(-A // block_rows) + E
    bmap = np.zeros((max_blocks, 3), np.int32)
    nb = np.zeros(1, np.int32)
    rc = lib().oracle_route_layout(_ptr(ids), T, E, k, block_rows, _ptr(counts), _ptr(offsets),
                                   _ptr(perm), _ptr(inv), _ptr(bmap), _ptr(nb))
    if rc != 0:
        raise ValueError("oracle_route_layout rejected its input")
    return dict(counts=counts, offsets=offsets, perm=perm, inv_perm=inv,
                block_map=bmap[: int(nb[0])].copy(), num_blocks=int(nb[0]))


def route(logits: np.ndarray, k: int, block_rows: int):
    ids, w = topk(logits, k)
    out = route_layout(ids, logits.shape[1], block_rows)
    out.update(ids=ids, w=w)
    return out


def expert_apply(x: np.ndarray, ex: dict, e: int) -> np.ndarray:
    keep = _Keep()
    xe = _c(x, np.uint16)
    exs = keep.experts(ex)
    d = xe.shape[0]
    I = ex["gate"][0].shape[1]
    y = np.empty(d, np.float64)
    lib().oracle_expert_apply(_ptr(xe), d, I, C.byref(exs), e, _ptr(y))
    return y


def forward(X: np.ndarray, routed: dict, shared: Optional[dict], ids: np.ndarray, w: np.ndarray,
            t_begin: int = 0, t_end: Optional[int] = None):
    """Returns (Y64 [n][d] float64, Y16 [n][d] uint16 bf16 bits) for tokens [t_begin, t_end)."""
    keep = _Keep()
    Xc = _c(X, np.uint16)
    T, d = Xc.shape
    t_end = T if t_end is None else t_end
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    k = ids.shape[1]
    I = routed["gate"][0].shape[1]
    r = keep.experts(routed)
    s = keep.experts(shared)
    I_sh = shared["gate"][0].shape[1] if shared is not None else 0
    n = t_end - t_begin
    Y64 = np.empty((n, d), np.float64)
    Y16 = np.empty((n, d), np.uint16)
    rc = lib().oracle_forward(_ptr(Xc), T, d, I, k, C.byref(r), C.byref(s) if s is not None else None, I_sh,
                              _ptr(ids), _ptr(w), t_begin, t_end, _ptr(Y64), _ptr(Y16))
    if rc != 0:
        raise ValueError("oracle_forward rejected its input")
    return Y64, Y16
