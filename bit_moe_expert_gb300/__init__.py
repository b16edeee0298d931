"""GB300-native 4-bit groupwise-affine mixture-of-experts layer (sm_103a).

Thin Python binding over the C ABI in include/moe.h.  The functions carry the C
names and only marshal arguments (torch tensors -> device pointers, the current
CUDA stream); every step of the layer runs in the CUDA library.  There is no
fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as C
import dataclasses
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libbitmoe.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_NONFINITE"}

# Every symbol the headers in include/ declare.
EXPORTED = ("moe_status_string", "moe_device_sm_count", "moe_prepack_bytes", "moe_prepack_codes",
            "moe_prepack_codes_bits", "moe_prepack_scales", "moe_dequant_experts",
            "moe_route_max_blocks", "moe_route_workspace_bytes", "moe_route", "moe_route_noalloc",
            "moe_route_noalloc_check_status",
            "moe_router_logits", "moe_route_x", "moe_layer_x", "moe_topk_wide",
            "moe_forward_workspace_bytes",
            "moe_forward", "moe_layer_workspace_bytes", "moe_layer", "moe_check_status", "moe_profile_enable", "moe_profile_kernel_count",
            "moe_profile_kernel_name", "moe_profile_read", "moe_profile_reset", "moe_debug_decode")


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


class _QMat(C.Structure):
    _fields_ = [("q", C.c_void_p), ("sb", C.c_void_p)]


class _Experts(C.Structure):
    _fields_ = [("gate", _QMat), ("up", _QMat), ("down", _QMat), ("n_experts", C.c_int), ("bits", C.c_int)]


class _Routing(C.Structure):
    _fields_ = [("ids", C.c_void_p), ("w", C.c_void_p), ("counts", C.c_void_p), ("offsets", C.c_void_p),
                ("perm", C.c_void_p), ("inv_perm", C.c_void_p), ("block_map", C.c_void_p),
                ("num_blocks", C.c_void_p), ("block_rows", C.c_int)]


_lib_handle = None


def lib(path: Optional[str] = None):
    """Loads the CUDA library (raises if it has not been built).  The environment
    variable BITMOE_LIB may name another build of it (for A/B comparisons)."""
    global _lib_handle
    if _lib_handle is None:
        p = path or os.environ.get("BITMOE_LIB") or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} (run __graft_entry__.build())")
        L = C.CDLL(p)
        L.moe_status_string.restype = C.c_char_p
        L.moe_status_string.argtypes = [C.c_int]
        L.moe_device_sm_count.restype = C.c_int
        L.moe_prepack_bytes.restype = C.c_size_t
        L.moe_prepack_bytes.argtypes = [C.c_int, C.c_int, C.c_int]
        L.moe_prepack_codes.restype = C.c_int
        L.moe_prepack_codes.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.moe_prepack_codes_bits.restype = C.c_int
        L.moe_prepack_codes_bits.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.moe_prepack_scales.restype = C.c_int
        L.moe_prepack_scales.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.moe_route_max_blocks.restype = C.c_int
        L.moe_route_max_blocks.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int]
        L.moe_route_workspace_bytes.restype = C.c_size_t
        L.moe_route_workspace_bytes.argtypes = [C.c_int, C.c_int, C.c_int]
        L.moe_route.restype = C.c_int
        L.moe_route.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.POINTER(_Routing),
                                C.c_void_p, C.c_size_t, C.c_void_p]
        L.moe_router_logits.restype = C.c_int
        L.moe_router_logits.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]
        L.moe_route_x.restype = C.c_int
        L.moe_route_x.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p,
                                  C.POINTER(_Routing), C.c_void_p, C.c_size_t, C.c_void_p]
        L.moe_topk_wide.restype = C.c_int
        L.moe_topk_wide.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]
        L.moe_dequant_experts.restype = C.c_int
        L.moe_dequant_experts.argtypes = [C.POINTER(_QMat), C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.moe_route_noalloc.restype = C.c_int
        L.moe_route_noalloc.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.POINTER(_Routing),
                                        C.c_void_p]
        L.moe_route_noalloc_check_status.restype = C.c_int
        L.moe_route_noalloc_check_status.argtypes = [C.c_void_p]
        L.moe_forward_workspace_bytes.restype = C.c_size_t
        L.moe_forward_workspace_bytes.argtypes = [C.c_int] * 6
        L.moe_forward.restype = C.c_int
        L.moe_forward.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.POINTER(_Experts),
                                  C.POINTER(_Experts), C.c_int, C.POINTER(_Routing), C.c_void_p, C.c_void_p,
                                  C.c_size_t, C.c_void_p]
        L.moe_layer_workspace_bytes.restype = C.c_size_t
        L.moe_layer_workspace_bytes.argtypes = [C.c_int] * 6
        L.moe_layer.restype = C.c_int
        L.moe_layer.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                C.POINTER(_Experts), C.POINTER(_Experts), C.c_int, C.POINTER(_Routing), C.c_void_p,
                                C.c_void_p, C.c_size_t, C.c_void_p]
        L.moe_layer_x.restype = C.c_int
        L.moe_layer_x.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                  C.POINTER(_Experts), C.POINTER(_Experts), C.c_int, C.c_void_p, C.POINTER(_Routing),
                                  C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]
        L.moe_check_status.restype = C.c_int
        L.moe_check_status.argtypes = [C.c_void_p, C.c_void_p]
        L.moe_profile_enable.restype = C.c_int
        L.moe_profile_enable.argtypes = [C.c_int]
        L.moe_profile_kernel_count.restype = C.c_int
        L.moe_profile_kernel_name.restype = C.c_char_p
        L.moe_profile_kernel_name.argtypes = [C.c_int]
        L.moe_profile_read.restype = C.c_int
        L.moe_profile_read.argtypes = [C.c_int, C.POINTER(C.c_double), C.POINTER(C.c_longlong)]
        L.moe_profile_reset.restype = None
        L.moe_debug_decode.restype = C.c_int
        L.moe_debug_decode.argtypes = [C.c_longlong, C.c_int]
        _lib_handle = L
    return _lib_handle


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def _stream(stream) -> int:
    if stream is not None:
        return stream.cuda_stream
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:  # the current stream's handle without building a Stream object (~0.2 against ~3 us)
        return raw(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


# ----------------------------------------------------------------------- data holders

@dataclasses.dataclass
class QMat:
    """One stacked packed matrix on the device: q int32 [E][K/64][N][2 bits] (group-major codes),
    sb int32 [E][K/64][N]."""
    q: "object"
    sb: "object"

    def _c(self) -> _QMat:
        # the C struct is built once and reused while q and sb are the same tensors (a call marshals
        # three matrices per expert set; rebuilding them cost several microseconds per call)
        c = self.__dict__.get("_cc")
        if c is None or c[0] is not self.q or c[1] is not self.sb:
            c = (self.q, self.sb, _QMat(_ptr(self.q), _ptr(self.sb)))
            self.__dict__["_cc"] = c
        return c[2]


@dataclasses.dataclass
class Experts:
    gate: QMat
    up: QMat
    down: QMat

    @property
    def n_experts(self) -> int:
        return int(self.gate.sb.shape[0])

    @property
    def I(self) -> int:
        return int(self.gate.sb.shape[2])

    @property
    def bits(self) -> int:
        """Bits per code: the prepacked rows hold 2 x bits words per group."""
        return int(self.gate.q.shape[3]) // 2

    def _c(self) -> _Experts:
        # rebuilt only when a matrix or one of its tensors was replaced (identity checks only)
        c = self.__dict__.get("_cc")
        g, u, dn = self.gate, self.up, self.down
        if (c is None or c[0] is not g or c[1] is not u or c[2] is not dn or c[3] is not g.q or c[4] is not g.sb
                or c[5] is not u.q or c[6] is not u.sb or c[7] is not dn.q or c[8] is not dn.sb):
            c = (g, u, dn, g.q, g.sb, u.q, u.sb, dn.q, dn.sb,
                 _Experts(g._c(), u._c(), dn._c(), self.n_experts, self.bits), self.I)
            self.__dict__["_cc"] = c
        return c[9]

    def _c_and_I(self):
        """The C struct and the intermediate width, from the same cache."""
        st = self._c()
        return st, self.__dict__["_cc"][10]


@dataclasses.dataclass
class Routing:
    """Device buffers written by moe_route."""
    ids: "object"
    w: "object"
    counts: "object"
    offsets: "object"
    perm: "object"
    inv_perm: "object"
    block_map: "object"
    num_blocks: "object"
    block_rows: int

    @staticmethod
    def empty(T: int, E: int, k: int, block_rows: int, device="cuda") -> "Routing":
        import torch
        i32 = dict(dtype=torch.int32, device=device)
        A = T * k
        mb = max(1, moe_route_max_blocks(T, E, k, block_rows))
        return Routing(ids=torch.empty((T, k), **i32), w=torch.empty((T, k), dtype=torch.float32, device=device),
                       counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
                       perm=torch.empty(max(A, 1), **i32), inv_perm=torch.empty(max(A, 1), **i32),
                       block_map=torch.empty((mb, 3), **i32), num_blocks=torch.zeros(1, **i32),
                       block_rows=block_rows)

    def _c(self) -> _Routing:
        c = self.__dict__.get("_cc")
        if (c is None or c[0] is not self.ids or c[1] is not self.w or c[2] is not self.counts
                or c[3] is not self.offsets or c[4] is not self.perm or c[5] is not self.inv_perm
                or c[6] is not self.block_map or c[7] is not self.num_blocks):
            bufs = (self.ids, self.w, self.counts, self.offsets, self.perm, self.inv_perm, self.block_map,
                    self.num_blocks)
            c = bufs + (_Routing(*(_ptr(b) for b in bufs), self.block_rows),)
            self.__dict__["_cc"] = c
        st = c[8]
        st.block_rows = self.block_rows
        return st


def workspace(nbytes: int, device="cuda"):
    """A zero-filled, 256-byte aligned device workspace."""
    import torch
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------- the C functions

def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def moe_device_sm_count() -> int:
    return int(lib().moe_device_sm_count())


def moe_prepack_bytes(E: int, N: int, K: int) -> int:
    return int(lib().moe_prepack_bytes(E, N, K))


def moe_prepack_codes(q, qp, stream=None, bits: int = 4) -> None:
    """q int32 [E][N][K*bits/32] (row-major codes) -> qp int32 [E][K/64][N][2 bits] (group-major)."""
    E, N, W = q.shape
    K = W * 32 // bits
    _check("moe_prepack_codes_bits", lib().moe_prepack_codes_bits(_ptr(q), E, N, K, bits, _ptr(qp), _stream(stream)))


def moe_prepack_scales(scale, bias, sb, stream=None) -> None:
    """scale, bias: int16/uint16-bit [E][N][K/64] device tensors; sb: int32 [E][K/64][N]."""
    E, N, G = scale.shape
    assert bias.shape == scale.shape and tuple(sb.shape) == (E, G, N)
    _check("moe_prepack_scales",
           lib().moe_prepack_scales(_ptr(scale), _ptr(bias), E, N, G * 64, _ptr(sb), _stream(stream)))


def moe_route_max_blocks(T: int, E: int, k: int, block_rows: int) -> int:
    return int(lib().moe_route_max_blocks(T, E, k, block_rows))


def moe_route_workspace_bytes(T: int, E: int, k: int) -> int:
    return int(lib().moe_route_workspace_bytes(T, E, k))


def moe_route(logits, k: int, block_rows: int, out: Routing, ws, stream=None) -> None:
    T, E = logits.shape
    r = out._c()
    _check("moe_route", lib().moe_route(_ptr(logits), T, E, k, block_rows, C.byref(r), _ptr(ws), ws.numel(),
                                        _stream(stream)))
    out.block_rows = r.block_rows


def moe_router_logits(X, W_r, logits, stream=None) -> None:
    """logits [T][E] fp32 = X [T][d] bf16 (int16 storage) times W_r [E][d] bf16, transposed."""
    T, d = X.shape
    E = W_r.shape[0]
    _check("moe_router_logits", lib().moe_router_logits(_ptr(X), T, d, _ptr(W_r), E, _ptr(logits), _stream(stream)))


def moe_route_x(X, W_r, k: int, block_rows: int, out: Routing, ws, logits, stream=None) -> None:
    """moe_router_logits into `logits`, then moe_route on them."""
    T, d = X.shape
    E = W_r.shape[0]
    r = out._c()
    _check("moe_route_x", lib().moe_route_x(_ptr(X), T, d, _ptr(W_r), E, k, block_rows, _ptr(logits), C.byref(r),
                                            _ptr(ws), ws.numel(), _stream(stream)))
    out.block_rows = r.block_rows


def moe_topk_wide(logits, K: int, values, indices, stream=None) -> None:
    """values [T][K] fp32 and indices [T][K] int32: each row's K largest entries of logits [T][V]."""
    T, V = logits.shape
    _check("moe_topk_wide", lib().moe_topk_wide(_ptr(logits), T, V, K, _ptr(values), _ptr(indices), _stream(stream)))


def moe_route_noalloc(logits, k: int, block_rows: int, out: Routing, stream=None) -> None:
    """moe_route without a workspace (for callers that cannot allocate device
    memory): uses the library's built-in scratch array; calls must not overlap
    on the GPU."""
    T, E = logits.shape
    r = out._c()
    _check("moe_route_noalloc", lib().moe_route_noalloc(_ptr(logits), T, E, k, block_rows, C.byref(r),
                                                        _stream(stream)))
    out.block_rows = r.block_rows


def moe_route_noalloc_check_status(stream=None) -> int:
    """Synchronises; the first device-side error recorded by moe_route_noalloc
    calls on the current device since the last check (0 if none), cleared."""
    return int(lib().moe_route_noalloc_check_status(_stream(stream)))


def moe_forward_workspace_bytes(T: int, d: int, I: int, E: int, k: int, I_shared: int) -> int:
    return int(lib().moe_forward_workspace_bytes(T, d, I, E, k, I_shared))


def moe_forward(X, routed: Experts, shared: Optional[Experts], routing: Routing, Y, ws, stream=None) -> None:
    T, d = X.shape
    k = int(routing.ids.shape[1])
    re = routed._c()
    se = shared._c() if shared is not None else None
    I_sh = shared.I if shared is not None else 0
    rr = routing._c()
    _check("moe_forward", lib().moe_forward(_ptr(X), T, d, routed.I, k, C.byref(re),
                                            C.byref(se) if se is not None else None, I_sh, C.byref(rr), _ptr(Y),
                                            _ptr(ws), ws.numel(), _stream(stream)))


def moe_layer_workspace_bytes(T: int, d: int, I: int, E: int, k: int, I_shared: int) -> int:
    return int(lib().moe_layer_workspace_bytes(T, d, I, E, k, I_shared))


def moe_layer(logits, X, routed: Experts, shared: Optional[Experts], k: int, block_rows: int, out: Routing, Y, ws,
              stream=None) -> None:
    """moe_route + moe_forward in one call (one launch on the decode path)."""
    T, d = X.shape
    re, I = routed._c_and_I()
    se, I_sh = shared._c_and_I() if shared is not None else (None, 0)
    r = out._c()
    _check("moe_layer", lib().moe_layer(_ptr(logits), _ptr(X), T, d, I, k, block_rows, C.byref(re),
                                        C.byref(se) if se is not None else None, I_sh, C.byref(r), _ptr(Y),
                                        _ptr(ws), ws.numel(), _stream(stream)))
    out.block_rows = r.block_rows


def moe_layer_x(X, W_r, routed: Experts, shared: Optional[Experts], k: int, block_rows: int, logits, out: Routing,
                Y, ws, stream=None) -> None:
    """moe_router_logits into `logits`, then moe_layer on them: the layer from the hidden state."""
    T, d = X.shape
    re = routed._c()
    se = shared._c() if shared is not None else None
    I_sh = shared.I if shared is not None else 0
    r = out._c()
    _check("moe_layer_x", lib().moe_layer_x(_ptr(X), T, d, _ptr(W_r), routed.I, k, block_rows, C.byref(re),
                                            C.byref(se) if se is not None else None, I_sh, _ptr(logits), C.byref(r),
                                            _ptr(Y), _ptr(ws), ws.numel(), _stream(stream)))
    out.block_rows = r.block_rows


def moe_check_status(ws, stream=None) -> int:
    return int(lib().moe_check_status(_ptr(ws), _stream(stream)))


def moe_profile_enable(on: bool) -> bool:
    return bool(lib().moe_profile_enable(1 if on else 0))


def moe_profile_reset() -> None:
    lib().moe_profile_reset()


def moe_debug_decode(wait_limit_cycles: int = 0, drop_cta: int = -1) -> None:
    """Test hook of the decode kernel: the limit of the wait at its barrier over
    the grid (cycles, 0 = default) and a CTA whose arrival there is skipped."""
    _check("moe_debug_decode", lib().moe_debug_decode(int(wait_limit_cycles), int(drop_cta)))


def moe_profile_read() -> dict:
    """{kernel name: (total device ms, launches)} for every kernel kind timed since the last reset."""
    L = lib()
    out = {}
    for i in range(L.moe_profile_kernel_count()):
        ms = C.c_double()
        n = C.c_longlong()
        _check("moe_profile_read", L.moe_profile_read(i, C.byref(ms), C.byref(n)))
        out[L.moe_profile_kernel_name(i).decode()] = (ms.value, n.value)
    return out


# ----------------------------------------------------------------------- weight preparation

def moe_dequant_experts(m: QMat, bits: int, W, stream=None) -> None:
    """W fp16 bits [E][N][K] (int16 tensor) = q * scale + bias of the prepacked matrix m."""
    E, G, N = m.sb.shape
    st = m._c()
    _check("moe_dequant_experts", lib().moe_dequant_experts(C.byref(st), int(E), int(N), int(G) * 64, int(bits),
                                                            _ptr(W), _stream(stream)))


def prepare_experts(ex: dict, device="cuda", stream=None) -> Experts:
    """Device copy of one expert set in the kernels' format.

    ex maps "gate", "up", "down" to (q, scale, bias): q uint32/int32 [E][N][K*bits/32]
    (4-, 3- or 2-bit codes, the width following from the shapes), scale and bias
    uint16/int16 bf16 bits [E][N][K/64], as NumPy arrays or torch tensors.  Codes and group parameters are reordered once with
    moe_prepack_codes and moe_prepack_scales (a one-time layout change, like
    loading a checkpoint).
    """
    import numpy as np
    import torch

    def dev(a, np_view, torch_dtype):
        if isinstance(a, np.ndarray):
            return torch.from_numpy(np.ascontiguousarray(a).view(np_view)).to(device)
        return a.to(device=device).view(torch_dtype).contiguous()

    mats = {}
    for name in ("gate", "up", "down"):
        q, s, b = ex[name]
        qd = dev(q, np.int32, torch.int32)
        sd = dev(s, np.int16, torch.int16)
        bd = dev(b, np.int16, torch.int16)
        E, N, G = sd.shape
        bits = 32 * int(qd.shape[2]) // (64 * G)
        if bits not in (2, 3, 4) or bits * 64 * G != 32 * int(qd.shape[2]):
            raise ValueError(f"{name}: codes [E][N][{qd.shape[2]}] do not match {G} groups of 4-, 3- or 2-bit codes")
        sb = torch.empty((E, G, N), dtype=torch.int32, device=device)
        moe_prepack_scales(sd, bd, sb, stream)
        qp = torch.empty((E, G, N, 2 * bits), dtype=torch.int32, device=device)
        moe_prepack_codes(qd, qp, stream, bits)
        del qd
        mats[name] = QMat(qp, sb)
    return Experts(**mats)
