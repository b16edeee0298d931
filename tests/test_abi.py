"""The C-ABI library builds, loads without a GPU, exports every function that
include/moe.h declares, and rejects bad arguments on the host with the
documented status codes (no compute calls here)."""
import ctypes as C
import os
import re
import subprocess

import pytest

import bit_moe_expert_gb300 as bm
from bit_moe_expert_gb300 import build as bbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def L():
    bbuild.build()
    return bm.lib()


def declared_functions():
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_and_binding_agree():
    assert declared_functions() == sorted(bm.EXPORTED)


def test_every_declared_symbol_is_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", bbuild.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(moe_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(L, name)


def test_profile_surface_without_gpu(L):
    names = [L.moe_profile_kernel_name(i).decode() for i in range(L.moe_profile_kernel_count())]
    assert "decode" in names and "gemm_gateup" in names and "route" in names
    assert L.moe_profile_kernel_name(-1) is None
    assert L.moe_profile_enable(0) == 0
    assert L.moe_profile_read(-1, C.byref(C.c_double()), C.byref(C.c_longlong())) == INVALID


def test_status_strings(L):
    for code, name in bm.STATUS_NAMES.items():
        assert bm.moe_status_string(code) == name
    assert bm.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def test_size_queries(L):
    assert bm.moe_route_max_blocks(512, 256, 8, 128) == 32 + 256
    assert bm.moe_route_max_blocks(0, 16, 2, 16) == 16
    assert bm.moe_prepack_bytes(256, 512, 2048) == 256 * 32 * 512 * 4
    assert bm.moe_prepack_bytes(1, 64, 100) == 0
    assert bm.moe_route_workspace_bytes(16, 16, 2) % 256 == 0
    a = bm.moe_forward_workspace_bytes(512, 2048, 512, 256, 8, 512)
    assert a % 256 == 0 and a >= 512 * 9 * 2048 * 4
    assert bm.moe_forward_workspace_bytes(-1, 2048, 512, 256, 8, 0) == 0


def _routing(fake=0x100000):
    return bm._Routing(*([fake] * 8), 0)


def test_route_rejects_bad_arguments(L):
    fake = 0x100000
    r = _routing(fake)
    ws_ok = bm.moe_route_workspace_bytes(16, 16, 2)
    call = lambda T, E, k, BM, ws=fake, nb=ws_ok, logits=fake: L.moe_route(logits, T, E, k, BM, C.byref(r), ws, nb, None)
    assert call(16, 0, 2, 16) == INVALID
    assert call(-1, 16, 2, 16) == INVALID
    assert call(16, 16, 0, 16) == INVALID
    assert call(16, 2000, 2, 16) == UNSUPPORTED
    assert call(16, 16, 17, 16) == UNSUPPORTED
    assert call(16, 64, 33, 16) == UNSUPPORTED
    assert call(16, 16, 2, 0) == UNSUPPORTED
    assert call(16, 16, 2, 129) == UNSUPPORTED
    assert call(16, 16, 2, 16, ws=0) == WORKSPACE
    assert call(16, 16, 2, 16, ws=fake + 16) == WORKSPACE          # not 256-byte aligned
    assert call(16, 16, 2, 16, nb=ws_ok - 1) == WORKSPACE
    assert call(16, 16, 2, 16, logits=0) == INVALID
    r0 = bm._Routing(*([fake] * 7), 0, 0)                          # num_blocks missing
    assert L.moe_route(fake, 16, 16, 2, 16, C.byref(r0), fake, ws_ok, None) == INVALID
    r1 = bm._Routing(0, *([fake] * 7), 0)                          # ids missing with T > 0
    assert L.moe_route(fake, 16, 16, 2, 16, C.byref(r1), fake, ws_ok, None) == INVALID


def test_forward_rejects_bad_arguments(L):
    fake = 0x100000
    q = bm._QMat(fake, fake)
    ex = bm._Experts(q, q, q, 16)
    sh = bm._Experts(q, q, q, 1)
    r = _routing(fake)
    need = bm.moe_forward_workspace_bytes(0, 256, 128, 16, 2, 128)

    def call(T=0, d=256, I=128, k=2, ex=ex, sh=sh, I_sh=128, ws=fake, nb=None, X=fake):
        nb = need if nb is None else nb
        return L.moe_forward(X, T, d, I, k, C.byref(ex), C.byref(sh) if sh is not None else None, I_sh,
                             C.byref(r), fake, ws, nb, None)

    assert call() == OK                      # T = 0 is a no-op
    assert call(d=100) == INVALID            # d not a multiple of 64
    assert call(I=96) == INVALID
    assert call(I_sh=0) == INVALID           # shared given but I_shared = 0
    assert call(sh=None) == INVALID          # I_shared > 0 without a shared expert
    assert call(sh=None, I_sh=0) == OK
    assert call(k=0) == INVALID
    assert call(k=17) == UNSUPPORTED         # k > E
    assert call(ex=bm._Experts(q, q, bm._QMat(fake, 0), 16)) == INVALID
    assert call(ex=bm._Experts(q, q, bm._QMat(fake + 4, fake), 16)) == INVALID   # misaligned
    assert call(ex=bm._Experts(q, q, q, 2000)) == UNSUPPORTED
    assert call(sh=bm._Experts(q, q, q, 2)) == INVALID
    assert call(ws=0) == WORKSPACE
    assert call(nb=need - 1) == WORKSPACE


def test_prepack_rejects_bad_arguments(L):
    fake = 0x100000
    assert L.moe_prepack_scales(fake, fake, 1, 64, 100, fake, None) == INVALID
    assert L.moe_prepack_scales(0, fake, 1, 64, 128, fake, None) == INVALID
    assert L.moe_prepack_scales(fake, fake, 0, 64, 128, fake, None) == INVALID
