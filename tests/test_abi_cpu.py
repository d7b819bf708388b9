"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the public header declares, and rejects invalid arguments on
the host before any CUDA call is made."""
import ctypes
import os
import re
import subprocess

import pytest

import layout_folding_gb300 as lf
from layout_folding_gb300 import build as lfbuild

EXPECTED = {"gemm_nt", "gemm_nt_xent", "matmul_k1", "lf_status_string", "lf_check_device_error",
            "lf_launch_count", "lf_last_gemm_plan", "lf_last_device_wait_code", "lf_set_test_hooks", "lf_set_tuning", "lf_device_query", "gemm_nt_xent_noalloc",
            "fp8_cast_dual", "rope_cos_sin", "gemm_layout", "lf_set_onepass_tile", "gemm_batched",
            "gemm_nt_xent_layout"}


@pytest.fixture(scope="module")
def L():
    lfbuild.build()
    return lf.lib()


def test_header_declares_the_boundary():
    assert set(lf.declared_functions()) >= EXPECTED


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", lf.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in lf.declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_status_strings(L):
    for code in range(8):
        s = L.lf_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.lf_status_string(99).decode() == "unknown status"


A16 = 1 << 20  # a 16-byte aligned fake address: validation fails before it is used
P = ctypes.c_void_p


@pytest.mark.parametrize("args,want", [
    ((None, A16, A16, 64, 256, 128), 1),
    ((A16, None, A16, 64, 256, 128), 1),
    ((A16, A16, None, 64, 256, 128), 1),
    ((A16, A16, A16, 0, 256, 128), 2),
    ((A16, A16, A16, 64, -1, 128), 2),
    ((A16, A16, A16, 64, 256, 0), 2),
    ((A16, A16, A16, 1 << 31, 256, 128), 2),
    ((A16 + 2, A16, A16, 64, 256, 128), 3),
    ((A16, A16 + 8, A16, 64, 256, 128), 3),
    ((A16, A16, A16 + 4, 64, 256, 128), 3),
    ((A16, A16, A16, 64, 250, 128), 3),      # N % 8 != 0
    ((A16, A16, A16, 64, 256, 100), 3),      # K % 8 != 0
    ((A16, A16, A16, 64, 12, 1), 3),         # K = 1 still needs N % 8 == 0
])
def test_gemm_nt_rejects_on_host(L, args, want):
    assert L.gemm_nt(*[P(a) if a is not None else None for a in args[:3]], *args[3:], None) == want


@pytest.mark.parametrize("args,want", [
    ((None, A16, A16, A16, None, 64, 256, 128), 1),
    ((A16, A16, None, A16, None, 64, 256, 128), 1),
    ((A16, A16, A16, None, None, 64, 256, 128), 1),
    ((A16, A16, A16, A16, None, 64, 256, 1), 2),      # K = 1 has no cross-entropy path
    ((A16, A16, A16, A16, None, 0, 256, 128), 2),
    ((A16, A16, A16 + 2, A16, None, 64, 256, 128), 3),
    ((A16, A16, A16, A16, A16 + 8, 64, 256, 128), 3),
    ((A16, A16, A16, A16, None, 64, 256, 132), 3),
])
def test_gemm_nt_xent_rejects_on_host(L, args, want):
    ptrs = [P(a) if a is not None else None for a in args[:5]]
    assert L.gemm_nt_xent(*ptrs, *args[5:], None) == want


def test_fp8_cast_dual_rejects_on_host(L):
    L.fp8_cast_dual.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 2 + [ctypes.c_void_p]
    assert L.fp8_cast_dual(None, P(A16), P(A16), P(A16), 4, 4, None) == 1
    assert L.fp8_cast_dual(P(A16), None, P(A16), P(A16), 4, 4, None) == 1
    assert L.fp8_cast_dual(P(A16), P(A16), P(A16), None, 4, 4, None) == 1
    assert L.fp8_cast_dual(P(A16), P(A16), P(A16), P(A16), 0, 4, None) == 2
    assert L.fp8_cast_dual(P(A16), P(A16), P(A16), P(A16), 4, -1, None) == 2
    assert L.fp8_cast_dual(P(A16), P(A16), P(A16), P(A16), 1 << 31, 4, None) == 2
    assert L.fp8_cast_dual(P(A16 + 1), P(A16), P(A16), P(A16), 4, 4, None) == 3


def test_rope_cos_sin_rejects_on_host(L):
    L.rope_cos_sin.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 2 + [ctypes.c_void_p]
    assert L.rope_cos_sin(None, P(A16), P(A16), None, 64, 16, None) == 1
    assert L.rope_cos_sin(P(A16), None, P(A16), None, 64, 16, None) == 1
    assert L.rope_cos_sin(P(A16), P(A16), None, P(A16), 64, 16, None) == 1
    assert L.rope_cos_sin(P(A16), P(A16), P(A16), None, 0, 16, None) == 2
    assert L.rope_cos_sin(P(A16), P(A16), P(A16), None, 64, 0, None) == 2
    assert L.rope_cos_sin(P(A16), P(A16 + 4), P(A16), None, 64, 16, None) == 3
    assert L.rope_cos_sin(P(A16 + 1), P(A16), P(A16), None, 64, 16, None) == 3
    assert L.rope_cos_sin(P(A16), P(A16), P(A16), P(A16 + 1), 64, 16, None) == 3


def test_gemm_layout_rejects_on_host(L):
    L.gemm_layout.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P] + [ctypes.c_int64] * 3 + [P]
    assert L.gemm_layout(None, 0, P(A16), 0, P(A16), 8, 8, 8, None) == 1
    assert L.gemm_layout(P(A16), 2, P(A16), 0, P(A16), 8, 8, 8, None) == 2     # no such layout
    assert L.gemm_layout(P(A16), 0, P(A16), -1, P(A16), 8, 8, 8, None) == 2
    assert L.gemm_layout(P(A16), 1, P(A16), 0, P(A16), 12, 8, 8, None) == 3    # X [K,M] pitch M*2 not 16-aligned
    assert L.gemm_layout(P(A16), 0, P(A16), 1, P(A16), 8, 8, 12, None) == 3    # X [M,K] pitch K*2 not 16-aligned
    assert L.gemm_layout(P(A16), 1, P(A16), 1, P(A16), 8, 12, 8, None) == 3    # N % 8
    assert L.gemm_layout(P(A16 + 8), 1, P(A16), 1, P(A16), 8, 8, 8, None) == 3
    assert L.gemm_layout(P(A16), 1, P(A16), 1, P(A16), 0, 8, 8, None) == 2


def test_gemm_nt_xent_layout_rejects_on_host(L):
    L.gemm_nt_xent_layout.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, P, P] + [ctypes.c_int64] * 3 + [P]
    f = L.gemm_nt_xent_layout
    assert f(None, 0, P(A16), 0, P(A16), P(A16), None, 8, 8, 8, None) == 1
    assert f(P(A16), 0, P(A16), 0, P(A16), None, None, 8, 8, 8, None) == 1      # loss is required
    assert f(P(A16), 2, P(A16), 0, P(A16), P(A16), None, 8, 8, 8, None) == 2     # no such layout
    assert f(P(A16), 0, P(A16), 3, P(A16), P(A16), None, 8, 8, 8, None) == 2
    assert f(P(A16), 1, P(A16), 1, P(A16), P(A16), None, 8, 8, 1, None) == 2     # K = 1
    assert f(P(A16), 1, P(A16), 0, P(A16), P(A16), None, 12, 8, 8, None) == 3    # X [K,M] pitch M*2
    assert f(P(A16), 0, P(A16), 1, P(A16), P(A16), None, 8, 8, 12, None) == 3    # X [M,K] pitch K*2
    assert f(P(A16), 1, P(A16), 1, P(A16), P(A16), None, 8, 12, 8, None) == 3    # N % 8
    assert f(P(A16), 1, P(A16), 1, P(A16), P(A16), P(A16 + 8), 8, 8, 8, None) == 3  # grad alignment
    assert f(P(A16), 1, P(A16), 1, P(A16), P(A16), None, 0, 8, 8, None) == 2


def test_gemm_batched_rejects_on_host(L):
    I = ctypes.c_int64
    L.gemm_batched.argtypes = [P, ctypes.c_int, I, I, P, ctypes.c_int, I, I, P, I, I, I, I, I, I, P]
    ok = dict(x=P(A16), xl=0, ldx=64, sx=64 * 64, w=P(A16), wl=0, ldw=64, sw=64 * 64, o=P(A16), ldo=64, so=64 * 64,
              b=2, M=64, N=64, K=64)

    def call(**kw):
        a = dict(ok, **kw)
        return L.gemm_batched(a["x"], a["xl"], a["ldx"], a["sx"], a["w"], a["wl"], a["ldw"], a["sw"], a["o"],
                              a["ldo"], a["so"], a["b"], a["M"], a["N"], a["K"], None)
    assert call(x=None) == 1
    assert call(xl=2) == 2
    assert call(b=0) == 2
    assert call(ldx=32) == 2          # K-major X rows shorter than K
    assert call(ldo=56) == 2          # out rows shorter than N
    assert call(so=64) == 2           # overlapping out matrices
    assert call(ldx=72 + 4) == 3      # pitch not a multiple of 8 elements
    assert call(sx=64 * 64 + 4) == 3
    assert call(o=P(A16 + 8)) == 3


def test_matmul_k1_rejects_on_host(L):
    assert L.matmul_k1(None, P(A16), P(A16), 4, 4, None) == 1
    assert L.matmul_k1(P(A16), P(A16), P(A16), 0, 4, None) == 2
    assert L.matmul_k1(P(A16 + 1), P(A16), P(A16), 4, 4, None) == 3


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        lf.gemm_nt(x, x)


def test_last_gemm_plan_accepts_null_pointers(L):
    L.lf_last_gemm_plan(None, None, None, None)      # every output is optional
    g = ctypes.c_int(-1)
    L.lf_last_gemm_plan(ctypes.byref(g), None, None, None)
    assert g.value == 0                              # no GEMM has run in this process


def test_last_gemm_plan_is_empty_before_any_gemm(L):
    # no GEMM has run in this process: the record is all zero, and reading it
    # touches no device
    assert lf.last_gemm_plan() == {"grid": 0, "cta_pairs": False, "stream_k": False, "tile_n": 0}


def test_wait_codes_match_the_header(L):
    # the binding's table of wait codes is the header's, and nothing has timed out yet
    text = open(lf.HEADER).read()
    block = text[text.index("int lf_last_device_wait_code") - 1200:text.index("int lf_last_device_wait_code")]
    codes = {int(c, 16) for c in re.findall(r"\*\s+(0x1[0-9a-f]{2}) ", block)}
    assert codes == set(lf.WAIT_CODES)
    assert lf.last_device_wait_code() == 0
