"""CPU oracle for the layout-folding hot path -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the bench's CPU-baseline
leg may import this package.  The CUDA library never loads it and shares no
code with it; the only thing both sides share is the seeded input generator,
which holds none of the method's arithmetic.

The arithmetic lives in ``oracle.c`` (plain loops, fp64); this module is the
ctypes marshalling around it.  Every function takes and returns numpy arrays;
bf16 data travels as ``uint16`` bit patterns.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, brute force, library cross-checks and invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2 -fopenmp, strict IEEE: no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        sig = {
            "oracle_gemm_nt": [P, P, I64, I64, I64, P],
            "oracle_gemm_nt_rows": [P, P, P, I64, I64, I64, P],
            "oracle_transpose_bf16": [P, I64, I64, P],
            "oracle_gemm_nn": [P, P, I64, I64, I64, P],
            "oracle_xent_logits": [P, P, I64, I64, P, P, P],
            "oracle_xent_bruteforce": [P, P, I64, I64, P],
            "oracle_xent_rows": [P, P, P, P, I64, I64, I64, P, P, P, P],
            "oracle_matmul_k1": [P, P, I64, I64, P],
            "oracle_matmul_k1_bf16": [P, P, I64, I64, P],
            "oracle_set_num_threads": [ctypes.c_int],
            "oracle_fp8_cast_dual": [P, I64, I64, ctypes.c_float, P, P],
            "oracle_rope_cos_sin": [P, P, I64, I64, P, P],
            "oracle_gemm_layout": [P, ctypes.c_int, P, ctypes.c_int, I64, I64, I64, P, I64, P],
            "oracle_gemm_batched": [P, ctypes.c_int, I64, I64, P, ctypes.c_int, I64, I64, I64, I64, I64, I64, P],
        }
        for name, argtypes in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_bf16_round.argtypes = [ctypes.c_float]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a) -> np.ndarray:
    """Accept a uint16 bf16-bit array (numpy) or a torch bf16 CPU tensor."""
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint16:
            raise TypeError("bf16 operands travel as uint16 bit patterns")
        return np.ascontiguousarray(a)
    import torch  # only for the tensor -> bits view
    if a.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def bf16_round(values) -> np.ndarray:
    """fp32 -> bf16 bits with round-to-nearest-even, element by element."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32).ravel()
    out = np.empty(v.shape, dtype=np.uint16)
    for i, f in enumerate(v):
        out[i] = lib.oracle_bf16_round(float(f))
    return out.reshape(np.shape(values))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm_nt(x, w) -> np.ndarray:
    """out[m,n] = sum_k x[m,k] w[n,k] in fp64; x [M,K], w [N,K] bf16."""
    x, w = _bits(x), _bits(w)
    M, K = x.shape
    N, K2 = w.shape
    assert K == K2
    out = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_nt(_p(x), _p(w), M, N, K, _p(out))
    return out


def gemm_nt_rows(x, w, rows) -> np.ndarray:
    """gemm_nt restricted to the listed rows of x: out [len(rows), N]."""
    x, w = _bits(x), _bits(w)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    M, K = x.shape
    N, K2 = w.shape
    assert K == K2 and (rows.size == 0 or (rows.min() >= 0 and rows.max() < M))
    out = np.empty((rows.size, N), dtype=np.float64)
    _load().oracle_gemm_nt_rows(_p(x), _p(w), _p(rows), rows.size, N, K, _p(out))
    return out


def transpose_bf16(w) -> np.ndarray:
    """wt[k,n] = w[n,k] (bf16 bits)."""
    w = _bits(w)
    N, K = w.shape
    wt = np.empty((K, N), dtype=np.uint16)
    _load().oracle_transpose_bf16(_p(w), N, K, _p(wt))
    return wt


def gemm_nn(x, wt) -> np.ndarray:
    """out[m,n] = sum_k x[m,k] wt[k,n] in fp64; wt [K,N] bf16."""
    x, wt = _bits(x), _bits(wt)
    M, K = x.shape
    K2, N = wt.shape
    assert K == K2
    out = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_nn(_p(x), _p(wt), M, N, K, _p(out))
    return out


def gemm_layout(x, x_mn: bool, w, w_mn: bool, rows=None) -> np.ndarray:
    """out[m,n] = sum_k X(m,k) W(n,k) in fp64 with X stored [M,K] (x_mn False)
    or [K,M] (x_mn True) and W stored [N,K] (w_mn False) or [K,N] (w_mn True);
    `rows` restricts the result to those rows m."""
    x, w = _bits(x), _bits(w)
    if x_mn:
        K, M = x.shape
    else:
        M, K = x.shape
    if w_mn:
        K2, N = w.shape
    else:
        N, K2 = w.shape
    assert K == K2
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = M if r is None else r.shape[0]
    out = np.empty((R, N), dtype=np.float64)
    _load().oracle_gemm_layout(_p(x), int(bool(x_mn)), _p(w), int(bool(w_mn)), M, N, K, _p(r),
                               0 if r is None else R, _p(out))
    return out


def gemm_batched(x, x_mn: bool, ldx: int, sx: int, w, w_mn: bool, ldw: int, sw: int,
                 batch: int, M: int, N: int, K: int) -> np.ndarray:
    """out[b, m, n] = sum_k X_b(m, k) W_b(n, k) in fp64 over flat bf16 storage:
    X_b(m, k) = x[b*sx + m*ldx + k] (x_mn False) or x[b*sx + k*ldx + m] (True),
    W_b(n, k) = w[b*sw + n*ldw + k] (w_mn False) or w[b*sw + k*ldw + n] (True)."""
    xb, wb = _bits(x).ravel(), _bits(w).ravel()
    need_x = (batch - 1) * sx + ((K - 1) * ldx + M if x_mn else (M - 1) * ldx + K)
    need_w = (batch - 1) * sw + ((K - 1) * ldw + N if w_mn else (N - 1) * ldw + K)
    assert xb.size >= need_x and wb.size >= need_w, "storage too small for the views"
    out = np.empty((batch, M, N), dtype=np.float64)
    _load().oracle_gemm_batched(_p(np.ascontiguousarray(xb)), int(bool(x_mn)), ldx, sx,
                                _p(np.ascontiguousarray(wb)), int(bool(w_mn)), ldw, sw, batch, M, N, K, _p(out))
    return out


def xent_logits(z, labels, want_grad: bool = True):
    """Cross-entropy of fp64 logits z [M,N]: returns (loss, lse, grad|None)."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    labels = np.ascontiguousarray(labels, dtype=np.int32)
    M, N = z.shape
    assert labels.shape == (M,)
    loss = np.empty(M, dtype=np.float64)
    lse = np.empty(M, dtype=np.float64)
    grad = np.empty((M, N), dtype=np.float64) if want_grad else None
    _load().oracle_xent_logits(_p(z), _p(labels), M, N, _p(loss), _p(lse), _p(grad))
    return loss, lse, grad


def xent_bruteforce(z, labels) -> np.ndarray:
    """-log(exp(z_L)/sum exp z) in long double, no max subtraction."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    labels = np.ascontiguousarray(labels, dtype=np.int32)
    M, N = z.shape
    loss = np.empty(M, dtype=np.float64)
    _load().oracle_xent_bruteforce(_p(z), _p(labels), M, N, _p(loss))
    return loss


def xent_rows(x, w, labels, rows, want_grad: bool = True):
    """GEMM + cross-entropy for the listed rows of x.

    Returns (z [R,N], loss [R], lse [R], grad [R,N] | None), all fp64.
    """
    x, w = _bits(x), _bits(w)
    labels = np.ascontiguousarray(labels, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    M, K = x.shape
    N, K2 = w.shape
    assert K == K2 and labels.shape == (M,)
    R = rows.size
    z = np.empty((R, N), dtype=np.float64)
    loss = np.empty(R, dtype=np.float64)
    lse = np.empty(R, dtype=np.float64)
    grad = np.empty((R, N), dtype=np.float64) if want_grad else None
    _load().oracle_xent_rows(_p(x), _p(w), _p(labels), _p(rows), R, N, K,
                             _p(z), _p(loss), _p(lse), _p(grad))
    return z, loss, lse, grad


def xent(x, w, labels, want_grad: bool = True):
    """GEMM + cross-entropy over every row (small shapes)."""
    M = _bits(x).shape[0]
    return xent_rows(x, w, labels, np.arange(M, dtype=np.int64), want_grad)


def matmul_k1(a, b) -> np.ndarray:
    """out[i,j] = a[i]*b[j], one fp32 multiply; a [M] or [M,1], b [N] or [1,N]."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32).ravel())
    b = np.ascontiguousarray(np.asarray(b, dtype=np.float32).ravel())
    M, N = a.size, b.size
    out = np.empty((M, N), dtype=np.float32)
    _load().oracle_matmul_k1(_p(a), _p(b), M, N, _p(out))
    return out


def matmul_k1_bf16(x, w) -> np.ndarray:
    """bf16 K=1 NT product: x [M,1], w [N,1] bits -> bf16 bits [M,N]."""
    x = _bits(x).ravel()
    w = _bits(w).ravel()
    M, N = x.size, w.size
    out = np.empty((M, N), dtype=np.uint16)
    _load().oracle_matmul_k1_bf16(_p(x), _p(w), M, N, _p(out))
    return out


def f32_to_e4m3(values) -> np.ndarray:
    """fp32 -> float8 E4M3 codes (round to nearest even), element by element."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32).ravel()
    out = np.empty(v.shape, dtype=np.uint8)
    for i, f in enumerate(v):
        out[i] = lib.oracle_f32_to_e4m3(float(f))
    return out.reshape(np.shape(values))


def fp8_cast_dual(x, scale: float):
    """(out [M,K], out_t [K,M]) E4M3 codes of clamp(x * scale, -448, 448)."""
    x = _bits(x)
    M, K = x.shape
    out = np.empty((M, K), dtype=np.uint8)
    out_t = np.empty((K, M), dtype=np.uint8)
    _load().oracle_fp8_cast_dual(_p(x), M, K, float(scale), _p(out), _p(out_t))
    return out, out_t


def rope_cos_sin(inv_freq, positions, with_sin: bool = True):
    """(cos [S, 2H], sin [S, 2H] | None) as bf16 bit patterns (uint16) of the
    RoPE segment: angle[s, c] = fp32(inv_freq[c mod H] * float(positions[s]))."""
    inv = _bits(inv_freq).ravel()
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64).ravel())
    H, S = inv.shape[0], pos.shape[0]
    cos_out = np.empty((S, 2 * H), dtype=np.uint16)
    sin_out = np.empty((S, 2 * H), dtype=np.uint16) if with_sin else None
    _load().oracle_rope_cos_sin(_p(inv), _p(pos), H, S, _p(cos_out), _p(sin_out))
    return cos_out, sin_out
