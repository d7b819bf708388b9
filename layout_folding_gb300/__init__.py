"""layout_folding_gb300 -- Python binding of liblayoutfold.so.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library (``include/layoutfold.h`` is the contract).  PyTorch is
used for device memory and the current stream.  There is no fallback: if the
library is missing or the device is not sm_103, the calls raise.

Entry points (same names as the C ABI):
  gemm_nt(x, w, out=None)                       -> out = x @ w.T   (bf16)
  gemm_nt_xent(x, w, labels, want_grad=False)   -> (loss fp32 [M], grad bf16 [M,N] | None)
  matmul_k1(a, b, out=None)                     -> out = a * b     (fp32, K=1)
  fp8_cast_dual(x, scale)                       -> (out e4m3 [M,K], out_t e4m3 [M,K] column-major)
  rope_cos_sin(inv_freq, positions)             -> (cos bf16 [S,2H], sin bf16 [S,2H])
  gemm_layout(x, w, x_mn, w_mn)                 -> out = X . W^T, X/W stored K-major or MN-major
  matmul(a, b)                                  -> a @ b for contiguous or transposed-view operands
  gemm_batched(...) / bmm(a, b)                 -> batched a @ b over strided views (pitches, batch strides)
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "liblayoutfold.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "layoutfold.h")

LF_OK = 0
STATUS_NAMES = {0: "LF_OK", 1: "LF_ERR_NULL", 2: "LF_ERR_SHAPE", 3: "LF_ERR_ALIGN", 4: "LF_ERR_LAUNCH",
                5: "LF_ERR_WORKSPACE", 6: "LF_ERR_DEVICE_TIMEOUT", 7: "LF_ERR_ARCH"}

_lock = threading.Lock()
_lib = None


class LayoutFoldError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        msg = lib().lf_status_string(status).decode() if _lib is not None else name
        super().__init__("%s: %s (%s)" % (where, name, msg))


def lib():
    """Load liblayoutfold.so (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("liblayoutfold.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.gemm_nt.argtypes = [P, P, P, I64, I64, I64, P]
        L.gemm_nt.restype = I32
        L.gemm_nt_xent.argtypes = [P, P, P, P, P, I64, I64, I64, P]
        L.gemm_nt_xent.restype = I32
        L.gemm_nt_xent_layout.argtypes = [P, I32, P, I32, P, P, P, I64, I64, I64, P]
        L.gemm_nt_xent_layout.restype = I32
        L.matmul_k1.argtypes = [P, P, P, I64, I64, P]
        L.matmul_k1.restype = I32
        L.fp8_cast_dual.argtypes = [P, P, P, P, I64, I64, P]
        L.fp8_cast_dual.restype = I32
        L.rope_cos_sin.argtypes = [P, P, P, P, I64, I64, P]
        L.rope_cos_sin.restype = I32
        L.gemm_layout.argtypes = [P, I32, P, I32, P, I64, I64, I64, P]
        L.gemm_layout.restype = I32
        L.gemm_batched.argtypes = [P, I32, I64, I64, P, I32, I64, I64, P, I64, I64, I64, I64, I64, I64, P]
        L.gemm_batched.restype = I32
        L.lf_status_string.argtypes = [I32]
        L.lf_status_string.restype = ctypes.c_char_p
        L.lf_check_device_error.argtypes = [P]
        L.lf_check_device_error.restype = I32
        L.lf_launch_count.argtypes = []
        L.lf_launch_count.restype = ctypes.c_uint64
        L.lf_last_gemm_plan.argtypes = [ctypes.POINTER(ctypes.c_int)] * 4
        L.lf_last_gemm_plan.restype = None
        L.lf_last_device_wait_code.argtypes = []
        L.lf_last_device_wait_code.restype = ctypes.c_int
        L.lf_device_query.argtypes = [P, P]
        L.lf_device_query.restype = I32
        L.lf_set_tuning.argtypes = [I32, I32]
        L.lf_set_tuning.restype = None
        L.lf_set_onepass_tile.argtypes = [I32]
        L.lf_set_onepass_tile.restype = None
        L.lf_set_test_hooks.argtypes = [I32, ctypes.c_uint64]
        L.lf_set_test_hooks.restype = None
        L.lf_set_xent_grad_path.argtypes = [I32]
        L.lf_set_xent_grad_path.restype = None
        L.lf_set_tile_band.argtypes = [I32]
        L.lf_set_tile_band.restype = None
        L.lf_set_tile_schedule.argtypes = [I32]
        L.lf_set_tile_schedule.restype = None
        L.lf_set_cooperative.argtypes = [I32]
        L.lf_set_cooperative.restype = None
        L.lf_test_occupy_sms.argtypes = [I32, ctypes.c_uint64, P]
        L.lf_test_occupy_sms.restype = I32
        L.gemm_nt_xent_noalloc.argtypes = [P, P, P, P, P, I64, I64, I64, P]
        L.gemm_nt_xent_noalloc.restype = I32
        _lib = L
        return L


def declared_functions(header: str = HEADER):
    """Names of the functions include/layoutfold.h declares."""
    with open(header) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)))


def _check(status: int, where: str):
    if status != LF_OK:
        raise LayoutFoldError(status, where)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _require(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def gemm_nt(x, w, out=None, stream=None):
    """out[..., n] = sum_k x[..., k] * w[n, k]; x bf16 [..., K], w bf16 [N, K]."""
    import torch
    _require(x, torch.bfloat16, "x")
    _require(w, torch.bfloat16, "w")
    K = x.shape[-1]
    N = w.shape[0]
    if w.dim() != 2 or w.shape[1] != K:
        raise ValueError("w must be [N, K] with K = x.shape[-1]")
    M = x.numel() // K if K else 0
    if out is None:
        out = torch.empty(*x.shape[:-1], N, dtype=torch.bfloat16, device=x.device)
    _require(out, torch.bfloat16, "out")
    if out.numel() != M * N:
        raise ValueError("out has the wrong size")
    _check(lib().gemm_nt(x.data_ptr(), w.data_ptr(), out.data_ptr(), M, N, K, _stream(stream)), "gemm_nt")
    return out


def gemm_nt_xent(x, w, labels, want_grad=False, loss=None, grad=None, stream=None, x_mn=False, w_mn=False):
    """Fused x @ w.T + row-wise cross-entropy.  Returns (loss fp32 [M], grad bf16 [M, N] or None).
    x is stored [M, K] (any leading dims flattened into M), or [K, M] with x_mn;
    w is stored [N, K], or [K, N] with w_mn -- read in place either way."""
    import torch
    _require(x, torch.bfloat16, "x")
    _require(w, torch.bfloat16, "w")
    _require(labels, torch.int32, "labels")
    if x_mn:
        if x.dim() != 2:
            raise ValueError("an [K, M] x must be 2-D")
        K, M = x.shape
    else:
        K = x.shape[-1]
        M = x.numel() // K
    if w.dim() != 2:
        raise ValueError("w must be 2-D")
    Kw, N = w.shape if w_mn else (w.shape[1], w.shape[0])
    if Kw != K:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, Kw))
    if labels.numel() != M:
        raise ValueError("labels must have M elements")
    if loss is None:
        loss = torch.empty(M, dtype=torch.float32, device=x.device)
    _require(loss, torch.float32, "loss")
    if want_grad and grad is None:
        grad = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    if grad is not None:
        _require(grad, torch.bfloat16, "grad")
        if grad.numel() != M * N:
            raise ValueError("grad must be [M, N]")
    gptr = grad.data_ptr() if grad is not None else None
    if x_mn or w_mn:
        _check(lib().gemm_nt_xent_layout(x.data_ptr(), LF_MN_MAJOR if x_mn else LF_K_MAJOR, w.data_ptr(),
                                         LF_MN_MAJOR if w_mn else LF_K_MAJOR, labels.data_ptr(), loss.data_ptr(),
                                         gptr, M, N, K, _stream(stream)), "gemm_nt_xent_layout")
    else:
        _check(lib().gemm_nt_xent(x.data_ptr(), w.data_ptr(), labels.data_ptr(), loss.data_ptr(), gptr, M, N, K,
                                  _stream(stream)), "gemm_nt_xent")
    return loss, grad


def matmul_k1(a, b, out=None, stream=None):
    """out[i, j] = a[i] * b[j]; a fp32 [M, 1], b fp32 [1, N] -> out fp32 [M, N]."""
    import torch
    _require(a, torch.float32, "a")
    _require(b, torch.float32, "b")
    M, N = a.numel(), b.numel()
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=a.device)
    _require(out, torch.float32, "out")
    if out.numel() != M * N:
        raise ValueError("out must be [M, N]")
    _check(lib().matmul_k1(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, _stream(stream)), "matmul_k1")
    return out


def fp8_cast_dual(x, scale, out=None, out_t=None, stream=None):
    """The float8 training cast in both layouts: x bf16 [M, K] (contiguous),
    scale fp32 one-element device tensor.  Returns (out, out_t), both
    float8_e4m3fn [M, K] holding clamp(x * scale, -448, 448) rounded to E4M3;
    out is row-major, out_t column-major (strides (1, M)).  Raw [M, K] / [K, M]
    uint8 buffers may be passed as out / out_t."""
    import torch
    _require(x, torch.bfloat16, "x")
    _require(scale, torch.float32, "scale")
    if x.dim() != 2 or scale.numel() != 1:
        raise ValueError("x must be 2-D and scale must hold one element")
    M, K = x.shape
    fp8 = torch.float8_e4m3fn
    if out is None:
        out = torch.empty(M, K, dtype=fp8, device=x.device)
    if out_t is None:
        out_t = torch.empty(K, M, dtype=fp8, device=x.device).t()
    for t, name in ((out, "out"), (out_t, "out_t")):
        if t.dtype not in (fp8, torch.uint8) or t.device != x.device or t.numel() != M * K:
            raise ValueError("%s must be a 1-byte tensor of M*K elements on x's device" % name)
    if tuple(out.shape) != (M, K) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, K] tensor")
    col_major = tuple(out_t.shape) == (M, K) and (M == 1 or out_t.stride() == (1, M))
    if not col_major and not (tuple(out_t.shape) == (K, M) and out_t.is_contiguous()):
        raise ValueError("out_t must be [M, K] column-major or a contiguous [K, M] tensor")
    _check(lib().fp8_cast_dual(x.data_ptr(), scale.data_ptr(), out.data_ptr(), out_t.data_ptr(), M, K,
                               _stream(stream)), "fp8_cast_dual")
    return out, out_t


def rope_cos_sin(inv_freq, positions, cos_out=None, sin_out=None, want_sin=True, stream=None):
    """The RoPE segment: inv_freq bf16 [H], positions int64 (any shape, S
    elements, contiguous).  Returns (cos, sin) bf16 [S, 2H] with
    cos[s, i] = cos[s, H + i] = bf16(cosf(fp32(inv_freq[i] * float(positions[s])))),
    sin likewise (None when want_sin is False and no sin_out is given)."""
    import torch
    _require(inv_freq, torch.bfloat16, "inv_freq")
    _require(positions, torch.int64, "positions")
    H, S = inv_freq.numel(), positions.numel()
    if cos_out is None:
        cos_out = torch.empty(S, 2 * H, dtype=torch.bfloat16, device=inv_freq.device)
    if sin_out is None and want_sin:
        sin_out = torch.empty(S, 2 * H, dtype=torch.bfloat16, device=inv_freq.device)
    for t, name in ((cos_out, "cos_out"), (sin_out, "sin_out")):
        if t is not None:
            _require(t, torch.bfloat16, name)
            if t.numel() != S * 2 * H:
                raise ValueError("%s must hold S * 2H elements" % name)
    _check(lib().rope_cos_sin(inv_freq.data_ptr(), positions.data_ptr(), cos_out.data_ptr(),
                              None if sin_out is None else sin_out.data_ptr(), H, S, _stream(stream)),
           "rope_cos_sin")
    return cos_out, sin_out


LF_K_MAJOR, LF_MN_MAJOR = 0, 1


def gemm_layout(x, w, x_mn=False, w_mn=False, out=None, stream=None):
    """out[m, n] = sum_k X[m, k] W[n, k] (bf16 out, fp32 accumulation) with
    x stored [M, K] (x_mn False) or [K, M] (x_mn True) and w stored [N, K]
    (w_mn False) or [K, N] (w_mn True); x and w contiguous bf16."""
    import torch
    _require(x, torch.bfloat16, "x")
    _require(w, torch.bfloat16, "w")
    if x.dim() != 2 or w.dim() != 2:
        raise ValueError("x and w must be 2-D")
    K, M = x.shape if x_mn else (x.shape[1], x.shape[0])
    Kw, N = w.shape if w_mn else (w.shape[1], w.shape[0])
    if K != Kw:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, Kw))
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _require(out, torch.bfloat16, "out")
    if out.numel() != M * N:
        raise ValueError("out must be [M, N]")
    _check(lib().gemm_layout(x.data_ptr(), LF_MN_MAJOR if x_mn else LF_K_MAJOR, w.data_ptr(),
                             LF_MN_MAJOR if w_mn else LF_K_MAJOR, out.data_ptr(), M, N, K, _stream(stream)),
           "gemm_layout")
    return out


def matmul(a, b, out=None, stream=None):
    """a @ b for 2-D bf16 a [M, K] and b [K, N], each either contiguous or the
    transpose of a contiguous tensor (a.t(), b.t() views): the transpose is
    folded into the GEMM's operand layout, never materialised."""
    def storage(t):
        if t.is_contiguous():
            return t, False
        if t.t().is_contiguous():
            return t.t(), True
        raise ValueError("operand must be contiguous or a transposed contiguous tensor")
    if a.dim() != 2 or b.dim() != 2:
        raise ValueError("a and b must be 2-D")
    xa, a_t = storage(a)      # a_t: a is a transposed view -> X stored [K, M]
    bb, b_t = storage(b)      # b_t: b is a transposed view of a [N, K] tensor -> W K-major
    return gemm_layout(xa, bb, x_mn=a_t, w_mn=not b_t, out=out, stream=stream)


def gemm_batched(x, x_mn, ldx, stride_x, w, w_mn, ldw, stride_w, out, ldo, stride_o, batch, M, N, K,
                 stream=None):
    """The raw batched entry point on bf16 CUDA tensors used as flat storage
    (element offsets; see gemm_batched in include/layoutfold.h)."""
    import torch
    for t, name in ((x, "x"), (w, "w"), (out, "out")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise TypeError("%s must be a bf16 CUDA tensor" % name)
    _check(lib().gemm_batched(x.data_ptr(), LF_MN_MAJOR if x_mn else LF_K_MAJOR, ldx, stride_x, w.data_ptr(),
                              LF_MN_MAJOR if w_mn else LF_K_MAJOR, ldw, stride_w, out.data_ptr(), ldo, stride_o,
                              batch, M, N, K, _stream(stream)), "gemm_batched")
    return out


def _strided_view(t, rows_are_k):
    """(mn_major, ld) of the last two dims of t: unit column stride -> rows of
    length t.shape[-1] with pitch stride(-2); unit row stride -> the transposed
    storage with pitch stride(-1).  `rows_are_k`: the view's rows index K (the
    [K, N] right operand), so a row-major view of it is the N-major W."""
    s_r, s_c = t.stride(-2), t.stride(-1)
    if s_c == 1:
        return (rows_are_k, s_r)
    if s_r == 1:
        return (not rows_are_k, s_c)
    raise ValueError("each matrix must have unit stride along one of its two dimensions")


def bmm(a, b, out=None, stream=None):
    """a @ b over batches of strided views: a [M, K] or [B, M, K], b [K, N] or
    [B, K, N] (a 2-D operand is shared by every batch), bf16, each matrix with a
    unit stride in one dimension (slices, transposes and batch strides are
    folded into the kernel's tensor maps, never copied).  Returns [B, M, N]
    (or [M, N] when both are 2-D)."""
    import torch
    if a.dim() not in (2, 3) or b.dim() not in (2, 3):
        raise ValueError("a and b must be 2-D or 3-D")
    M, K = a.shape[-2], a.shape[-1]
    K2, N = b.shape[-2], b.shape[-1]
    if K != K2:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    B = max(a.shape[0] if a.dim() == 3 else 1, b.shape[0] if b.dim() == 3 else 1)
    for t in (a, b):
        if t.dim() == 3 and t.shape[0] not in (1, B):
            raise ValueError("batch sizes differ")
    x_mn, ldx = _strided_view(a, rows_are_k=False)
    w_mn, ldw = _strided_view(b, rows_are_k=True)
    sx = a.stride(0) if a.dim() == 3 and a.shape[0] == B and B > 1 else 0
    sw = b.stride(0) if b.dim() == 3 and b.shape[0] == B and B > 1 else 0
    if out is None:
        out = torch.empty(B, M, N, dtype=torch.bfloat16, device=a.device)
    if out.dim() == 2:
        out3 = out.unsqueeze(0)
    else:
        out3 = out
    if tuple(out3.shape) != (B, M, N) or out3.stride(-1) != 1:
        raise ValueError("out must be [B, M, N] with unit column stride")
    gemm_batched(a, x_mn, ldx, sx, b, w_mn, ldw, sw, out3, out3.stride(-2), out3.stride(0) if B > 1 else 0,
                 B, M, N, K, stream=stream)
    return out3[0] if a.dim() == 2 and b.dim() == 2 and out.dim() == 3 else out


# which device-side wait gave up (lf_last_device_wait_code)
WAIT_CODES = {0x101: "operand ring slot never freed", 0x102: "operand stage never landed",
              0x103: "accumulator never released", 0x104: "accumulator never completed",
              0x105: "unwinding did not finish", 0x106: "stream-K partial never arrived",
              0x107: "own stream-K partial write incomplete", 0x108: "one-pass group member never published",
              0x109: "partial copy into shared memory never landed",
              0x10A: "claimed tile index never arrived"}


def last_device_wait_code() -> int:
    """Code of the wait behind the last device timeout reported (0: none)."""
    return int(lib().lf_last_device_wait_code())


def check_device_error(stream=None):
    """Synchronise the stream; raise LayoutFoldError if a device wait timed
    out (its message names the wait that gave up)."""
    status = lib().lf_check_device_error(_stream(stream))
    where = "lf_check_device_error"
    if status == 6:
        code = last_device_wait_code()
        where += " [wait 0x%x: %s]" % (code, WAIT_CODES.get(code, "unknown"))
    _check(status, where)


def launch_count() -> int:
    return int(lib().lf_launch_count())


def last_gemm_plan():
    """Schedule of the last tensor-core GEMM launch in this process: grid
    (CTAs), cta_pairs (bool), stream_k (bool) and tile_n."""
    v = [ctypes.c_int(0) for _ in range(4)]
    lib().lf_last_gemm_plan(*[ctypes.byref(x) for x in v])
    return {"grid": v[0].value, "cta_pairs": bool(v[1].value), "stream_k": bool(v[2].value), "tile_n": v[3].value}


def device_query():
    """(SM count, co-resident CTA pairs of the pair GEMM kernel) of the current device."""
    sms, pairs = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().lf_device_query(ctypes.byref(sms), ctypes.byref(pairs)), "lf_device_query")
    return sms.value, pairs.value


def set_tuning(l2_prefetch_kblocks: int = -1, gemm_variant: int = -1):
    """L2-prefetch distance in K blocks (-1 = default, off) and GEMM tile
    variant (1 = single CTA, 2 = CTA pair, 3 = CTA pair + stream-K, -1 =
    automatic)."""
    lib().lf_set_tuning(int(l2_prefetch_kblocks), int(gemm_variant))


def set_onepass_tile(width: int = 0):
    """N-tile width of the one-pass cross-entropy kernel (128..256, multiple
    of 32); 0 = automatic."""
    lib().lf_set_onepass_tile(int(width))


def set_xent_grad_path(path: int = 0):
    """Gradient form of the cross-entropy on CTA pairs: 1 = one pass, 2 = exp
    pass + rescale, 3 = recompute pass, 0 = automatic."""
    lib().lf_set_xent_grad_path(int(path))


def set_tile_band(m_blocks: int = -1):
    """Whole-tile band height in 256-row blocks (0 = one band, -1 = automatic)."""
    lib().lf_set_tile_band(int(m_blocks))


def set_tile_schedule(mode: int = -1):
    """Whole tiles on CTA pairs: 0 = fixed assignment, 1 = claimed at run time,
    -1 = automatic."""
    lib().lf_set_tile_schedule(int(mode))


def set_cooperative(enable: bool = True):
    """Launch the CTA-waiting kernels with (True) or without (False) the
    cooperative attribute -- False only for profilers that cannot replay it."""
    lib().lf_set_cooperative(1 if enable else 0)


def set_test_hooks(inject_stall: bool, wait_timeout_ns: int = 0):
    lib().lf_set_test_hooks(1 if inject_stall else 0, int(wait_timeout_ns))


def occupy_sms(ctas: int, duration_ns: int, stream=None):
    """Test hook: hold `ctas` SMs (200 KiB of shared memory each) for
    duration_ns on `stream`, standing in for another application's kernels."""
    _check(lib().lf_test_occupy_sms(int(ctas), int(duration_ns), _stream(stream)), "lf_test_occupy_sms")
