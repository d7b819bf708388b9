"""The allocation-free cross-entropy entry point, gemm_nt_xent_noalloc.

It exists for callers that cannot allocate device memory during a call --
code inside CUDA-graph capture, programs whose allocator owns the whole GPU,
latency-critical paths that cannot take a first-use cudaMalloc.  It keeps its
scratch in a fixed device array inside the library.  These tests call it
through the C ABI (ctypes, no binding) and check its outputs against the
allocating entry point, gemm_nt_xent, within the parity tolerances (loss
relative error <= 1e-3, gradient absolute error <= 2e-3), on two calls in a
row with different shapes, so stale scratch from the first call cannot leak
into the second.  The file sorts last so a failure here stops a run only
after every other test has run.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import layout_folding_gb300 as lf
from layout_folding_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _noalloc():
    fn = lf.lib().gemm_nt_xent_noalloc
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, x, w, lab, loss, grad):
    M, K = x.shape
    N = w.shape[0]
    return fn(x.data_ptr(), w.data_ptr(), lab.data_ptr(), loss.data_ptr(),
              grad.data_ptr() if grad is not None else None, M, N, K,
              torch.cuda.current_stream().cuda_stream)


def _inputs(M, N, K, seed_shift):
    x = synthetic.bf16_normal((M, K), 1.0, 10 + seed_shift).to(DEV)
    w = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 20 + seed_shift).to(DEV)
    lab = synthetic.labels_uniform(M, N, 30 + seed_shift)
    lab[0], lab[1] = 0, N - 1
    return x, w, lab.to(DEV)


def test_noalloc_matches_gemm_nt_xent_on_two_calls_in_a_row():
    torch.cuda.set_device(0)
    fn = _noalloc()
    cases = [(384, 4104, 520, True), (200, 1000, 136, True)]
    for i, (M, N, K, want_grad) in enumerate(cases):
        x, w, lab = _inputs(M, N, K, i)
        ref_loss, ref_grad = lf.gemm_nt_xent(x, w, lab, want_grad=want_grad)
        loss = torch.full((M,), float("nan"), dtype=torch.float32, device=DEV)
        grad = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV) if want_grad else None
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _call(fn, x, w, lab, loss, grad) == 0
        torch.cuda.synchronize()
        if i > 0:   # after the first call's one-time set-up nothing is allocated
            assert torch.cuda.mem_get_info()[0] == free_before
        rl, l = ref_loss.double().cpu().numpy(), loss.double().cpu().numpy()
        assert np.all(np.isfinite(l))
        assert np.max(np.abs(l - rl) / np.abs(rl)) <= 1e-3
        g, rg = grad.double().cpu().numpy(), ref_grad.double().cpu().numpy()
        assert np.max(np.abs(g - rg)) <= 2e-3


def test_noalloc_loss_only_and_oversize_rejected():
    torch.cuda.set_device(0)
    fn = _noalloc()
    x, w, lab = _inputs(256, 2048, 256, 5)
    ref_loss, _ = lf.gemm_nt_xent(x, w, lab)
    loss = torch.empty(256, dtype=torch.float32, device=DEV)
    assert _call(fn, x, w, lab, loss, None) == 0
    torch.cuda.synchronize()
    rl = ref_loss.double().cpu().numpy()
    assert np.max(np.abs(loss.double().cpu().numpy() - rl) / np.abs(rl)) <= 1e-3
    # scratch need 16384 * 1024 * 8 bytes > 32 MiB: rejected on the host with
    # LF_ERR_WORKSPACE (5) before anything is enqueued (buffers are real and
    # in bounds for K = 8 regardless)
    M, N, K = 16384, 262144, 8
    xb = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    wb = torch.zeros(N, K, dtype=torch.bfloat16, device=DEV)
    lb = torch.zeros(M, dtype=torch.int32, device=DEV)
    lo = torch.zeros(M, dtype=torch.float32, device=DEV)
    assert _call(fn, xb, wb, lb, lo, None) == 5
    lf.check_device_error()
