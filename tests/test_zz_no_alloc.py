"""The allocation-free cross-entropy entry point, gemm_nt_xent_noalloc.

It exists for callers that cannot allocate device memory during a call --
code inside CUDA-graph capture, programs whose allocator owns the whole GPU,
latency-critical paths that cannot take a first-use cudaMalloc.  It keeps its
scratch in a fixed device array inside the library.  These tests call it
through the C ABI (ctypes, no binding) and check its outputs against the CPU
oracle and against the allocating entry point, gemm_nt_xent, within the
parity tolerances (loss relative error <= 1e-3, gradient absolute error
<= 2e-3), on two calls in a row with different shapes, so stale scratch from
the first call cannot leak into the second.  A stalled device wait (the
library's test hook) must turn every output NaN and leave the context usable.
The file sorts last so a failure here stops a run only after every other test
has run.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import layout_folding_gb300 as lf
import oracle
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
    x = synthetic.bf16_normal((M, K), 1.0, 10 + seed_shift)
    w = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 20 + seed_shift)
    lab = synthetic.labels_uniform(M, N, 30 + seed_shift)
    lab[0], lab[1] = 0, N - 1
    return x, w, lab


def test_noalloc_matches_oracle_on_two_calls_in_a_row():
    torch.cuda.set_device(0)
    fn = _noalloc()
    cases = [(384, 4104, 520), (200, 1000, 136)]
    for i, (M, N, K) in enumerate(cases):
        x, w, lab = _inputs(M, N, K, i)
        xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
        loss = torch.full((M,), float("nan"), dtype=torch.float32, device=DEV)
        grad = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        n0 = lf.launch_count()
        assert _call(fn, xd, wd, ld, loss, grad) == 0
        torch.cuda.synchronize()
        assert lf.launch_count() - n0 == 4      # partials, combine, gradient, poison check
        if i > 0:   # after the first call's one-time set-up nothing is allocated
            assert torch.cuda.mem_get_info()[0] == free_before
        _, rloss, _, rgrad = oracle.xent(x, w, lab.numpy())
        got_l = loss.double().cpu().numpy()
        got_g = grad.double().cpu().numpy()
        assert np.all(np.isfinite(got_l))
        assert np.max(np.abs(got_l - rloss) / np.abs(rloss)) <= 1e-3
        assert np.max(np.abs(got_g - rgrad)) <= 2e-3
        # and the allocating entry point agrees within the same tolerances
        ref_loss, ref_grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        rl = ref_loss.double().cpu().numpy()
        assert np.max(np.abs(got_l - rl) / np.abs(rl)) <= 1e-3
        assert np.max(np.abs(got_g - ref_grad.double().cpu().numpy())) <= 2e-3


def test_noalloc_loss_only_and_oversize_rejected():
    torch.cuda.set_device(0)
    fn = _noalloc()
    x, w, lab = _inputs(256, 2048, 256, 5)
    loss = torch.empty(256, dtype=torch.float32, device=DEV)
    assert _call(fn, x.to(DEV), w.to(DEV), lab.to(DEV), loss, None) == 0
    torch.cuda.synchronize()
    _, rloss, _, _ = oracle.xent(x, w, lab.numpy(), want_grad=False)
    assert np.max(np.abs(loss.double().cpu().numpy() - rloss) / np.abs(rloss)) <= 1e-3
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


def test_noalloc_stalled_wait_poisons_outputs_and_context_survives():
    """The test hook stalls the first operand stage of CTA 0; with a 200 ms
    limit the bounded wait gives up, every loss and every gradient element of
    the call comes back NaN, and the next call is correct again."""
    torch.cuda.set_device(0)
    fn = _noalloc()
    M, N, K = 256, 1024, 256
    x, w, lab = _inputs(M, N, K, 7)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    loss = torch.zeros(M, dtype=torch.float32, device=DEV)
    grad = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    lf.set_test_hooks(True, 200_000_000)
    try:
        assert _call(fn, xd, wd, ld, loss, grad) == 0
        torch.cuda.synchronize()
    finally:
        lf.set_test_hooks(False, 0)
    assert torch.isnan(loss).all()
    assert torch.isnan(grad.float()).all()
    assert _call(fn, xd, wd, ld, loss, grad) == 0
    torch.cuda.synchronize()
    _, rloss, _, rgrad = oracle.xent(x, w, lab.numpy())
    assert np.max(np.abs(loss.double().cpu().numpy() - rloss) / np.abs(rloss)) <= 1e-3
    assert np.max(np.abs(grad.double().cpu().numpy() - rgrad)) <= 2e-3
    lf.check_device_error()
