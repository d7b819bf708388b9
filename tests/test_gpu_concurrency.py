"""Calls from several streams and host threads, and kernels whose CTAs wait on
each other while other work holds part of the GPU.

The library's per-device workspace (stream-K partial slots and flags, the
cross-entropy partials, the one-pass flags and stash) is shared by every call
on a device.  Calls on different streams are ordered on the GPU by an event
(no host synchronisation), so two streams issuing the same kinds of calls with
different inputs must each get their own, correct result.

The one-pass cross-entropy ("Allow reductions in matmul epilogues": reusing
the row reduction in the epilogue needs every CTA of a row of tiles resident
at once) and the stream-K split wait on other CTAs; they are launched
cooperatively.  A test kernel holds 40 SMs for 300 ms on another stream -- a
stand-in for another application's kernels -- while such a call is made with a
200 ms wait limit: the call must give the oracle's result or report a clean
device timeout, and the context must stay usable.
"""
import math
import threading

import numpy as np
import pytest
import torch

import layout_folding_gb300 as lf
import oracle
from layout_folding_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def f64(t):
    return t.detach().float().cpu().double().numpy()


@pytest.fixture(scope="module", autouse=True)
def _device():
    lf.lib()
    torch.cuda.set_device(0)
    lf.check_device_error()
    yield
    lf.set_test_hooks(False, 0)
    lf.set_tuning(-1, -1)
    torch.cuda.synchronize()
    lf.check_device_error()


def _gemm_rows_ok(out, x, w, rows, what):
    ref = oracle.gemm_nt_rows(x, w, rows)
    err = np.abs(f64(out)[rows] - ref).max()
    assert err <= 1e-2 * np.abs(ref).max(), "%s: max err %g" % (what, err)


def test_two_streams_gemm_nt_streamk_projection():
    """The projection shape runs stream-K (partial slots and epoch flags in the
    workspace); two streams, different inputs, three rounds back to back."""
    M, N, K = 768, 5120, 13824
    xa = synthetic.bf16_normal((M, K), 0.02, 100)
    xb = synthetic.bf16_normal((M, K), 0.02, 101)
    wa = synthetic.bf16_normal((N, K), 0.02, 102)
    wb = synthetic.bf16_normal((N, K), 0.02, 103)
    xad, xbd, wad, wbd = xa.to(DEV), xb.to(DEV), wa.to(DEV), wb.to(DEV)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(sa):
            oa = lf.gemm_nt(xad, wad)
        with torch.cuda.stream(sb):
            ob = lf.gemm_nt(xbd, wbd)
        assert lf.last_gemm_plan()["stream_k"]
        outs.append((oa, ob))
    torch.cuda.synchronize()
    lf.check_device_error()
    rows = np.array([0, 255, 256, 511, 512, 767])
    for oa, ob in outs:
        _gemm_rows_ok(oa, xa, wa, rows, "stream a")
        _gemm_rows_ok(ob, xb, wb, rows, "stream b")


def test_two_streams_xent_with_gradient():
    M, N, K = 1024, 8192, 256
    xa, wa = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    xb = synthetic.bf16_normal((M, K), 1.0, 200)
    wb = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 201)
    la = synthetic.labels_uniform(M, N, seed=202)
    lb = synthetic.labels_uniform(M, N, seed=203)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    args_a = (xa.to(DEV), wa.to(DEV), la.to(DEV))
    args_b = (xb.to(DEV), wb.to(DEV), lb.to(DEV))
    torch.cuda.synchronize()
    with torch.cuda.stream(sa):
        ra = lf.gemm_nt_xent(*args_a, want_grad=True)
    with torch.cuda.stream(sb):
        rb = lf.gemm_nt_xent(*args_b, want_grad=True)
    with torch.cuda.stream(sa):
        ra_loss_only = lf.gemm_nt_xent(*args_a, want_grad=False)
    torch.cuda.synchronize()
    lf.check_device_error()
    rows = np.array([0, 1, 255, 256, 700, 1023])
    for (x, w, lab), (loss, grad), what in (((xa, wa, la), ra, "a"), ((xb, wb, lb), rb, "b")):
        _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
        assert (np.abs(f64(loss)[rows] - rloss) / np.abs(rloss)).max() <= 1e-3, what
        assert np.abs(f64(grad)[rows] - rgrad).max() <= 2e-3, what
    _, rloss, _, _ = oracle.xent_rows(xa, wa, la.numpy(), rows, want_grad=False)
    assert (np.abs(f64(ra_loss_only[0])[rows] - rloss) / np.abs(rloss)).max() <= 1e-3


def test_two_host_threads_on_their_own_streams():
    """Host threads race to enqueue workspace-using calls; the ordering lock
    and the events keep each result intact."""
    M, N, K = 512, 4096, 264
    jobs = []
    for t in range(4):
        x = synthetic.bf16_normal((M, K), 1.0, 300 + t)
        w = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 310 + t)
        lab = synthetic.labels_uniform(M, N, seed=320 + t)
        jobs.append((x, w, lab))
    dev_in = [(x.to(DEV), w.to(DEV), lab.to(DEV)) for x, w, lab in jobs]
    results = [None] * len(jobs)
    errors = []

    def run(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                outs = []
                for _ in range(3):
                    outs.append(lf.gemm_nt_xent(*dev_in[i], want_grad=(i % 2 == 0)))
                s.synchronize()
            results[i] = outs
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(jobs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    lf.check_device_error()
    rows = np.array([0, 100, 255, 256, 511])
    for i, (x, w, lab) in enumerate(jobs):
        _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows, want_grad=(i % 2 == 0))
        for loss, grad in results[i]:
            assert (np.abs(f64(loss)[rows] - rloss) / np.abs(rloss)).max() <= 1e-3, i
            if grad is not None:
                assert np.abs(f64(grad)[rows] - rgrad).max() <= 2e-3, i


def _under_occupation(call, check):
    """Hold 40 SMs for 300 ms on another stream, then make `call` on the
    current stream with a 200 ms wait limit.  Returns "correct" or "timeout";
    anything else fails."""
    other = torch.cuda.Stream()
    torch.cuda.synchronize()
    lf.check_device_error()
    lf.set_test_hooks(False, 200_000_000)
    try:
        lf.occupy_sms(40, 300_000_000, stream=other)
        result = call()
        torch.cuda.synchronize()
        try:
            lf.check_device_error()
            outcome = "correct"
        except lf.LayoutFoldError as e:
            assert e.status == 6, e           # only a clean device timeout is acceptable
            outcome = "timeout"
    finally:
        lf.set_test_hooks(False, 0)
    if outcome == "correct":
        check(result)
    print("co-residency outcome:", outcome)
    return outcome


def test_onepass_while_other_kernels_hold_sms():
    M, N, K = 512, 32768, 256          # one-pass: 74 pairs busy, more than the 56 left free
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=41)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    rows = np.array([0, 255, 256, 511])

    def check(res):
        _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
        assert (np.abs(f64(res[0])[rows] - rloss) / np.abs(rloss)).max() <= 1e-3
        assert np.abs(f64(res[1])[rows] - rgrad).max() <= 2e-3

    lf.set_xent_grad_path(1)                          # the one-pass kernel (its pairs wait on each other)
    try:
        lf.gemm_nt_xent(xd, wd, ld, want_grad=True)   # set-up outside the occupied window
        n0 = lf.launch_count()
        _under_occupation(lambda: lf.gemm_nt_xent(xd, wd, ld, want_grad=True), check)
        # occupier + the one pass (or + the exp pass and rescale, had the
        # cooperative launch been refused)
        assert lf.launch_count() - n0 in (2, 3)
        loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)   # the context is usable
        lf.check_device_error()
    finally:
        lf.set_xent_grad_path(0)
    check((loss, grad))


def test_streamk_while_other_kernels_hold_sms():
    M, N, K = 768, 5120, 13824
    x, w = synthetic.make_gemm_inputs(M, N, K, 0.02, 0.02)
    xd, wd = x.to(DEV), w.to(DEV)
    lf.gemm_nt(xd, wd)
    rows = np.array([0, 300, 767])
    _under_occupation(lambda: lf.gemm_nt(xd, wd), lambda out: _gemm_rows_ok(out, x, w, rows, "stream-K"))
    out = lf.gemm_nt(xd, wd)
    lf.check_device_error()
    _gemm_rows_ok(out, x, w, rows, "after")
