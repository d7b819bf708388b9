"""Failure detection without a GPU fault: a device-side wait that nothing
satisfies must run out after its limit, be reported through
lf_check_device_error as LF_ERR_DEVICE_TIMEOUT, and leave the CUDA context
usable.  The stall is made by the library's test hook (the first CTA never
arms its first stage, so its MMA wait can never complete); every other wait is
bounded too, so all CTAs unwind: copies in flight land, issued MMAs drain and
TMEM is freed before they exit.  No trap, no assert, no bad address."""
import math

import numpy as np
import pytest
import torch

import layout_folding_gb300 as lf
import oracle
from layout_folding_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("variant", [1, 2, 3, 5], ids=["cta1", "pair", "pair_streamk", "pair_claimed"])
def test_stalled_wait_times_out_and_context_survives(variant):
    # pair_claimed: whole tiles claimed at run time, enough tiles (256) that
    # the other pairs go on claiming while the stalled pair unwinds; the
    # launch's last CTA still resets the tile counter, so the next call is right
    torch.cuda.set_device(0)
    M, N, K = (1024, 16384, 512) if variant == 5 else (256, 1024, 512)
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    xd, wd = x.to(DEV), w.to(DEV)
    lf.check_device_error()                      # start from a clean error word
    lf.set_tuning(-1, 2 if variant == 5 else variant)
    lf.set_tile_schedule(1 if variant == 5 else -1)
    lf.set_test_hooks(True, 200_000_000)         # 200 ms limit per wait
    try:
        lf.gemm_nt(xd, wd)
        with pytest.raises(lf.LayoutFoldError) as info:
            lf.check_device_error()
        assert info.value.status == 6            # LF_ERR_DEVICE_TIMEOUT
        assert lf.last_device_wait_code() in lf.WAIT_CODES   # the wait that gave up is named
        assert "wait 0x" in str(info.value)
    finally:
        lf.set_test_hooks(False, 0)
    try:
        lf.check_device_error()                  # the word was cleared by the read
        out = lf.gemm_nt(xd, wd)
        lf.check_device_error()
    finally:
        lf.set_tuning(-1, -1)
        lf.set_tile_schedule(-1)
    ref = oracle.gemm_nt(x, w)
    got = out.float().cpu().double().numpy()
    assert np.abs(got - ref).max() <= 1e-2 * np.abs(ref).max()


@pytest.mark.parametrize("path", [1, 2], ids=["one_pass", "exp_rescale"])
def test_stalled_wait_in_cross_entropy_gradient_times_out(path):
    # the one-pass gradient kernel: a stalled pair also stalls its group's
    # flag waits; the exp pass: a stalled CTA; every wait is bounded, the
    # error is reported, the context lives, and the next call is right
    torch.cuda.set_device(0)
    lf.set_xent_grad_path(path)
    M, N, K = 512, 2048, 256
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    lf.check_device_error()
    lf.set_tuning(-1, 2)
    lf.set_test_hooks(True, 200_000_000)
    try:
        lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        with pytest.raises(lf.LayoutFoldError) as info:
            lf.check_device_error()
        assert info.value.status == 6
    finally:
        lf.set_test_hooks(False, 0)
    try:
        loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        lf.check_device_error()
    finally:
        lf.set_tuning(-1, -1)
        lf.set_xent_grad_path(0)
    _, rloss, _, rgrad = oracle.xent(x, w, lab.numpy())
    got = loss.double().cpu().numpy()
    assert np.max(np.abs(got - rloss) / np.abs(rloss)) <= 1e-3
    assert np.max(np.abs(grad.double().cpu().numpy() - rgrad)) <= 2e-3


@pytest.mark.parametrize("kind", ["layout_tt", "batched"])
def test_stalled_wait_times_out_in_layout_and_batched_variants(kind):
    # the MN-major operand and batched (3-D tensor map) variants of the pair
    # kernel share the bounded waits: same error, same clean unwind
    torch.cuda.set_device(0)
    M, N, K = 256, 1024, 512
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    xd, wd = x.to(DEV), w.to(DEV)
    xt, wt = xd.t().contiguous(), wd.t().contiguous()

    def call():
        if kind == "layout_tt":
            return lf.gemm_layout(xt, wt, x_mn=True, w_mn=True)
        return lf.bmm(xd.view(2, M // 2, K), wd.t())

    lf.check_device_error()
    lf.set_test_hooks(True, 200_000_000)
    try:
        call()
        with pytest.raises(lf.LayoutFoldError) as info:
            lf.check_device_error()
        assert info.value.status == 6
    finally:
        lf.set_test_hooks(False, 0)
    out = call()
    lf.check_device_error()
    ref = oracle.gemm_nt(x, w)
    got = out.reshape(M, N).float().cpu().double().numpy()
    assert np.abs(got - ref).max() <= 1e-2 * np.abs(ref).max()


@pytest.mark.parametrize("variant", [1, 2], ids=["cta1", "pair"])
def test_stalled_wait_in_whole_row_cross_entropy_times_out(variant):
    # N <= 256 (the single-launch whole-row epilogue): same bounded waits
    torch.cuda.set_device(0)
    M, N, K = 256, 256, 256
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    lf.check_device_error()
    lf.set_tuning(-1, variant)
    lf.set_test_hooks(True, 200_000_000)
    try:
        lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        with pytest.raises(lf.LayoutFoldError) as info:
            lf.check_device_error()
        assert info.value.status == 6
    finally:
        lf.set_test_hooks(False, 0)
    try:
        loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        lf.check_device_error()
    finally:
        lf.set_tuning(-1, -1)
    _, rloss, _, rgrad = oracle.xent(x, w, lab.numpy())
    assert np.max(np.abs(loss.double().cpu().numpy() - rloss) / np.abs(rloss)) <= 1e-3
    assert np.max(np.abs(grad.double().cpu().numpy() - rgrad)) <= 2e-3

