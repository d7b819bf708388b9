"""GPU parity of the GEMM with either operand in either stored layout (the
transpose folded into the operand layout) against the oracle.

Tolerance as for gemm_nt: max|gpu - ref| <= 1e-2 * max|ref|, plus the
element-wise diagnostic (bf16 rounding 2^-8 |ref| + 1e-3 max|ref| for the fp32
summation order).  The MN-major variants run the same MMAs over the same K
order as the K-major one, so they are also compared with gemm_nt on the
transposed copies.
"""
import numpy as np
import pytest
import torch

import layout_folding_gb300 as lf
import oracle
from layout_folding_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LAYOUTS = [(True, False), (False, True), (True, True)]


def f64(t):
    return t.detach().float().cpu().double().numpy()


def check_close(got, ref):
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    assert err.max() <= 1e-2 * scale, (err.max(), scale)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-3 * scale)


def stored(x, w, x_mn, w_mn):
    """Device copies of X [M,K] and W [N,K] in the requested stored layouts."""
    xs = x.t().contiguous() if x_mn else x
    ws = w.t().contiguous() if w_mn else w
    return xs.to(DEV), ws.to(DEV)


@pytest.mark.parametrize("x_mn,w_mn", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (600, 1032, 264), (1240, 2056, 136), (128, 256, 64),
                                   (8, 512, 1024), (520, 264, 72)])
def test_layouts_match_oracle(M, N, K, x_mn, w_mn):
    x = synthetic.bf16_normal((M, K), 1.0, 31)
    w = synthetic.bf16_normal((N, K), 1.0 / np.sqrt(K), 32)
    xs, ws = stored(x, w, x_mn, w_mn)
    out = lf.gemm_layout(xs, ws, x_mn=x_mn, w_mn=w_mn)
    torch.cuda.synchronize()
    ref = oracle.gemm_layout(xs.cpu(), x_mn, ws.cpu(), w_mn)
    check_close(f64(out), ref)


@pytest.mark.parametrize("x_mn,w_mn", LAYOUTS)
def test_layouts_agree_with_gemm_nt(x_mn, w_mn):
    M, N, K = 768, 1024, 1000
    x = synthetic.bf16_normal((M, K), 1.0, 33)
    w = synthetic.bf16_normal((N, K), 1.0 / 32, 34)
    xs, ws = stored(x, w, x_mn, w_mn)
    out = lf.gemm_layout(xs, ws, x_mn=x_mn, w_mn=w_mn)
    nt = lf.gemm_nt(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    d = (out.float() - nt.float()).abs().max().item()
    assert d <= 1e-2 * nt.float().abs().max().item()


@pytest.mark.parametrize("variant", [2, 3])
def test_layouts_whole_tiles_and_streamk(variant):
    """Both pair schedules (whole tiles, stream-K) with W N-major."""
    M, N, K = 512, 768, 2048
    x = synthetic.bf16_normal((M, K), 1.0, 35)
    w = synthetic.bf16_normal((N, K), 1.0 / 45, 36)
    xs, ws = stored(x, w, False, True)
    try:
        lf.set_tuning(gemm_variant=variant)
        out = lf.gemm_layout(xs, ws, x_mn=False, w_mn=True)
        torch.cuda.synchronize()
    finally:
        lf.set_tuning()
    check_close(f64(out), oracle.gemm_layout(xs.cpu(), False, ws.cpu(), True))
    lf.check_device_error()


def test_headline_shape_with_the_traced_transposed_weight():
    """The traced program's shape (X [768, 13824], W [5120, 13824]) with W
    given as the [K, N] array the trace's transpose would have materialised:
    sampled rows against the oracle."""
    M, N, K = 768, 5120, 13824
    x = synthetic.bf16_normal((M, K), 0.02, 0)
    w = synthetic.bf16_normal((N, K), 0.02, 1)
    xs, ws = stored(x, w, False, True)
    out = lf.gemm_layout(xs, ws, x_mn=False, w_mn=True)
    torch.cuda.synchronize()
    rows = [0, 1, 127, 128, 255, 256, 383, 511, 640, 767]
    ref = oracle.gemm_layout(x, False, ws.cpu(), True, rows=rows)
    check_close(f64(out[rows]), ref)


def test_matmul_folds_transposed_views():
    M, N, K = 384, 520, 200
    a = synthetic.bf16_normal((M, K), 1.0, 37).to(DEV)
    b = synthetic.bf16_normal((K, N), 0.1, 38).to(DEV)
    ref = oracle.gemm_nn(a.cpu(), b.cpu())
    for aa in (a, a.t().contiguous().t()):
        for bb in (b, b.t().contiguous().t()):
            n0 = lf.launch_count()
            out = lf.matmul(aa, bb)
            torch.cuda.synchronize()
            assert lf.launch_count() - n0 == 1      # one kernel, no transpose copy
            check_close(f64(out), ref)


def test_k1_any_layout():
    M, N = 64, 4096
    a = synthetic.bf16_normal((M, 1), 1.0, 39)
    w = synthetic.bf16_normal((N, 1), 1.0, 40)
    out = lf.gemm_layout(a.reshape(1, M).to(DEV), w.reshape(1, N).to(DEV), x_mn=True, w_mn=True)
    torch.cuda.synchronize()
    ref = oracle.matmul_k1_bf16(a.reshape(M), w.reshape(N))
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), ref)


def test_invalid_layout_and_alignment_raise():
    x = torch.zeros(16, 12, dtype=torch.bfloat16, device=DEV)   # X stored [K=16, M=12]: pitch 24 B
    w = torch.zeros(16, 16, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(lf.LayoutFoldError):
        lf.gemm_layout(x, w, x_mn=True, w_mn=True)
