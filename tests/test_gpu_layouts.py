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
# (192, 320, 136): rows multiples of 64 whose last 128-row slice is half inside the
# matrix, so one 64-row half of the 3-D view's box reads zeros past the edge
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (600, 1032, 264), (1240, 2056, 136), (128, 256, 64),
                                   (8, 512, 1024), (520, 264, 72), (192, 320, 136)])
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


@pytest.fixture
def grad_path(request):
    """Force one gradient form of the cross-entropy for the test."""
    lf.set_xent_grad_path(request.param)
    yield request.param
    lf.set_xent_grad_path(0)


# launches per call of each gradient form: one pass; exp pass + rescale;
# partials + combine + recompute pass
GRAD_LAUNCHES = {1: 1, 2: 2, 3: 3}


@pytest.mark.parametrize("grad_path", [1, 2], ids=["one_pass", "exp_rescale"], indirect=True)
@pytest.mark.parametrize("x_mn,w_mn", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(600, 1032, 264), (256, 2048, 128), (520, 776, 136)])
def test_xent_layouts_match_oracle(M, N, K, x_mn, w_mn, grad_path):
    """gemm_nt_xent with X stored [K,M] and/or W stored [K,N] (read in place),
    the gradient by the one-pass kernel or by the exp pass + rescale: loss
    (rel 1e-3) and gradient (abs 2e-3) of every row against the oracle on the
    logical operands, with labels on tile edges."""
    x = synthetic.bf16_normal((M, K), 1.0, 41)
    w = synthetic.bf16_normal((N, K), 1.0 / np.sqrt(K), 42)
    lab = synthetic.labels_uniform(M, N, seed=43)
    lab[0], lab[1], lab[2], lab[3] = 0, N - 1, min(255, N - 1), min(256, N - 1)
    xs, ws = stored(x, w, x_mn, w_mn)
    ld = lab.to(DEV)
    n0 = lf.launch_count()
    loss, grad = lf.gemm_nt_xent(xs, ws, ld, want_grad=True, x_mn=x_mn, w_mn=w_mn)
    n1 = lf.launch_count()
    loss_only, none = lf.gemm_nt_xent(xs, ws, ld, x_mn=x_mn, w_mn=w_mn)
    torch.cuda.synchronize()
    lf.check_device_error()
    assert none is None
    assert n1 - n0 == GRAD_LAUNCHES[grad_path]
    rows = list(range(M))
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    for got in (loss, loss_only):
        rel = np.abs(f64(got) - rloss) / np.abs(rloss)
        assert rel.max() <= 1e-3, rel.max()
    assert np.abs(f64(grad) - rgrad).max() <= 2e-3


def test_xent_layout_k_major_is_gemm_nt_xent():
    """Two K-major operands through the layout entry point are gemm_nt_xent
    itself (the same launches), bit for bit."""
    M, N, K = 512, 4096, 256
    x = synthetic.bf16_normal((M, K), 1.0, 44).to(DEV)
    w = synthetic.bf16_normal((N, K), 1.0 / 16, 45).to(DEV)
    lab = synthetic.labels_uniform(M, N, seed=46).to(DEV)
    na = lf.launch_count()
    loss_a, grad_a = lf.gemm_nt_xent(x, w, lab, want_grad=True)
    na = lf.launch_count() - na
    lib = lf.lib()
    loss_b = torch.empty_like(loss_a)
    grad_b = torch.empty_like(grad_a)
    n0 = lf.launch_count()
    assert lib.gemm_nt_xent_layout(x.data_ptr(), lf.LF_K_MAJOR, w.data_ptr(), lf.LF_K_MAJOR, lab.data_ptr(),
                                   loss_b.data_ptr(), grad_b.data_ptr(), M, N, K,
                                   torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert lf.launch_count() - n0 == na
    assert torch.equal(loss_a, loss_b) and torch.equal(grad_a, grad_b)


@pytest.mark.parametrize("grad_path", [1, 2], ids=["one_pass", "exp_rescale"], indirect=True)
def test_xent_layout_large_vocab_w_stored_kn_sampled(grad_path):
    """The LM-head shape with the weight stored [K, N] (as a tied embedding
    read transposed): 4096 x 32768 x 4096, sampled rows, every column."""
    M, N, K = 4096, 32768, 4096
    x = synthetic.bf16_normal((M, K), 1.0, 47)
    w = synthetic.bf16_normal((N, K), 1.0 / 64, 48)
    lab = synthetic.labels_uniform(M, N, seed=49)
    xs, ws = stored(x, w, False, True)
    loss, grad = lf.gemm_nt_xent(xs, ws, lab.to(DEV), want_grad=True, w_mn=True)
    torch.cuda.synchronize()
    lf.check_device_error()
    rows = [0, 1, 255, 256, 2047, 4095]
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    rel = np.abs(f64(loss)[rows] - rloss) / np.abs(rloss)
    assert rel.max() <= 1e-3, rel.max()
    assert np.abs(f64(grad)[rows] - rgrad).max() <= 2e-3


@pytest.mark.parametrize("grad_path", [2, 3], ids=["exp_rescale", "recompute"], indirect=True)
@pytest.mark.parametrize("x_mn,w_mn", LAYOUTS)
def test_xent_layouts_two_pass_wide_vocab(x_mn, w_mn, grad_path):
    """A vocabulary too wide for one pass (N = 40992) with the operands in
    other layouts: the exp pass + rescale, or partials, combine and the
    recompute pass, all reading the stored layouts; sampled rows, every
    column, against the oracle."""
    M, N, K = 256, 40992, 136
    x = synthetic.bf16_normal((M, K), 1.0, 50)
    w = synthetic.bf16_normal((N, K), 1.0 / np.sqrt(K), 51)
    lab = synthetic.labels_uniform(M, N, seed=52)
    lab[0], lab[1] = 0, N - 1
    xs, ws = stored(x, w, x_mn, w_mn)
    n0 = lf.launch_count()
    loss, grad = lf.gemm_nt_xent(xs, ws, lab.to(DEV), want_grad=True, x_mn=x_mn, w_mn=w_mn)
    torch.cuda.synchronize()
    lf.check_device_error()
    assert lf.launch_count() - n0 == GRAD_LAUNCHES[grad_path]
    rows = [0, 1, 127, 128, 255]
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    rel = np.abs(f64(loss)[rows] - rloss) / np.abs(rloss)
    assert rel.max() <= 1e-3, rel.max()
    assert np.abs(f64(grad)[rows] - rgrad).max() <= 2e-3


@pytest.mark.parametrize("grad_path", [1], ids=["one_pass"], indirect=True)
@pytest.mark.parametrize("x_mn,w_mn", LAYOUTS)
def test_xent_layouts_one_pass_multi_round(x_mn, w_mn, grad_path):
    """Several rounds of the one-pass kernel with MN-major operands (M = 1536:
    6 row blocks; N = 16384 at 256- or 224-wide tiles), every row."""
    M, N, K = 1536, 16384, 136
    x = synthetic.bf16_normal((M, K), 1.0, 53)
    w = synthetic.bf16_normal((N, K), 1.0 / np.sqrt(K), 54)
    lab = synthetic.labels_uniform(M, N, seed=55)
    xs, ws = stored(x, w, x_mn, w_mn)
    n0 = lf.launch_count()
    loss, grad = lf.gemm_nt_xent(xs, ws, lab.to(DEV), want_grad=True, x_mn=x_mn, w_mn=w_mn)
    torch.cuda.synchronize()
    lf.check_device_error()
    assert lf.launch_count() - n0 == 1
    rows = list(range(M))
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    rel = np.abs(f64(loss) - rloss) / np.abs(rloss)
    assert rel.max() <= 1e-3, rel.max()
    assert np.abs(f64(grad) - rgrad).max() <= 2e-3
