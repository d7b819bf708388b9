"""GPU parity of the GEMM over batches of strided views (row pitches, batch
strides, a shared operand, any stored layout) against the oracle.

Tolerance as for gemm_nt: max|gpu - ref| <= 1e-2 * max|ref| per batch, plus
the element-wise diagnostic 2^-8 |ref| + 1e-3 max|ref|.
"""
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


def check_close(got, ref):
    for b in range(ref.shape[0]):
        err = np.abs(got[b] - ref[b])
        scale = np.abs(ref[b]).max()
        assert err.max() <= 1e-2 * scale, (b, err.max(), scale)
        assert np.all(err <= 2.0 ** -8 * np.abs(ref[b]) + 1e-3 * scale)


@pytest.mark.parametrize("x_mn,w_mn", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("B,M,N,K,pad", [(3, 200, 264, 136, 24), (2, 520, 1032, 72, 8), (1, 256, 256, 128, 64)])
def test_batched_padded_views_match_oracle(B, M, N, K, pad, x_mn, w_mn):
    rows_x, cols_x = (K, M) if x_mn else (M, K)
    rows_w, cols_w = (K, N) if w_mn else (N, K)
    ldx, ldw = cols_x + pad, cols_w + pad
    sx, sw = rows_x * ldx + 8 * pad, rows_w * ldw + 16     # batches not packed either
    x = synthetic.bf16_normal((B * sx,), 1.0, 51)
    w = synthetic.bf16_normal((B * sw,), 1.0 / np.sqrt(K), 52)
    ldo, so = N + 16, M * (N + 16) + 64
    out = torch.zeros(B * so, dtype=torch.bfloat16, device=DEV)
    lf.gemm_batched(x.to(DEV), x_mn, ldx, sx, w.to(DEV), w_mn, ldw, sw, out, ldo, so, B, M, N, K)
    torch.cuda.synchronize()
    ref = oracle.gemm_batched(x, x_mn, ldx, sx, w, w_mn, ldw, sw, B, M, N, K)
    o = out.cpu()
    got = np.stack([f64(o[b * so:b * so + M * ldo].view(M, ldo)[:, :N]) for b in range(B)])
    check_close(got, ref)
    # nothing written outside the out views
    mask = torch.ones(B * so, dtype=torch.bool)
    for b in range(B):
        mask[b * so:b * so + M * ldo].view(M, ldo)[:, :N] = False
    assert int(o[mask].view(torch.int16).count_nonzero()) == 0


def test_shared_operands_batch_stride_zero():
    B, M, N, K = 4, 256, 512, 192
    x = synthetic.bf16_normal((B * M * K,), 1.0, 53)
    w = synthetic.bf16_normal((N * K,), 0.1, 54)
    out = torch.empty(B * M * N, dtype=torch.bfloat16, device=DEV)
    lf.gemm_batched(x.to(DEV), False, K, M * K, w.to(DEV), False, K, 0, out, N, M * N, B, M, N, K)
    torch.cuda.synchronize()
    check_close(f64(out.view(B, M, N)), oracle.gemm_batched(x, False, K, M * K, w, False, K, 0, B, M, N, K))
    # one X, batched W
    wb = synthetic.bf16_normal((B * N * K,), 0.1, 55)
    lf.gemm_batched(x.to(DEV), False, K, 0, wb.to(DEV), False, K, N * K, out, N, M * N, B, M, N, K)
    torch.cuda.synchronize()
    check_close(f64(out.view(B, M, N)), oracle.gemm_batched(x, False, K, 0, wb, False, K, N * K, B, M, N, K))


@pytest.mark.parametrize("variant", [2, 3])
def test_batched_whole_tiles_and_streamk(variant):
    B, M, N, K = 3, 384, 512, 1536
    x = synthetic.bf16_normal((B, M, K), 1.0, 56)
    w = synthetic.bf16_normal((B, N, K), 1.0 / 40, 57)
    try:
        lf.set_tuning(gemm_variant=variant)
        out = lf.bmm(x.to(DEV), w.to(DEV).transpose(1, 2))
        torch.cuda.synchronize()
    finally:
        lf.set_tuning()
    lf.check_device_error()
    ref = oracle.gemm_batched(x, False, K, M * K, w, False, K, N * K, B, M, N, K)
    check_close(f64(out), ref)


def test_bmm_folds_slices_and_transposes():
    """Slices (padded rows), transposed views and a broadcast right operand,
    one launch each, against the oracle on the same storage."""
    B, M, N, K = 2, 304, 264, 200               # M % 8 == 0: the transposed left operand's pitch
    big = synthetic.bf16_normal((B, M, K + 56), 1.0, 58).to(DEV)
    a = big[:, :, 8:8 + K]                        # rows of 256 with an offset of 8 elements
    bt = synthetic.bf16_normal((N, K), 0.1, 59).to(DEV)
    for bb in (bt.t(), bt.t().contiguous()):      # W K-major (transposed view) or N-major
        n0 = lf.launch_count()
        out = lf.bmm(a, bb)
        torch.cuda.synchronize()
        assert lf.launch_count() - n0 == 1
        ref = np.stack([oracle.gemm_nt(a[i].contiguous().cpu(), bt.cpu()) for i in range(B)])
        check_close(f64(out), ref)
    # a transposed left operand
    at = synthetic.bf16_normal((B, K, M), 1.0, 60).to(DEV)
    out = lf.bmm(at.transpose(1, 2), bt.t())
    torch.cuda.synchronize()
    ref = np.stack([oracle.gemm_nt(at[i].t().contiguous().cpu(), bt.cpu()) for i in range(B)])
    check_close(f64(out), ref)


def test_headline_shape_as_four_batches():
    """The traced projection's FLOPs split into four batched N slices of the
    same W: sampled rows of every batch against the oracle."""
    M, N, K, B = 768, 5120, 13824, 4
    x = synthetic.bf16_normal((M, K), 0.02, 0)
    w = synthetic.bf16_normal((N, K), 0.02, 1)
    Nb = N // B
    out = torch.empty(B, M, Nb, dtype=torch.bfloat16, device=DEV)
    lf.gemm_batched(x.to(DEV), False, K, 0, w.to(DEV), False, K, Nb * K, out, Nb, M * Nb, B, M, Nb, K)
    torch.cuda.synchronize()
    rows = [0, 255, 256, 511, 767]
    for b in range(B):
        ref = oracle.gemm_nt_rows(x, w[b * Nb:(b + 1) * Nb].contiguous(), rows)
        check_close(f64(out[b][rows])[None], ref[None])
