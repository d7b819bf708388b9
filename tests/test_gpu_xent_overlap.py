"""The cross-entropy gradient's rescale overlapped with its exp pass.

With the exp pass and the rescale pass ("Allow reductions in matmul
epilogues": fp16 exp(z - tile max) parked in the gradient buffer, then each
row rescaled once its log-sum-exp is known) and the overlap switched on (an
option; the automatic choice leaves it off), the GEMM's whole tiles walk bands
of row blocks and its epilogue warps, between tiles, rescale the rows of every
band whose tiles are all finished (except the last band); the rescale kernel
then does only the units the GEMM did not take.  Both run one routine per
unit, so the results must be bit-identical with the overlap off, whatever the
band height, tile schedule or operand layout, and must match the oracle.  The
units the GEMM took are read back (lf_last_xent_overlap) to show that the
overlap ran.
"""
import math

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
    lf.set_xent_grad_path(2)
    yield
    lf.set_xent_grad_path(0)
    lf.set_xent_overlap(None)
    lf.set_tile_band(-1)
    lf.set_tile_schedule(-1)
    lf.set_tuning(-1, -1)
    lf.check_device_error()


def inputs(M, N, K, seed):
    x = synthetic.bf16_normal((M, K), 1.0, seed)
    w = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), seed + 1)
    lab = synthetic.labels_uniform(M, N, seed=seed + 2)
    # both ends of the row and tile edges; a label in a unit's last tile
    lab[:5] = torch.tensor([0, N - 1, 255, 256, min(8191, N - 1)], dtype=lab.dtype)
    return x, w, lab


def units_per_row(N):
    tiles = -(-N // 256)       # 256-column tiles of a row
    return -(-tiles // 32)     # a unit: 32 tiles of one row


def run(call, overlap):
    lf.set_xent_overlap(overlap)
    try:
        loss, grad = call()
        taken, total = lf.last_xent_overlap()
        lf.check_device_error()
    finally:
        lf.set_xent_overlap(None)
    return loss, grad, taken, total


def check_oracle(x, w, lab, loss, grad, rows, what):
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    rel = np.abs(f64(loss)[rows] - rloss) / np.abs(rloss)
    assert rel.max() <= 1e-3, "%s: loss rel err %g" % (what, rel.max())
    err = np.abs(f64(grad)[rows] - rgrad).max()
    assert err <= 2e-3, "%s: grad abs err %g" % (what, err)


# (M, N, K): two bands of 4 row blocks over ~7 waves of tiles; ragged rows
# (8 rows in the last block) and ragged columns (81 tiles: units of 32, 32
# and 17 tiles, the last tile 8 columns wide); a row block count that does not
# halve evenly (bands of 3 and 2)
@pytest.mark.parametrize("M,N,K", [(2048, 16384, 512), (1800, 20488, 256), (1280, 12288, 264)])
def test_overlap_matches_rescale_kernel_bitwise(M, N, K):
    x, w, lab = inputs(M, N, K, 300)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)

    def call():
        return lf.gemm_nt_xent(xd, wd, ld, want_grad=True)

    loss0, grad0, taken0, total0 = run(call, False)
    loss1, grad1, taken1, total1 = run(call, True)
    mb = (M + 255) // 256
    band = (mb + 1) // 2
    upr = units_per_row(N)
    assert total0 == total1 == M * upr
    assert taken0 == 0
    assert 0 < taken1 <= band * 256 * upr, (taken1, band * 256 * upr)
    assert torch.equal(loss0, loss1)
    assert torch.equal(grad0, grad1)
    rows = np.unique(np.array([0, 1, 2, 3, 4, 255, 256, band * 256 - 1, band * 256, M - 1]))
    check_oracle(x, w, lab, loss1, grad1, rows, "overlap %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("bands", [2, 1], ids=["four_bands", "eight_bands"])
def test_overlap_with_more_bands(bands):
    """Forced band heights: 4 or 8 bands, so several bands finish while the
    launch runs and their units are taken in order."""
    M, N, K = 2048, 16384, 264
    x, w, lab = inputs(M, N, K, 310)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    lf.set_tile_band(bands)
    try:
        ref = run(lambda: lf.gemm_nt_xent(xd, wd, ld, want_grad=True), False)
        got = run(lambda: lf.gemm_nt_xent(xd, wd, ld, want_grad=True), True)
    finally:
        lf.set_tile_band(-1)
    nb = 8 // bands
    assert 0 < got[2] <= (nb - 1) * bands * 256 * units_per_row(N)
    assert torch.equal(ref[0], got[0])
    assert torch.equal(ref[1], got[1])
    check_oracle(x, w, lab, got[0], got[1], np.array([0, 1, 511, 512, 1023, 1024, 2047]), "bands %d" % bands)


def test_overlap_one_band_is_off():
    """A band height of all row blocks (lf_set_tile_band(0)) leaves no finished
    band to overlap: the rescale kernel does every unit."""
    M, N, K = 1024, 8192, 136
    x, w, lab = inputs(M, N, K, 320)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    lf.set_tile_band(0)
    try:
        loss, grad, taken, total = run(lambda: lf.gemm_nt_xent(xd, wd, ld, want_grad=True), True)
    finally:
        lf.set_tile_band(-1)
    assert taken == 0 and total == M * units_per_row(N)
    check_oracle(x, w, lab, loss, grad, np.array([0, 1, 255, 256, M - 1]), "one band")


def test_overlap_with_claimed_tiles():
    M, N, K = 2048, 16384, 136
    x, w, lab = inputs(M, N, K, 330)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    lf.set_tuning(-1, 2)
    try:
        lf.set_tile_schedule(0)
        ref = run(lambda: lf.gemm_nt_xent(xd, wd, ld, want_grad=True), False)
        lf.set_tile_schedule(1)
        got = run(lambda: lf.gemm_nt_xent(xd, wd, ld, want_grad=True), True)
    finally:
        lf.set_tile_schedule(-1)
        lf.set_tuning(-1, -1)
    assert got[2] > 0
    assert torch.equal(ref[0], got[0])
    assert torch.equal(ref[1], got[1])


@pytest.mark.parametrize("x_mn,w_mn", [(False, True), (True, True)])
def test_overlap_operand_layouts(x_mn, w_mn):
    M, N, K = 1536, 16384, 264
    x, w, lab = inputs(M, N, K, 340)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    xa = xd.t().contiguous() if x_mn else xd
    wa = wd.t().contiguous() if w_mn else wd

    def call():
        return lf.gemm_nt_xent(xa, wa, ld, want_grad=True, x_mn=x_mn, w_mn=w_mn)

    ref = run(call, False)
    got = run(call, True)
    assert got[2] > 0
    assert torch.equal(ref[0], got[0])
    assert torch.equal(ref[1], got[1])
    check_oracle(x, w, lab, got[0], got[1], np.array([0, 1, 767, 768, M - 1]), "layout")


def test_overlap_back_to_back_and_interleaved():
    """The control words are left zero by each launch's last CTA: overlapped
    calls of different shapes, with the overlap switched off in between and a
    claimed-tile GEMM (which shares the word block) between them."""
    shapes = [(2048, 16384, 136), (1280, 12288, 72), (2048, 16384, 136)]
    ins = [inputs(M, N, K, 350 + 10 * i) for i, (M, N, K) in enumerate(shapes)]
    dev = [tuple(t.to(DEV) for t in v) for v in ins]
    gx, gw = synthetic.make_gemm_inputs(1024, 16384, 136, 1.0, 1.0 / math.sqrt(136))
    gxd, gwd = gx.to(DEV), gw.to(DEV)
    outs = []
    for rnd in range(2):
        for i, (xd, wd, ld) in enumerate(dev):
            lf.set_xent_overlap(not (rnd == 1 and i == 1))   # on, except once
            outs.append((i, lf.gemm_nt_xent(xd, wd, ld, want_grad=True)))
            lf.set_tuning(-1, 2)
            lf.set_tile_schedule(1)
            lf.gemm_nt(gxd, gwd)
            lf.set_tile_schedule(-1)
            lf.set_tuning(-1, -1)
    lf.set_xent_overlap(None)
    torch.cuda.synchronize()
    lf.check_device_error()
    for i, (loss, grad) in outs:
        x, w, lab = ins[i]
        M = x.shape[0]
        check_oracle(x, w, lab, loss, grad, np.array([0, 2, 255, 256, M // 2, M - 1]), "sequence %d" % i)
    for i in range(3):
        a = [o for j, o in outs if j == i]
        assert torch.equal(a[0][0], a[1][0]) and torch.equal(a[0][1], a[1][1])


def test_overlap_while_other_kernels_hold_sms():
    """No step of the overlap waits for another CTA: with a test kernel holding
    40 SMs for 300 ms, the CTAs that start late find their bands' units taken
    or left to the rescale kernel, and the result is the same, bit for bit."""
    M, N, K = 2048, 16384, 264
    x, w, lab = inputs(M, N, K, 360)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    ref = run(lambda: lf.gemm_nt_xent(xd, wd, ld, want_grad=True), False)
    other = torch.cuda.Stream()
    torch.cuda.synchronize()
    lf.set_xent_overlap(True)
    try:
        lf.occupy_sms(40, 300_000_000, stream=other)
        loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        torch.cuda.synchronize()
        lf.check_device_error()
    finally:
        lf.set_xent_overlap(None)
    assert torch.equal(ref[0], loss)
    assert torch.equal(ref[1], grad)


def test_overlap_in_graph_replays():
    """Captured into a CUDA graph (no per-launch flags: the control words reset
    themselves), replayed with new inputs: each replay's result equals the
    eager call's on the same inputs."""
    M, N, K = 2048, 16384, 136
    xb = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
    wb = torch.empty(N, K, dtype=torch.bfloat16, device=DEV)
    lb = torch.empty(M, dtype=torch.int32, device=DEV)
    loss = torch.empty(M, dtype=torch.float32, device=DEV)
    grad = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    x, w, lab = inputs(M, N, K, 370)
    xb.copy_(x)
    wb.copy_(w)
    lb.copy_(lab)
    lf.set_xent_overlap(True)
    try:
        lf.gemm_nt_xent(xb, wb, lb, want_grad=True, loss=loss, grad=grad)   # workspaces before capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                lf.gemm_nt_xent(xb, wb, lb, want_grad=True, loss=loss, grad=grad)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for seed in (380, 390, 400):
            x, w, lab = inputs(M, N, K, seed)
            xb.copy_(x)
            wb.copy_(w)
            lb.copy_(lab)
            graph.replay()
            torch.cuda.synchronize()
            lf.check_device_error()
            taken, _ = lf.last_xent_overlap()   # the replay's count (the eager call below makes its own)
            assert taken > 0, seed
            eager = lf.gemm_nt_xent(x.to(DEV), w.to(DEV), lab.to(DEV), want_grad=True)
            torch.cuda.synchronize()
            assert torch.equal(eager[0], loss), seed
            assert torch.equal(eager[1], grad), seed
            check_oracle(x, w, lab, loss, grad, np.array([0, 1, 1023, 1024, M - 1]), "replay %d" % seed)
    finally:
        lf.set_xent_overlap(None)
