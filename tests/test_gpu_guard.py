"""Bounds evidence without a memory checker: every output of every entry point
is placed inside a larger device buffer whose head and tail (64 KiB each) hold
a position-dependent canary pattern.  After the call, every canary byte must
be unchanged, and the output itself must match the CPU oracle (so the writes
landed where they belong, not merely inside the buffer).

This covers the places where a kernel computes addresses it could get wrong:
the TMA-store clipping of ragged row and column edges, the masked plain stores,
the swapped (transposed) store of skinny problems, the stream-K partial slots
and the one-pass stash (library workspace, whose misuse would show up as
corrupted outputs), the vectorised and scalar paths of the bandwidth kernels.

The cross-entropy's optional gradient ("Allow reductions in matmul epilogues",
fusion example: the softmax-minus-onehot tensor is an optional second output)
is checked the other way round as well: with grad_or_null = NULL, a sentinel
[M, N] buffer -- including the very buffer a previous call wrote its gradient
to -- must stay byte-identical.
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
GUARD = 64 * 1024


def _pattern(n, salt):
    i = torch.arange(n, dtype=torch.int64, device=DEV)
    return ((i * 131 + 7 + salt) % 251 + 3).to(torch.uint8)


class Guarded:
    """A typed [shape] tensor at byte offset GUARD of a canary-filled buffer."""

    def __init__(self, shape, dtype, salt=0):
        self.numel = int(np.prod(shape))
        self.nbytes = self.numel * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.empty(GUARD + self.nbytes + GUARD, dtype=torch.uint8, device=DEV)
        self.want = _pattern(self.raw.numel(), salt)
        self.raw.copy_(self.want)
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)

    def check(self, what):
        torch.cuda.synchronize()
        head_bad = (self.raw[:GUARD] != self.want[:GUARD]).nonzero()
        tail_bad = (self.raw[GUARD + self.nbytes:] != self.want[GUARD + self.nbytes:]).nonzero()
        assert head_bad.numel() == 0, "%s: %d canary bytes before the output overwritten, first at -%d" % (
            what, head_bad.numel(), GUARD - int(head_bad[0]))
        assert tail_bad.numel() == 0, "%s: %d canary bytes after the output overwritten, first at +%d" % (
            what, tail_bad.numel(), int(tail_bad[0]))


def f64(t):
    return t.detach().float().cpu().double().numpy()


@pytest.fixture(scope="module", autouse=True)
def _device():
    lf.lib()
    torch.cuda.set_device(0)
    lf.check_device_error()
    yield
    lf.set_tuning(-1, -1)
    lf.set_onepass_tile(0)
    lf.check_device_error()


def _gemm_bound(got, ref, what):
    err = np.abs(got - ref).max()
    assert err <= 1e-2 * np.abs(ref).max(), "%s: max err %g" % (what, err)


# ------------------------------------------------------------------ gemm_nt

@pytest.mark.parametrize("variant,M,N,K", [
    (1, 200, 520, 264),       # single CTA, ragged M and N
    (2, 257, 1032, 136),      # CTA pairs, whole tiles, ragged edges in both
    (3, 300, 1288, 4104),     # CTA pairs, stream-K (partial slots), ragged
    (3, 768, 5120, 13824),    # the projection shape, stream-K as planned
    (4, 33, 1032, 264),       # swapped operands (transposed store), skinny X
    (4, 1, 4096, 4096),       # swapped, a single row
    (5, 1800, 20488, 72),     # CTA pairs, whole tiles claimed at run time, ragged
], ids=["cta1", "pair", "streamk", "streamk_projection", "swapped", "swapped_m1", "pair_claimed"])
def test_gemm_nt_writes_only_its_output(variant, M, N, K):
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    out = Guarded((M, N), torch.bfloat16, salt=variant)
    lf.set_tuning(-1, 2 if variant == 5 else variant)
    lf.set_tile_schedule(1 if variant == 5 else -1)
    try:
        lf.gemm_nt(x.to(DEV), w.to(DEV), out.t)
        lf.check_device_error()
    finally:
        lf.set_tuning(-1, -1)
        lf.set_tile_schedule(-1)
    out.check("gemm_nt variant %d %dx%dx%d" % (variant, M, N, K))
    rows = np.unique(np.array([0, M // 3, M // 2, M - 1]))
    _gemm_bound(f64(out.t)[rows], oracle.gemm_nt_rows(x, w, rows), "gemm_nt")


def test_gemm_nt_k1_writes_only_its_output():
    x = synthetic.bf16_normal((37, 1), 2.0, 0)
    w = synthetic.bf16_normal((264, 1), 0.5, 1)
    out = Guarded((37, 264), torch.bfloat16, salt=9)
    lf.gemm_nt(x.to(DEV), w.to(DEV), out.t)
    out.check("gemm_nt K=1")
    want = oracle.matmul_k1_bf16(x, w)
    assert np.array_equal(out.t.cpu().view(torch.int16).numpy().view(np.uint16), want)


# ------------------------------------------------------------- gemm_nt_xent

def _xent_guarded(x, w, lab, want_grad, what, rows=None):
    M, N = x.shape[0], w.shape[0]
    loss = Guarded((M,), torch.float32, salt=1)
    grad = Guarded((M, N), torch.bfloat16, salt=2) if want_grad else None
    lf.gemm_nt_xent(x.to(DEV), w.to(DEV), lab.to(DEV), loss=loss.t, grad=grad.t if grad else None)
    lf.check_device_error()
    loss.check(what + " loss")
    if grad:
        grad.check(what + " grad")
    rows = np.arange(M) if rows is None else rows
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows, want_grad=want_grad)
    rel = np.abs(f64(loss.t)[rows] - rloss) / np.abs(rloss)
    assert rel.max() <= 1e-3, "%s: loss rel err %g" % (what, rel.max())
    if grad:
        assert np.abs(f64(grad.t)[rows] - rgrad).max() <= 2e-3, what


@pytest.mark.parametrize("width", [128, 160, 192, 224, 256])
def test_xent_onepass_writes_only_its_outputs(width):
    M, N, K = 600, 1032, 264
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=21)
    lab[0], lab[M - 1] = 0, N - 1
    lf.set_onepass_tile(width)
    try:
        _xent_guarded(x, w, lab, True, "one-pass width %d" % width)
    finally:
        lf.set_onepass_tile(0)


@pytest.mark.parametrize("variant", [1, 2, 3], ids=["cta1", "pair", "pair_streamk"])
def test_xent_loss_only_writes_only_its_output(variant):
    M, N, K = 257, 2056, 136
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=22)
    lf.set_tuning(-1, variant)
    try:
        _xent_guarded(x, w, lab, False, "loss only variant %d" % variant)
    finally:
        lf.set_tuning(-1, -1)


@pytest.mark.parametrize("variant", [1, 2, 3], ids=["cta1", "pair", "pair_streamk"])
@pytest.mark.parametrize("want_grad", [True, False], ids=["grad", "loss"])
def test_xent_whole_row_writes_only_its_outputs(variant, want_grad):
    # N = 136 <= 256: the single-launch whole-row epilogue, ragged M and N
    M, N, K = 261, 136, 520
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=26)
    lf.set_tuning(-1, variant)
    try:
        _xent_guarded(x, w, lab, want_grad, "whole row variant %d" % variant)
    finally:
        lf.set_tuning(-1, -1)


@pytest.mark.parametrize("variant", [1, 2], ids=["cta1", "pair"])
def test_xent_two_pass_gradient_writes_only_its_outputs(variant):
    # N = 40992: too wide for one pass on the pairs (the single-CTA kernel is
    # always two-pass); the last 256-column tile is 32 wide
    M, N, K = 260, 40992, 136
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=23)
    lab[0], lab[1] = N - 1, 256 * 160
    lf.set_tuning(-1, variant)
    try:
        _xent_guarded(x, w, lab, True, "two-pass variant %d" % variant,
                      rows=np.array([0, 1, 100, 255, 256, 259]))
    finally:
        lf.set_tuning(-1, -1)


@pytest.mark.parametrize("x_mn,w_mn", [(True, False), (False, True), (True, True)])
def test_xent_layouts_write_only_their_outputs(x_mn, w_mn):
    M, N, K = 264, 1032, 200
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=24)
    xs = x.to(DEV).t().contiguous() if x_mn else x.to(DEV)
    ws = w.to(DEV).t().contiguous() if w_mn else w.to(DEV)
    loss = Guarded((M,), torch.float32, salt=3)
    grad = Guarded((M, N), torch.bfloat16, salt=4)
    lf.gemm_nt_xent(xs, ws, lab.to(DEV), loss=loss.t, grad=grad.t, x_mn=x_mn, w_mn=w_mn)
    lf.check_device_error()
    loss.check("xent layout loss")
    grad.check("xent layout grad")
    rows = np.array([0, 131, 263])
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    assert (np.abs(f64(loss.t)[rows] - rloss) / np.abs(rloss)).max() <= 1e-3
    assert np.abs(f64(grad.t)[rows] - rgrad).max() <= 2e-3


def _xent_c(x, w, lab, loss, grad_ptr):
    M, K = x.shape
    N = w.shape[0]
    return lf.lib().gemm_nt_xent(x.data_ptr(), w.data_ptr(), lab.data_ptr(), loss.data_ptr(), grad_ptr,
                                 M, N, K, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("variant", [1, 2, 3], ids=["cta1", "pair", "pair_streamk"])
def test_xent_null_grad_writes_nothing_of_size_mn(variant):
    """grad_or_null = NULL through the C ABI: a sentinel-filled [M, N] buffer,
    which a previous call with a gradient wrote to, stays byte-identical; the
    loss is still right."""
    M, N, K = 384, 4104, 264
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=25)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    grad = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    loss = torch.empty(M, dtype=torch.float32, device=DEV)
    lf.set_tuning(-1, variant)
    try:
        assert _xent_c(xd, wd, ld, loss, grad.data_ptr()) == 0     # writes grad
        lf.check_device_error()
        sentinel = _pattern(M * N * 2, 77)
        grad.view(torch.uint8).view(-1).copy_(sentinel)
        other = torch.empty(M * N * 2, dtype=torch.uint8, device=DEV)
        other.copy_(sentinel)
        loss.fill_(float("nan"))
        assert _xent_c(xd, wd, ld, loss, None) == 0                # loss only
        lf.check_device_error()
    finally:
        lf.set_tuning(-1, -1)
    assert torch.equal(grad.view(torch.uint8).view(-1), sentinel)
    assert torch.equal(other, sentinel)
    rows = np.array([0, 1, 200, M - 1])
    _, rloss, _, _ = oracle.xent_rows(x, w, lab.numpy(), rows, want_grad=False)
    assert (np.abs(f64(loss)[rows] - rloss) / np.abs(rloss)).max() <= 1e-3


# ------------------------------------------------- gemm_layout / gemm_batched

@pytest.mark.parametrize("x_mn,w_mn", [(False, True), (True, False), (True, True)])
def test_gemm_layout_writes_only_its_output(x_mn, w_mn):
    M, N, K = 264, 1288, 200
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    xs = x.to(DEV).t().contiguous() if x_mn else x.to(DEV)
    ws = w.to(DEV).t().contiguous() if w_mn else w.to(DEV)
    out = Guarded((M, N), torch.bfloat16, salt=5)
    lf.gemm_layout(xs, ws, x_mn=x_mn, w_mn=w_mn, out=out.t)
    lf.check_device_error()
    out.check("gemm_layout")
    rows = np.array([0, 100, 263])
    _gemm_bound(f64(out.t)[rows], oracle.gemm_nt_rows(x, w, rows), "gemm_layout")


def test_gemm_batched_writes_only_its_outputs():
    # 3 batches of 136 x 264 (ragged against the 256 x 256 tiles), out rows
    # padded to a pitch of 272, the gaps between rows and batches canaried too
    B, M, N, K, ldo = 3, 136, 264, 72, 272
    x = synthetic.bf16_normal((B, M, K), 1.0, 31)
    w = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 32)
    stride_o = M * ldo + 64
    out = Guarded((B * stride_o,), torch.bfloat16, salt=6)
    before = out.raw.clone()
    lf.gemm_batched(x.to(DEV), False, K, M * K, w.to(DEV), False, K, 0, out.t, ldo, stride_o, B, M, N, K)
    lf.check_device_error()
    out.check("gemm_batched")
    flat = out.t.cpu()
    raw_before = before[GUARD:GUARD + out.nbytes].view(torch.bfloat16).cpu()
    for b in range(B):
        ref = oracle.gemm_nt(x[b], w)
        blk = flat[b * stride_o: b * stride_o + M * ldo].view(M, ldo)
        _gemm_bound(f64(blk[:, :N]), ref, "batch %d" % b)
        # the pitch padding and the batch gap keep their canary bytes
        old = raw_before[b * stride_o: b * stride_o + M * ldo].view(M, ldo)
        assert torch.equal(blk[:, N:].view(torch.int16), old[:, N:].view(torch.int16)), "row padding written"
        gap = slice(b * stride_o + M * ldo, (b + 1) * stride_o)
        assert torch.equal(flat[gap].view(torch.int16), raw_before[gap].view(torch.int16)), "batch gap written"


# ------------------------------------------------------- bandwidth kernels

@pytest.mark.parametrize("M,N,offset", [(64, 4096, 0), (7, 13, 0), (3, 1000, 1)])
def test_matmul_k1_writes_only_its_output(M, N, offset):
    rng = np.random.default_rng(M * 7 + N)
    a = torch.from_numpy(rng.standard_normal(M).astype(np.float32))
    b = torch.from_numpy(rng.standard_normal(N).astype(np.float32))
    out = Guarded((M * N + offset,), torch.float32, salt=7)
    view = out.t[offset:].view(M, N)        # offset 1: unaligned output, scalar kernel
    before = out.t[:offset].clone()
    lf.matmul_k1(a.to(DEV).reshape(M, 1), b.to(DEV).reshape(1, N), view)
    out.check("matmul_k1")
    assert torch.equal(out.t[:offset], before)
    want = oracle.matmul_k1(a.numpy(), b.numpy())
    assert np.array_equal(view.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("H,S", [(64, 4096), (7, 33)])
def test_rope_writes_only_its_outputs(H, S):
    inv, pos = synthetic.rope_operands(H, S)
    cos = Guarded((S, 2 * H), torch.bfloat16, salt=8)
    sin = Guarded((S, 2 * H), torch.bfloat16, salt=9)
    lf.rope_cos_sin(inv.to(DEV), pos.to(DEV), cos_out=cos.t, sin_out=sin.t)
    cos.check("rope cos")
    sin.check("rope sin")
    rc, rs = oracle.rope_cos_sin(inv, pos.numpy())
    for got, ref in ((cos.t, rc), (sin.t, rs)):
        g = got.cpu().view(torch.int16).numpy().view(np.uint16).astype(np.int64)
        r = ref.astype(np.int64)
        go = np.where(g < 0x8000, g, -(g & 0x7FFF))
        ro = np.where(r < 0x8000, r, -(r & 0x7FFF))
        assert np.abs(go - ro).max() <= 1


@pytest.mark.parametrize("M,K", [(256, 4096), (100, 36)])
def test_fp8_cast_writes_only_its_outputs(M, K):
    xs = synthetic.bf16_normal((M, K), 1.0, 15)
    scale = torch.tensor([10.0], dtype=torch.float32, device=DEV)
    out = Guarded((M, K), torch.uint8, salt=10)
    out_t = Guarded((K, M), torch.uint8, salt=11)
    lf.fp8_cast_dual(xs.to(DEV), scale, out=out.t, out_t=out_t.t)
    out.check("fp8 out")
    out_t.check("fp8 out_t")
    rq, rq_t = oracle.fp8_cast_dual(xs, 10.0)
    assert np.array_equal(out.t.cpu().numpy(), rq)
    assert np.array_equal(out_t.t.cpu().numpy(), rq_t)
