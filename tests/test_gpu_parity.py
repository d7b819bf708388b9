"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, on the
same seeded inputs.

Tolerances (stated for the path): GEMM max|gpu - ref| <= 1e-2 * max|ref|
(plus a stricter element-wise diagnostic: the bf16 rounding bound 2^-8|ref|
plus 1e-3 * max|ref| for fp32 summation order); per-row loss relative error
<= 1e-3; gradient absolute error <= 2e-3; the K=1 path bit-exact.
Full-size workloads are checked on sampled rows (every column of each sampled
row), small ones in full.
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
_cache = {}


def workload(name):
    if name not in _cache:
        _cache[name] = synthetic.make_workload(name)
    return _cache[name]


def f64(t):
    return t.detach().float().cpu().double().numpy()


def sample_rows(M, k=24, seed=0, extra=()):
    rng = np.random.default_rng(seed)
    base = {0, M - 1, min(127, M - 1), min(128, M - 1), M // 2}
    base.update(int(r) for r in rng.integers(0, M, size=k))
    base.update(r for r in extra if 0 <= r < M)
    return np.array(sorted(base), dtype=np.int64)


def assert_gemm_close(got, ref, what=""):
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    assert err.max() <= 1e-2 * scale, "%s: max err %g vs bound %g" % (what, err.max(), 1e-2 * scale)
    bad = err > (2.0 ** -8) * np.abs(ref) + 1e-3 * scale
    assert not bad.any(), "%s: %d elements outside the element-wise bound, first at %s" % (
        what, bad.sum(), np.argwhere(bad)[0])


def assert_loss_close(got, ref, what=""):
    rel = np.abs(got - ref) / np.abs(ref)
    assert rel.max() <= 1e-3, "%s: loss rel err %g at row %d" % (what, rel.max(), rel.argmax())


def assert_grad_close(got, ref, what=""):
    err = np.abs(got - ref)
    assert err.max() <= 2e-3, "%s: grad abs err %g at %s" % (what, err.max(), np.unravel_index(err.argmax(), err.shape))


@pytest.fixture(scope="module", autouse=True)
def _device():
    lf.lib()
    torch.cuda.set_device(0)
    yield
    lf.check_device_error()


@pytest.fixture(params=[1, 2, 3], ids=["cta1", "pair", "pair_streamk"])
def variant(request):
    """Run the test on the single-CTA (128x256) kernel, the CTA-pair (256x256,
    cta_group::2) kernel by whole tiles, and the CTA-pair kernel with the K
    iterations split evenly over all pairs (stream-K)."""
    lf.set_tuning(-1, request.param)
    yield request.param
    lf.check_device_error()
    lf.set_tuning(-1, -1)


# -------------------------------------------------------------- gemm_nt

def test_gemm_nt_tiny_full(variant):
    inp = workload("tiny")
    x, w = inp["x"], inp["w"]
    out = lf.gemm_nt(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    assert out.shape == (64, 256) and out.dtype == torch.bfloat16
    assert_gemm_close(f64(out), oracle.gemm_nt(x, w), "tiny")


@pytest.mark.parametrize("M,N,K", [(200, 520, 200), (130, 264, 72), (1, 8, 8), (257, 1032, 4104)])
def test_gemm_nt_ragged_full(M, N, K, variant):
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    out = lf.gemm_nt(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    assert_gemm_close(f64(out), oracle.gemm_nt(x, w), "ragged %dx%dx%d" % (M, N, K))


def test_gemm_nt_persistent_many_tiles(variant):
    # more tiles than SMs: every CTA runs several tiles through both TMEM buffers
    M, N, K = 1280, 8192, 512
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    out = lf.gemm_nt(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    rows = sample_rows(M, k=40, seed=3)
    assert_gemm_close(f64(out)[rows], oracle.gemm_nt_rows(x, w, rows), "persistent")


def test_gemm_nt_onehot_rows_select_weight_columns_exactly(variant):
    M, N, K = 256, 512, 256
    w = synthetic.bf16_normal((N, K), 1.0, 5)
    ks = (np.arange(M) * 37 + 11) % K
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    x[torch.arange(M), torch.from_numpy(ks)] = 1.0
    out = lf.gemm_nt(x.to(DEV), w.to(DEV)).cpu()
    want = w.t()[torch.from_numpy(ks)]            # row m = column ks[m] of W^T = W[:, ks[m]]
    assert torch.equal(out.view(torch.int16), want.contiguous().view(torch.int16))


def test_gemm_nt_projection_full_size(variant):
    wl = synthetic.WORKLOADS["nt_projection"]
    inp = workload("nt_projection")
    x, w = inp["x"], inp["w"]
    assert tuple(x.shape) == (384, 2, 13824)
    out = lf.gemm_nt(x.to(DEV), w.to(DEV))       # [384,2,13824] viewed as [768,13824]
    torch.cuda.synchronize()
    assert tuple(out.shape) == (384, 2, 5120)
    rows = sample_rows(wl.M, k=20, seed=1, extra=(255, 256, 511, 512, 640))
    ref = oracle.gemm_nt_rows(x.reshape(wl.M, wl.K), w, rows)
    assert_gemm_close(f64(out.reshape(wl.M, wl.N))[rows], ref, "nt_projection")


@pytest.mark.parametrize("M,N,K", [(768, 5120, 512), (640, 6000, 136), (700, 4984, 4104)])
def test_gemm_nt_automatic_schedule_full(M, N, K):
    """The planner's own choice (whole tiles or stream-K, by the K blocks the
    split saves against its fixed cost) on shapes with fewer 256x256 tiles
    than CTA pairs: every element against the oracle."""
    lf.set_tuning(-1, -1)
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    out = lf.gemm_nt(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    lf.check_device_error()
    assert_gemm_close(f64(out), oracle.gemm_nt(x, w), "auto %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K,stream_k", [(768, 5120, 13824, True), (768, 5120, 4096, False),
                                             (512, 8192, 4096, False), (640, 6000, 4096, False)])
def test_gemm_nt_automatic_schedule_choice(M, N, K, stream_k):
    """The planner splits K over the CTA pairs only where that saves each
    pair more than ~32 K blocks: the projection shape (216 -> 172.8 K blocks
    per pair) is split, the K = 4096 shapes (64 -> 51..61) run whole tiles."""
    lf.set_tuning(-1, -1)
    pairs = lf.device_query()[1]
    x, w = synthetic.make_gemm_inputs(M, N, K, 0.02, 0.02)
    lf.gemm_nt(x.to(DEV), w.to(DEV))
    plan = lf.last_gemm_plan()
    torch.cuda.synchronize()
    lf.check_device_error()
    assert plan["cta_pairs"] and plan["tile_n"] == 256, plan
    if pairs == 76:                       # the split's share depends on the pair count
        assert plan["stream_k"] == stream_k, plan


def test_gemm_nt_k1_routes_to_pointwise_bitexact():
    x = synthetic.bf16_normal((96, 1), 2.0, 0)
    w = synthetic.bf16_normal((264, 1), 0.5, 1)
    before = lf.launch_count()
    out = lf.gemm_nt(x.to(DEV), w.to(DEV)).cpu()
    assert lf.launch_count() - before == 1
    want = oracle.matmul_k1_bf16(x, w)
    assert np.array_equal(out.view(torch.int16).numpy().view(np.uint16), want)


def test_gemm_nt_is_one_launch_and_allocates_nothing():
    M, N, K = 768, 5120, 1024
    x, w = synthetic.make_gemm_inputs(M, N, K, 0.02, 0.02)
    xd, wd = x.to(DEV), w.to(DEV)
    out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    lf.gemm_nt(xd, wd, out)          # first call: any one-time setup happens here
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    before = lf.launch_count()
    lf.gemm_nt(xd, wd, out)
    torch.cuda.synchronize()
    assert lf.launch_count() - before == 1
    # no transposed copy of W (K*N*2 bytes) appears anywhere on the device
    assert abs(torch.cuda.mem_get_info()[0] - free0) < K * N * 2 // 4


# --------------------------------------------------------- gemm_nt_xent

def _xent_check(x, w, lab, rows=None, what=""):
    M = x.reshape(-1, x.shape[-1]).shape[0]
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
    loss_only, none = lf.gemm_nt_xent(xd, wd, ld, want_grad=False)
    torch.cuda.synchronize()
    assert none is None
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    _, rloss, _, rgrad = oracle.xent_rows(x.reshape(M, -1), w, lab.numpy(), rows)
    assert_loss_close(f64(loss)[rows], rloss, what)
    assert_loss_close(f64(loss_only)[rows], rloss, what + " (loss only)")
    assert_grad_close(f64(grad)[rows], rgrad, what)
    return loss, grad


def test_xent_tiny_full(variant):
    inp = workload("tiny")
    _xent_check(inp["x"], inp["w"], inp["labels"], what="tiny")


@pytest.mark.parametrize("M,N,K", [(200, 1000, 136), (64, 8, 64), (129, 776, 520), (600, 1032, 264), (1240, 18952, 136)])
def test_xent_ragged_full(M, N, K, variant):
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N)
    edges = [0, N - 1, min(255, N - 1), min(256, N - 1), min(767, N - 1), min(768, N - 1)]
    for i, e in enumerate(edges):
        lab[i] = e
    _xent_check(x, w, lab, what="ragged %dx%dx%d" % (M, N, K))


def test_xent_zero_weight_gives_ln_n(variant):
    M, N, K = 192, 2048, 128
    x = synthetic.bf16_normal((M, K), 1.0, 0)
    w = torch.zeros(N, K, dtype=torch.bfloat16)
    lab = synthetic.labels_uniform(M, N)
    loss, grad = lf.gemm_nt_xent(x.to(DEV), w.to(DEV), lab.to(DEV), want_grad=True)
    assert np.allclose(f64(loss), math.log(N), rtol=1e-6, atol=0)
    want = np.full((M, N), 1.0 / N)
    want[np.arange(M), lab.numpy()] -= 1.0
    assert_grad_close(f64(grad), want, "zero weight")


def test_xent_large_logits(variant):
    M, N, K = 256, 1536, 256
    x, w = synthetic.make_gemm_inputs(M, N, K, 30.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N)
    _xent_check(x, w, lab, what="large logits")


def test_xent_launch_counts():
    inp = workload("tiny")
    xd, wd, ld = inp["x"].to(DEV), inp["w"].to(DEV), inp["labels"].to(DEV)
    lf.gemm_nt_xent(xd, wd, ld)
    b0 = lf.launch_count()
    lf.gemm_nt_xent(xd, wd, ld)
    b1 = lf.launch_count()
    lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
    b2 = lf.launch_count()
    assert (b1 - b0, b2 - b1) == (1, 1)     # N = 256: the whole row in one tile, one launch


def test_xent_onepass_gradient_is_one_launch():
    # on CTA pairs the gradient comes from the same pass (no combine kernel,
    # no recompute GEMM); without a gradient it stays partials + combine
    M, N, K = 512, 2048, 256
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    lf.set_tuning(-1, 2)
    lf.set_xent_grad_path(1)
    try:
        lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        b0 = lf.launch_count()
        loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        b1 = lf.launch_count()
        lf.gemm_nt_xent(xd, wd, ld, want_grad=False)
        b2 = lf.launch_count()
        lf.check_device_error()
    finally:
        lf.set_tuning(-1, -1)
        lf.set_xent_grad_path(0)
    assert (b1 - b0, b2 - b1) == (1, 2)
    rows = sample_rows(M, k=16, seed=9)
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    assert_loss_close(f64(loss)[rows], rloss, "one-pass")
    assert_grad_close(f64(grad)[rows], rgrad, "one-pass")


def test_xent_grad_full_size(variant):
    wl = synthetic.WORKLOADS["xent_grad"]
    inp = workload("xent_grad")
    lab = inp["labels"].clone()
    lab[1], lab[2], lab[3] = 0, wl.N - 1, 256 * 77
    rows = sample_rows(wl.M, k=28, seed=4, extra=(1, 2, 3))
    _xent_check(inp["x"], inp["w"], lab, rows=rows, what="xent_grad")


def test_xent_loss_only_full_size(variant):
    wl = synthetic.WORKLOADS["xent_loss"]
    inp = workload("xent_loss")
    lab = inp["labels"].clone()
    lab[1], lab[2], lab[3] = 0, wl.N - 1, 256 * 400
    xd, wd, ld = inp["x"].to(DEV), inp["w"].to(DEV), lab.to(DEV)
    loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=False)
    torch.cuda.synchronize()
    assert grad is None
    rows = sample_rows(wl.M, k=20, seed=5, extra=(1, 2, 3))
    _, rloss, _, _ = oracle.xent_rows(inp["x"], inp["w"], lab.numpy(), rows, want_grad=False)
    assert_loss_close(f64(loss)[rows], rloss, "xent_loss")
    assert np.all(np.isfinite(f64(loss))) and np.all(f64(loss) > 0)


# ------------------------------------------------------------- matmul_k1

def test_matmul_k1_rope_bitexact_and_permuted_view():
    inp = workload("k1_rope")
    a, b = inp["a"], inp["b"]
    out = lf.matmul_k1(a.to(DEV), b.to(DEV)).cpu()
    want = oracle.matmul_k1(a.numpy(), b.numpy())
    assert out.shape == (64, 4096)
    assert np.array_equal(out.numpy().view(np.uint32), want.view(np.uint32))
    perm = out.t()                                   # the page's [4096, 64] permute
    assert perm.shape == (4096, 64)
    assert np.array_equal(perm.numpy().view(np.uint32), want.T.view(np.uint32))


@pytest.mark.parametrize("M,N,offset", [(7, 13, 0), (3, 4096, 1), (64, 1 << 20, 0), (1, 1, 0), (70000, 8, 0)])
def test_matmul_k1_shapes_bitexact(M, N, offset):
    rng = np.random.default_rng(M + N)
    a = torch.from_numpy((rng.standard_normal(M) * 100).astype(np.float32))
    b = torch.from_numpy((rng.standard_normal(N + offset) * 0.01).astype(np.float32))
    bd = b.to(DEV)[offset:]                          # offset 1: not 16-byte aligned -> scalar path
    out = lf.matmul_k1(a.to(DEV).reshape(M, 1), bd.reshape(1, N)).cpu()
    want = oracle.matmul_k1(a.numpy(), b.numpy()[offset:])
    assert np.array_equal(out.numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("width", [128, 160, 192, 224, 256])
def test_xent_onepass_every_tile_width(width):
    """The one-pass kernel at each N-tile width it can choose, on a shape whose
    last tile is ragged in a different way for each (N = 1032: 136 columns at
    224, 72 at 160, ...), every row against the oracle."""
    M, N, K = 600, 1032, 264
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=11)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    lf.set_onepass_tile(width)
    try:
        b0 = lf.launch_count()
        loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        b1 = lf.launch_count()
        lf.check_device_error()
    finally:
        lf.set_onepass_tile(0)
    assert b1 - b0 == 1
    rows = list(range(M))
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    assert_loss_close(f64(loss), rloss, "width %d" % width)
    assert_grad_close(f64(grad), rgrad, "width %d" % width)


@pytest.mark.parametrize("path", [2, 3], ids=["exp_rescale", "recompute"])
@pytest.mark.parametrize("variant", [2, 3])
def test_xent_two_pass_gradient_on_pairs(variant, path):
    """A vocabulary too wide for one pass (N = 40992: 161 tiles, more than two
    per resident pair; the last tile 32 columns wide) on CTA pairs, by whole
    tiles or stream-K: the exp pass (partials and fp16 exp(z - tile max) into
    grad) and the rescale pass; or partials, combine, and the recompute pass
    writing the gradient.  Sampled rows, every column, against the oracle."""
    M, N, K = 512, 40992, 256
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=12)
    lab[5] = N - 1
    lab[6] = 0
    lab[7] = 256 * 160                      # first column of the ragged last tile
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    lf.set_tuning(-1, variant)
    lf.set_xent_grad_path(path)
    try:
        b0 = lf.launch_count()
        loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        b1 = lf.launch_count()
        lf.check_device_error()
    finally:
        lf.set_tuning(-1, -1)
        lf.set_xent_grad_path(0)
    # exp pass + rescale, or partials GEMM, combine, gradient GEMM
    assert b1 - b0 == (2 if path == 2 else 3)
    rows = sample_rows(M, k=12, seed=13, extra=(5, 6, 7))
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    assert_loss_close(f64(loss)[rows], rloss, "two-pass")
    assert_grad_close(f64(grad)[rows], rgrad, "two-pass")


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (8, 2056, 13824), (16, 4096, 4096), (33, 1032, 264),
                                   (64, 5120, 13824), (100, 520, 2048), (128, 32768, 512), (64, 256, 128)])
def test_skinny_gemm_swapped_operands(M, N, K):
    """M <= 128 runs with the operands swapped (W's rows on the MMA's 256-row
    side, X's rows as its N, the accumulator stored transposed), whole tiles or
    stream-K as the planner picks; every element against the oracle."""
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    n0 = lf.launch_count()
    out = lf.gemm_nt(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    assert lf.launch_count() - n0 == 1
    lf.check_device_error()
    ref = oracle.gemm_nt(x, w)
    got = f64(out)
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    assert err.max() <= 1e-2 * scale
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-3 * scale)


@pytest.mark.parametrize("variant", [2, 3])
def test_skinny_gemm_swapped_whole_tiles_and_streamk(variant):
    M, N, K = 48, 3000 - 3000 % 8, 1536
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lf.set_tuning(-1, 4)                     # force the swapped path ...
    try:
        out_auto = lf.gemm_nt(x.to(DEV), w.to(DEV))
        lf.set_tuning(-1, variant)           # ... and compare with the given pair schedule
        out_v = lf.gemm_nt(x.to(DEV), w.to(DEV))
        torch.cuda.synchronize()
    finally:
        lf.set_tuning(-1, -1)
    lf.check_device_error()
    ref = oracle.gemm_nt(x, w)
    for out in (out_auto, out_v):
        err = np.abs(f64(out) - ref)
        assert err.max() <= 1e-2 * np.abs(ref).max()


def test_matmul_k1_bandwidth_shape_sampled_bitexact():
    """The bench's bandwidth case, [64,1] x [1, 8388608] (2 GiB out), in the
    bench's launch configuration: sampled rows bit-exact against the oracle,
    and the whole output against the fp32 broadcast product on the device
    (one fp32 multiply per element, so any correct kernel is bit-identical)."""
    N = 1 << 23
    a, _ = synthetic.k1_operands(64, 4096)
    b = torch.arange(N, dtype=torch.float32).reshape(1, N)
    ad, bd = a.to(DEV), b.to(DEV)
    out = lf.matmul_k1(ad, bd)
    torch.cuda.synchronize()
    assert out.shape == (64, N)
    rows = [0, 1, 31, 63]
    want = oracle.matmul_k1(a.numpy()[rows], b.numpy())
    got = out[rows].cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert torch.equal(out, ad.reshape(64, 1) * bd)


@pytest.mark.parametrize("width", [224, 256])
def test_xent_onepass_multi_round(width):
    """Several rounds of the one-pass kernel (M = 1500: 6 row blocks, the last
    one ragged; N = 16384: at 224 columns 74 tiles, the last 32 wide), so the
    rounds after the first walk their first tile's K blocks downwards; every
    row against the oracle."""
    M, N, K = 1500, 16384, 136
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=12)
    lab[0], lab[1], lab[2] = 0, N - 1, 16352
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    lf.set_onepass_tile(width)
    try:
        b0 = lf.launch_count()
        loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        b1 = lf.launch_count()
        lf.check_device_error()
    finally:
        lf.set_onepass_tile(0)
    assert b1 - b0 == 1
    rows = list(range(M))
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    assert_loss_close(f64(loss), rloss, "multi-round width %d" % width)
    assert_grad_close(f64(grad), rgrad, "multi-round width %d" % width)


# ------------------------------------------ gradient by exp pass + rescale

@pytest.fixture
def exp_path():
    lf.set_xent_grad_path(2)
    yield
    lf.set_xent_grad_path(0)
    lf.set_tile_band(-1)


@pytest.mark.parametrize("M,N,K", [(600, 1032, 264), (257, 264, 72), (129, 4104, 520), (1500, 16384, 136)])
def test_xent_exp_rescale_ragged_full(M, N, K, exp_path):
    """The exp pass + rescale on ragged shapes (last row block and last
    256-column tile partial; N = 264: the last tile 8 columns wide), labels at 0,
    N - 1 and tile edges; every row, every column against the oracle."""
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=61)
    for i, e in enumerate([0, N - 1, min(255, N - 1), min(256, N - 1), min(N - 8, 4096)]):
        lab[i] = e
    n0 = lf.launch_count()
    loss, grad = lf.gemm_nt_xent(x.to(DEV), w.to(DEV), lab.to(DEV), want_grad=True)
    torch.cuda.synchronize()
    assert lf.launch_count() - n0 == 2
    lf.check_device_error()
    _, rloss, _, rgrad = oracle.xent(x, w, lab.numpy())
    assert_loss_close(f64(loss), rloss, "exp/rescale %dx%dx%d" % (M, N, K))
    assert_grad_close(f64(grad), rgrad, "exp/rescale %dx%dx%d" % (M, N, K))


def test_xent_exp_rescale_near_ties_across_tiles(exp_path):
    """Rows whose softmax mass sits on three near-equal logits in different
    256-column tiles (columns 3, 5 and 700; probabilities about 1/3 each, the
    range where the fp16 intermediate's rounding matters most), the label on
    one of them or elsewhere; and rows dominated by one logit (p > 1/2, which
    must be its tile's maximum, where e = 1 exactly)."""
    M, N, K = 512, 1024, 128
    w = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 62).float()
    w[5] = w[3]
    w[700] = w[3] + 0.01 * synthetic.bf16_normal((K,), 1.0, 63).float()
    d = w[3] / w[3].norm()
    g = torch.Generator().manual_seed(64)
    scale = torch.where(torch.arange(M) % 2 == 0, torch.tensor(12.0), torch.tensor(40.0))
    x = scale[:, None] * d[None, :] + 0.05 * torch.randn(M, K, generator=g)
    # every 4th row: one dominant logit (column 900, p about 0.94 -- large
    # enough to sit at its tile's max, small enough that the loss, about 0.06,
    # is resolved in fp32: a loss near 0 cancels lse against z[label] to noise)
    x[::4] = 10.0 * w[900] / w[900].norm() + 0.05 * torch.randn(M // 4, K, generator=g)
    x, w = x.to(torch.bfloat16), w.to(torch.bfloat16)
    lab = synthetic.labels_uniform(M, N, seed=65)
    lab[1::4], lab[2::4] = 3, 700
    lab[::8] = 900
    loss, grad = lf.gemm_nt_xent(x.to(DEV), w.to(DEV), lab.to(DEV), want_grad=True)
    torch.cuda.synchronize()
    lf.check_device_error()
    _, rloss, _, rgrad = oracle.xent(x, w, lab.numpy())
    p = rgrad + (np.arange(N)[None, :] == lab.numpy()[:, None])
    assert (p.max(axis=1) > 0.8).sum() >= M // 8 and ((p > 0.25) & (p < 0.5)).sum() >= M
    assert_loss_close(f64(loss), rloss, "near ties")
    assert_grad_close(f64(grad), rgrad, "near ties")


def test_xent_exp_rescale_zero_weight_and_large_logits(exp_path):
    M, N, K = 192, 2048, 128
    x = synthetic.bf16_normal((M, K), 1.0, 0)
    w = torch.zeros(N, K, dtype=torch.bfloat16)
    lab = synthetic.labels_uniform(M, N)
    loss, grad = lf.gemm_nt_xent(x.to(DEV), w.to(DEV), lab.to(DEV), want_grad=True)
    assert np.allclose(f64(loss), math.log(N), rtol=1e-6, atol=0)
    want = np.full((M, N), 1.0 / N)
    want[np.arange(M), lab.numpy()] -= 1.0
    assert_grad_close(f64(grad), want, "zero weight")
    x, w = synthetic.make_gemm_inputs(256, 1536, 256, 30.0, 1.0 / 16)
    lab = synthetic.labels_uniform(256, 1536)
    _xent_check(x, w, lab, what="exp/rescale large logits")


def test_xent_exp_rescale_banded_tile_order(exp_path):
    """Whole tiles in bands of 2 and 3 row blocks (the order used when X is too
    large to stay in L2): the same results as one band, bit for bit."""
    M, N, K = 1800, 3080, 136        # 8 row blocks, the last ragged
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=66)
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    outs = []
    for band in (0, 2, 3):
        lf.set_tile_band(band)
        loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
        out = lf.gemm_nt(xd, wd)
        outs.append((loss, grad, out))
    lf.check_device_error()
    for loss, grad, out in outs[1:]:
        assert torch.equal(loss, outs[0][0]) and torch.equal(grad, outs[0][1]) and torch.equal(out, outs[0][2])
    rows = sample_rows(M, k=20, seed=67)
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    assert_loss_close(f64(outs[0][0])[rows], rloss, "banded")
    assert_grad_close(f64(outs[0][1])[rows], rgrad, "banded")
    assert_gemm_close(f64(outs[0][2])[rows], oracle.gemm_nt_rows(x, w, rows), "banded gemm")


def test_xent_exp_rescale_grad_full_size(exp_path):
    """The 4096 x 32768 x 4096 workload through the exp pass + rescale, in the
    bench's configuration; sampled rows with labels at 0, N - 1 and a tile edge."""
    wl = synthetic.WORKLOADS["xent_grad"]
    inp = workload("xent_grad")
    lab = inp["labels"].clone()
    lab[1], lab[2], lab[3] = 0, wl.N - 1, 256 * 77
    rows = sample_rows(wl.M, k=28, seed=68, extra=(1, 2, 3))
    _xent_check(inp["x"], inp["w"], lab, rows=rows, what="xent_grad exp/rescale")


def test_xent_grad_large_vocab_full_size():
    """The 8192 x 128256 x 4096 vocabulary with the gradient, automatic form
    (the exp pass + rescale: two launches), as the bench runs it; sampled rows,
    every column, labels at 0, N - 1 and tile edges."""
    wl = synthetic.WORKLOADS["xent_loss"]
    inp = workload("xent_loss")
    lab = inp["labels"].clone()
    lab[1], lab[2], lab[3], lab[4] = 0, wl.N - 1, 256 * 400, 256 * 500 + 255
    xd, wd, ld = inp["x"].to(DEV), inp["w"].to(DEV), lab.to(DEV)
    n0 = lf.launch_count()
    loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
    torch.cuda.synchronize()
    assert lf.launch_count() - n0 == 2
    lf.check_device_error()
    rows = sample_rows(wl.M, k=12, seed=69, extra=(1, 2, 3, 4))
    _, rloss, _, rgrad = oracle.xent_rows(inp["x"], inp["w"], lab.numpy(), rows)
    assert_loss_close(f64(loss)[rows], rloss, "large vocab grad")
    assert_grad_close(f64(grad[torch.from_numpy(rows).to(DEV)]), rgrad, "large vocab grad")



@pytest.mark.parametrize("form", [(2, 1), (2, 2), (2, 3), (1, 0)],
                         ids=["pair_one_pass", "pair_exp_rescale", "pair_recompute", "cta1_recompute"])
def test_xent_labels_outside_range(form):
    """A label outside [0, N) (no ignore-index exists): that row's loss is NaN
    and its gradient row is the softmax without the -1 term, in every form;
    the other rows are unaffected."""
    variant, path = form
    M, N, K = 264, 1032, 136
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=71)
    bad = {0: -1, 1: N, 2: N + 5, 3: 1 << 30, 4: -(1 << 30), 200: N + 8}
    for r, v in bad.items():
        lab[r] = v
    lf.set_tuning(-1, variant)
    lf.set_xent_grad_path(path)
    try:
        loss, grad = lf.gemm_nt_xent(x.to(DEV), w.to(DEV), lab.to(DEV), want_grad=True)
        loss_only, _ = lf.gemm_nt_xent(x.to(DEV), w.to(DEV), lab.to(DEV), want_grad=False)
        lf.check_device_error()
    finally:
        lf.set_tuning(-1, -1)
        lf.set_xent_grad_path(0)
    _, rloss, _, rgrad = oracle.xent(x, w, lab.numpy())
    got_l, got_lo = f64(loss), f64(loss_only)
    badrows = np.array(sorted(bad))
    good = np.setdiff1d(np.arange(M), badrows)
    assert np.all(np.isnan(rloss[badrows]))
    assert np.all(np.isnan(got_l[badrows])) and np.all(np.isnan(got_lo[badrows]))
    assert_loss_close(got_l[good], rloss[good], "good rows")
    assert_loss_close(got_lo[good], rloss[good], "good rows, loss only")
    assert_grad_close(f64(grad), rgrad, "out-of-range labels")   # bad rows: softmax only


@pytest.mark.parametrize("M,N,K", [(64, 256, 128), (1, 8, 8), (200, 136, 264), (600, 256, 72), (129, 248, 4104)])
def test_xent_whole_row_in_one_tile(M, N, K, variant):
    """N <= 256: every row lies in one N tile, so loss and gradient come from
    one epilogue in one launch (single CTA, CTA pairs, and CTA pairs with the
    K loop split by stream-K, whose owners add the partials in each pass);
    every row and column against the oracle, labels at 0 and N - 1."""
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=81)
    lab[0] = N - 1
    if M > 1:
        lab[M - 1] = 0
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    n0 = lf.launch_count()
    loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
    n1 = lf.launch_count()
    loss_only, _ = lf.gemm_nt_xent(xd, wd, ld)
    n2 = lf.launch_count()
    lf.check_device_error()
    assert (n1 - n0, n2 - n1) == (1, 1)
    _, rloss, _, rgrad = oracle.xent(x, w, lab.numpy())
    assert_loss_close(f64(loss), rloss, "whole row")
    assert_loss_close(f64(loss_only), rloss, "whole row, loss only")
    assert_grad_close(f64(grad), rgrad, "whole row")



@pytest.mark.parametrize("N,launches", [(20000 * 256, 2), (49153 * 256, 3)], ids=["80KiB_scales", "past_limit"])
def test_xent_gradient_very_wide_rows(N, launches):
    """Rows so wide that the rescale kernel keeps 20,000 tile scales (80 KiB)
    in shared memory -- past the 48 KiB default, so the launch opts in to more;
    and one tile past its 49,152-tile limit, where the recompute form runs.
    M = 130 (CTA pairs), K = 8; sampled rows, every column, against the oracle."""
    M, K = 130, 8
    x = synthetic.bf16_normal((M, K), 1.0, 91)
    w = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 92)
    lab = synthetic.labels_uniform(M, N, seed=93)
    lab[0], lab[64], lab[129] = 0, N - 1, 256 * 12345 + 255
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    n0 = lf.launch_count()
    loss, grad = lf.gemm_nt_xent(xd, wd, ld, want_grad=True)
    torch.cuda.synchronize()
    assert lf.launch_count() - n0 == launches
    lf.check_device_error()
    rows = np.array([0, 64, 129])
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
    assert_loss_close(f64(loss)[rows], rloss, "very wide rows")
    assert_grad_close(f64(grad[torch.from_numpy(rows).to(DEV)]), rgrad, "very wide rows")
    del grad
    torch.cuda.empty_cache()
