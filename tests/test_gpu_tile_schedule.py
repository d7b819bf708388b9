"""Whole tiles claimed at run time, and calls captured into CUDA graphs.

A CTA pair of the whole-tile GEMM either takes a fixed list of tiles (pair i:
tiles i, i + pairs, ...) or starts with tile i and claims every further tile,
in the tile order, from a counter in the library's workspace, handing each
claimed index to its MMA issuer, its epilogue warps and the other CTA through
a ring of shared-memory slots.  Either way every tile is computed whole by one
pair over the same K order, so the outputs must be bit-identical to the fixed
assignment's, and they must match the oracle.  The counter is zeroed by the
pair that claims last, so launches of every kind may follow each other in any
order.

A call made while its stream is being captured into a graph plans only forms
whose CTAs do not wait on each other's flags (the flags carry a per-launch
epoch that every replay would repeat): replays with new inputs must give new,
correct results, claimed tiles included.
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
    yield
    lf.set_tile_schedule(-1)
    lf.set_tuning(-1, -1)
    lf.set_xent_grad_path(0)
    lf.set_test_hooks(False, 0)
    lf.check_device_error()


def both_schedules(call):
    """call() under the fixed assignment and with claimed tiles (CTA pairs,
    whole tiles); returns both results."""
    lf.set_tuning(-1, 2)
    try:
        lf.set_tile_schedule(0)
        fixed = call()
        lf.set_tile_schedule(1)
        claimed = call()
        torch.cuda.synchronize()
        lf.check_device_error()
    finally:
        lf.set_tile_schedule(-1)
        lf.set_tuning(-1, -1)
    return fixed, claimed


def gemm_ok(got, x, w, rows, what):
    ref = oracle.gemm_nt_rows(x, w, rows)
    err = np.abs(f64(got)[rows] - ref).max()
    assert err <= 1e-2 * np.abs(ref).max(), "%s: max err %g" % (what, err)


# (M, N, K): one tile per pair and fewer tiles than pairs; about two waves
# with ragged edges; many waves of single-K-block tiles (the ring's slots are
# reused fastest there: every pair publishes an entry per K block); many
# waves, a deeper K loop
@pytest.mark.parametrize("M,N,K", [(200, 520, 200), (700, 4984, 264), (2048, 16384, 64), (1024, 24576, 520)])
def test_claimed_tiles_match_fixed_assignment_bitwise(M, N, K):
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    xd, wd = x.to(DEV), w.to(DEV)
    fixed, claimed = both_schedules(lambda: lf.gemm_nt(xd, wd))
    assert torch.equal(fixed, claimed)
    rows = np.unique(np.array([r for r in (0, 255, 256, M // 2, M - 1) if r < M]))
    gemm_ok(claimed, x, w, rows, "gemm_nt %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("x_mn,w_mn", [(True, False), (False, True), (True, True)])
def test_claimed_tiles_operand_layouts(x_mn, w_mn):
    M, N, K = 1280, 6144, 264
    x = synthetic.bf16_normal((M, K), 1.0, 61)
    w = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 62)
    xs = (x.t().contiguous() if x_mn else x).to(DEV)
    ws = (w.t().contiguous() if w_mn else w).to(DEV)
    fixed, claimed = both_schedules(lambda: lf.gemm_layout(xs, ws, x_mn=x_mn, w_mn=w_mn))
    assert torch.equal(fixed, claimed)
    gemm_ok(claimed, x, w, np.array([0, 300, 700, M - 1]), "layout")


def test_claimed_tiles_batched_views():
    B, M, N, K = 4, 512, 4104, 136
    x = synthetic.bf16_normal((B * M, K), 1.0, 63)
    w = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 64)
    xd, wd = x.to(DEV).view(B, M, K), w.to(DEV)
    fixed, claimed = both_schedules(lambda: lf.bmm(xd, wd.t()))
    assert torch.equal(fixed, claimed)
    gemm_ok(claimed.reshape(B * M, N), x, w, np.array([0, 511, 512, 1500, B * M - 1]), "batched")


def test_claimed_tiles_skinny_swapped_store():
    M, N, K = 48, 65536, 264     # the swapped (transposed-store) form: tiles along N
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    xd, wd = x.to(DEV), w.to(DEV)
    lf.set_tuning(-1, 4)
    try:
        lf.set_tile_schedule(0)
        fixed = lf.gemm_nt(xd, wd)
        lf.set_tile_schedule(1)
        claimed = lf.gemm_nt(xd, wd)
        torch.cuda.synchronize()
        lf.check_device_error()
    finally:
        lf.set_tile_schedule(-1)
        lf.set_tuning(-1, -1)
    assert torch.equal(fixed, claimed)
    gemm_ok(claimed, x, w, np.arange(M), "swapped")


@pytest.mark.parametrize("form", ["loss", "exp_rescale", "whole_row"])
def test_claimed_tiles_cross_entropy(form):
    M, N, K = {"loss": (1536, 20000, 136), "exp_rescale": (1024, 16392, 264), "whole_row": (24576, 200, 72)}[form]
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    lab = synthetic.labels_uniform(M, N, seed=65)
    lab[:3] = torch.tensor([0, N - 1, min(256, N - 1)], dtype=lab.dtype)   # both ends and a tile edge
    xd, wd, ld = x.to(DEV), w.to(DEV), lab.to(DEV)
    want_grad = form != "loss"
    lf.set_xent_grad_path(2 if form == "exp_rescale" else 0)
    try:
        fixed, claimed = both_schedules(lambda: lf.gemm_nt_xent(xd, wd, ld, want_grad=want_grad))
    finally:
        lf.set_xent_grad_path(0)
    assert torch.equal(fixed[0], claimed[0])
    if want_grad:
        assert torch.equal(fixed[1], claimed[1])
    rows = np.unique(np.array([0, 1, 2, 255, 256, M // 2, M - 1]))
    _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows, want_grad=want_grad)
    rel = np.abs(f64(claimed[0])[rows] - rloss) / np.abs(rloss)
    assert rel.max() <= 1e-3, rel.max()
    if want_grad:
        assert np.abs(f64(claimed[1])[rows] - rgrad).max() <= 2e-3


def test_claimed_tiles_in_every_sequence_of_launch_kinds():
    """Claimed-tile, stream-K and one-pass launches back to back, twice over
    with new inputs: each claimed-tile launch starts from the zero counter its
    predecessor left, so every result is right."""
    shapes = {"claimed": (1024, 16384, 136), "streamk": (768, 5120, 4104), "onepass": (512, 8192, 136)}
    for rnd in range(2):
        ins = {}
        for i, (k, (M, N, K)) in enumerate(shapes.items()):
            x = synthetic.bf16_normal((M, K), 1.0, 70 + 10 * rnd + i)
            w = synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 71 + 10 * rnd + i)
            ins[k] = (x, w, synthetic.labels_uniform(M, N, seed=72 + 10 * rnd + i))
        dev = {k: tuple(t.to(DEV) for t in v) for k, v in ins.items()}
        outs = []
        try:
            for order in (("claimed", "streamk", "onepass", "claimed"), ("onepass", "onepass", "streamk", "streamk")):
                for k in order:
                    x, w, lab = dev[k]
                    if k == "claimed":
                        lf.set_tuning(-1, 2)
                        lf.set_tile_schedule(1)
                        outs.append((k, lf.gemm_nt(x, w)))
                    elif k == "streamk":
                        lf.set_tuning(-1, 3)
                        outs.append((k, lf.gemm_nt(x, w)))
                    else:
                        lf.set_tuning(-1, -1)
                        lf.set_xent_grad_path(1)
                        outs.append((k, lf.gemm_nt_xent(x, w, lab, want_grad=True)))
                    lf.set_tuning(-1, -1)
                    lf.set_tile_schedule(-1)
                    lf.set_xent_grad_path(0)
            torch.cuda.synchronize()
            lf.check_device_error()
        finally:
            lf.set_tuning(-1, -1)
            lf.set_tile_schedule(-1)
            lf.set_xent_grad_path(0)
        for k, res in outs:
            x, w, lab = ins[k]
            rows = np.array([0, 255, 256, x.shape[0] - 1])
            if k == "onepass":
                _, rloss, _, rgrad = oracle.xent_rows(x, w, lab.numpy(), rows)
                assert (np.abs(f64(res[0])[rows] - rloss) / np.abs(rloss)).max() <= 1e-3
                assert np.abs(f64(res[1])[rows] - rgrad).max() <= 2e-3
            else:
                gemm_ok(res, x, w, rows, k)


def test_graph_replays_with_new_inputs():
    """Capture the projection GEMM (stream-K when called eagerly), a claimed-
    tile GEMM and the cross-entropy with gradient (forced to the one-pass
    kernel when called eagerly) into a CUDA graph, then replay it with new
    inputs copied into the captured buffers."""
    M1, N1, K1 = 768, 5120, 4104      # stream-K when eager
    M2, N2, K2 = 1024, 16384, 136     # claimed whole tiles
    M3, N3, K3 = 512, 8192, 136       # one-pass cross-entropy when eager
    x1 = torch.empty(M1, K1, dtype=torch.bfloat16, device=DEV)
    w1 = torch.empty(N1, K1, dtype=torch.bfloat16, device=DEV)
    x2 = torch.empty(M2, K2, dtype=torch.bfloat16, device=DEV)
    w2 = torch.empty(N2, K2, dtype=torch.bfloat16, device=DEV)
    x3 = torch.empty(M3, K3, dtype=torch.bfloat16, device=DEV)
    w3 = torch.empty(N3, K3, dtype=torch.bfloat16, device=DEV)
    l3 = torch.empty(M3, dtype=torch.int32, device=DEV)
    o1 = torch.empty(M1, N1, dtype=torch.bfloat16, device=DEV)
    o2 = torch.empty(M2, N2, dtype=torch.bfloat16, device=DEV)
    loss3 = torch.empty(M3, dtype=torch.float32, device=DEV)
    grad3 = torch.empty(M3, N3, dtype=torch.bfloat16, device=DEV)
    bufs = {"x1": x1, "w1": w1, "x2": x2, "w2": w2, "x3": x3, "w3": w3, "l3": l3}

    def fill(seed):
        host = {
            "x1": synthetic.bf16_normal((M1, K1), 1.0, seed), "w1": synthetic.bf16_normal((N1, K1), 1.0 / 64, seed + 1),
            "x2": synthetic.bf16_normal((M2, K2), 1.0, seed + 2),
            "w2": synthetic.bf16_normal((N2, K2), 1.0 / math.sqrt(K2), seed + 3),
            "x3": synthetic.bf16_normal((M3, K3), 1.0, seed + 4),
            "w3": synthetic.bf16_normal((N3, K3), 1.0 / math.sqrt(K3), seed + 5),
            "l3": synthetic.labels_uniform(M3, N3, seed=seed + 6)}
        for k, t in host.items():
            bufs[k].copy_(t)
        return host

    plans = []

    def calls():
        lf.set_tuning(-1, 3)
        lf.gemm_nt(x1, w1, o1)
        plans.append(lf.last_gemm_plan()["stream_k"])
        lf.set_tuning(-1, 2)
        lf.set_tile_schedule(1)
        lf.gemm_nt(x2, w2, o2)
        lf.set_tuning(-1, -1)
        lf.set_tile_schedule(-1)
        lf.set_xent_grad_path(1)
        n0 = lf.launch_count()
        lf.gemm_nt_xent(x3, w3, l3, want_grad=True, loss=loss3, grad=grad3)
        plans.append(lf.launch_count() - n0)
        lf.set_xent_grad_path(0)

    try:
        fill(100)
        calls()                          # eager: allocates the workspaces before capture
        torch.cuda.synchronize()
        lf.check_device_error()
        assert plans == [True, 1]        # eager: stream-K; the one-pass kernel (one launch)
        plans.clear()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                calls()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        assert plans == [False, 2]       # captured: whole tiles; the exp pass and the rescale
        for seed in (200, 300, 400):
            host = fill(seed)
            graph.replay()
            torch.cuda.synchronize()
            lf.check_device_error()
            rows = np.array([0, 255, 256, 500])
            gemm_ok(o1, host["x1"], host["w1"], rows, "projection replay %d" % seed)
            gemm_ok(o2, host["x2"], host["w2"], rows, "claimed replay %d" % seed)
            _, rloss, _, rgrad = oracle.xent_rows(host["x3"], host["w3"], host["l3"].numpy(), rows)
            assert (np.abs(f64(loss3)[rows] - rloss) / np.abs(rloss)).max() <= 1e-3, seed
            assert np.abs(f64(grad3)[rows] - rgrad).max() <= 2e-3, seed
    finally:
        lf.set_tuning(-1, -1)
        lf.set_tile_schedule(-1)
        lf.set_xent_grad_path(0)


def test_claimed_tiles_from_two_streams():
    """The tile counter is per-device workspace: claimed-tile calls on two
    streams are ordered on the GPU like every other workspace user, and each
    gets its own result."""
    M, N, K = 1024, 16384, 136
    ins = [synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K)) for _ in range(2)]
    ins[1] = (synthetic.bf16_normal((M, K), 1.0, 91), synthetic.bf16_normal((N, K), 1.0 / math.sqrt(K), 92))
    dev = [(x.to(DEV), w.to(DEV)) for x, w in ins]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    lf.set_tuning(-1, 2)
    lf.set_tile_schedule(1)
    try:
        torch.cuda.synchronize()
        for _ in range(3):
            for i in range(2):
                with torch.cuda.stream(streams[i]):
                    outs.append((i, lf.gemm_nt(*dev[i])))
        torch.cuda.synchronize()
        lf.check_device_error()
    finally:
        lf.set_tile_schedule(-1)
        lf.set_tuning(-1, -1)
    rows = np.array([0, 255, 256, 700, M - 1])
    for i, out in outs:
        gemm_ok(out, ins[i][0], ins[i][1], rows, "stream %d" % i)


def test_claimed_tiles_while_other_kernels_hold_sms():
    """Claimed tiles need no co-resident grid: with a test kernel holding 40 SMs
    for 300 ms, the pairs that start late claim fewer tiles (or none) and the
    result is the same, bit for bit."""
    M, N, K = 2048, 16384, 264
    x, w = synthetic.make_gemm_inputs(M, N, K, 1.0, 1.0 / math.sqrt(K))
    xd, wd = x.to(DEV), w.to(DEV)
    lf.set_tuning(-1, 2)
    try:
        lf.set_tile_schedule(0)
        fixed = lf.gemm_nt(xd, wd)
        lf.set_tile_schedule(1)
        other = torch.cuda.Stream()
        torch.cuda.synchronize()
        lf.occupy_sms(40, 300_000_000, stream=other)
        claimed = lf.gemm_nt(xd, wd)
        torch.cuda.synchronize()
        lf.check_device_error()
    finally:
        lf.set_tile_schedule(-1)
        lf.set_tuning(-1, -1)
    assert torch.equal(fixed, claimed)
