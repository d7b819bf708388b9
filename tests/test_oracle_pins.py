"""Pins for the CPU oracle: it is checked against things other than itself --
closed forms, hand-derived values, brute force, library routines and
invariants -- so that a plausible mistake in it (a dropped term, a wrong sign
or index, a transposed operand) fails at least one check.  The same pin
functions are run against deliberately broken oracles (mutants written here,
on the CPU) to show that each pin can fail.

Sources: "Strength reduction: fold transpose into a subsequent GEMM call"
(NT GEMM), "Allow reductions in matmul epilogues" (cross-entropy epilogue),
"Feature request: Schedule a small matmul op as a reduction (or pointwise) op"
(K=1 matmul).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from layout_folding_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(shape, std, seed):
    return synthetic.bf16_normal(shape, std, seed)


def _f64(t):
    return t.float().double().numpy()


# ----------------------------------------------------------------- GEMM pins

def gemm_pin_failures(gemm_nt):
    """Run every GEMM pin against an implementation ``gemm_nt(x, w) -> f64``;
    return the list of pins that fail."""
    bad = []
    # (1) rank-1 closed form with distinct row/column/depth factors; a
    #     transposed operand or a wrong index gives a different matrix.
    M, N, K = 5, 7, 24
    a = np.arange(1, M + 1)              # row factor of X
    b = np.arange(2, N + 2) * 3 - 10     # row factor of W (signed)
    c = (np.arange(K) % 5) - 2           # depth factor of X
    d = (np.arange(K) % 3) + 1           # depth factor of W
    x = torch.tensor(np.outer(a, c), dtype=torch.bfloat16)
    w = torch.tensor(np.outer(b, d), dtype=torch.bfloat16)
    cd = sum(int(ci) * int(di) for ci, di in zip(c, d))
    want = np.array([[int(ai) * int(bj) * cd for bj in b] for ai in a], dtype=np.float64)
    got = gemm_nt(x, w)
    if got.shape != want.shape or not np.array_equal(got, want):
        bad.append("rank1_closed_form")
    # (2) one-hot rows of X select columns of W exactly.
    M, N, K = 6, 9, 16
    w = _bf16((N, K), 1.0, 11)
    ks = [(3 * m + 1) % K for m in range(M)]
    xo = torch.zeros(M, K, dtype=torch.bfloat16)
    for m, k in enumerate(ks):
        xo[m, k] = 1.0
    got = gemm_nt(xo, w)
    want = np.stack([_f64(w)[:, k] for k in ks])
    if got.shape != want.shape or not np.array_equal(got, want):
        bad.append("onehot_selects_columns")
    # (3) numpy float64 X @ W.T on random inputs (library routine).
    M, N, K = 9, 13, 40
    x = _bf16((M, K), 1.0, 21)
    w = _bf16((N, K), 1.0, 22)
    want = _f64(x) @ _f64(w).T
    got = gemm_nt(x, w)
    if got.shape != want.shape or not np.allclose(got, want, rtol=1e-12, atol=1e-12):
        bad.append("numpy_f64_matmul")
    return bad


def test_gemm_nt_pins():
    assert gemm_pin_failures(oracle.gemm_nt) == []


def test_gemm_nt_equals_transpose_then_gemm():
    # The traced program's path (materialised transpose, then GEMM) and the NT
    # GEMM are the same product; with the same summation order they agree bit
    # for bit.
    x = _bf16((11, 56), 1.0, 31)
    w = _bf16((17, 56), 1.0, 32)
    wt = oracle.transpose_bf16(w)
    assert wt.shape == (56, 17)
    assert np.array_equal(oracle.gemm_nt(x, w), oracle.gemm_nn(x, wt))


def test_transpose_is_a_transpose():
    w = _bf16((5, 8), 1.0, 33)
    bits = w.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.transpose_bf16(w), bits.T)


def test_gemm_rows_equal_full_rows():
    x = _bf16((12, 32), 1.0, 41)
    w = _bf16((10, 32), 1.0, 42)
    rows = np.array([0, 3, 11, 3], dtype=np.int64)
    assert np.array_equal(oracle.gemm_nt_rows(x, w, rows), oracle.gemm_nt(x, w)[rows])


def test_gemm_scaling_by_two_is_exact():
    x = _bf16((4, 24), 1.0, 51)
    w = _bf16((6, 24), 1.0, 52)
    assert np.array_equal(oracle.gemm_nt(x * 2, w), 2.0 * oracle.gemm_nt(x, w))


def test_gemm_mutants_fail_pins():
    def transposed_operand(x, w):      # reads W as if it were [K,N]
        xx, ww = _f64(x), _f64(w)
        K = xx.shape[1]
        wt = ww.reshape(-1)[: K * ww.shape[0]].reshape(K, ww.shape[0])
        return xx @ wt

    def dropped_last_term(x, w):       # loop bound off by one
        xx, ww = _f64(x), _f64(w)
        return xx[:, :-1] @ ww[:, :-1].T

    def reversed_row_index(x, w):      # writes row m of the product into row M-1-m
        xx, ww = _f64(x), _f64(w)
        return (xx @ ww.T)[::-1]

    for mutant in (transposed_operand, dropped_last_term, reversed_row_index):
        assert gemm_pin_failures(mutant), mutant.__name__


# ------------------------------------------------------- cross-entropy pins

def xent_pin_failures(xent_logits):
    """Run every cross-entropy pin against ``xent_logits(z, labels) ->
    (loss, lse, grad)``; return the failing pins."""
    bad = []
    with open(os.path.join(GOLDEN, "xent_closed_forms.json")) as f:
        cases = json.load(f)["cases"]
    # (1) hand-derived closed forms (golden fixture).
    for i, cs in enumerate(cases):
        z = np.array([[math.log(r) + cs["shift"] for r in cs["ratios"]]])
        loss, _, grad = xent_logits(z, np.array([cs["label"]], dtype=np.int32))
        num, den = cs["loss_ln_of"]
        if not math.isclose(loss[0], math.log(num / den), rel_tol=1e-12, abs_tol=1e-12):
            bad.append("closed_form_loss_%d" % i)
        want_g = np.array([p / q for p, q in cs["grad"]])
        if not np.allclose(grad[0], want_g, rtol=0, atol=1e-13):
            bad.append("closed_form_grad_%d" % i)
    rng = np.random.default_rng(7)
    M, N = 16, 37
    z = rng.normal(0.0, 3.0, size=(M, N))
    lab = rng.integers(0, N, size=M).astype(np.int32)
    lab[0], lab[1] = 0, N - 1
    loss, lse, grad = xent_logits(z, lab)
    # (2) brute force -log(exp z_L / sum exp z) in long double.
    if not np.allclose(loss, oracle.xent_bruteforce(z, lab), rtol=1e-12, atol=1e-13):
        bad.append("bruteforce")
    # (3) loss >= 0 and lse >= max z.
    if not (np.all(loss >= 0) and np.all(lse >= z.max(axis=1))):
        bad.append("nonnegative")
    # (4) equal logits give ln N.
    for NN in (2, 256, 32768):
        zz = np.full((2, NN), 0.75)
        l2, _, _ = xent_logits(zz, np.array([0, NN - 1], dtype=np.int32))
        if not np.allclose(l2, math.log(NN), rtol=1e-13, atol=0):
            bad.append("equal_logits_lnN_%d" % NN)
    # (5) two classes: loss = softplus(z_other - z_L).
    z2 = rng.normal(0.0, 4.0, size=(8, 2))
    l2lab = (np.arange(8) % 2).astype(np.int32)
    l2, _, _ = xent_logits(z2, l2lab)
    want = [math.log1p(math.exp(z2[i, 1 - l2lab[i]] - z2[i, l2lab[i]])) for i in range(8)]
    if not np.allclose(l2, want, rtol=1e-12, atol=1e-14):
        bad.append("two_class_softplus")
    # (6) shift invariance per row.
    shift = rng.normal(0, 50, size=(M, 1))
    ls, _, gs = xent_logits(z + shift, lab)
    if not (np.allclose(ls, loss, rtol=1e-9, atol=1e-9) and np.allclose(gs, grad, atol=1e-12)):
        bad.append("shift_invariance")
    # (7) grad rows sum to zero, entries in (-1,1), exactly one negative at L.
    if not np.all(np.abs(grad.sum(axis=1)) <= 1e-12):
        bad.append("grad_rows_sum_zero")
    neg = grad < 0
    if not (np.all(np.abs(grad) < 1) and np.all(neg.sum(axis=1) == 1)
            and np.all(neg[np.arange(M), lab])):
        bad.append("grad_sign_pattern")
    # (8) central finite differences of the loss w.r.t. z.
    h = 1e-6
    zf = z[:3]
    lf = lab[:3]
    _, _, gf = xent_logits(zf, lf)
    fd = np.empty_like(zf)
    for n in range(N):
        e = np.zeros_like(zf)
        e[:, n] = h
        lp, _, _ = xent_logits(zf + e, lf)
        lm, _, _ = xent_logits(zf - e, lf)
        fd[:, n] = (lp - lm) / (2 * h)
    if not np.allclose(fd, gf, atol=1e-7, rtol=0):
        bad.append("finite_differences")
    # (9) extreme magnitudes need the max subtraction: no overflow, exact-ish.
    zb = np.array([[1000.0, 1000.0 + math.log(3.0), -1000.0]])
    lb, _, _ = xent_logits(zb, np.array([1], dtype=np.int32))
    if not (np.isfinite(lb[0]) and math.isclose(lb[0], math.log(4.0 / 3.0), rel_tol=1e-12)):
        bad.append("large_logits")
    return bad


def test_xent_pins():
    assert xent_pin_failures(oracle.xent_logits) == []


def test_xent_label_out_of_range_is_nan():
    z = np.zeros((3, 5))
    loss, lse, grad = oracle.xent_logits(z, np.array([-1, 5, 2], dtype=np.int32))
    assert np.isnan(loss[0]) and np.isnan(loss[1]) and loss[2] == pytest.approx(math.log(5))
    assert np.allclose(grad[0], 0.2) and np.allclose(grad[1], 0.2)


def test_xent_rows_equals_gemm_then_logits():
    x = _bf16((8, 64), 1.0, 61)
    w = _bf16((40, 64), 0.125, 62)
    lab = synthetic.labels_uniform(8, 40).numpy()
    z, loss, lse, grad = oracle.xent(x, w, lab)
    z2 = oracle.gemm_nt(x, w)
    assert np.array_equal(z, z2)
    l2, s2, g2 = oracle.xent_logits(z2, lab)
    assert np.array_equal(loss, l2) and np.array_equal(lse, s2) and np.array_equal(grad, g2)


def test_xent_zero_weight_gives_ln_n_and_uniform_grad():
    # W = 0 makes every logit 0: loss = ln N and grad = 1/N - onehot.
    M, N, K = 4, 256, 128
    x = _bf16((M, K), 1.0, 0)
    w = torch.zeros(N, K, dtype=torch.bfloat16)
    lab = np.array([0, 255, 128, 7], dtype=np.int32)
    _, loss, _, grad = oracle.xent(x, w, lab)
    assert np.allclose(loss, math.log(N), rtol=1e-15, atol=0)
    want = np.full((M, N), 1.0 / N)
    want[np.arange(M), lab] -= 1.0
    assert np.allclose(grad, want, rtol=0, atol=1e-15)


def test_xent_mutants_fail_pins():
    def literal_sum_reading(z, lab):   # sum_n (lse - where(onehot, z, 0)) = N*lse - z_L
        loss, lse, grad = oracle.xent_logits(z, lab)
        return z.shape[1] * lse - z[np.arange(len(lab)), lab], lse, grad

    def grad_sign_flipped(z, lab):     # onehot - softmax
        loss, lse, grad = oracle.xent_logits(z, lab)
        return loss, lse, -grad

    def dropped_max_in_lse(z, lab):    # lse = log sum exp(z - m), forgetting + m
        loss, lse, grad = oracle.xent_logits(z, lab)
        mx = z.max(axis=1)
        return loss - mx, lse - mx, grad

    def label_off_by_one(z, lab):      # reads z at L+1
        lab2 = np.minimum(lab + 1, z.shape[1] - 1).astype(np.int32)
        loss, lse, _ = oracle.xent_logits(z, lab2)
        _, _, grad = oracle.xent_logits(z, lab)
        return loss, lse, grad

    def grad_missing_onehot(z, lab):   # softmax without the -1
        loss, lse, grad = oracle.xent_logits(z, lab)
        g = grad.copy()
        g[np.arange(len(lab)), lab] += 1.0
        return loss, lse, g

    for mutant in (literal_sum_reading, grad_sign_flipped, dropped_max_in_lse,
                   label_off_by_one, grad_missing_onehot):
        assert xent_pin_failures(mutant), mutant.__name__


# ---------------------------------------------------------------- K=1 pins

def test_matmul_k1_is_broadcast_multiply():
    a, b = synthetic.k1_operands(64, 4096)
    got = oracle.matmul_k1(a.numpy(), b.numpy())
    want = a.numpy().astype(np.float32) * b.numpy().astype(np.float32)   # numpy fp32 broadcast
    assert got.dtype == np.float32 and got.shape == (64, 4096)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # a[0] = 1: row 0 is b exactly; column 0 (position 0) is all zeros.
    assert np.array_equal(got[0], b.numpy().ravel())
    assert np.all(got[:, 0] == 0)


def test_k1_operands_follow_the_rope_definition():
    a, b = synthetic.k1_operands(64, 4096)
    for i in (0, 1, 17, 63):
        assert a[i, 0].item() == np.float32(10000.0 ** (-(2.0 * i) / 128.0))
    assert a[0, 0].item() == 1.0
    assert b[0, 4095].item() == 4095.0 and b[0, 0].item() == 0.0


def test_matmul_k1_random_values_bitexact():
    rng = np.random.default_rng(3)
    a = rng.standard_normal(33).astype(np.float32) * 1e3
    b = rng.standard_normal(77).astype(np.float32) * 1e-3
    got = oracle.matmul_k1(a, b)
    want = a[:, None] * b[None, :]
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_bf16_round_matches_torch():
    vals = np.array([0.0, -0.0, 1.0, 1.00390625, 1.001953125, 1.005859375, 3.14159,
                     -2.7182817, 1e-40, 6.5e4, 3.4e38, -3.4e38, float("inf"), 1.0 + 2 ** -8,
                     1.0 + 3 * 2 ** -9, 255.5, 257.0, 259.0], dtype=np.float32)
    rng = np.random.default_rng(5)
    vals = np.concatenate([vals, rng.standard_normal(500).astype(np.float32) * 10])
    got = oracle.bf16_round(vals)
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_matmul_k1_bf16_matches_library_rounding():
    x = _bf16((19, 1), 3.0, 71)
    w = _bf16((24, 1), 0.5, 72)
    got = oracle.matmul_k1_bf16(x, w)
    want = (x.float() * w.float().t()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_page_shapes_fixture_matches_workloads():
    with open(os.path.join(GOLDEN, "page_shapes.json")) as f:
        pages = json.load(f)
    wl = synthetic.WORKLOADS["nt_projection"]
    nt = pages["nt_projection"]
    assert list(wl.x_shape) == nt["activation"]
    assert [wl.M, wl.K] == nt["activation_2d"] and [wl.N, wl.K] == nt["weight"]
    assert [wl.K, wl.N] == nt["transposed_weight"] and [wl.M, wl.N] == nt["output_2d"]
    assert nt["output"][0] * nt["output"][1] == wl.M
    k1 = synthetic.WORKLOADS["k1_rope"]
    pk = pages["k1_rope"]
    assert [k1.M, k1.K] == pk["a"][1:] and [k1.K, k1.N] == pk["b"][1:]
    assert [k1.M, k1.N] == pk["out"][1:] and [k1.N, k1.M] == pk["out_permuted"][1:]


# ------------------------------------------------ fp8 cast + dual layout pins
# "Improve the Inductor generated kernel for the pattern of output1 =
# pointwise(intput); output2 = transpose(output1)" (pytorch issue 130015).

def test_e4m3_hand_derived_codes():
    with open(os.path.join(GOLDEN, "e4m3_codes.json")) as f:
        cases = json.load(f)["cases"]
    vals = np.array([v for v, _ in cases], dtype=np.float32)
    want = np.array([c for _, c in cases], dtype=np.uint8)
    assert np.array_equal(oracle.f32_to_e4m3(vals), want)


def test_e4m3_matches_library_conversion():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.uniform(-448, 448, 3000), rng.normal(0, 1, 3000), rng.normal(0, 0.01, 2000),
        np.ldexp(rng.integers(0, 8, 500), -9) + np.ldexp(1, -10),     # subnormal midpoints
        np.arange(-448, 449, 0.5)]).astype(np.float32)
    got = oracle.f32_to_e4m3(vals)
    want = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_fp8_cast_dual_layout_and_clamp():
    x = synthetic.bf16_normal((37, 53), 30.0, 3)          # |x * 10| often > 448: exercises the clamp
    out, out_t = oracle.fp8_cast_dual(x, 10.0)
    assert out.shape == (37, 53) and out_t.shape == (53, 37)
    assert np.array_equal(out_t, out.T)                    # the column-major copy holds the same codes
    ref = (x.float() * torch.tensor(10.0)).clamp(-448, 448).to(torch.float8_e4m3fn)
    assert np.array_equal(out, ref.view(torch.uint8).numpy())
    assert np.sum(out == 126) + np.sum(out == 254) > 0     # some values clamped to +-448


def test_fp8_cast_dual_mutants_fail():
    x = synthetic.bf16_normal((16, 24), 30.0, 4)
    out, out_t = oracle.fp8_cast_dual(x, 10.0)
    ref = (x.float() * 10.0).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    no_clamp = (x.float() * 10.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()   # forgotten clamp
    truncating = np.sign(x.float().numpy()) * np.floor(np.abs(x.float().numpy() * 10.0))  # wrong rounding
    assert not np.array_equal(no_clamp, ref)
    assert not np.array_equal(oracle.f32_to_e4m3(np.clip(truncating, -448, 448)), ref)
    assert not np.array_equal(out_t, out)                  # the second layout really is transposed


# --------------------------------------------------------------- RoPE segment
# "Feature request: Schedule a small matmul op as a reduction (or pointwise)
# op", the Mistral forward listing T3 .. T26: angle = fp32(inv_freq[i] *
# float(position)), the permute to [S, H], the pad/cat duplicate to 2H
# columns, cos (and sin) in fp32, rounded to bf16.

def _bf16_bits_to_f64(b):
    return oracle.bf16_bits_to_f64(np.asarray(b, dtype=np.uint16))


def rope_pin_failures(rope):
    """Names of the pins `rope(inv_freq_bf16_tensor, positions) -> (cos, sin)`
    (uint16 bf16 codes, [S, 2H]) violates."""
    failed = []
    with open(os.path.join(GOLDEN, "rope_cos_sin.json")) as f:
        g = json.load(f)
    inv = torch.tensor(g["inv_freq"], dtype=torch.bfloat16)
    c, s = rope(inv, g["positions"])
    H = len(g["inv_freq"])
    want_c = np.array([[int(v, 16) for v in r] for r in g["cos_first_half"]], dtype=np.uint16)
    want_s = np.array([[int(v, 16) for v in r] for r in g["sin_first_half"]], dtype=np.uint16)
    if c.shape != (4, 2 * H) or not np.array_equal(c[:, :H], want_c) or not np.array_equal(s[:, :H], want_s):
        failed.append("golden")
    # the second half of the row repeats the first (pad + cat of the same freqs)
    inv64, pos = synthetic.rope_operands(64, 300)
    c, s = rope(inv64, pos.numpy())
    if c.shape != (300, 128) or not (np.array_equal(c[:, :64], c[:, 64:]) and np.array_equal(s[:, :64], s[:, 64:])):
        failed.append("duplicate halves")
    # position 0: angle 0 for every frequency
    if not (np.all(c[0] == 0x3F80) and np.all(s[0] == 0)):
        failed.append("position zero")
    # cos^2 + sin^2 = 1 within two bf16 roundings
    cf, sf = _bf16_bits_to_f64(c), _bf16_bits_to_f64(s)
    if np.max(np.abs(cf * cf + sf * sf - 1.0)) > 2 * 2.0 ** -8:
        failed.append("pythagoras")
    # double angle with power-of-two frequencies: angle(2p) = 2 * angle(p) exactly
    inv_p2 = torch.tensor([2.0 ** -k for k in range(8)], dtype=torch.bfloat16)
    p = np.arange(0, 200, dtype=np.int64)
    c1, s1 = rope(inv_p2, p)
    c2, s2 = rope(inv_p2, 2 * p)
    a_c, a_s = _bf16_bits_to_f64(c1), _bf16_bits_to_f64(s1)
    b_c, b_s = _bf16_bits_to_f64(c2), _bf16_bits_to_f64(s2)
    if (np.max(np.abs(b_c - (2 * a_c * a_c - 1))) > 0.02 or np.max(np.abs(b_s - 2 * a_s * a_c)) > 0.02):
        failed.append("double angle")
    # negative positions: cos even, sin odd, bit for bit
    cn, sn = rope(inv_p2, -p)
    if not (np.array_equal(cn, c1) and np.array_equal(sn[1:], s1[1:] ^ 0x8000)):
        failed.append("parity")
    return failed


def _oracle_rope(inv, pos):
    return oracle.rope_cos_sin(inv, pos)


def test_rope_pins():
    assert rope_pin_failures(_oracle_rope) == []


def test_rope_operands_follow_the_page_shapes():
    inv, pos = synthetic.rope_operands()
    assert inv.dtype == torch.bfloat16 and inv.shape == (64,) and pos.dtype == torch.int64 and pos.shape == (4096,)
    assert float(inv[0]) == 1.0 and np.all(np.diff(inv.float().numpy()) < 0)
    c, s = oracle.rope_cos_sin(inv, pos)
    assert c.shape == (4096, 128) and s.shape == (4096, 128)


def test_rope_mutants_fail_pins():
    def swapped(inv, pos):
        c, s = _oracle_rope(inv, pos)
        return s, c

    def no_cat(inv, pos):
        c, s = _oracle_rope(inv, pos)
        H = c.shape[1] // 2
        c, s = c.copy(), s.copy()
        c[:, H:] = 0
        s[:, H:] = 0
        return c, s

    def reversed_freqs(inv, pos):                  # wrong index into inv_freq
        return _oracle_rope(torch.flip(inv, [0]), pos)

    def no_freq(inv, pos):                         # angle = position (dropped factor)
        return _oracle_rope(torch.ones_like(inv), pos)

    def off_by_one(inv, pos):
        return _oracle_rope(inv, np.asarray(pos) + 1)

    def sin_negated(inv, pos):
        c, s = _oracle_rope(inv, pos)
        return c, s ^ np.uint16(0x8000)

    for m in (swapped, no_cat, reversed_freqs, no_freq, off_by_one, sin_negated):
        assert rope_pin_failures(m), m.__name__


# ------------------------------------------------------- operand layouts
# "Strength reduction: fold transpose into a subsequent GEMM call": the
# product must not depend on which stored layout an operand arrives in.

def layout_pin_failures(gemm_layout):
    failed = []
    x = _bf16((37, 72), 1.0, 21)
    w = _bf16((45, 72), 1.0, 22)
    ref = oracle.gemm_nt(x, w)                      # pinned on its own above
    xt = oracle.transpose_bf16(x)                   # [K, M]
    wt = oracle.transpose_bf16(w)                   # [K, N]
    for x_mn, w_mn in ((False, False), (True, False), (False, True), (True, True)):
        got = gemm_layout(xt if x_mn else x, x_mn, wt if w_mn else w, w_mn)
        if got.shape != ref.shape or not np.array_equal(got, ref):
            failed.append("transpose identity %d%d" % (x_mn, w_mn))
    # one-hot rows of X stored M-major select columns of W stored N-major, exactly
    K, M, N = 40, 16, 24
    xo = np.zeros((K, M), dtype=np.float32)
    for m in range(M):
        xo[(3 * m) % K, m] = 1.0
    xo = torch.from_numpy(xo).to(torch.bfloat16)
    wn = _bf16((K, N), 1.0, 23)
    got = gemm_layout(xo, True, wn, True)
    want = np.stack([_f64(wn)[(3 * m) % K] for m in range(M)])
    if not np.array_equal(got, want):
        failed.append("one-hot")
    # row subset equals the full rows
    full = gemm_layout(xt, True, w, False)
    sub = gemm_layout(xt, True, w, False, rows=[0, 5, 36])
    if not np.array_equal(sub, full[[0, 5, 36]]):
        failed.append("rows")
    return failed


def test_gemm_layout_pins():
    assert layout_pin_failures(oracle.gemm_layout) == []


def test_gemm_layout_mutants_fail_pins():
    def ignores_x_layout(x, x_mn, w, w_mn, rows=None):     # reads X as if K-major
        xb = oracle._bits(x)
        xb = xb.reshape(xb.shape[1], xb.shape[0]) if x_mn else xb
        return oracle.gemm_layout(xb, False, w, w_mn, rows)

    def transposed_w(x, x_mn, w, w_mn, rows=None):          # flips W's layout flag
        wb = oracle._bits(w)
        return oracle.gemm_layout(x, x_mn, wb.reshape(wb.shape[1], wb.shape[0]), not w_mn, rows)

    def dropped_last_k(x, x_mn, w, w_mn, rows=None):
        out = oracle.gemm_layout(x, x_mn, w, w_mn, rows)
        xb, wb = oracle._bits(x), oracle._bits(w)
        xl = oracle.bf16_bits_to_f64(xb[-1] if x_mn else xb[:, -1])
        wl = oracle.bf16_bits_to_f64(wb[-1] if w_mn else wb[:, -1])
        if rows is not None:
            xl = xl[list(rows)]
        return out - np.outer(xl, wl)

    for m in (ignores_x_layout, transposed_w, dropped_last_k):
        assert layout_pin_failures(m), m.__name__



# ------------------------------------------------ batched, strided views

def batched_pin_failures(gemm_batched):
    failed = []
    B, M, N, K = 3, 20, 24, 40
    ldx, ldw = 56, 48                               # padded rows: views of wider tensors
    xs = _bf16((B, M, ldx), 1.0, 41)
    ws = _bf16((B, N, ldw), 1.0, 42)
    got = gemm_batched(xs, False, ldx, M * ldx, ws, False, ldw, N * ldw, B, M, N, K)
    for b in range(B):                              # each batch is the 2-D product of its slices
        ref = oracle.gemm_nt(xs[b, :, :K].contiguous(), ws[b, :, :K].contiguous())
        if not np.array_equal(got[b], ref):
            failed.append("slice %d" % b)
    # MN-major views: the transposed storage of the same operands
    xt = torch.stack([xs[b, :, :K].t().contiguous() for b in range(B)])       # [B, K, M]
    wt = torch.stack([ws[b, :, :K].t().contiguous() for b in range(B)])       # [B, K, N]
    got_t = gemm_batched(xt, True, M, K * M, wt, True, N, K * N, B, M, N, K)
    if not np.array_equal(got_t, got):
        failed.append("layouts")
    # one W for every batch (batch stride 0)
    got_bc = gemm_batched(xs, False, ldx, M * ldx, ws[0], False, ldw, 0, B, M, N, K)
    for b in range(B):
        if not np.array_equal(got_bc[b], oracle.gemm_nt(xs[b, :, :K].contiguous(), ws[0, :, :K].contiguous())):
            failed.append("broadcast %d" % b)
    return failed


def test_gemm_batched_pins():
    assert batched_pin_failures(oracle.gemm_batched) == []


def test_gemm_batched_mutants_fail_pins():
    def ignores_ld(x, x_mn, ldx, sx, w, w_mn, ldw, sw, B, M, N, K):      # assumes dense rows
        return oracle.gemm_batched(x, x_mn, K if not x_mn else M, sx, w, w_mn, ldw, sw, B, M, N, K)

    def first_batch_only(x, x_mn, ldx, sx, w, w_mn, ldw, sw, B, M, N, K):
        return oracle.gemm_batched(x, x_mn, ldx, 0, w, w_mn, ldw, sw, B, M, N, K)

    def w_batch_ignored(x, x_mn, ldx, sx, w, w_mn, ldw, sw, B, M, N, K):
        return oracle.gemm_batched(x, x_mn, ldx, sx, w, w_mn, ldw, 0, B, M, N, K)

    for m in (ignores_ld, first_batch_only, w_batch_ignored):
        assert batched_pin_failures(m), m.__name__
