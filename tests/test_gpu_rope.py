"""GPU parity of the fused RoPE segment (K=1 matmul, permute, pad/cat, cos/sin,
bf16) against the oracle.

Tolerance, from the arithmetic: the angle is one fp32 multiply on both sides
(bit-identical); the oracle then takes the cosine in fp64, rounds it to fp32
(the listing's cosf result) and to bf16.  CUDA's cosf/sinf are within 2 fp32
ulp of the exact value, so the bf16 result can differ from the oracle's only
where the exact value lies within 2 fp32 ulp of a bf16 rounding boundary: by
one bf16 ulp, on a small fraction of elements (bounded here by 0.1 %).  The
cat duplicate is checked bit for bit.
"""
import numpy as np
import pytest
import torch

import layout_folding_gb300 as lf
import oracle
from layout_folding_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def ordered(bits):
    """bf16 codes -> integers in value order (+0 and -0 both 0), so that
    adjacent representable values differ by 1."""
    b = np.asarray(bits, dtype=np.int64)
    return np.where(b < 0x8000, b, -(b & 0x7FFF))


def bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check(inv_cpu, pos_cpu, want_sin=True, max_mismatch=1e-3, **kw):
    inv, pos = inv_cpu.to(DEV), pos_cpu.to(DEV)
    c, s = lf.rope_cos_sin(inv, pos, want_sin=want_sin, **kw)
    torch.cuda.synchronize()
    rc, rs = oracle.rope_cos_sin(inv_cpu, pos_cpu.numpy(), with_sin=want_sin)
    outs = [(bits(c).reshape(rc.shape), rc)]
    if want_sin:
        outs.append((bits(s).reshape(rs.shape), rs))
    else:
        assert s is None
    H = inv_cpu.numel()
    for got, ref in outs:
        d = np.abs(ordered(got) - ordered(ref))
        assert d.max() <= 1, "more than one bf16 ulp from the oracle"
        assert (d != 0).mean() <= max_mismatch
        assert np.array_equal(got[:, :H], got[:, H:]), "the two halves of the cat differ"
    return c, s


def test_page_shape_mistral_4096_positions():
    inv, pos = synthetic.rope_operands(64, 4096)
    c, s = check(inv, pos)
    assert c.shape == (4096, 128) and s.shape == (4096, 128)


def test_long_context_positions():
    inv, pos = synthetic.rope_operands(64, 65536, max_position=32768)
    check(inv, pos)


def test_cos_only():
    inv, pos = synthetic.rope_operands(64, 1000)
    check(inv, pos, want_sin=False)


@pytest.mark.parametrize("H,S", [(13, 100), (1, 1), (8, 3), (64, 1), (24, 777)])
def test_odd_sizes(H, S):
    inv, pos = synthetic.rope_operands(H, S)
    check(inv, pos)


def test_unaligned_outputs_take_the_elementwise_path():
    inv, pos = synthetic.rope_operands(64, 300)
    H, S = 64, 300
    raw_c = torch.zeros(S * 2 * H + 8, dtype=torch.bfloat16, device=DEV)
    raw_s = torch.zeros(S * 2 * H + 8, dtype=torch.bfloat16, device=DEV)
    co, so = raw_c[1:1 + S * 2 * H], raw_s[3:3 + S * 2 * H]
    check(inv, pos, cos_out=co, sin_out=so)
    assert int(raw_c[:1].view(torch.int16).count_nonzero()) == 0 and int(raw_c[1 + S * 2 * H:].view(torch.int16).count_nonzero()) == 0
    assert int(raw_s[:3].view(torch.int16).count_nonzero()) == 0


def test_negative_and_large_positions():
    """Negative ids (cos even, sin odd) and ids far beyond any context length,
    whose angles leave the short argument-reduction range and whose int64 ->
    fp32 conversion rounds."""
    inv, _ = synthetic.rope_operands(64, 1)
    rng = np.random.default_rng(5)
    pos = torch.from_numpy(np.concatenate([-np.arange(0, 512), rng.integers(1 << 17, 1 << 26, 512),
                                           rng.integers(-(1 << 40), 1 << 40, 64)]).astype(np.int64))
    check(inv, pos)


def test_launches_one_kernel():
    inv, pos = synthetic.rope_operands(64, 4096)
    inv, pos = inv.to(DEV), pos.to(DEV)
    lf.rope_cos_sin(inv, pos)
    n0 = lf.launch_count()
    lf.rope_cos_sin(inv, pos)
    assert lf.launch_count() - n0 == 1


def test_bench_shape_2_20_positions_sampled():
    """The bench's bandwidth case: 2^20 positions (32 sequences of 32768),
    H = 64, with sine; sampled positions against the oracle (the same
    one-ulp bound), the whole output checked for the cat duplicate."""
    S = 1 << 20
    inv_cpu, pos_cpu = synthetic.rope_operands(64, S, max_position=32768)
    inv, pos = inv_cpu.to(DEV), pos_cpu.to(DEV)
    c, s = lf.rope_cos_sin(inv, pos)
    torch.cuda.synchronize()
    assert c.shape == (S, 128) and s.shape == (S, 128)
    assert torch.equal(c[:, :64], c[:, 64:]) and torch.equal(s[:, :64], s[:, 64:])
    idx = np.unique(np.concatenate([[0, 1, 32767, 32768, S - 1],
                                    np.random.default_rng(11).integers(0, S, 4096)]))
    rc, rs = oracle.rope_cos_sin(inv_cpu, pos_cpu.numpy()[idx])
    for got, ref in ((bits(c[torch.from_numpy(idx).to(DEV)]), rc), (bits(s[torch.from_numpy(idx).to(DEV)]), rs)):
        d = np.abs(ordered(got.reshape(ref.shape)) - ordered(ref))
        assert d.max() <= 1, "more than one bf16 ulp from the oracle"
        assert (d != 0).mean() <= 1e-3
