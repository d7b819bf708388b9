"""GPU parity of the fused float8 cast (both layouts) against the oracle.

The cast is integer-valued at the output (one E4M3 code per element), so the
bar is bit-exact: every code equal to the oracle's, in both layouts.  NaN
inputs must give a NaN code (0x7F or 0xFF: the sign of a NaN is not fixed by
the cast).  Small shapes are checked in full; the page's 4096 x 4096 case on
sampled rows of out (every column) plus the property out_t == out^T over the
whole tensor.
"""
import numpy as np
import pytest
import torch

import layout_folding_gb300 as lf
import oracle
from layout_folding_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run(x_cpu, scale, **kw):
    x = x_cpu.to(DEV)
    s = torch.tensor([scale], dtype=torch.float32, device=DEV)
    out, out_t = lf.fp8_cast_dual(x, s, **kw)
    torch.cuda.synchronize()
    return out, out_t


def codes(t):
    """uint8 codes of an [M, K] fp8 tensor of any strides, row-major on the CPU."""
    return t.contiguous().view(torch.uint8).cpu().numpy() if t.dtype != torch.uint8 else t.contiguous().cpu().numpy()


def check_full(x_cpu, scale, **kw):
    out, out_t = run(x_cpu, scale, **kw)
    ref, ref_t = oracle.fp8_cast_dual(x_cpu, scale)
    got = codes(out)
    got_t = codes(out_t.t()) if tuple(out_t.shape) == tuple(x_cpu.shape) else codes(out_t)
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(got_t, ref_t)
    return out, out_t


@pytest.mark.parametrize("M,K", [(64, 64), (128, 4096), (48, 80), (16, 16), (80, 1040), (1040, 48), (4, 4),
                                 (20, 36), (68, 132), (1028, 260)])
def test_vector_path_tiles_and_ragged_tails(M, K):
    x = synthetic.bf16_normal((M, K), 1.0, 11)
    check_full(x, 10.0)


@pytest.mark.parametrize("M,K", [(1, 1), (1, 4096), (17, 33), (3, 64), (64, 3), (250, 130)])
def test_scalar_path_odd_shapes(M, K):
    x = synthetic.bf16_normal((M, K), 1.0, 12)
    check_full(x, 10.0)


def test_unaligned_pointers_take_the_scalar_path():
    M, K = 64, 128
    big = synthetic.bf16_normal((M * K + 8,), 1.0, 13)
    x_cpu = big[1:1 + M * K].view(M, K)          # 2-byte aligned, not 16
    x = big.to(DEV)[1:1 + M * K].view(M, K)
    s = torch.tensor([10.0], device=DEV)
    raw = torch.zeros(M * K + 16, dtype=torch.uint8, device=DEV)
    raw_t = torch.zeros(M * K + 16, dtype=torch.uint8, device=DEV)
    out = raw[3:3 + M * K].view(M, K)
    out_t = raw_t[5:5 + M * K].view(K, M)
    lf.fp8_cast_dual(x, s, out=out, out_t=out_t)
    torch.cuda.synchronize()
    ref, ref_t = oracle.fp8_cast_dual(x_cpu, 10.0)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    np.testing.assert_array_equal(out_t.cpu().numpy(), ref_t)
    # nothing outside the two views was written
    assert int(raw[:3].count_nonzero()) == 0 and int(raw[3 + M * K:].count_nonzero()) == 0
    assert int(raw_t[:5].count_nonzero()) == 0 and int(raw_t[5 + M * K:].count_nonzero()) == 0


def test_eight_byte_aligned_input():
    M, K = 64, 128
    big = synthetic.bf16_normal((M * K + 8,), 1.0, 18)
    x_cpu = big[4:4 + M * K].view(M, K)          # 8-byte aligned, not 16
    x = big.to(DEV)[4:4 + M * K].view(M, K)
    s = torch.tensor([10.0], device=DEV)
    raw = torch.zeros(M * K + 16, dtype=torch.uint8, device=DEV)
    raw_t = torch.zeros(M * K + 16, dtype=torch.uint8, device=DEV)
    out = raw[4:4 + M * K].view(M, K)
    out_t = raw_t[8:8 + M * K].view(K, M)
    lf.fp8_cast_dual(x, s, out=out, out_t=out_t)
    torch.cuda.synchronize()
    ref, ref_t = oracle.fp8_cast_dual(x_cpu, 10.0)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    np.testing.assert_array_equal(out_t.cpu().numpy(), ref_t)
    assert int(raw[:4].count_nonzero()) == 0 and int(raw[4 + M * K:].count_nonzero()) == 0
    assert int(raw_t[:8].count_nonzero()) == 0 and int(raw_t[8 + M * K:].count_nonzero()) == 0


@pytest.mark.parametrize("scale", [1.0, 10.0, 2.0 ** -20, 1e30])
def test_every_bf16_bit_pattern(scale):
    """All 65536 bf16 values (zeros, subnormals, normals, infinities, NaNs) as a
    [256, 256] input: ties, saturation at 448, underflow to signed zero."""
    bits = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    out, out_t = run(x, scale)
    ref, ref_t = oracle.fp8_cast_dual(x, scale)
    got, got_t = codes(out), codes(out_t.t())
    is_nan = np.isnan(x.float().numpy())
    assert is_nan.sum() > 0
    np.testing.assert_array_equal(got[~is_nan], ref[~is_nan])
    np.testing.assert_array_equal(got_t[~is_nan.T], ref_t[~is_nan.T])
    assert np.all((got[is_nan] & 0x7F) == 0x7F) and np.all((got_t[is_nan.T] & 0x7F) == 0x7F)


def test_output_dtype_and_strides_match_the_page():
    x = synthetic.bf16_normal((96, 160), 1.0, 14)
    out, out_t = check_full(x, 10.0)
    assert out.dtype == torch.float8_e4m3fn and out_t.dtype == torch.float8_e4m3fn
    assert out.stride() == (160, 1) and out_t.stride() == (1, 96)
    assert torch.equal(out.view(torch.uint8), out_t.contiguous().view(torch.uint8))


def test_page_shape_4096x4096_scale_10():
    """The page's example: M = K = 4096, randn bf16 input, scale 10."""
    M = K = 4096
    x_cpu = synthetic.bf16_normal((M, K), 1.0, 15)
    out, out_t = run(x_cpu, 10.0)
    # property at full size: the column-major copy holds exactly the same codes
    assert torch.equal(out.view(torch.uint8), out_t.contiguous().view(torch.uint8))
    rows = sorted({0, 1, 63, 64, 2047, 4095} | set(np.random.default_rng(3).integers(0, M, 58).tolist()))
    ref, _ = oracle.fp8_cast_dual(x_cpu[rows], 10.0)
    np.testing.assert_array_equal(out.view(torch.uint8)[rows].cpu().numpy(), ref)
    # a few full columns of out_t's storage (rows of the [K, M] array)
    cols = [0, 15, 16, 4095]
    ref_cols, _ = oracle.fp8_cast_dual(x_cpu[:, cols].contiguous(), 10.0)
    np.testing.assert_array_equal(out_t.view(torch.uint8)[:, cols].cpu().numpy(), ref_cols)


def test_launches_one_kernel():
    x = synthetic.bf16_normal((256, 256), 1.0, 16).to(DEV)
    s = torch.tensor([10.0], device=DEV)
    lf.fp8_cast_dual(x, s)
    n0 = lf.launch_count()
    lf.fp8_cast_dual(x, s)
    assert lf.launch_count() - n0 == 1


def test_four_row_tiles_with_ragged_tails():
    """Large enough for the 256-row tile variant (at least 16 tiles per SM),
    with a partial last row slab (M % 256 = 48) and a partial last column tile
    (K % 64 = 16): sampled rows against the oracle, all of out_t by transposition."""
    M, K = 256 * 40 + 48, 64 * 63 + 16
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ((M + 255) // 256) * ((K + 63) // 64) >= 16 * sms
    x_cpu = synthetic.bf16_normal((M, K), 1.0, 17)
    out, out_t = run(x_cpu, 10.0)
    assert torch.equal(out.view(torch.uint8), out_t.contiguous().view(torch.uint8))
    rows = sorted({0, 63, 64, 191, 255, 256, M - 49, M - 48, M - 17, M - 16, M - 1}
                  | set(np.random.default_rng(4).integers(0, M, 40).tolist()))
    ref, _ = oracle.fp8_cast_dual(x_cpu[rows], 10.0)
    np.testing.assert_array_equal(out.view(torch.uint8)[rows].cpu().numpy(), ref)
    cols = [0, 63, 64, K - 17, K - 16, K - 1]
    ref_cols, _ = oracle.fp8_cast_dual(x_cpu[:, cols].contiguous(), 10.0)
    np.testing.assert_array_equal(out_t.view(torch.uint8)[:, cols].cpu().numpy(), ref_cols)


def test_bench_shape_16384_sampled():
    """The bench's bandwidth case, 16384 x 16384 with scale 10 (the four-row
    tile path): the two layouts hold the same codes everywhere, sampled rows
    and columns match the oracle bit for bit."""
    M = K = 16384
    x_cpu = synthetic.bf16_normal((M, K), 1.0, 15)
    out, out_t = run(x_cpu, 10.0)
    assert torch.equal(out.view(torch.uint8), out_t.contiguous().view(torch.uint8))
    rows = sorted({0, 255, 256, 8191, M - 1} | set(np.random.default_rng(4).integers(0, M, 27).tolist()))
    ref, _ = oracle.fp8_cast_dual(x_cpu[rows], 10.0)
    np.testing.assert_array_equal(out.view(torch.uint8)[rows].cpu().numpy(), ref)
    cols = [0, 63, 64, K - 1]
    ref_cols, _ = oracle.fp8_cast_dual(x_cpu[:, cols].contiguous(), 10.0)
    np.testing.assert_array_equal(out_t.view(torch.uint8)[:, cols].cpu().numpy(), ref_cols)
