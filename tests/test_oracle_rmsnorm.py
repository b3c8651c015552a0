"""Pins of the oracle's fused RMSNorm producer (FA4 write-up, "Fused
RMSNorm+Quantize") and of its fp32-input quantizers.  CPU only."""
import numpy as np
import torch

from oracle import oracle as orc


def _bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def test_rmsnorm_matches_fp64_definition_within_fp32_rounding():
    """y = x / sqrt(mean(x^2) + eps) * w against the fp64 formula: a few fp32
    ulps (the fp32 sequence rounds each step once)."""
    x = _bf16((37, 3, 128), 1)
    w = np.random.default_rng(2).uniform(0.5, 1.5, 128).astype(np.float32)
    y = orc.rmsnorm_f32(x, w, 1e-6)
    xd = x.float().double().numpy()
    ref = xd / np.sqrt((xd * xd).mean(-1, keepdims=True) + 1e-6) * w.astype(np.float64)
    np.testing.assert_allclose(y, ref, rtol=6e-7 * 8, atol=1e-30)


def test_rmsnorm_is_scale_invariant_and_exact_for_powers_of_two():
    """With eps = 0 scaling x by 2^k leaves every fp32 step exact up to that
    power, so y is bit-identical; mean(y^2) = 1 for w = 1 to fp32 rounding."""
    x = _bf16((16, 2, 64), 3)
    y0 = orc.rmsnorm_f32(x, None, 0.0)
    for k in (-6, 3, 9):
        y1 = orc.rmsnorm_f32((x.float() * 2.0 ** k).to(torch.bfloat16), None, 0.0)
        np.testing.assert_array_equal(y0, y1)
    np.testing.assert_allclose((y0.astype(np.float64) ** 2).mean(-1), 1.0, rtol=1e-6)


def test_rmsnorm_zero_row_and_constant_row():
    """An all-zero row gives zeros (r = 0 by the reading) even with eps = 0; a
    constant row c gives sign(c) * w exactly when eps = 0 and |c| is a power
    of two."""
    x = torch.zeros((2, 1, 128), dtype=torch.bfloat16)
    x[1] = -0.25
    w = np.linspace(0.5, 2.0, 128).astype(np.float32)
    y = orc.rmsnorm_f32(x, w, 0.0)
    assert not y[0].any()
    np.testing.assert_array_equal(y[1, 0], -w)


def test_f32_quantizers_equal_the_bf16_ones_on_bf16_values():
    """The fp32-input quantizers follow the same rules: on values that are
    bf16 numbers they return the bf16 quantizers' codes and scales."""
    x = _bf16((70, 2, 128), 4)
    cu = np.array([0, 33, 70], np.int32)
    xf = x.float().numpy()
    for a, b in ((orc.quant_row(x), orc.quant_row_f32(xf)),
                 (orc.quant_tok(x, cu), orc.quant_tok_f32(xf, cu)),
                 (orc.quant_tokblock(x, cu, True), orc.quant_tokblock_f32(xf, cu, True))):
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])
