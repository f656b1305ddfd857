"""The FP8 quantization oracle against its pins (CPU only)."""
import math

import numpy as np
import pytest
import torch

from oracle import fp8


def test_e4m3_round_matches_torch_on_random_values():
    """torch's float8_e4m3fn conversion (round to nearest even) on values inside +-448."""
    g = np.random.default_rng(0)
    x = np.concatenate([g.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x[np.abs(x) <= 448.0].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).float().double().numpy()
    np.testing.assert_array_equal(fp8.e4m3_round(x.astype(np.float64)), ref)


@pytest.mark.parametrize("x,v", [(448.0, 448.0), (449.0, 448.0), (1000.0, 448.0), (2.0 ** -9, 2.0 ** -9),
                                 (2.0 ** -10, 0.0), (3 * 2.0 ** -11, 2.0 ** -9), (0.1, 0.1015625),
                                 (1.0 + 1 / 16, 1.0), (1.0 + 3 / 16, 1.25), (-240.0, -240.0)])
def test_e4m3_round_special_values(x, v):
    """Saturation at 448, subnormal spacing 2^-9, ties to even (1 + 1/16 -> 1, 1 + 3/16 -> 1.25)."""
    assert fp8.e4m3_round(x) == v


def test_codes_round_trip_and_match_torch_bits():
    grid = fp8.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = ~np.isnan(grid)
    codes = fp8.e4m3_encode(grid[finite])
    np.testing.assert_array_equal(fp8.e4m3_decode(codes), grid[finite])
    t = torch.from_numpy(grid[finite].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # +0 and -0 aside, the codes are torch's
    assert np.array_equal(codes[grid[finite] != 0], t[grid[finite] != 0])
    assert grid[finite].max() == 448.0 and np.nanmin(grid[grid > 0]) == 2.0 ** -9


def test_hadamard_is_orthogonal_and_keeps_scores():
    g = np.random.default_rng(1)
    for d in (4, 64, 128):
        signs = g.choice([-1.0, 1.0], size=d)
        r = fp8.hadamard(d, signs)
        np.testing.assert_allclose(r @ r.T, np.eye(d), atol=1e-12)
        q, k = g.standard_normal((5, d)), g.standard_normal((7, d))
        np.testing.assert_allclose((q @ r) @ (k @ r).T, q @ k.T, atol=1e-10)
    h2 = fp8.hadamard(2) * math.sqrt(2)
    np.testing.assert_array_equal(h2, [[1, 1], [1, -1]])


def test_rotation_spreads_an_outlier_dimension():
    """One dimension 50x larger: the page's reason for incoherent processing.
    After the rotation the largest magnitude is far closer to the RMS value."""
    g = np.random.default_rng(2)
    x = g.standard_normal((1, 1, 256, 128))
    x[..., 7] *= 50.0
    signs = g.choice([-1.0, 1.0], size=128)
    y = x[0, 0] @ fp8.hadamard(128, signs)
    ratio_before = np.abs(x).max() / np.sqrt((x ** 2).mean())
    ratio_after = np.abs(y).max() / np.sqrt((y ** 2).mean())
    assert ratio_after < ratio_before / 3


def test_quantize_tiles_map_amax_to_448_and_bound_the_error():
    g = np.random.default_rng(3)
    x = g.standard_normal((2, 3, 300, 64))
    codes, scales = fp8.quantize(x)
    assert scales.shape == (2, 3, 3)
    back = fp8.dequantize(codes, scales)
    for t in range(3):
        blk = x[:, :, t * 128:(t + 1) * 128]
        np.testing.assert_allclose(np.abs(blk).reshape(2, 3, -1).max(axis=2) / 448.0, scales[:, :, t])
    # relative error of e4m3 rounding: half a unit in the last place (2^-4), or 2^-10 * scale when subnormal
    per_row = np.repeat(scales, 128, axis=2)[:, :, :300, None]
    assert np.all(np.abs(back - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * per_row) + 1e-12)


def test_transposed_and_per_head_layouts():
    g = np.random.default_rng(4)
    x = g.standard_normal((1, 2, 130, 64))
    codes, scales = fp8.quantize(x, per_head=True, transpose=True)
    assert codes.shape == (1, 2, 64, 130) and scales.shape == (1, 2)
    back = fp8.dequantize(codes, scales, transpose=True)
    np.testing.assert_allclose(back, x, rtol=2.0 ** -4, atol=2.0 ** -10 * scales.max())


def test_rotated_quantized_scores_stay_close():
    """Scores from the rotated, quantized Q and K approximate Q K^T."""
    g = np.random.default_rng(5)
    q = g.standard_normal((1, 1, 128, 128))
    k = g.standard_normal((1, 1, 128, 128))
    signs = g.choice([-1.0, 1.0], size=128)
    qq = fp8.dequantize(*fp8.quantize(q, signs))
    kq = fp8.dequantize(*fp8.quantize(k, signs))
    s_ref = q[0, 0] @ k[0, 0].T
    s = qq[0, 0] @ kq[0, 0].T
    assert np.abs(s - s_ref).max() < 0.05 * np.abs(s_ref).max()
