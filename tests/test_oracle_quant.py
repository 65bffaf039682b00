"""Pins of the oracle's E4M3 weight quantization (oracle/quant.py).

The encoding is checked against torch's float8_e4m3fn type (a library
routine) on all 256 codes and on rounding inputs chosen at and between the
representable values; scaling and saturation against their definitions."""

import numpy as np
import torch

from oracle import quant


def _torch_codes(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_every_code_decodes_like_the_library_type():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = quant.e4m3_value(codes)
    assert np.isnan(got).sum() == 2 and (np.isnan(got) == np.isnan(want)).all()
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])
    assert np.nanmax(got) == quant.E4M3_MAX == 448.0


def test_rounding_matches_the_library_type_within_range():
    pos = quant.e4m3_value(np.arange(127, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2                       # exact ties
    near = np.concatenate([mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20)])
    rng = np.random.default_rng(0)
    rand = np.concatenate([rng.normal(size=4000) * s for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    x = np.concatenate([pos, mids, near, rand, [1e-12, 2.0 ** -10, 3 * 2.0 ** -11]])
    x = x[np.abs(x) <= 448.0].astype(np.float32)
    x = np.concatenate([x, -x])
    np.testing.assert_array_equal(quant.e4m3_round(x), _torch_codes(x))


def test_ties_go_to_an_even_mantissa_and_overflow_saturates():
    # 1.0625 lies halfway between 1.0 (code 0x38) and 1.125 (0x39): even wins
    assert quant.e4m3_round(np.float32(1.0625)) == 0x38
    # 1.1875 lies halfway between 1.125 (0x39) and 1.25 (0x3A)
    assert quant.e4m3_round(np.float32(1.1875)) == 0x3A
    assert quant.e4m3_round(np.float32(1e6)) == 0x7E
    assert quant.e4m3_round(np.float32(-449.0)) == 0xFE
    assert quant.e4m3_round(np.float32(-1e-12)) == 0x80


def test_row_scales_put_each_rows_largest_magnitude_at_448():
    rng = np.random.default_rng(1)
    w = (rng.normal(size=(64, 300)) * rng.uniform(1e-3, 10, size=(64, 1))).astype(np.float32)
    w[5] = 0.0
    codes, s = quant.quantize_rows(w)
    assert s.dtype == np.float32 and s[5] == 1.0 and (codes[5] == 0).all()
    for r in range(64):
        if r == 5:
            continue
        assert s[r] == np.float32(np.abs(w[r]).max() / np.float32(448.0))
        j = np.abs(w[r]).argmax()
        assert abs(quant.e4m3_value(codes[r, j])) == 448.0


def test_dequantization_error_is_within_half_a_step():
    """Normal E4M3 values are 2^-3 apart relative to their binade, subnormals
    2^-9 apart (times the row scale): rounding to nearest is off by at most
    half of that."""
    rng = np.random.default_rng(2)
    w = (rng.normal(size=(32, 512)) * 0.02).astype(np.float32)
    codes, s = quant.quantize_rows(w)
    wq = quant.dequantize_rows(codes, s)
    x = w.astype(np.float64) / s[:, None]
    step = np.where(np.abs(x) >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 1e-30))) - 3),
                    2.0 ** -9)
    assert (np.abs(wq - w) <= 0.5 * step * s[:, None] * (1 + 1e-6) + 1e-30).all()
