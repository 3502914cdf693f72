"""Pins of the blockwise FP8 (E4M3) weight encoding reference.

Checked against torch's float8_e4m3fn dtype (a library implementation of
the same format), against every tie between neighbouring E4M3 values,
against the format's own closed forms (largest value 448, smallest
subnormal 2^-9), and against the page's statement that the dequantised
weights differ from the originals by up to ~6% of the block maximum.
"""
import numpy as np
import pytest
import torch

from oracle import fp8_oracle as f8

ALL = np.arange(256, dtype=np.uint8)
FINITE = ALL[~np.isnan(f8.e4m3_decode(ALL))]


def test_decode_matches_torch_for_every_code():
    mine = f8.e4m3_decode(ALL)
    ref = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(mine)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.isnan(mine).sum() == 2  # S.1111.111
    assert np.nanmax(mine) == 448.0 and np.nanmin(np.abs(mine[mine != 0])) == 2.0 ** -9


def test_encode_inverts_decode():
    assert np.array_equal(f8.e4m3_encode(f8.e4m3_decode(FINITE)), FINITE)


def test_rounding_matches_torch_including_every_tie():
    vals = np.unique(f8.e4m3_decode(FINITE[FINITE < 128]))          # non-negative finite values
    mids = ((vals[:-1].astype(np.float64) + vals[1:]) / 2).astype(np.float32)  # exact midpoints (ties)
    rng = np.random.default_rng(1)
    x = np.concatenate([mids, -mids, vals, rng.standard_normal(50000).astype(np.float32) * 40,
                        rng.standard_normal(5000).astype(np.float32) * 1e-3]).astype(np.float32)
    mine = f8.e4m3_round(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(mine, ref)
    # ties go to the even mantissa
    assert f8.e4m3_round(np.float32(1.0625)) == 1.0 and f8.e4m3_round(np.float32(1.1875)) == 1.25


def test_rounding_saturates_at_448():
    assert list(f8.e4m3_round(np.array([448.0, 470.0, 1e6, -1e6], dtype=np.float32))) == [448, 448, 448, -448]


def test_blockwise_scale_puts_the_block_maximum_at_448():
    rng = np.random.default_rng(2)
    w = torch.from_numpy(rng.standard_normal(128 * 64).astype(np.float32) * 0.02).to(torch.bfloat16)
    codes, scales = f8.quantize_blockwise(w)
    blocks = w.float().numpy().reshape(-1, 128)
    amax_pos = np.abs(blocks).argmax(axis=1)
    top = codes.reshape(-1, 128)[np.arange(64), amax_pos]
    assert set(np.unique(top & 0x7F).tolist()) == {0x7E}          # |code| = 448
    np.testing.assert_array_equal(scales, (np.abs(blocks).max(axis=1) / np.float32(448)).astype(np.float32))


def test_dequantised_weights_within_the_pages_six_percent():
    """Per value, |w' - w| <= 2^-4 of its block maximum (3 mantissa bits)
    plus one bf16 rounding: 'up to ~6% of the block maximum'."""
    rng = np.random.default_rng(3)
    w = torch.from_numpy(rng.standard_normal(128 * 500).astype(np.float32) * rng.uniform(1e-3, 1, 128 * 500)
                         .astype(np.float32)).to(torch.bfloat16)
    codes, scales = f8.quantize_blockwise(w)
    back = f8.dequantize_blockwise(codes, scales).float().numpy().reshape(-1, 128)
    orig = w.float().numpy().reshape(-1, 128)
    amax = np.abs(orig).max(axis=1, keepdims=True)
    rel = np.abs(back - orig) / amax
    assert rel.max() <= 2.0 ** -4 * (1 + 2.0 ** -8) + 2.0 ** -9
    assert rel.max() > 0.01  # the bound is reached in order of magnitude, not vacuous


def test_zero_block_and_exact_values():
    w = torch.zeros(256, dtype=torch.bfloat16)
    w[128:] = torch.tensor([448.0, -224.0, 1.0, 0.5] * 32, dtype=torch.bfloat16)
    codes, scales = f8.quantize_blockwise(w)
    assert scales[0] == 1.0 and not codes[:128].any()
    assert scales[1] == 1.0  # amax 448 -> scale 1: every value is exact
    assert torch.equal(f8.dequantize_blockwise(codes, scales), w)


def test_rejects_partial_blocks():
    with pytest.raises(ValueError):
        f8.quantize_blockwise(torch.zeros(100, dtype=torch.bfloat16))
