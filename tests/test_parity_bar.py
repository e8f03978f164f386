"""The parity bar itself (CPU): rounding to bf16 and the two assertions of
assert_parity, so a weakened bar cannot pass unnoticed."""
import numpy as np
import pytest
import torch

from _parity import assert_parity, round_to


def test_round_to_bf16_matches_torch_on_float32_values():
    # torch rounds float32 -> bf16 to nearest even; on values exact in float32 a single
    # fp64 rounding must agree with it.
    x = np.random.default_rng(0).standard_normal(200000).astype(np.float32)
    x = np.concatenate([x, np.float32([1.00390625, 1.01171875, -1.00390625, 0.0, 3.0])])
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(round_to(x.astype(np.float64), torch.bfloat16), want)


def test_round_to_ties_go_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: even significand is 1.
    assert round_to(np.array([1 + 2**-8]), torch.bfloat16)[0] == 1.0
    assert round_to(np.array([1 + 3 * 2**-8]), torch.bfloat16)[0] == 1 + 2**-6


def _bf16(a):
    return torch.tensor(a, dtype=torch.float64).to(torch.bfloat16)


def test_bar_accepts_correctly_rounded_output():
    # Attention outputs are averages of N(0,1) rows: mostly small, a few large.
    ref = np.random.default_rng(1).standard_normal(4096) * 0.2
    ref[:8] = [2.5, -3.7, 5.1, -7.9, 2.0, 1.99, 0.999, -0.5]
    assert_parity(_bf16(round_to(ref, torch.bfloat16)), ref)


def test_bar_rejects_a_small_value_off_by_more_than_1e_2():
    ref = np.full(64, 0.3)
    got = round_to(ref, torch.bfloat16)
    got[5] += 0.0117  # 0.0117 from the rounded oracle (6 ulps at 0.3)
    with pytest.raises(AssertionError):
        assert_parity(_bf16(got), ref)


def test_bar_rejects_large_value_two_ulps_off():
    ref = np.full(64, 3.0)
    got = round_to(ref, torch.bfloat16)
    got[0] = 3.0 + 2 * 2**-6  # two bf16 ulps above the exact value
    with pytest.raises(AssertionError):
        assert_parity(_bf16(got), ref)


def test_bar_rejects_mean_error():
    ref = np.linspace(-0.5, 0.5, 4096)
    got = ref + 2e-3  # every element within max-abs, the mean far off
    with pytest.raises(AssertionError):
        assert_parity(_bf16(got), ref)


def test_mean_bar_ignores_only_the_output_rounding():
    # Rows equal to single V values of an FP8 cache (code * 0.02) are not bf16 numbers: the
    # correctly rounded output differs from them by ~1e-3 on average, which passes; the same
    # rows shifted by 1.5e-3 do not.
    codes = np.random.default_rng(3).standard_normal(8192) / 0.02
    ref = np.round(codes) * 0.02
    st = assert_parity(_bf16(round_to(ref, torch.bfloat16)), ref)
    assert st["mean_abs"] > 5e-4 and st["mean_abs_vs_rounded"] == 0.0
    # A bias of 1.5e-3 on rows of magnitude < 0.25 (bf16 spacing <= 2^-10) fails the mean bar
    # while every element stays within max-abs.
    small = ref * 0.1
    with pytest.raises(AssertionError, match="mean-abs"):
        assert_parity(_bf16(small + 1.5e-3), small)
