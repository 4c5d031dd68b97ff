"""Checks of the test harness's own helpers (no GPU)."""
import numpy as np

from harness import max_abs_err_bf16_large, rne_bf16


def test_rne_bf16_matches_torch_rounding_of_binary32_values():
    import torch
    x = (np.random.default_rng(4).standard_normal(100000) * 16).astype(np.float32).astype(np.float64)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(rne_bf16(x), want)


def test_rne_bf16_ties_go_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: even (1) wins;
    # 1 + 3 * 2^-8 lies between 1 + 2^-7 and 1 + 2^-6: even (1 + 2^-6) wins
    assert rne_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert rne_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert rne_bf16(np.array([-(1 + 2.0 ** -8)]))[0] == -1.0
    assert rne_bf16(np.array([0.0]))[0] == 0.0


def test_large_outputs_are_held_to_the_rounded_oracle_only():
    want = np.array([5.02, 1.0])  # bf16 values in [4, 8) are 2^-5 apart: 5.02 rounds to 5.03125
    got = np.array([5.03125, 1.0])
    assert max_abs_err_bf16_large(got, want) == 0.0
    # below 4 the comparison is with the oracle itself
    assert max_abs_err_bf16_large(np.array([1.0 + 2.0 ** -7]), np.array([1.0])) == 2.0 ** -7
