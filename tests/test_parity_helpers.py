"""The GPU parity tests' comparison helper, checked on the CPU against values
worked out by hand from the bf16 format (8 significant bits)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from tests._gpu import MAX_ABS, MEAN_ABS, ULP_LOG, bf16_ulps, compare


def test_bf16_ulps_by_hand():
    want = np.array([1.0, 1.0, 3.0, -0.5, 0.0, 1.0 + 2.0 ** -8, 100.0])
    got = np.array([1.0, 1.0 + 2.0 ** -7, 3.0 + 2.0 ** -6, -0.5 - 2.0 ** -9, 0.0, 1.0, 100.5])
    # 1 + 2^-8 rounds (to even) to 1; the ulp of [2^e, 2^(e+1)) is 2^(e-7); 100 is in
    # [64, 128): ulp 0.5.
    assert np.array_equal(bf16_ulps(got, want), [0.0, 1.0, 1.0, 0.5, 0.0, 0.0, 1.0])


def test_compare_logs_and_enforces_the_bounds():
    want = np.linspace(-1, 1, 64).reshape(4, 16)
    got = torch.from_numpy(want).to(torch.bfloat16)
    n = len(ULP_LOG)
    mx, mean = compare(got, want, "rounded copy")
    assert len(ULP_LOG) == n + 1 and ULP_LOG[-1][3] == 0.0
    assert mx <= 2.0 ** -9 and mean <= mx
    bad = want.copy()
    bad[0, 0] += 2 * MAX_ABS
    with pytest.raises(AssertionError, match="bf16 ulps"):
        compare(got, bad, "one large error")
    shifted = want + 2 * MEAN_ABS
    with pytest.raises(AssertionError):
        compare(got, shifted, "biased")
    del ULP_LOG[n:]  # the session summary reports parity cases only
