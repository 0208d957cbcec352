"""The parity checker itself, on host arrays (no GPU): at the magnitudes of
the largest workload (N = 1048576, where the attention output has rms about
sqrt(e / N) = 0.0016) the absolute bar alone passes an all-zero output, while
the signal-relative bars of gpu_util reject it, reject a uniformly 10 % small
output and a gradient with a flipped sign, and still pass an output that
carries the rounding a correct bf16 kernel makes."""
import math

import numpy as np
import pytest
import torch

from gpu_util import REL_MAX, REL_RMS, TOL_OUT, check_close, error_stats

BF16 = torch.bfloat16
N5 = 1048576


def reference(seed, rms, shape=(256, 128)):
    """A stand-in reference tensor of the given rms (sampled rows x d)."""
    return np.random.default_rng(seed).standard_normal(shape) * rms


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).float().to(BF16).double().numpy()


def correct_kernel(ref, seed):
    """What a correct bf16 kernel returns: the exact result plus the noise of
    p rounded to bf16 (rms 2^-9 / sqrt(3) of the signal), rounded to bf16."""
    g = np.random.default_rng(seed)
    noise = g.standard_normal(ref.shape) * (2.0 ** -9 / math.sqrt(3)) * np.sqrt(np.mean(ref ** 2))
    return bf16_round(ref + noise)


def passes(got, ref, tol_abs=TOL_OUT[BF16]):
    try:
        check_close(got, ref, BF16, "checker test", tol_abs)
        return True
    except AssertionError:
        return False


def test_absolute_bar_alone_is_vacuous_at_workload5_magnitudes():
    ref = reference(1, math.sqrt(math.e / N5))
    assert np.abs(ref).max() < TOL_OUT[BF16]
    assert error_stats(np.zeros_like(ref), ref)["abs"] <= TOL_OUT[BF16]


def test_correct_rounding_passes():
    for seed, rms in ((2, math.sqrt(math.e / N5)), (3, math.sqrt(math.e / 131072)), (4, 0.3)):
        ref = reference(seed, rms)
        st = error_stats(correct_kernel(ref, seed + 100), ref)
        assert st["rel_max"] <= REL_MAX[BF16] / 2 and st["rel_rms"] <= REL_RMS[BF16] / 2, st
        assert passes(correct_kernel(ref, seed + 100), ref)


@pytest.mark.parametrize("rms", [math.sqrt(math.e / N5), math.sqrt(math.e / 131072)])
def test_planted_mistakes_fail(rms):
    ref = reference(5, rms)
    good = correct_kernel(ref, 6)
    assert passes(good, ref)
    assert not passes(np.zeros_like(ref), ref)             # nothing written
    assert not passes(bf16_round(0.9 * ref), ref)          # 10 % too small
    assert not passes(bf16_round(1.1 * ref), ref)          # 10 % too large
    assert not passes(-good, ref)                          # sign flipped (a dK with -tau)
    shifted = good.copy()
    shifted[:, 0] = good[:, 1]                             # one column from its neighbour
    assert not passes(shifted, ref)


def test_one_bad_row_fails():
    """A single wrong row among 256 (one tile lane) still trips max-abs."""
    ref = reference(7, math.sqrt(math.e / N5))
    got = correct_kernel(ref, 8)
    got[17] = 0.0
    assert not passes(got, ref)
