"""The sparse MLA kernel's two CTAs swap half-tile scores as fp16 differences
to the half's maximum (log2 domain).  These CPU checks confirm the rounding
bound that argument relies on: the rebuilt scores change the softmax weights
by less than the bf16 rounding that P gets anyway."""

import numpy as np
import pytest


def _rebuild(z):
    """z (fp32, log2 domain, one half-tile row) -> m + fp32(fp16(z - m))."""
    z = z.astype(np.float32)
    m = np.float32(z.max())
    d = (z - m).astype(np.float16).astype(np.float32)
    return (m + d).astype(np.float32)


@pytest.mark.parametrize("scale", [0.5, 4.0, 30.0])
def test_exp2_relative_error_near_the_max(scale):
    rng = np.random.default_rng(7)
    z = (rng.standard_normal(200000) * scale).astype(np.float32)
    zr = _rebuild(z)
    m = z.max()
    d = z.astype(np.float64) - m
    rel = np.abs(np.exp2(zr.astype(np.float64) - m) - np.exp2(d)) / np.exp2(d)
    near = d > -2.0
    # fp16 spacing below |d| = 2 is 2^-10, so rounding errs by <= 2^-11 in d
    # (plus fp32 rounding of m + d, a few 1e-6 at |z| ~ 100)
    assert rel[near].max() <= np.log(2.0) * 2.0 ** -11 + 1e-5
    # everywhere, the absolute error of a weight relative to the maximum weight
    # stays below the bf16 rounding of P (2^-9 relative)
    absw = np.abs(np.exp2(zr.astype(np.float64) - m) - np.exp2(d))
    assert absw.max() <= 2.0 ** -9


def test_softmax_of_rebuilt_scores_within_bf16_rounding():
    rng = np.random.default_rng(11)
    for _ in range(50):
        z = (rng.standard_normal((2, 32)) * rng.uniform(0.1, 20.0)).astype(np.float32)
        exact = np.concatenate([z[0], z[1]]).astype(np.float64)
        rebuilt = np.concatenate([_rebuild(z[0]), _rebuild(z[1])]).astype(np.float64)
        p = np.exp2(exact - exact.max()); p /= p.sum()
        q = np.exp2(rebuilt - rebuilt.max()); q /= q.sum()
        assert np.abs(p - q).max() <= 2.0 ** -9 * p.max()


def test_masked_rows_stay_masked():
    z = np.array([1.5, -np.inf, 0.25, -np.inf], dtype=np.float32)
    zr = _rebuild(z)
    assert np.isneginf(zr[1]) and np.isneginf(zr[3])
    assert zr[0] == np.float32(1.5)
