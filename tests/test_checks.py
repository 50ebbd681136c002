"""Pins for the comparison helpers (CPU only).

The bf16 logits check accepts exactly the bf16 values that are the
round-to-nearest-even image of some value within the fp32 tolerance of the
oracle. These tests build such values with PyTorch's own bf16 cast and check
that one bf16 step further out is rejected.
"""

import numpy as np
import pytest
import torch

from tests.checks import ATOL, RTOL, assert_logits_close, bf16_rounding_interval, tol


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_rounding_interval_contains_exactly_what_rounds_to_it():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(20000) * np.exp2(rng.integers(-20, 20, 20000))).astype(np.float32)
    b = _bf16(x)
    lo, hi = bf16_rounding_interval(b)
    assert np.all(lo <= x) and np.all(x <= hi)
    # just outside the interval the value rounds elsewhere
    eps = np.abs(b) * 2.0 ** -20 + 1e-45
    assert np.all(_bf16((hi + eps).astype(np.float32)) != b)
    assert np.all(_bf16((lo - eps).astype(np.float32)) != b)
    # the half-gap is between 2^-9 and 2^-8 of |b|
    assert np.all(hi - b <= np.abs(b) * 2.0 ** -8 + 1e-45) and np.all(hi - b >= np.abs(b) * 2.0 ** -9 * 0.999)


def test_bf16_check_accepts_rounded_in_band_values_and_rejects_one_step_out():
    rng = np.random.default_rng(1)
    o = rng.standard_normal(5000) * 3
    t = tol(o)
    g = (o + rng.uniform(-1, 1, o.shape) * t).astype(np.float32)     # any fp32 result within tau
    b = _bf16(g)
    assert_logits_close(b, o, "in band", bf16=True)
    # the fp32 check without the bf16 allowance rejects some of the same values
    with pytest.raises(AssertionError):
        assert_logits_close(b, o, "no bf16 allowance")
    # one bf16 step beyond the value at the edge of the band is rejected
    edge = _bf16((o + 1.001 * t).astype(np.float32))
    lo, _ = bf16_rounding_interval(edge)
    far = np.where(lo > o + t, edge, np.nextafter(edge, np.inf))
    bits = (far.astype(np.float32).view(np.uint32) >> 16).astype(np.uint32)
    step = ((np.where(far >= 0, bits + 1, bits - 1)) << 16).view(np.float32)
    for i in range(0, 5000, 97):
        with pytest.raises(AssertionError):
            assert_logits_close(step[i:i + 1], o[i:i + 1], "one step out", bf16=True)


def test_tolerance_constants():
    assert ATOL == 1e-3 and RTOL == 2e-3
    assert tol(0.0) == ATOL and tol(-10.0) == ATOL + RTOL * 10
