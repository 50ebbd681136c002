"""Comparison helpers shared by the parity tests and the smoke entry point.

Tolerances are the ones the problem statement fixes for floating-point logits:
``|gpu - oracle| <= 1e-3 + 2e-3 * |oracle|``. Top-k index sets must be exact
except where oracle values tie within that tolerance at the k-th value.

bf16 outputs. A kernel that writes bf16 computes an fp32 value ``g`` and stores
it rounded to nearest even once. The check for such an output ``b`` is exact:
``b`` must be the rounding of SOME value within the fp32 tolerance of the
oracle, i.e. the interval of reals that round to ``b`` must meet
``[o - tau(o), o + tau(o)]``. That interval is ``b`` plus or minus half the gap
to each bf16 neighbour, so the allowance is the actual local half ulp (between
2^-9 and 2^-8 of |b|), never a blanket relative term.

For the tie band of the top-k check an additive bound is needed instead. With
an 8-bit significand the rounding error of one store is at most 2^-8 of the
stored magnitude (1 + 2^-8 rounds to 1), so
``|b - o| <= tau(o) + 2^-8 (|o| + tau(o))``.
"""

from __future__ import annotations

import numpy as np

ATOL = 1e-3
RTOL = 2e-3

# worst-case relative rounding error of one round-to-nearest bf16 store
BF16_UNIT_ROUNDOFF = 2.0 ** -8


def tol(x, bf16: bool = False):
    """The fp32 tolerance tau(x); with ``bf16`` the additive bound of one bf16 store on top."""
    t = ATOL + RTOL * np.abs(x)
    if bf16:
        t = (1.0 + BF16_UNIT_ROUNDOFF) * t + BF16_UNIT_ROUNDOFF * np.abs(x)
    return t


def bf16_rounding_interval(b):
    """[lo, hi]: the reals whose round-to-nearest-even bf16 value is ``b`` (closed at both ends).

    ``b`` holds finite values exactly representable in bf16. The neighbours are
    the adjacent bf16 bit patterns; the interval runs halfway to each of them.
    Including both tie points makes the check at most one tie point looser.
    """
    b = np.asarray(b, dtype=np.float32)
    bits = (b.view(np.uint32) >> 16).astype(np.int64)
    mag = bits & 0x7FFF
    sign = np.where(bits & 0x8000, -1.0, 1.0)

    def val(m):
        return (np.asarray(m, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)

    up = val(np.minimum(mag + 1, 0x7F80))       # next larger magnitude (+inf past the largest)
    down = np.where(mag > 0, val(np.maximum(mag - 1, 0)), -val(1))  # below zero: the -smallest
    m = val(mag)
    hi_mag = np.where(np.isinf(up), np.inf, (m + up) / 2)
    lo_mag = (m + down) / 2
    lo = np.where(sign > 0, lo_mag, -hi_mag)
    hi = np.where(sign > 0, hi_mag, -lo_mag)
    return lo, hi


def assert_logits_close(got, ref, what: str = "logits", bf16: bool = False) -> None:
    """Finite oracle entries within tolerance; -inf entries exactly -inf.

    ``bf16``: ``got`` was stored as bf16; each entry must be the rounding of a
    value within tau of the oracle (see the module docstring).
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf), f"{what}: -inf pattern differs " \
        f"({int(np.sum(np.isneginf(got) != ninf))} entries)"
    fin = ~ninf
    g, o = got[fin], ref[fin]
    t = tol(o)
    if bf16:
        assert np.all(np.isfinite(g)), f"{what}: non-finite bf16 output"
        lo, hi = bf16_rounding_interval(g)
        bad = (lo > o + t) | (hi < o - t)
        err = np.maximum(lo - (o + t), (o - t) - hi)
    else:
        err = np.abs(g - o)
        bad = err > t
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {int(fin.sum())} entries out of tolerance, "
                           f"worst excess {float(np.max(err - (0 if bf16 else t))):.3e}")


def assert_topk_row(sel, ref_values, k: int, what: str = "topk", bf16: bool = False) -> None:
    """Tie-tolerant check of one row of request-local indices.

    ``ref_values``: oracle scores of the row's visible columns (index i = column ks + i).
    Requires exactly min(k, n) unique valid indices followed by -1, every oracle
    index clearly above the k-th value selected, and no selected index clearly below it.
    ``bf16``: the selection ran on bf16 scores, so the tie band includes one store's rounding.
    """
    sel = np.asarray(sel, dtype=np.int64)
    ref_values = np.asarray(ref_values, dtype=np.float64)
    n = len(ref_values)
    m = min(k, n)
    assert len(sel) >= k
    valid = sel[:k]
    assert np.all(valid[:m] >= 0) and np.all(valid[:m] < n), f"{what}: index out of range"
    assert np.all(valid[m:] == -1), f"{what}: tail is not -1"
    chosen = valid[:m]
    assert len(np.unique(chosen)) == m, f"{what}: duplicate indices"
    if n <= k:
        assert np.array_equal(chosen, np.arange(n)), f"{what}: all-visible row must list 0..n-1"
        return
    vk = np.sort(ref_values)[::-1][k - 1]
    t = tol(vk, bf16)
    must = np.nonzero(ref_values > vk + t)[0]
    missing = np.setdiff1d(must, chosen)
    assert missing.size == 0, f"{what}: {missing.size} clearly-larger indices not selected"
    assert np.all(ref_values[chosen] >= vk - t), f"{what}: selected an index clearly below the threshold"


def assert_topk_values_exact(sel, values, k: int, what: str = "topk") -> None:
    """When ``values`` are the exact selection input: the chosen values are the top-k multiset."""
    sel = np.asarray(sel, dtype=np.int64)
    values = np.asarray(values)
    n = len(values)
    m = min(k, n)
    chosen = sel[:m]
    assert np.all(sel[m:k] == -1)
    assert len(np.unique(chosen)) == m and np.all((chosen >= 0) & (chosen < n)), what
    want = np.sort(values.astype(np.float64))[::-1][:m]
    got = np.sort(values[chosen].astype(np.float64))[::-1]
    assert np.array_equal(got, want), f"{what}: selected values differ from the top-{k} values"
