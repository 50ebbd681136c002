"""Comparison helpers shared by the parity tests and the smoke entry point.

Tolerances are the ones the problem statement fixes for floating-point logits:
``|gpu - oracle| <= 1e-3 + 2e-3 * |oracle|``. Top-k index sets must be exact
except where oracle values tie within that tolerance at the k-th value.
"""

from __future__ import annotations

import numpy as np

ATOL = 1e-3
RTOL = 2e-3


# A bf16 output carries its own rounding on top of the kernel's arithmetic:
# |bf16(x) - x| <= 2^-9 |x|; the check widens the relative term by 2^-8 for it.
BF16_REL = 2.0 ** -8


def tol(x, rel_extra: float = 0.0):
    return ATOL + (RTOL + rel_extra) * np.abs(x)


def assert_logits_close(got, ref, what: str = "logits", rel_extra: float = 0.0) -> None:
    """Finite oracle entries within tolerance; -inf entries exactly -inf."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf), f"{what}: -inf pattern differs " \
        f"({int(np.sum(np.isneginf(got) != ninf))} entries)"
    fin = ~ninf
    err = np.abs(got[fin] - ref[fin])
    bad = err > tol(ref[fin], rel_extra)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {int(fin.sum())} entries out of tolerance, "
                           f"worst abs err {err.max():.3e}")


def assert_topk_row(sel, ref_values, k: int, what: str = "topk", rel_extra: float = 0.0) -> None:
    """Tie-tolerant check of one row of request-local indices.

    ``ref_values``: oracle scores of the row's visible columns (index i = column ks + i).
    Requires exactly min(k, n) unique valid indices followed by -1, every oracle
    index clearly above the k-th value selected, and no selected index clearly below it.
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
    t = tol(vk, rel_extra)
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
