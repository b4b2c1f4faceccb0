"""Pins for the oracle's budget rules and top-m selection.

Sources: "Practical Online KV Cache Compaction for LLM Agents" (tutorial page): keep the top-m
positions by s_j; keep ratio 0.2 (drop 80%).  ActKV analysis page, budget paragraph: initial
budget 512 entries, x1.75 per growth step, cap 30 000, never shrinks.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle


def brute_force_keep(s, m):
    """The unique S, |S| = m, with: for j in S and k not in S, s_j > s_k or (s_j == s_k and j < k)."""
    n = len(s)
    found = []
    for S in itertools.combinations(range(n), m):
        inside = set(S)
        ok = all(s[j] > s[k] or (s[j] == s[k] and j < k)
                 for j in inside for k in range(n) if k not in inside)
        if ok:
            found.append(S)
    assert len(found) == 1, "the tie-break makes the keep set unique"
    return list(found[0])


@pytest.mark.parametrize("seed", range(6))
def test_select_matches_brute_force_over_all_subsets(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 13))
    # coarse values force many ties
    s = rng.integers(0, 5, size=n).astype(float) / 4.0
    for m in range(0, n + 1):
        got = oracle.select(s, m)
        assert list(got) == brute_force_keep(list(s), m), (s, m)


def test_select_continuous_scores_brute_force():
    rng = np.random.default_rng(99)
    s = rng.random(14)
    for m in (0, 1, 5, 13, 14):
        assert list(oracle.select(s, m)) == brute_force_keep(list(s), m)


def test_identical_scores_keep_lowest_positions():
    assert list(oracle.select(np.full(20, 0.05), 7)) == list(range(7))


def test_keep_is_ascending_and_clamped():
    rng = np.random.default_rng(3)
    s = rng.random(50)
    k = oracle.select(s, 20)
    assert np.all(np.diff(k) > 0)
    assert len(oracle.select(s, 80)) == 50
    assert len(oracle.select(s, 0)) == 0


def test_select_rejects_nonfinite():
    s = np.array([0.1, np.nan, 0.3])
    with pytest.raises(RuntimeError):
        oracle.select(s, 1)


def test_ratio_budget_values():
    # ceil(0.2 n), exact rational arithmetic
    for n in (1, 5, 12, 100, 512, 1536, 8192, 32768, 131072, 99991):
        want = min(n, -(-Fraction(n) * Fraction(1, 5) // 1))
        assert oracle.budget_ratio(n, 0.2) == want
    assert oracle.budget_ratio(512, 0.2) == 103          # the tiny workload's m
    assert oracle.budget_ratio(1536, 0.2) == 308
    assert oracle.budget_ratio(32768, 0.2) == 6554
    assert oracle.budget_ratio(131072, 0.2) == 26215
    assert oracle.budget_ratio(100, 0.07) == 7           # 0.07*100 = 7.000000000000001 in fp64
    assert oracle.budget_ratio(10, 1.5) == 10
    assert oracle.budget_ratio(10, -0.5) == 0
    assert oracle.budget_ratio(0, 0.2) == 0


def test_actkv_budget_values():
    # floor(512 * (7/4)^k), capped at 30000 -- exact rationals
    for k in range(12):
        want = min(30000, int(Fraction(512) * Fraction(7, 4) ** k))
        assert oracle.budget_actkv(k) == want
    assert [oracle.budget_actkv(k) for k in range(7)] == [512, 896, 1568, 2744, 4802, 8403, 14706]
    # monotone (the ratchet never shrinks) and capped
    vals = [oracle.budget_actkv(k) for k in range(20)]
    assert all(a <= b for a, b in zip(vals, vals[1:])) and vals[-1] == 30000


def test_select_cache_offsets():
    """Ragged sequences: keep [L][H][Mtot] with sequence b at offset sum of earlier min(m, n)."""
    rng = np.random.default_rng(5)
    n = [7, 3, 10]
    m = [2, 5, 0]
    L, H = 2, 3
    scores = rng.random((L, H, sum(n)))
    keep = oracle.select_cache(scores, [0, 0, 0], n, m)
    assert keep.shape == (L, H, 2 + 3 + 0)
    for l in range(L):
        for h in range(H):
            assert list(keep[l, h, :2]) == brute_force_keep(list(scores[l, h, :7]), 2)
            assert list(keep[l, h, 2:5]) == [0, 1, 2]
