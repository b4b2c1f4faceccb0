"""Pins for the oracle's ActKV scoring: action attention, action-critical entries, LRFU.

Source: "ActKV 解剖" (zhichai.net analysis of ActKV), first component: per KV entry, the
attention scores of all action tokens are gathered; entries within the top 90% are
action-critical; LRFU (the page-cache algorithm scoring entries by recency and frequency) is
driven by "hit by action attention" instead of "accessed", with decay lambda = 0.5.  LRFU's
combined recency-frequency value is sum_k F(t - t_k), F(x) = (1/2)^(lambda x) (Lee et al.):
lambda = 0 is LFU (a count of hits), large lambda approaches LRU (the last hit dominates).
"""
import numpy as np
import pytest

import oracle
from tests.test_oracle_compact import make_cache


def test_action_attention_rows_sum_to_one_each():
    rng = np.random.default_rng(1)
    for R, n in ((1, 7), (5, 40), (16, 3)):
        a, _ = oracle.action_dense(rng.standard_normal((R, 8)), rng.standard_normal((n, 8)), 0.4)
        assert abs(a.sum() - R) < 1e-12
        assert np.all(a >= 0) and np.all(a <= R)


def test_action_attention_closed_form():
    """d = 1, scale = 1, keys (0, ln 3): the row q = 1 gives alpha = (1/4, 3/4), the row q = -1
    gives (3/4, 1/4); one row alone is its alpha, both rows sum to (1, 1)."""
    K = np.array([[0.0], [np.log(3.0)]])
    a1, _ = oracle.action_dense(np.array([[1.0]]), K, 1.0)
    assert np.allclose(a1, [0.25, 0.75], rtol=0, atol=1e-15)
    a2, _ = oracle.action_dense(np.array([[1.0], [-1.0]]), K, 1.0)
    assert np.allclose(a2, [1.0, 1.0], rtol=0, atol=1e-15)


def test_action_attention_single_row_is_its_softmax():
    """R = 1: a_j = alpha_1j = exp(L_j) / sum exp(L), which is also the token-eviction score."""
    rng = np.random.default_rng(2)
    q, K = rng.standard_normal((1, 6)), rng.standard_normal((30, 6))
    a, _ = oracle.action_dense(q, K, 0.5)
    L = 0.5 * (K @ q[0])
    want = np.exp(L - L.max()) / np.exp(L - L.max()).sum()
    assert np.allclose(a, want, rtol=1e-13, atol=0)
    s, _ = oracle.score_dense(q, K, 0.5)
    assert np.allclose(a, s, rtol=1e-13, atol=0)


@pytest.mark.parametrize("a,frac,want", [
    ([0.5, 0.3, 0.15, 0.05], 0.9, [1, 1, 1, 0]),
    ([0.4, 0.25, 0.25, 0.1], 0.9, [1, 1, 1, 0]),   # boundary tie: both 0.25 kept
    ([6, 3, 3, 1, 1], 0.9, [1, 1, 1, 1, 1]),       # the crossing lands on a tie at 1
    ([0.5, 0.0, 0.5], 1.0, [1, 0, 1]),             # zero mass is never critical
    ([0.2, 0.7, 0.1], 0.5, [0, 1, 0]),
    ([0.2, 0.7, 0.1], 0.0, [0, 0, 0]),             # top 0%: nothing
    ([0.0, 0.0], 0.9, [0, 0]),
])
def test_action_hits_examples(a, frac, want):
    assert list(oracle.action_hits(np.array(a, float), frac).astype(int)) == want


def test_action_hits_characterisation():
    """For random masses the hit set is the unique set that (i) is closed upward in a, (ii)
    carries at least frac of the mass, and (iii) stops carrying it once the group of its
    smallest value is removed."""
    rng = np.random.default_rng(5)
    for trial in range(300):
        n = int(rng.integers(1, 25))
        a = rng.choice([0.0, 0.5, 1.0, 2.0, 3.0], size=n) if trial % 3 == 0 else rng.random(n) ** 3
        frac = float(rng.choice([0.5, 0.9, 0.99, 1.0]))
        hit = oracle.action_hits(a, frac)
        total = a.sum()
        if total == 0:
            assert not hit.any()
            continue
        assert hit.any()
        tau = a[hit].min()
        assert np.array_equal(hit, a >= tau)                       # (i)
        assert a[hit].sum() >= frac * total - 1e-12 * total          # (ii)
        assert a[a > tau].sum() < frac * total                       # (iii)


def lrfu_steps(hit_seq, lam):
    """Runs lrfu_cache on a one-slot unit for a sequence of hit / miss steps."""
    c = make_cache([2], 1, 1, 4, 1, seed=0)
    crf = np.zeros(c["tags"].shape, np.float64)
    out = []
    for h in hit_seq:
        # two entries; entry 0 holds all the mass when hit, none otherwise
        a = np.array([[[1.0, 0.0] if h else [0.0, 1.0]]])
        v, hits = oracle.lrfu_cache(crf, c["bt"], [0], [2], a, 0.9, lam)
        assert hits[0, 0, 0] == bool(h)
        out.append(v[0, 0, 0])
    return np.array(out)


def test_lrfu_closed_form():
    """crf after steps with hits h_k equals sum_k h_k 2^(-lambda (T - k))."""
    hist = [1, 0, 1, 1, 0, 0, 1, 0]
    for lam in (0.5, 1.0, 0.25):
        got = lrfu_steps(hist, lam)
        for T in range(1, len(hist) + 1):
            want = sum(h * 2.0 ** (-lam * (T - k)) for k, h in enumerate(hist[:T], start=1))
            assert abs(got[T - 1] - want) < 1e-13


def test_lrfu_lambda_zero_is_lfu_and_large_lambda_is_lru():
    hist = [1, 1, 1, 0, 0, 0]
    assert lrfu_steps(hist, 0.0)[-1] == 3.0                   # LFU: the hit count
    recent = lrfu_steps([0, 0, 0, 0, 0, 1], 20.0)[-1]
    frequent = lrfu_steps([1, 1, 1, 1, 1, 0], 20.0)[-1]
    assert recent > frequent                                    # LRU: the last hit wins


def test_lrfu_reads_and_writes_slots_through_the_block_table():
    """crf_out equals the per-slot state gathered through the (shuffled) block table, and
    slots outside the segments are untouched."""
    rng = np.random.default_rng(8)
    c = make_cache([37, 20], 2, 2, 8, 1, seed=3)
    crf = rng.random(c["tags"].shape)
    before = crf.copy()
    a = rng.random((2, 2, 37 + 12))
    seg_start, seg_end = [0, 8], [37, 20]
    v, hits = oracle.lrfu_cache(crf, c["bt"], seg_start, seg_end, a, 0.9, 0.5)
    touched = np.zeros(crf.shape, bool)
    off = 0
    for b in range(2):
        for j in range(seg_end[b] - seg_start[b]):
            slot = seg_start[b] + j
            pg, o = c["bt"][b, slot // 8], slot % 8
            for l in range(2):
                for h in range(2):
                    assert crf[l, pg, h, o] == v[l, h, off + j]
                    want = 2 ** -0.5 * before[l, pg, h, o] + hits[l, h, off + j]
                    assert abs(crf[l, pg, h, o] - want) < 1e-15
                    touched[l, pg, h, o] = True
        off += seg_end[b] - seg_start[b]
    assert np.array_equal(crf[~touched], before[~touched])
