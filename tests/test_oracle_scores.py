"""Pins for the oracle's scores (token-eviction attention-mass score, LSE recovery).

Source: "Practical Online KV Cache Compaction for LLM Agents" (tutorial page), design-space
section: s_j(Q,K) = ((1/q) sum_i alpha_ij^2)^(1/2); ActKV analysis page, system-engineering
paragraph: alpha = exp(logits - LSE).  None of these tests re-implements the oracle's
formula: they check closed forms, invariants and library special cases.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def test_closed_form_two_rows_two_keys():
    """d=1, scale=1, rows (1), (-1), keys (0), (ln 3): alpha rows (1/4, 3/4), (3/4, 1/4)."""
    with open(os.path.join(GOLDEN, "score_closed_form.json")) as f:
        g = json.load(f)
    Q = np.array(g["Q"], float)
    K = np.array([[0.0], [math.log(3.0)]])
    s, lse = oracle.score_dense(Q, K, g["scale"])
    np.testing.assert_allclose(s, [math.sqrt(5 / 16)] * 2, rtol=1e-14)
    np.testing.assert_allclose(lse, [math.log(4.0), math.log(4.0 / 3.0)], rtol=1e-14)
    assert s[0] == pytest.approx(s[1], rel=1e-15)  # an exact tie


def test_single_row_is_softmax():
    """q = 1 proxy row: s_j = alpha_1j (the softmax of the scaled logits)."""
    Q = rand((1, 16), 1)
    K = rand((37, 16), 2)
    scale = 0.25
    s, lse = oracle.score_dense(Q, K, scale)
    logits = scale * (K @ Q[0])
    np.testing.assert_allclose(s, scipy.special.softmax(logits), rtol=1e-12)
    np.testing.assert_allclose(lse[0], scipy.special.logsumexp(logits), rtol=1e-13)


def test_rows_sum_to_one_via_lse():
    """exp(L_ij - LSE_i) is a probability row: sums to 1 for every proxy row."""
    Q = rand((9, 8), 3, 2.0)
    K = rand((50, 8), 4, 2.0)
    scale = 1 / math.sqrt(8)
    s, lse = oracle.score_dense(Q, K, scale)
    L = scale * Q @ K.T
    np.testing.assert_allclose(np.exp(L - lse[:, None]).sum(1), 1.0, atol=1e-12)


def test_mean_of_squares_over_rows():
    """Two independent rows: s^2 is the mean of the two single-row s^2 (the 1/q average)."""
    K = rand((23, 4), 5)
    q1, q2 = rand((1, 4), 6), rand((1, 4), 7)
    s1, _ = oracle.score_dense(q1, K, 0.7)
    s2, _ = oracle.score_dense(q2, K, 0.7)
    s12, _ = oracle.score_dense(np.vstack([q1, q2]), K, 0.7)
    np.testing.assert_allclose(s12 ** 2, (s1 ** 2 + s2 ** 2) / 2, rtol=1e-12)


def test_duplicate_rows_invariant():
    Q = rand((5, 8), 8)
    K = rand((40, 8), 9)
    s, _ = oracle.score_dense(Q, K, 0.3)
    s2, _ = oracle.score_dense(np.vstack([Q, Q, Q]), K, 0.3)
    np.testing.assert_allclose(s2, s, rtol=1e-13)


def test_key_shift_invariance():
    """K_j += v for all j adds a per-row constant to the logits: alpha and s unchanged."""
    Q = rand((6, 8), 10)
    K = rand((31, 8), 11)
    v = rand((8,), 12, 3.0)
    s, lse = oracle.score_dense(Q, K, 0.4)
    s2, lse2 = oracle.score_dense(Q, K + v, 0.4)
    np.testing.assert_allclose(s2, s, rtol=1e-11)
    np.testing.assert_allclose(lse2 - lse, 0.4 * Q @ v, rtol=1e-11, atol=1e-11)


def test_key_permutation_equivariance():
    Q = rand((4, 8), 13)
    K = rand((29, 8), 14)
    perm = np.random.default_rng(15).permutation(29)
    s, lse = oracle.score_dense(Q, K, 0.5)
    sp, lsep = oracle.score_dense(Q, K[perm], 0.5)
    np.testing.assert_allclose(sp, s[perm], rtol=1e-13)
    np.testing.assert_allclose(lsep, lse, rtol=1e-13)


def test_zero_queries_and_identical_keys_are_uniform():
    n = 17
    s, lse = oracle.score_dense(np.zeros((3, 8)), rand((n, 8), 16), 1.0)
    np.testing.assert_allclose(s, 1.0 / n, rtol=1e-14)
    np.testing.assert_allclose(lse, math.log(n), rtol=1e-14)
    Kid = np.tile(rand((1, 8), 17), (n, 1))
    s, _ = oracle.score_dense(rand((5, 8), 18), Kid, 1.0)
    np.testing.assert_allclose(s, 1.0 / n, rtol=1e-13)


def test_sum_of_squares_bounds():
    """sum_j s_j^2 = mean_i sum_j alpha_ij^2, which lies in [1/n, 1]."""
    for seed in range(5):
        n = 10 + seed * 7
        s, _ = oracle.score_dense(rand((4, 6), 100 + seed, 3.0), rand((n, 6), 200 + seed, 3.0), 1.0)
        tot = float((s ** 2).sum())
        assert 1.0 / n - 1e-12 <= tot <= 1.0 + 1e-12
        assert np.all(s >= 0) and np.all(s <= 1.0 + 1e-15)


def test_scale_enters_logits():
    """scale multiplies the logits: scale 2 on K equals scale 1 on 2K."""
    Q = rand((3, 5), 19)
    K = rand((12, 5), 20)
    s1, l1 = oracle.score_dense(Q, K, 2.0)
    s2, l2 = oracle.score_dense(Q, 2 * K, 1.0)
    np.testing.assert_allclose(s1, s2, rtol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13)


def test_one_dominant_key():
    """A key with a huge logit for every row takes alpha ~ 1: s ~ 1 there, ~0 elsewhere."""
    K = rand((20, 4), 21)
    Q = np.abs(rand((6, 4), 22)) + 0.5  # every row has positive entries
    K[7] = 30.0  # logit >= 60 above the others' typical scale for every row
    s, _ = oracle.score_dense(Q, K, 1.0)
    assert s[7] > 0.999
    assert np.argmax(s) == 7


def test_nonfinite_rejected():
    Q = rand((2, 4), 23)
    K = rand((5, 4), 24)
    K[2, 1] = np.inf
    with pytest.raises(RuntimeError):
        oracle.score_dense(Q, K, 1.0)


def _paged_cache(n_list, L, H, P, d, seed, shuffle=True):
    """Tiny paged cache whose token keys are known: token j of sequence b, layer l, head h has key
    Ktrue[b][l][h][j], written through an explicit block table (independent of the oracle)."""
    rng = np.random.default_rng(seed)
    blocks = [-(-n // P) for n in n_list]
    num_pages = sum(blocks) + 3
    pages = rng.permutation(num_pages) if shuffle else np.arange(num_pages)
    max_blocks = max(blocks)
    bt = np.full((len(n_list), max_blocks), -1, np.int32)
    pool = rng.standard_normal((L, num_pages, H, P, d)).astype(np.float32)
    Ktrue = []
    it = 0
    for b, n in enumerate(n_list):
        bt[b, :blocks[b]] = pages[it:it + blocks[b]]
        it += blocks[b]
        kt = rng.standard_normal((L, H, n, d)).astype(np.float32)
        kt = (kt.view(np.uint32) & 0xFFFF0000).view(np.float32)  # exactly bf16-representable
        for j in range(n):
            pool[:, bt[b, j // P], :, j % P, :] = kt[:, :, j, :]
        Ktrue.append(kt)
    bits = (pool.view(np.uint32) >> 16).astype(np.uint16)
    return bits, bt, Ktrue, num_pages


def test_score_cache_gathers_through_block_table():
    n_list = [13, 40, 8]
    L, H, P, d, R = 2, 2, 4, 8, 3
    bits, bt, Ktrue, _ = _paged_cache(n_list, L, H, P, d, 31)
    rng = np.random.default_rng(32)
    qf = rng.standard_normal((len(n_list), L, H, R, d)).astype(np.float32)
    qf = (qf.view(np.uint32) & 0xFFFF0000).view(np.float32)
    qbits = (qf.view(np.uint32) >> 16).astype(np.uint16)
    s0 = np.zeros(3, np.int32)
    s1 = np.array(n_list, np.int32)
    nbk = np.array([-(-n // P) for n in n_list], np.int32)
    scores, lse = oracle.score_cache(bits, bt, nbk, s0, s1, s1, qbits, 0.5)
    off = np.concatenate([[0], np.cumsum(n_list)])
    for b in range(3):
        for l in range(L):
            for h in range(H):
                s, ls = oracle.score_dense(qf[b, l, h].astype(float), Ktrue[b][l, h].astype(float), 0.5)
                np.testing.assert_allclose(scores[l, h, off[b]:off[b + 1]], s, rtol=1e-14)
                np.testing.assert_allclose(lse[b, l, h], ls, rtol=1e-14)


def test_score_cache_segment_offset_and_mask():
    """A segment starting at a block boundary scores only its own keys; masked units untouched."""
    L, H, P, d, R = 1, 2, 4, 8, 2
    bits, bt, Ktrue, _ = _paged_cache([24], L, H, P, d, 41)
    rng = np.random.default_rng(42)
    qf = rng.standard_normal((1, L, H, R, d)).astype(np.float32)
    qf = (qf.view(np.uint32) & 0xFFFF0000).view(np.float32)
    qbits = (qf.view(np.uint32) >> 16).astype(np.uint16)
    nbk = np.array([6], np.int32)
    mask = np.array([[[True, False]]])
    scores, _ = oracle.score_cache(bits, bt, nbk, [8], [20], [24], qbits, 1.0, unit_mask=mask)
    s, _ = oracle.score_dense(qf[0, 0, 0].astype(float), Ktrue[0][0, 0, 8:20].astype(float), 1.0)
    np.testing.assert_allclose(scores[0, 0], s, rtol=1e-14)
    assert np.all(np.isnan(scores[0, 1]))


@pytest.mark.parametrize("s0,s1,seq_len", [(2, 12, 24), (4, 13, 24), (0, 25, 24)])
def test_score_cache_rejects_bad_segments(s0, s1, seq_len):
    bits, bt, _, _ = _paged_cache([24], 1, 1, 4, 8, 51)
    q = np.zeros((1, 1, 1, 1, 8), np.uint16)
    with pytest.raises(RuntimeError):
        oracle.score_cache(bits, bt, np.array([6], np.int32), [s0], [s1], [seq_len], q, 1.0)
