"""Pins for the oracle's layout variants of eviction.

Source: "IntentKV: Cross-Turn Intent-Aware KV Cache Pruning" (gist.science summary), section on
layout-preserving eviction: an evicted position is redirected to a sentinel dead slot whose K/V
are constants that remove its attention contribution (K = -10^4, V = 0) while every surviving
row, its position and its slot identity stay unchanged; the same page objects that in-place
compaction renumbers positions.  The order-preserving compaction into fresh pages answers that
objection by moving every survivor, in logical order, into newly allocated pages (the paged
cache's free stack, as in the ActKV analysis page's "return the emptied blocks to the
scheduler").

Each property is checked from the pages' statements and from independent oracle functions
(the logical view), not by restating the oracle's loops.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_compact import make_cache


def keep_of(mask):
    return np.array([j for j, b in enumerate(mask) if b], np.int32)


def unit_keep(keeps, L, H):
    """keep array [L][H][Mtot] from per-sequence keep lists shared by every unit."""
    row = np.concatenate(keeps) if keeps else np.zeros(0, np.int32)
    return np.broadcast_to(row, (L, H, row.size)).copy().astype(np.int32)


def test_sentinel_value_is_bf16_of_minus_1e4():
    """The sentinel key element is the bf16 nearest to -10^4 (a library conversion)."""
    want = torch.tensor(-1.0e4, dtype=torch.bfloat16).view(torch.int16).item() & 0xFFFF
    assert oracle.sentinel_k_bits() == want == 0xC61C
    as_i16 = want - 0x10000 if want >= 0x8000 else want
    assert torch.tensor([as_i16], dtype=torch.int16).view(torch.bfloat16).item() == -9984.0


@pytest.mark.parametrize("n", range(1, 11))
def test_sentinel_exhaustive(n):
    """Every keep mask: retained slots and everything outside the segment keep their bytes and
    tags; every evicted slot holds K = bf16(-1e4) in all d elements, V = +0, tag -1; the block
    table and the allocator are not touched (nothing is freed)."""
    P, d, L, H = 4, 3, 1, 2
    c = make_cache([n, 5], L, H, P, d, seed=n)
    ks = oracle.sentinel_k_bits()
    for mask in itertools.product((0, 1), repeat=n):
        kp = keep_of(mask)
        keep = unit_keep([kp, np.array([1, 3], np.int32)], L, H)
        k, v, tags = c["k"].copy(), c["v"].copy(), c["tags"].copy()
        oracle.evict_sentinel(k, v, tags, 0, L, c["bt"], [0, 0], [n, 5], [len(kp), 2], keep)
        touched = np.zeros(tags.shape, bool)
        for b, (nn, kept) in enumerate(((n, set(kp.tolist())), (5, {1, 3}))):
            for j in range(nn):
                pg, off = c["bt"][b, j // P], j % P
                if j in kept:
                    continue
                touched[:, pg, :, off] = True
                assert np.all(k[:, pg, :, off] == ks)
                assert np.all(v[:, pg, :, off] == 0)
                assert np.all(tags[:, pg, :, off] == -1)
        assert np.array_equal(k[~touched], c["k"][~touched])
        assert np.array_equal(v[~touched], c["v"][~touched])
        assert np.array_equal(tags[~touched], c["tags"][~touched])


def test_sentinel_slot_carries_no_attention_mass():
    """With the sentinel key, a dead slot's softmax weight vanishes next to live keys for
    queries whose element sum is positive (the pages' intent for K = -10^4)."""
    rng = np.random.default_rng(3)
    d = 16
    q = np.abs(rng.standard_normal((4, d))) + 0.1
    K = rng.standard_normal((6, d))
    K[2] = -9984.0
    s, _ = oracle.score_dense(q, K, 1.0 / np.sqrt(d))
    assert s[2] < 1e-300 or s[2] == 0.0


def run_fresh(c, seg_start, seg_end, m, keep):
    k, v, tags = c["k"].copy(), c["v"].copy(), c["tags"].copy()
    bt, nbk = c["bt"].copy(), c["nblocks"].copy()
    fi, ft = c["free_ids"].copy(), c["free_top"].copy()
    fresh = oracle.fresh_pages(fi, int(ft[0]), c["P"], seg_start, seg_end, m)
    oracle.compact_fresh(k, v, tags, 0, c["L"], bt, seg_start, seg_end, m, keep, fresh)
    oracle.commit_fresh(bt, nbk, fi, ft, c["P"], seg_start, seg_end, m, fresh)
    return dict(k=k, v=v, tags=tags, bt=bt, nblocks=nbk, free_ids=fi, free_top=ft), fresh


@pytest.mark.parametrize("n", range(1, 11))
def test_fresh_exhaustive(n):
    """Every keep mask (m < n): walking the new block table over the first X = ceil(m/P)
    blocks of the segment gives slot r = the r-th survivor (bytes equal to the independent
    order-preserving logical view, tag = its logical position, so physical order is strictly
    monotone), slots m..X*P-1 dead; the other sequence is untouched; the pages popped are the
    stack's top X, every old page of the segment returns to the stack, and the mapped pages
    plus the free pages are every page of the pool exactly once."""
    P, d, L, H = 4, 3, 2, 1
    c = make_cache([n, 6], L, H, P, d, seed=10 + n, extra_pages=4)
    num_pages = c["k"].shape[1]
    for mask in itertools.product((0, 1), repeat=n):
        kp = keep_of(mask)
        m = [len(kp), 6]
        keep = unit_keep([kp, np.arange(6, dtype=np.int32)], L, H)
        views = [oracle.logical_view(c["k"], c["v"], c["tags"], l, 0,
                                     c["bt"][0], 0, kp) for l in range(L)]
        out, fresh = run_fresh(c, [0, 0], [n, 6], m, keep)
        if len(kp) == n:  # keeps everything: a no-op
            for key in out:
                assert np.array_equal(out[key], c[key]), key
            continue
        X = -(-len(kp) // P)
        nb = -(-n // P)
        top0 = int(c["free_top"][0])
        assert list(fresh) == list(c["free_ids"][top0 - 1 - np.arange(X)]) if X else len(fresh) == 0
        assert out["nblocks"][0] == c["nblocks"][0] - (nb - X)
        assert list(out["bt"][0, :X]) == list(fresh)
        for l in range(L):
            Kc, Vc, pos = views[l]
            for r in range(X * P):
                pg, off = out["bt"][0, r // P], r % P
                if r < len(kp):
                    assert np.array_equal(out["k"][l, pg, 0, off], Kc[r])
                    assert np.array_equal(out["v"][l, pg, 0, off], Vc[r])
                    assert out["tags"][l, pg, 0, off] == pos[r] == kp[r]
                else:
                    assert out["tags"][l, pg, 0, off] == -1
        # sequence 1 (keeps everything) keeps its row and bytes
        assert np.array_equal(out["bt"][1], c["bt"][1])
        # allocator conservation
        top = int(out["free_top"][0])
        assert top == top0 - X + nb
        assert list(out["free_ids"][top0 - X:top]) == list(c["bt"][0, :nb])
        mapped = [int(x) for b in range(2) for x in out["bt"][b, :out["nblocks"][b]]]
        free = [int(x) for x in out["free_ids"][:top]]
        assert sorted(mapped + free) == list(range(num_pages))
        assert np.all(out["bt"][0, out["nblocks"][0]:] == -1)


def test_fresh_later_blocks_shift_and_two_active_sequences():
    """Blocks after the segment shift down by nb - X; pops of every active sequence come before
    any page returns, so no sequence receives a page another one is still copying from."""
    P, d, L, H = 4, 2, 1, 1
    c = make_cache([20, 13], L, H, P, d, seed=7, extra_pages=6)
    seg_start, seg_end = [4, 0], [12, 13]
    k0 = np.array([1, 2, 6], np.int32)
    k1 = np.array([0, 5, 9, 12], np.int32)
    keep = unit_keep([k0, k1], L, H)
    out, fresh = run_fresh(c, seg_start, seg_end, [3, 4], keep)
    # sequence 0: blocks 1..2 of its row (segment) -> 1 fresh page; blocks 3, 4 shift down by 1
    assert out["bt"][0, 1] == fresh[0]
    assert list(out["bt"][0, 2:4]) == list(c["bt"][0, 3:5])
    assert out["nblocks"][0] == 4 and out["bt"][0, 4] == -1
    # sequence 1: 4 blocks -> 1 fresh page
    assert out["bt"][1, 0] == fresh[1] and out["nblocks"][1] == 1
    old_pages = set(c["bt"][0, 1:3]) | set(c["bt"][1, :4])
    assert not old_pages & set(fresh.tolist())
    for r, j in enumerate(k1):
        assert out["tags"][0, fresh[1], 0, r] == j


def test_fresh_stack_too_small_is_an_error():
    P, d = 4, 2
    c = make_cache([16], 1, 1, P, d, seed=1, extra_pages=0)
    assert int(c["free_top"][0]) == 0
    with pytest.raises(RuntimeError):
        oracle.fresh_pages(c["free_ids"], 0, P, [0], [16], [5])


def test_fresh_zero_budget_frees_every_block():
    P, d = 4, 2
    c = make_cache([10], 1, 1, P, d, seed=2, extra_pages=1)
    keep = np.zeros((1, 1, 0), np.int32)
    out, fresh = run_fresh(c, [0], [10], [0], keep)
    assert len(fresh) == 0 and out["nblocks"][0] == 0
    assert int(out["free_top"][0]) == int(c["free_top"][0]) + 3
