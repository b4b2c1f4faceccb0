"""Pins for the oracle's slot plan, compaction and block release.

Source: ActKV analysis page (zhichai.net), system-engineering paragraph: the last X logical
blocks are the target region, retained entries outside it are paired one-to-one with holes
inside it, one parallel copy runs (so no source is also a destination), and the emptied blocks
go back to the scheduler; token eviction keeps the raw K/V unmodified ("Practical Online KV
Cache Compaction" tutorial page).  Chain Cache (SparseEngine page): the logical prefix is kept
apart from physical storage, so logical positions travel with the entries (tags).

The exhaustive test enumerates every keep mask of small segments and checks the properties the
pages fix, without restating the oracle's walk.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def make_cache(lengths, L, H, P, d, seed, extra_pages=2, starts=None):
    """A tiny cache with unique K/V bytes per slot; tags = logical positions."""
    rng = np.random.default_rng(seed)
    blocks = [-(-n // P) for n in lengths]
    num_pages = sum(blocks) + extra_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    max_blocks = max(blocks) + 1
    bt = np.full((len(lengths), max_blocks), -1, np.int32)
    it = 0
    for b, nb in enumerate(blocks):
        bt[b, :nb] = perm[it:it + nb]
        it += nb
    free_ids = np.zeros(num_pages, np.int32)
    free_ids[:num_pages - it] = perm[it:][::-1]
    free_top = np.array([num_pages - it], np.int32)
    nblocks = np.array(blocks, np.int32)
    k = rng.integers(0, 65535, size=(L, num_pages, H, P, d), dtype=np.uint16)
    v = rng.integers(0, 65535, size=(L, num_pages, H, P, d), dtype=np.uint16)
    tags = np.full((L, num_pages, H, P), -1, np.int32)
    for b, n in enumerate(lengths):
        for j in range(n):
            tags[:, bt[b, j // P], :, j % P] = j
    return dict(k=k, v=v, tags=tags, bt=bt, nblocks=nblocks, free_ids=free_ids, free_top=free_top,
                P=P, d=d, L=L, H=H)


def run_oracle(c, seg_start, seg_end, m, keep):
    k, v, tags = c["k"].copy(), c["v"].copy(), c["tags"].copy()
    bt, nbk = c["bt"].copy(), c["nblocks"].copy()
    fi, ft = c["free_ids"].copy(), c["free_top"].copy()
    oracle.compact_layers(k, v, tags, 0, c["L"], bt, seg_start, seg_end, m, keep)
    oracle.free_blocks(bt, nbk, fi, ft, c["P"], seg_start, seg_end, m)
    return dict(k=k, v=v, tags=tags, bt=bt, nblocks=nbk, free_ids=fi, free_top=ft)


def slot_loc(c, b, slot):
    return c["bt"][b, slot // c["P"]], slot % c["P"]


def test_golden_slot_plan_example():
    with open(os.path.join(GOLDEN, "slot_plan_example.json")) as f:
        g = json.load(f)
    P, n = g["P"], g["n"]
    c = make_cache([n], 1, 1, P, 4, 0)
    keep = np.array(g["keep"], np.int32).reshape(1, 1, -1)
    out = run_oracle(c, [0], [n], [len(g["keep"])], keep)
    for slot_s, tag in g["tags_after_in_target"].items():
        pg, off = slot_loc(c, 0, int(slot_s))
        assert out["tags"][0, pg, 0, off] == tag
    for src, dst in g["moves"]:
        ps, os_ = slot_loc(c, 0, src)
        pd, od = slot_loc(c, 0, dst)
        assert np.array_equal(out["k"][0, pd, 0, od], c["k"][0, ps, 0, os_])
        assert np.array_equal(out["v"][0, pd, 0, od], c["v"][0, ps, 0, os_])
    freed = [c["bt"][0, i] for i in g["freed_blocks"]]
    top0 = int(c["free_top"][0])
    assert list(out["free_ids"][top0:top0 + len(freed)]) == freed
    assert int(out["free_top"][0]) == top0 + len(freed)
    assert list(out["bt"][0, :2]) == list(c["bt"][0, 1:3])
    assert out["nblocks"][0] == 2 and out["bt"][0, 2] == -1


def check_unit_properties(c, out, b, l, h, s0, n, keep):
    """The properties the pages fix for one unit, checked from the outside."""
    P = c["P"]
    m = len(keep)
    nb = -(-n // P)
    X = -(-m // P)
    Bs = (nb - X) * P
    keep_set = set(int(x) for x in keep)
    target = range(Bs, Bs + X * P)

    def kv(cache, slot):
        pg, off = slot_loc(c, b, s0 + slot)  # physical location under the OLD block table
        return (cache["k"][l, pg, h, off].tobytes(), cache["v"][l, pg, h, off].tobytes(),
                int(cache["tags"][l, pg, h, off]))

    # slots outside the target region are byte-for-byte untouched
    for slot in range(0, Bs):
        assert kv(out, slot) == kv(c, slot)
    # retained entries inside T never move
    for slot in target:
        if slot < n and slot in keep_set:
            assert kv(out, slot) == kv(c, slot)
    # every retained entry appears exactly once among T's live slots, with its own bytes
    live = [kv(out, slot) for slot in target if kv(out, slot)[2] != -1]
    want = sorted(kv(c, j) for j in keep_set)
    assert sorted(live) == want
    # dead slots of T: X*P - m of them, bytes untouched
    dead = [slot for slot in target if kv(out, slot)[2] == -1]
    assert len(dead) == X * P - m
    for slot in dead:
        assert kv(out, slot)[:2] == kv(c, slot)[:2]
    # one parallel copy: every destination is a hole (not a retained slot), every source lies
    # before T; moved entries keep ascending order among themselves
    outside = sorted(j for j in keep_set if j < Bs)
    moved_dst = []
    for j in outside:
        hits = [slot for slot in target if kv(out, slot) == kv(c, j)]
        assert len(hits) >= 1
        dst = [s for s in hits if not (s < n and s in keep_set)]
        assert len(dst) == 1
        moved_dst.append(dst[0])
    assert moved_dst == sorted(moved_dst)
    holes = [slot for slot in target if not (slot < n and slot in keep_set)]
    assert len(outside) <= len(holes)
    # the logical view (order-preserving, out of place) equals T's live slots sorted by tag
    kc, vc, pos = oracle.logical_view(c["k"], c["v"], c["tags"], l, h, c["bt"][b], s0,
                                      np.array(sorted(keep_set), np.int32))
    live_sorted = sorted(live, key=lambda e: e[2])
    assert [e[2] for e in live_sorted] == list(pos)
    assert [e[0] for e in live_sorted] == [r.tobytes() for r in kc]
    assert [e[1] for e in live_sorted] == [r.tobytes() for r in vc]
    return nb - X


@pytest.mark.parametrize("n,P", [(8, 4), (10, 4), (11, 4), (6, 2)])
def test_exhaustive_keep_masks(n, P):
    """Every keep mask of a segment of n slots (P = 4 or 2), whole-sequence segment."""
    c = make_cache([n], 1, 1, P, 2, 7)
    for mask in range(1 << n):
        keep = [j for j in range(n) if mask >> j & 1]
        out = run_oracle(c, [0], [n], [len(keep)], np.array(keep, np.int32).reshape(1, 1, -1))
        freed = check_unit_properties(c, out, 0, 0, 0, 0, n, keep)
        top0 = int(c["free_top"][0])
        assert int(out["free_top"][0]) == top0 + freed
        assert list(out["free_ids"][top0:top0 + freed]) == list(c["bt"][0, :freed])
        nb = -(-n // P)
        assert out["nblocks"][0] == nb - freed
        assert list(out["bt"][0, :nb - freed]) == list(c["bt"][0, freed:nb])
        assert np.all(out["bt"][0, nb - freed:] == -1)


def test_exhaustive_inner_segment_multi_unit():
    """Segment in the middle of a sequence, 2 layers x 2 heads with different keep sets."""
    P, n, s0 = 4, 8, 4
    c = make_cache([20], 2, 2, P, 3, 9)
    rng = np.random.default_rng(1)
    for trial in range(200):
        m = int(rng.integers(0, n + 1))
        keep = np.stack([np.stack([np.sort(rng.choice(n, m, replace=False)) for _ in range(2)])
                         for _ in range(2)]).astype(np.int32)
        out = run_oracle(c, [s0], [s0 + n], [m], keep)
        for l in range(2):
            for h in range(2):
                freed = check_unit_properties(c, out, 0, l, h, s0, n, list(keep[l, h]))
        # blocks after the segment shift down, the first freed blocks go to the free stack
        sb = s0 // P
        assert list(out["bt"][0, :sb]) == list(c["bt"][0, :sb])
        assert list(out["bt"][0, sb:5 - freed]) == list(c["bt"][0, sb + freed:5])
        top0 = int(c["free_top"][0])
        assert list(out["free_ids"][top0:top0 + freed]) == list(c["bt"][0, sb:sb + freed])


def test_multi_sequence_free_order_and_edge_budgets():
    P = 4
    lengths = [13, 9, 16]
    c = make_cache(lengths, 1, 1, P, 2, 11)
    m = [0, 9, 5]  # m = 0 frees all; m = n frees none; partial last block
    rng = np.random.default_rng(2)
    keeps = [np.array([], np.int32), np.arange(9, dtype=np.int32),
             np.sort(rng.choice(16, 5, replace=False)).astype(np.int32)]
    keep = np.concatenate(keeps).reshape(1, 1, -1)
    out = run_oracle(c, [0, 0, 0], lengths, m, keep)
    freed = [c["bt"][0, :4].tolist(), [], c["bt"][2, :2].tolist()]
    top0 = int(c["free_top"][0])
    flat = sum(freed, [])
    assert list(out["free_ids"][top0:top0 + len(flat)]) == flat
    assert list(out["nblocks"]) == [0, 3, 2]
    for b, kp in enumerate(keeps):
        check_unit_properties(c, out, b, 0, 0, 0, lengths[b], list(kp))


def test_partial_last_block_holes_fill_past_segment_end():
    """n = 13, P = 4, keep {0, 1, 4..12}: X = 3, T = slots 4..15; the only holes are 13..15,
    past the segment end inside its last block, and they receive positions 0 and 1."""
    P, n = 4, 13
    c = make_cache([n], 1, 1, P, 2, 13)
    keep = np.array([0, 1] + list(range(4, 13)), np.int32)
    out = run_oracle(c, [0], [n], [len(keep)], keep.reshape(1, 1, -1))
    tags_T = []
    for s in range(4, 16):
        pg, off = slot_loc(c, 0, s)
        tags_T.append(int(out["tags"][0, pg, 0, off]))
    assert tags_T == list(range(4, 13)) + [0, 1, -1]
    assert int(out["nblocks"][0]) == 3


def test_rejects_unsorted_or_out_of_range_keep():
    c = make_cache([8], 1, 1, 4, 2, 17)
    with pytest.raises(RuntimeError):
        run_oracle(c, [0], [8], [2], np.array([5, 3], np.int32).reshape(1, 1, -1))
    with pytest.raises(RuntimeError):
        run_oracle(c, [0], [8], [2], np.array([3, 8], np.int32).reshape(1, 1, -1))
