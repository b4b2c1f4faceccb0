"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded
inputs.  Scores, LSE and keep sets follow the rules in tests/parity.py; compaction is checked
bit-exact given a selection that comes from the oracle or from the seeded generator (never from
the CUDA path)."""
import numpy as np
import pytest
import torch

import oracle
import online_kv_cache_gb300 as kvc
import workloads
from tests import parity as PT

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from online_kv_cache_gb300 import build
    build.build()
    kvc.kvc_read_device_status(clear=True)


def full_check(case, label, check_lse=True):
    """Score + select against the oracle on every unit, then compaction bit-exact given the
    oracle's keep sets.  Returns (max score error, in-band selection differences)."""
    m_orc = PT.oracle_budgets(case)
    m_lib = PT.lib_budgets(case)
    assert m_orc == m_lib, "budget helpers disagree"
    pristine = PT.host_state(case)
    snap = case.snapshot()
    s_orc, lse_orc = PT.oracle_scores(case)
    keep_orc = oracle.select_cache(s_orc, case.seg_start, case.seg_end, m_orc)

    cp = PT.compactor(case, m_lib)
    cp.score(case.q, case.spec.scale, True)
    cp.select()
    torch.cuda.synchronize()
    s_gpu = cp.scores.cpu().numpy()[:, :, :cp.Ntot]
    k_gpu = cp.keep.cpu().numpy()[:, :, :cp.Mtot]
    worst = PT.check_scores(s_gpu, s_orc, label)
    if check_lse:
        lse_gpu = cp.lse.cpu().numpy()
        for b in range(case.spec.B):
            if case.seg_end[b] > case.seg_start[b]:
                PT.check_lse(lse_gpu[b], lse_orc[b], f"{label} lse b={b}")
    diffs = 0
    L, H = case.spec.L, case.spec.H
    noff, moff = PT.unit_offsets(case, m_orc)
    for l in range(L):
        for h in range(H):
            for b in range(case.spec.B):
                diffs += PT.check_keep(k_gpu[l, h, moff[b]:moff[b + 1]], keep_orc[l, h, moff[b]:moff[b + 1]],
                                       s_orc[l, h, noff[b]:noff[b + 1]], int(moff[b + 1] - moff[b]),
                                       f"{label} l={l} h={h} b={b}")
    # compaction given the oracle's selection
    keep_dev = torch.from_numpy(np.ascontiguousarray(keep_orc)).to(DEV)
    cp.plan_compact(keep_dev if keep_orc.size else None)
    cp.compact()
    cp.free_pages()
    torch.cuda.synchronize()
    PT.device_status_clean()
    PT.assert_state_equal(PT.host_state(case), PT.oracle_compaction(pristine, case, m_orc, keep_orc),
                          label)
    # the chain on the GPU's own selection, when it equals the oracle's, gives the same bytes
    if diffs == 0:
        case.restore(snap)
        PT.run_chain(case, m_lib)
        torch.cuda.synchronize()
        PT.device_status_clean()
        PT.assert_state_equal(PT.host_state(case),
                              PT.oracle_compaction(PT.host_state_from(snap), case, m_orc, keep_orc),
                              label + " (own selection)")
    return worst, diffs


def test_tiny_workload():
    case = workloads.build(workloads.spec("tiny"), 0, DEV)
    planted = case.planted[0].cpu().numpy()  # [L][H][4] segment positions
    m = PT.lib_budgets(case)
    assert m == [103]
    cp = PT.compactor(case, m)
    cp.score(case.q, case.spec.scale)
    cp.select()
    torch.cuda.synchronize()
    keep = cp.keep.cpu().numpy()
    for h in range(case.spec.H):
        assert set(planted[0, h].tolist()) <= set(keep[0, h].tolist()), "planted keys must survive"
    case2 = workloads.build(workloads.spec("tiny"), 0, DEV)
    worst, diffs = full_check(case2, "tiny")
    assert diffs == 0


MICRO = [
    # d, P, G, q, lengths, budget
    (64, 16, 2, 8, (512,), ("ratio", 0.2)),
    (128, 16, 8, 16, (1, 15, 16, 17, 32, 129), ("ratio", 0.2)),
    (128, 8, 4, 1, (7, 8, 9, 300), ("ratio", 0.5)),
    (64, 32, 1, 1, (4097,), ("ratio", 0.2)),
    (128, 64, 4, 25, (200, 1000), ("ratio", 0.1)),
    (128, 16, 8, 64, (2048, 777), ("ratio", 0.2)),          # R = 512: two pass-2 chunks
    (64, 16, 4, 75, (640,), ("ratio", 0.3)),                # R = 300: padded rows
    (128, 32, 16, 256, (1536,), ("ratio", 0.2)),            # R = 4096
    (128, 16, 8, 16, (5000, 3000, 9000), ("actkv", (0, 1, 2))),
]


@pytest.mark.parametrize("d,P,G,q,lengths,budget", MICRO)
def test_micro_shapes(d, P, G, q, lengths, budget):
    sp = workloads.custom(L=2, H=2, G=G, d=d, P=P, q=q, lengths=lengths, budget=budget,
                          shuffle_pages=True)
    case = workloads.build(sp, 1, DEV)
    full_check(case, f"micro d={d} P={P} R={sp.R} n={lengths}")


@pytest.mark.parametrize("grid", ["3", "1"])
@pytest.mark.parametrize("shape", [(128, 16, 8, 64, (2048, 1500, 700)), (64, 32, 4, 8, (3000, 130)),
                                   (128, 16, 16, 128, (900,))])
def test_many_items_per_cta(monkeypatch, grid, shape):
    """A persistent grid of 1 or 3 CTAs walks every work item: rings and Q sub-tile barriers wrap
    many times, items of different lengths and row groups follow each other."""
    d, P, G, q, lengths = shape
    monkeypatch.setenv("KVC_GRID_LIMIT", grid)
    sp = workloads.custom(L=2, H=2, G=G, d=d, P=P, q=q, lengths=lengths, shuffle_pages=True)
    case = workloads.build(sp, 7, DEV)
    full_check(case, f"grid={grid} d={d} R={sp.R} n={lengths}")


@pytest.mark.parametrize("mode", ["zero", "one", "n-1", "all"])
def test_edge_budgets(mode):
    sp = workloads.custom(L=1, H=2, G=4, d=128, P=16, q=8, lengths=(100, 47, 16), shuffle_pages=True)
    case = workloads.build(sp, 2, DEV)
    n = PT.seg_lengths(case)
    m = {"zero": [0] * 3, "one": [1] * 3, "n-1": [x - 1 for x in n], "all": n}[mode]
    pristine = PT.host_state(case)
    s_orc, _ = PT.oracle_scores(case)
    keep_orc = oracle.select_cache(s_orc, case.seg_start, case.seg_end, m)
    cp = PT.compactor(case, m)
    cp.score(case.q, sp.scale)
    cp.select()
    torch.cuda.synchronize()
    k_gpu = cp.keep.cpu().numpy()[:, :, :cp.Mtot]
    noff, moff = PT.unit_offsets(case, m)
    for l in range(sp.L):
        for h in range(sp.H):
            for b in range(sp.B):
                PT.check_keep(k_gpu[l, h, moff[b]:moff[b + 1]], keep_orc[l, h, moff[b]:moff[b + 1]],
                              s_orc[l, h, noff[b]:noff[b + 1]], int(moff[b + 1] - moff[b]), mode)
    keep_dev = torch.from_numpy(np.ascontiguousarray(keep_orc)).to(DEV) if keep_orc.size else None
    cp.plan_compact(keep_dev)
    cp.compact()
    cp.free_pages()
    torch.cuda.synchronize()
    PT.device_status_clean()
    PT.assert_state_equal(PT.host_state(case), PT.oracle_compaction(pristine, case, m, keep_orc), mode)


def test_segments_inside_sequences():
    """Segments that start past slot 0 and end before the sequence end; a sequence with no
    segment; a segment ending at a ragged sequence end."""
    sp = workloads.custom(L=2, H=2, G=4, d=128, P=16, q=8, lengths=(1000, 333, 520),
                          shuffle_pages=True)
    case = workloads.build(sp, 3, DEV, with_q=False)
    case.seg_start = [160, 0, 96]
    case.seg_end = [800, 0, 520]
    workloads.make_q(case, 3)
    full_check(case, "inner segments")


def test_given_selection_random_keeps():
    """Compaction alone, bit-exact, for seeded random keep sets (any selection)."""
    sp = workloads.custom(L=3, H=2, G=2, d=64, P=8, q=2, lengths=(257, 64, 1023, 8),
                          shuffle_pages=True)
    case = workloads.build(sp, 4, DEV)
    for trial, ratio in enumerate((0.0, 0.05, 0.2, 0.6, 1.0)):
        m = [oracle.budget_ratio(x, ratio) for x in PT.seg_lengths(case)]
        snap = case.snapshot()
        pristine = PT.host_state(case)
        keep = workloads.random_keep(case, m, 100 + trial)
        cp = PT.compactor(case, m)
        cp.plan_compact(keep.contiguous() if keep.numel() else None)
        cp.compact()
        cp.free_pages()
        torch.cuda.synchronize()
        PT.device_status_clean()
        PT.assert_state_equal(PT.host_state(case),
                              PT.oracle_compaction(pristine, case, m, keep.cpu().numpy()),
                              f"random keep ratio={ratio}")
        case.restore(snap)


def test_logical_view_after_compaction():
    """T's live slots gathered by ascending tag reproduce the oracle's order-preserving view."""
    sp = workloads.custom(L=2, H=2, G=4, d=128, P=16, q=8, lengths=(700, 260), shuffle_pages=True)
    case = workloads.build(sp, 5, DEV)
    m = PT.lib_budgets(case)
    pristine = PT.host_state(case)
    cp = PT.run_chain(case, m)
    torch.cuda.synchronize()
    keep = cp.keep.cpu().numpy()[:, :, :cp.Mtot]
    after = PT.host_state(case)
    moff = np.concatenate([[0], np.cumsum(m)])
    P = sp.P
    for l in range(sp.L):
        for h in range(sp.H):
            for b in range(sp.B):
                kb = keep[l, h, moff[b]:moff[b + 1]]
                Kc, Vc, pos = oracle.logical_view(pristine["k"], pristine["v"], pristine["tags"], l, h,
                                                  pristine["bt"][b], case.seg_start[b], kb)
                n = case.seg_end[b] - case.seg_start[b]
                nb, X = -(-n // P), -(-len(kb) // P)
                row = after["bt"][b]
                slots = [(row[blk] , off) for blk in range(X) for off in range(P)]  # new rows: T first
                live = [(after["tags"][l, pg, h, off], after["k"][l, pg, h, off], after["v"][l, pg, h, off])
                        for pg, off in slots if after["tags"][l, pg, h, off] >= 0]
                live.sort(key=lambda e: e[0])
                assert [e[0] for e in live] == list(pos)
                assert np.array_equal(np.array([e[1] for e in live]).reshape(Kc.shape), Kc)
                assert np.array_equal(np.array([e[2] for e in live]).reshape(Vc.shape), Vc)


@pytest.mark.parametrize("d,R", [(128, 128), (128, 512), (64, 256)])
def test_rising_logits(d, R):
    """Key norms grow along the sequence (x1 at slot 0 to x24 at the end), so each row's
    largest logits sit in the last tiles, far above every earlier tile: the LSE pass
    must move its running reference up mid-item without overflowing or losing mass."""
    sp = workloads.custom(L=1, H=2, G=4, d=d, P=16, q=R // 4, lengths=(3000, 1300),
                          budget=("ratio", 0.2), shuffle_pages=True)
    case = workloads.build(sp, 7, DEV)
    P = sp.P
    for b, n in enumerate(sp.lengths):
        slots = torch.arange(n, device=DEV)
        pages = case.block_table[b].long()[slots // P]
        grow = (1.0 + 23.0 * slots.float() / max(1, n - 1)).view(-1, 1, 1, 1)
        view = case.k_pool.permute(1, 3, 0, 2, 4)
        view[pages, slots % P] = (view[pages, slots % P].float() * grow).to(torch.bfloat16)
    full_check(case, f"rising logits d={d} R={R}")


@pytest.mark.parametrize("distinct", [1, 3])
def test_exact_ties_keep_lowest_positions(distinct):
    """Keys drawn from `distinct` vectors: scores tie exactly on both sides, and the lower
    position wins, so the GPU keep sets equal the oracle's exactly."""
    sp = workloads.custom(L=1, H=2, G=4, d=128, P=16, q=8, lengths=(1000, 4096), shuffle_pages=True)
    case = workloads.build(sp, 9, DEV, with_q=False)
    g = torch.Generator(device=DEV)
    g.manual_seed(123)
    basis = torch.randn((distinct, sp.d), generator=g, device=DEV).to(torch.bfloat16)
    pick = torch.randint(0, distinct, case.k_pool.shape[:-1], generator=g, device=DEV)
    case.k_pool.copy_(basis[pick])
    workloads.make_q(case, 9)
    m = PT.lib_budgets(case)
    s_orc, _ = PT.oracle_scores(case)
    keep_orc = oracle.select_cache(s_orc, case.seg_start, case.seg_end, m)
    cp = PT.compactor(case, m)
    cp.score(case.q, sp.scale)
    cp.select()
    torch.cuda.synchronize()
    k_gpu = cp.keep.cpu().numpy()[:, :, :cp.Mtot]
    assert np.array_equal(k_gpu, keep_orc)
    if distinct == 1:
        noff, moff = PT.unit_offsets(case, m)
        for b in range(sp.B):
            assert np.array_equal(k_gpu[0, 0, moff[b]:moff[b + 1]], np.arange(m[b]))


@pytest.mark.parametrize("lengths,tied", [
    ((9000, 20000), True),             # one CTA, then a cluster of 2
    ((70000,), True),                  # a cluster of 4: ties straddle the CTAs' slices
    ((140000, 3000, 65536), True),     # a cluster of 8 for every unit of the launch
    ((140000, 33000), False),          # continuous scores
])
def test_selection_across_cluster_sizes(lengths, tied):
    """The selection alone, on seeded scores fed in directly: segments long enough that a unit
    is split across a thread-block cluster of 1, 2, 4 or 8 CTAs.  With few distinct score
    levels the m-th score ties across CTA boundaries, and the lower positions must win across
    the cluster; the keep sets equal the oracle's sort-based top-m exactly."""
    sp = workloads.custom(L=1, H=2, G=2, d=64, P=16, q=2, lengths=lengths)
    case = workloads.build(sp, 4, DEV, with_q=False)
    m = [oracle.budget_ratio(n, 0.2) for n in PT.seg_lengths(case)]
    cp = PT.compactor(case, m)
    g = torch.Generator(device=DEV).manual_seed(77)
    if tied:
        s = torch.randint(0, 12, (sp.L, sp.H, cp.Ntot), generator=g, device=DEV).float() / 8.0
    else:
        s = torch.rand((sp.L, sp.H, cp.Ntot), generator=g, device=DEV)
    cp.scores[:, :, :cp.Ntot] = s
    cp.select()
    torch.cuda.synchronize()
    PT.device_status_clean()
    keep_orc = oracle.select_cache(s.cpu().numpy().astype(np.float64), case.seg_start, case.seg_end, m)
    assert np.array_equal(cp.keep.cpu().numpy()[:, :, :cp.Mtot], keep_orc)


def test_free_stack_overflow_pushes_nothing():
    """A free stack with room for fewer pages than the release returns (the push runs as a
    cluster of CTAs that share the stack top): KVC_DEV_FREE_STACK is set, no page id is written
    and the stack top stays."""
    sp = workloads.custom(L=1, H=2, G=2, d=64, P=16, q=2, lengths=(700, 333, 96), shuffle_pages=True)
    case = workloads.build(sp, 13, DEV, with_q=False)
    m = [oracle.budget_ratio(n, 0.2) for n in PT.seg_lengths(case)]
    keep = workloads.random_keep(case, m, 5)
    cp = PT.compactor(case, m)
    cp.plan_compact(keep.contiguous())
    top = int(case.free_top.item())
    small = kvc.Allocator(case.free_ids[:top + 2], case.free_top)  # capacity top + 2
    ids_before = case.free_ids.cpu().clone()
    kvc.kvc_free_pages(cp.cache, cp.segs, cp.m, small, cp.plan)
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status(clear=True) == kvc.KVC_DEV_FREE_STACK
    assert int(case.free_top.item()) == top
    assert torch.equal(case.free_ids.cpu(), ids_before)


def test_selection_at_the_longest_segment():
    """Selection at its longest segment, 2^20 - 4096 positions, with 304 units (8 KV heads x 38
    sequences), so that each unit runs in one CTA: the case where a warp's 16-bit bin counts
    come closest to 2^16.  Sequences of even index hold one score everywhere (every count of a
    pass lands in one bin; the lowest m positions win), the others seeded uniform scores.  The
    oracle's sort-based top-m is compared on three sampled units; on every unit the properties
    that hold at any size: m strictly ascending positions inside the segment, every kept score
    >= every evicted one, and among scores equal to the smallest kept one the kept positions
    come first.  Selection reads only the scores, so the pools are a token page."""
    n, B, H, P = (1 << 20) - 4096, 38, 8, 64
    nb = n // P
    k_pool = torch.zeros((1, 1, H, P, 64), dtype=torch.bfloat16, device=DEV)
    v_pool = torch.zeros_like(k_pool)
    tags = torch.zeros((1, 1, H, P), dtype=torch.int32, device=DEV)
    block_table = torch.zeros((B, nb), dtype=torch.int32, device=DEV)
    nblocks = torch.full((B,), nb, dtype=torch.int32, device=DEV)
    cache = kvc.Cache(k_pool, v_pool, tags, block_table, nblocks)
    segs = kvc.Segments([0] * B, [n] * B, [n] * B)
    mb = oracle.budget_ratio(n, 0.2)
    m = [mb] * B
    g = torch.Generator(device=DEV).manual_seed(2024)
    scores = torch.rand((1, H, B * n), generator=g, device=DEV)
    for b in range(0, B, 2):
        scores[:, :, b * n:(b + 1) * n] = 0.5
    keep = torch.full((1, H, B * mb), -1, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(256, kvc.kvc_select_workspace_size(cache, segs, m)), dtype=torch.uint8, device=DEV)
    kvc.kvc_select_topm(cache, segs, scores, m, keep, ws)
    torch.cuda.synchronize()
    PT.device_status_clean()
    lowest = torch.arange(mb, dtype=torch.int32, device=DEV)
    for h in range(H):
        for b in range(B):
            s = scores[0, h, b * n:(b + 1) * n]
            k = keep[0, h, b * mb:(b + 1) * mb]
            if b % 2 == 0:
                assert torch.equal(k, lowest), (h, b)
                continue
            assert int(k[0]) >= 0 and int(k[-1]) < n and bool((k[1:] > k[:-1]).all()), (h, b)
            kept = torch.zeros(n, dtype=torch.bool, device=DEV)
            kept[k.long()] = True
            t = s[k.long()].min()
            assert bool((s[~kept] <= t).all()), (h, b)
            tie = s == t
            if bool((tie & ~kept).any()):
                assert int(torch.nonzero(tie & kept).max()) < int(torch.nonzero(tie & ~kept).min()), (h, b)
    for (h, b) in ((0, 1), (5, 19), (7, 37)):
        s = scores[0, h, b * n:(b + 1) * n].cpu().numpy().astype(np.float64)
        want = oracle.select_cache(s[None, None, :], [0], [n], [mb])[0, 0]
        assert np.array_equal(keep[0, h, b * mb:(b + 1) * mb].cpu().numpy(), want), (h, b)


@pytest.mark.parametrize("lengths,tied", [
    ((2, 3, 17, 1024), True),    # every unit sorted whole (the launch's longest segment <= 1024)
    ((2, 3, 17, 1024), False),
    ((1025, 40), True),          # one position more: the radix path for the whole launch
])
def test_short_unit_selection(lengths, tied):
    """The selection of short units (sorted whole in shared memory) and just above its limit
    (radix passes), on seeded scores fed in directly, with exact ties: the keep sets equal the
    oracle's sort-based top-m exactly, budgets 1 .. n - 1 included."""
    sp = workloads.custom(L=2, H=2, G=2, d=64, P=16, q=2, lengths=lengths)
    case = workloads.build(sp, 6, DEV, with_q=False)
    n = PT.seg_lengths(case)
    m = [max(1, min(x - 1, oracle.budget_ratio(x, 0.3))) for x in n]
    cp = PT.compactor(case, m)
    g = torch.Generator(device=DEV).manual_seed(91)
    if tied:
        s = torch.randint(0, 6, (sp.L, sp.H, cp.Ntot), generator=g, device=DEV).float() / 4.0
    else:
        s = torch.rand((sp.L, sp.H, cp.Ntot), generator=g, device=DEV)
    cp.scores[:, :, :cp.Ntot] = s
    cp.select()
    torch.cuda.synchronize()
    PT.device_status_clean()
    keep_orc = oracle.select_cache(s.cpu().numpy().astype(np.float64), case.seg_start, case.seg_end, m)
    assert np.array_equal(cp.keep.cpu().numpy()[:, :, :cp.Mtot], keep_orc)
