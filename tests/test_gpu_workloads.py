"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times.

* Scores and keep sets are compared with the oracle on sampled units (the oracle computes them
  unit by unit); every unit is checked for the properties that hold at any size.
* Compaction is checked bit-exact over the whole cache given a seeded selection (layer slices
  at a time, so host memory stays bounded).
* The multi-turn schedule (20 turns, delay-1 compaction) is checked against the oracle after
  every turn, then for block-table / logical-position continuity and freed-page totals.
"""
import math

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


# Units compared with the oracle at full size, beyond every unit of one seeded layer.  The
# Qwen3-shaped cache gets the most: its attention sinks make the selection band tightest there.
EXTRA_UNITS = {"qwen3-30b-a3b": 32, "batched-ragged": 16, "batched-ragged-sinks": 16, "long-context": 16}


def sample_units(case, k, seed):
    """Every (b, l, h) unit of one seeded layer, plus k more seeded units (the first and the last
    unit of the cache among them); active sequences only."""
    sp = case.spec
    active = [b for b in range(sp.B) if case.seg_end[b] > case.seg_start[b]]
    rng = np.random.default_rng(seed)
    layer = int(rng.integers(sp.L))
    units = {(b, layer, h) for b in active for h in range(sp.H)}
    extra = {(active[0], 0, 0), (active[-1], sp.L - 1, sp.H - 1)}
    total = min(len(units) + k, len(active) * sp.L * sp.H)
    while len(extra - units) < k and len(units | extra) < total:
        extra.add((int(rng.choice(active)), int(rng.integers(sp.L)), int(rng.integers(sp.H))))
    return sorted(units | extra)


def check_live_tags(case, m, keep_gpu):
    """After the chain: for every unit, the live tags of the segment's new first X blocks are
    exactly the kept positions (tags of a fresh sequence are its slot numbers)."""
    sp = case.spec
    n = PT.seg_lengths(case)
    _, moff = PT.unit_offsets(case, m)
    bt = case.block_table
    for b in range(sp.B):
        if n[b] == 0:
            continue
        X = -(-min(m[b], n[b]) // sp.P)
        sb = case.seg_start[b] // sp.P
        pages = bt[b, sb:sb + X].long()
        tags = case.tags[:, pages].permute(0, 2, 1, 3).reshape(sp.L, sp.H, X * sp.P)  # [L][H][X*P]
        live = torch.sort(tags, dim=-1).values[:, :, X * sp.P - min(m[b], n[b]):]
        want = keep_gpu[:, :, moff[b]:moff[b + 1]].to(torch.int32) + case.seg_start[b]
        assert torch.equal(live, want), f"sequence {b}: live tags differ from the keep set"


@pytest.mark.parametrize("name", ["qwen3-30b-a3b", "batched-ragged", "batched-ragged-sinks", "long-context"])
def test_full_size(name):
    sp = workloads.spec(name, 0)
    case = workloads.build(sp, 0, DEV)
    m = PT.lib_budgets(case)
    assert m == PT.oracle_budgets(case)
    snap = case.snapshot()
    nblocks0 = case.nblocks.clone()
    top0 = int(case.free_top.item())
    cp = PT.run_chain(case, m, want_lse=True)
    torch.cuda.synchronize()
    PT.device_status_clean()
    s_gpu = cp.scores[:, :, :cp.Ntot]
    k_gpu = cp.keep[:, :, :cp.Mtot]

    # properties on every unit
    n = PT.seg_lengths(case)
    noff, moff = PT.unit_offsets(case, m)
    assert torch.isfinite(s_gpu).all() and (s_gpu >= 0).all()
    for b in range(sp.B):
        kb = k_gpu[:, :, moff[b]:moff[b + 1]]
        if kb.shape[-1] > 1:
            assert (kb[:, :, 1:] > kb[:, :, :-1]).all(), "keep not ascending"
        if kb.numel():
            assert kb.min() >= 0 and kb.max() < n[b]
    if case.planted and case.planted[0] is not None and sp.qdist == "aligned":
        # Q-aligned heavy hitters outscore the median key of their unit
        pl = case.planted[0].long()
        s0 = s_gpu[:, :, :n[0]]
        med = s0.median(dim=-1).values.unsqueeze(-1)
        assert (torch.gather(s0, 2, pl) > med).float().mean() > 0.99
    check_live_tags(case, m, k_gpu)
    freed = sum(-(-x // sp.P) - -(-min(a, x) // sp.P) for a, x in zip(m, n))
    assert int(case.free_top.item()) == top0 + freed
    assert int((nblocks0 - case.nblocks).sum().item()) == freed

    # every unit of one layer plus seeded units against the oracle (all host threads)
    case.restore(snap)
    units = sample_units(case, EXTRA_UNITS[name], 1)
    mask = np.zeros((sp.B, sp.L, sp.H), bool)
    for u in units:
        mask[u] = True
    s_orc, lse_orc = PT.oracle_scores(case, mask)
    s_gpu_np = s_gpu.cpu().numpy()
    k_gpu_np = k_gpu.cpu().numpy()
    lse_gpu = cp.lse.cpu().numpy()
    worst, inband = 0.0, 0
    for (b, l, h) in units:
        so = s_orc[l, h, noff[b]:noff[b + 1]]
        worst = max(worst, PT.check_scores(s_gpu_np[l, h, noff[b]:noff[b + 1]], so, f"{name} unit {(b, l, h)}"))
        PT.check_lse(lse_gpu[b, l, h], lse_orc[b, l, h], f"{name} lse {(b, l, h)}")
        ko = oracle.select(so, m[b])
        inband += PT.check_keep(k_gpu_np[l, h, moff[b]:moff[b + 1]], ko, so, min(m[b], n[b]), f"{name} keep {(b, l, h)}")
    print(f"{name}: {len(units)} units against the oracle, worst score error {worst:.2e}, "
          f"{inband} in-band selection differences")

    # compaction of the whole cache given a seeded selection, bit-exact, a few layers at a time
    keep = workloads.random_keep(case, m, 11)
    cp2 = PT.compactor(case, m)
    cp2.plan_compact(keep.contiguous())
    cp2.compact()
    cp2.free_pages()
    torch.cuda.synchronize()
    PT.device_status_clean()
    keep_np = keep.cpu().numpy()
    step = max(1, 4 if sp.L > 4 else sp.L)
    for l0 in range(0, sp.L, step):
        l1 = min(sp.L, l0 + step)
        pristine = {"k": PT.bits(snap[0][l0:l1]), "v": PT.bits(snap[1][l0:l1]), "tags": PT.i32(snap[2][l0:l1])}
        oracle.compact_layers(pristine["k"], pristine["v"], pristine["tags"], l0, sp.L, PT.i32(snap[3]),
                              case.seg_start, case.seg_end, m, keep_np)
        assert np.array_equal(PT.bits(case.k_pool[l0:l1]), pristine["k"]), f"K layers {l0}..{l1}"
        assert np.array_equal(PT.bits(case.v_pool[l0:l1]), pristine["v"]), f"V layers {l0}..{l1}"
        assert np.array_equal(PT.i32(case.tags[l0:l1]), pristine["tags"]), f"tags layers {l0}..{l1}"
    st = {"bt": PT.i32(snap[3]), "nblocks": PT.i32(snap[4]), "free_ids": PT.i32(snap[5]),
          "free_top": PT.i32(snap[6])}
    oracle.free_blocks(st["bt"], st["nblocks"], st["free_ids"], st["free_top"], sp.P, case.seg_start,
                       case.seg_end, m)
    for key, t in (("bt", case.block_table), ("nblocks", case.nblocks), ("free_ids", case.free_ids),
                   ("free_top", case.free_top)):
        assert np.array_equal(PT.i32(t), st[key]), key


def test_multi_turn_schedule():
    """20 turns x 1536 tokens; at the end of turn t >= 2 the segment of turn t-1 is compacted with
    turn t's proxy queries (delay 1).  Each compaction is checked against the oracle (scores,
    keep sets, then the state bit-exact given the oracle's selection); at the end the block table
    walks the frozen segments in order with the right logical positions."""
    ms = workloads.MultiTurnSpec()
    m_seg = kvc.kvc_budget_from_ratio(ms.tokens, ms.ratio)
    assert m_seg == oracle.budget_ratio(ms.tokens, ms.ratio) == 308
    X = -(-m_seg // ms.P)
    mt = workloads.MultiTurn(ms, 0, DEV, kept_blocks=X)
    mt.append_turn()
    keeps = {}
    top_init = mt.num_pages  # the free stack before any turn
    for t in range(2, ms.turns + 1):
        mt.append_turn()
        s0, s1 = mt.prepare_compaction()
        case = mt.case
        m = [m_seg]
        pristine = PT.host_state(case)
        s_orc, lse_orc = PT.oracle_scores(case)
        keep_orc = oracle.select_cache(s_orc, case.seg_start, case.seg_end, m)
        cp = PT.compactor(case, m)
        cp.score(case.q, case.spec.scale, True)
        cp.select()
        torch.cuda.synchronize()
        PT.check_scores(cp.scores.cpu().numpy()[:, :, :cp.Ntot], s_orc, f"turn {t}")
        PT.check_lse(cp.lse.cpu().numpy()[0], lse_orc[0], f"turn {t} lse")
        k_gpu = cp.keep.cpu().numpy()[:, :, :cp.Mtot]
        for l in range(ms.L):
            for h in range(ms.H):
                PT.check_keep(k_gpu[l, h], keep_orc[l, h], s_orc[l, h], m_seg, f"turn {t} l={l} h={h}")
        # planted keys of this compaction survive
        pl = case.planted[0].cpu().numpy()
        for l in range(ms.L):
            for h in range(ms.H):
                assert set(pl[l, h].tolist()) <= set(k_gpu[l, h].tolist())
        cp.plan_compact(torch.from_numpy(np.ascontiguousarray(keep_orc)).to(DEV))
        cp.compact()
        cp.free_pages()
        torch.cuda.synchronize()
        PT.device_status_clean()
        PT.assert_state_equal(PT.host_state(case), PT.oracle_compaction(pristine, case, m, keep_orc),
                              f"turn {t}")
        keeps[t - 1] = keep_orc
        mt.compacted(X)
        assert int(case.free_top.item()) == top_init - 96 * t + 76 * (t - 1)
    case = mt.case
    assert int(case.nblocks[0].item()) == 20 * 96 - 19 * 76 == 476
    assert int(case.free_top.item()) == top_init - 476  # 1444 pages freed in 19 compactions
    # continuity: segments 1..19 hold X blocks each, then the 96 blocks of turn 20
    bt = case.block_table[0].cpu().numpy()
    tags = case.tags.cpu().numpy()
    last_max = -1
    for seg in range(1, ms.turns):
        blocks = bt[(seg - 1) * X:seg * X]
        live = tags[:, blocks].transpose(0, 2, 1, 3).reshape(ms.L, ms.H, X * ms.P)
        for l in range(ms.L):
            for h in range(ms.H):
                got = np.sort(live[l, h][live[l, h] >= 0])
                want = ms.tokens * (seg - 1) + keeps[seg][l, h]
                assert np.array_equal(got, want), f"segment {seg} l={l} h={h}"
        lo = ms.tokens * (seg - 1)
        assert live.max() < ms.tokens * seg and live[live >= 0].min() >= lo > last_max
        last_max = live.max()
    tail = bt[19 * X:19 * X + 96]
    tail_tags = tags[:, tail].transpose(0, 2, 1, 3).reshape(ms.L, ms.H, -1)
    assert np.array_equal(tail_tags[0, 0], np.arange(ms.tokens * 19, ms.tokens * 20))
    assert (bt[476:] == -1).all()


def test_external_lse_path():
    """kvc_score_alpha with a caller-supplied LSE (here the oracle's, in fp32) gives the oracle's
    scores; kvc_score_lse + kvc_score_alpha equals kvc_score."""
    sp = workloads.custom(L=2, H=2, G=8, d=128, P=16, q=16, lengths=(3000, 777), shuffle_pages=True)
    case = workloads.build(sp, 21, DEV)
    m = PT.lib_budgets(case)
    s_orc, lse_orc = PT.oracle_scores(case)
    cp = PT.compactor(case, m)
    cp.score(case.q, sp.scale, True)
    torch.cuda.synchronize()
    ref = cp.scores.clone()
    cp.scores.zero_()
    cp.score_lse(case.q, sp.scale, True)
    cp.score_alpha(case.q, sp.scale)
    torch.cuda.synchronize()
    assert torch.equal(cp.scores, ref)
    lse_in = torch.from_numpy(lse_orc.astype(np.float32)).to(DEV).contiguous()
    cp.scores.zero_()
    cp.score_alpha(case.q, sp.scale, lse_in)
    torch.cuda.synchronize()
    PT.check_scores(cp.scores.cpu().numpy()[:, :, :cp.Ntot], s_orc, "external LSE")
    PT.device_status_clean()
