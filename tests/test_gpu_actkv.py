"""GPU parity of ActKV's eviction score (action attention, action-critical entries, LRFU) with
the oracle.

Source: "ActKV 解剖" (zhichai.net analysis of ActKV), first component: the attention of all
action tokens toward each KV entry, the entries within the top 90% counted as action-critical,
and LRFU (lambda = 0.5) driven by those hits.  The LRFU value travels with its entry through
the compaction (the per-slot aux state of the cache).
"""
import numpy as np
import pytest
import torch

import online_kv_cache_gb300 as kvc
import oracle
import workloads
from tests import parity as PT

pytestmark = pytest.mark.gpu
DEV = "cuda"
CRF_RTOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from online_kv_cache_gb300 import build
    build.build()
    kvc.kvc_read_device_status(clear=True)


def actkv_compactor(case, m, aux):
    return kvc.Compactor(case.k_pool, case.v_pool, case.tags, case.block_table, case.nblocks,
                         case.free_ids, case.free_top, case.seg_start, case.seg_end, case.seq_len,
                         m, case.spec.R, aux=aux)


def check_hits(h_gpu, h_orc, a, frac, what, band=1e-6):
    """Hit sets agree except for entries whose action mass sits at the 90% boundary: their value
    lies between the values at cumulative fractions frac -/+ band of the oracle's ordering."""
    diff = np.flatnonzero(h_gpu != h_orc)
    if diff.size == 0:
        return 0
    order = np.argsort(-a, kind="stable")
    cum = np.cumsum(a[order]) / a.sum()
    lo_v = a[order][min(np.searchsorted(cum, frac + band), a.size - 1)]
    hi_v = a[order][min(np.searchsorted(cum, frac - band), a.size - 1)]
    ok = (a[diff] >= lo_v) & (a[diff] <= hi_v)
    assert np.all(ok), f"{what}: {int((~ok).sum())} hit differences away from the boundary"
    return int(diff.size)


@pytest.mark.parametrize("d,P,G,q,lengths", [
    (128, 16, 8, 16, (700, 129, 1)),
    (64, 32, 2, 3, (4097,)),
    (128, 16, 8, 64, (2048, 777)),     # R = 512: two chunks of pass 2
    (128, 32, 16, 40, (1536,)),        # R = 640: two row groups, finished by score_finalize
])
def test_action_attention(d, P, G, q, lengths):
    sp = workloads.custom(L=2, H=2, G=G, d=d, P=P, q=q, lengths=lengths, shuffle_pages=True)
    case = workloads.build(sp, 2, DEV)
    m = PT.lib_budgets(case)
    cp = PT.compactor(case, m)
    cp.score_action(case.q, sp.scale)
    torch.cuda.synchronize()
    PT.device_status_clean()
    a_gpu = cp.attn.cpu().numpy()[:, :, :cp.Ntot].astype(np.float64)
    a_orc, _ = oracle.score_cache(case.k_pool, case.block_table, case.nblocks, case.seg_start,
                                  case.seg_end, case.seq_len, case.q, sp.scale, action=True)
    big = a_orc >= 1e-30
    rel = np.abs(a_gpu[big] - a_orc[big]) / a_orc[big]
    assert rel.max() <= PT.SCORE_RTOL, f"max relative error {rel.max():.3e}"
    assert np.all(a_gpu[~big] <= 1e-27)
    # every row's attention sums to 1, so each unit's mass is R
    noff, _ = PT.unit_offsets(case, m)
    for b in range(sp.B):
        tot = a_gpu[:, :, noff[b]:noff[b + 1]].sum(-1)
        assert np.allclose(tot, sp.R, rtol=1e-4)


def test_lrfu_steps_match_oracle():
    """Four LRFU steps with fresh seeded action masses each time (the kernel alone: both sides
    read the same fp32 masses and start from the same seeded state, then evolve on their own).
    Hit sets agree up to the 90% boundary band; the LRFU values agree wherever the two hit
    histories of an entry agree."""
    sp = workloads.custom(L=2, H=2, G=2, d=64, P=16, q=2, lengths=(1000, 257, 64),
                          shuffle_pages=True)
    case = workloads.build(sp, 6, DEV, with_q=False)
    num_pages = case.k_pool.shape[1]
    g = torch.Generator(device=DEV).manual_seed(5)
    aux = torch.rand((sp.L, num_pages, sp.H, sp.P), generator=g, device=DEV)
    crf_orc = aux.cpu().numpy().astype(np.float64)  # the seeded state, shared input
    m = PT.lib_budgets(case)
    cp = actkv_compactor(case, m, aux)
    noff, _ = PT.unit_offsets(case, m)
    agree = None
    for step in range(4):
        # heavy-tailed masses, as attention is: a few large entries and a long tail
        a = torch.rand((sp.L, sp.H, cp.Ntot), generator=g, device=DEV) ** 8
        cp.attn = a.contiguous()
        hits = torch.zeros((sp.L, sp.H, cp.Ntot), dtype=torch.uint8, device=DEV)
        cp.lrfu(0.9, 0.5, hits)
        torch.cuda.synchronize()
        PT.device_status_clean()
        a_np = a.cpu().numpy().astype(np.float64)
        v_orc, h_orc = oracle.lrfu_cache(crf_orc, case.block_table.cpu().numpy(), case.seg_start,
                                         case.seg_end, a_np, 0.9, 0.5)
        h_gpu = hits.cpu().numpy().astype(bool)
        for l in range(sp.L):
            for h in range(sp.H):
                for b in range(sp.B):
                    sl = slice(noff[b], noff[b + 1])
                    check_hits(h_gpu[l, h, sl], h_orc[l, h, sl], a_np[l, h, sl], 0.9,
                               f"step {step} l={l} h={h} b={b}")
        agree = (h_gpu == h_orc) if agree is None else (agree & (h_gpu == h_orc))
        v_gpu = cp.scores.cpu().numpy()[:, :, :cp.Ntot]
        assert np.allclose(v_gpu[agree], v_orc[agree], rtol=CRF_RTOL, atol=1e-6)
        assert np.any(h_gpu) and np.any(~h_gpu)


def test_actkv_chain_moves_lrfu_values_with_entries():
    """score_action -> LRFU -> top-m by LRFU value on the GPU, against the oracle's own chain
    (fp64 action attention, one LRFU step from the same seeded history, sort-based top-m): hit
    sets up to the boundary band, LRFU values, keep sets up to the 1e-4 band.  Then the oracle's
    keep sets drive the GPU compaction with a seeded per-slot state: the cache equals the
    oracle's compaction bit for bit and every surviving entry carries its own state value to
    its new slot."""
    sp = workloads.custom(L=2, H=2, G=4, d=128, P=16, q=8, lengths=(3000, 900),
                          shuffle_pages=True, budget=("actkv", (1, 0)))
    case = workloads.build(sp, 8, DEV)
    num_pages = case.k_pool.shape[1]
    g = torch.Generator(device=DEV).manual_seed(1)
    aux = torch.rand((sp.L, num_pages, sp.H, sp.P), generator=g, device=DEV)  # an earlier history
    aux_start = aux.cpu().numpy().copy()
    m = PT.lib_budgets(case)
    cp = actkv_compactor(case, m, aux)
    hits = torch.zeros_like(cp.scores, dtype=torch.uint8)
    cp.score_action(case.q, sp.scale)
    cp.lrfu(0.9, 0.5, hits)
    cp.select()
    torch.cuda.synchronize()
    PT.device_status_clean()
    crf = cp.scores.cpu().numpy()[:, :, :cp.Ntot].astype(np.float64)
    keep = cp.keep.cpu().numpy()[:, :, :cp.Mtot]
    # the oracle's own chain
    a_orc, _ = oracle.score_cache(case.k_pool, case.block_table, case.nblocks, case.seg_start,
                                  case.seg_end, case.seq_len, case.q, sp.scale, action=True)
    crf_pool = aux_start.astype(np.float64)
    v_orc, h_orc = oracle.lrfu_cache(crf_pool, case.block_table.cpu().numpy(), case.seg_start,
                                     case.seg_end, a_orc, 0.9, 0.5)
    keep_orc = oracle.select_cache(v_orc, case.seg_start, case.seg_end, m)
    h_gpu = hits.cpu().numpy()[:, :, :cp.Ntot].astype(bool)
    noff, moff = PT.unit_offsets(case, m)
    for l in range(sp.L):
        for h in range(sp.H):
            for b in range(sp.B):
                sl = slice(noff[b], noff[b + 1])
                check_hits(h_gpu[l, h, sl], h_orc[l, h, sl], a_orc[l, h, sl], 0.9,
                           f"chain l={l} h={h} b={b}", band=1e-4)
    same = h_gpu == h_orc
    assert np.allclose(crf[same], v_orc[same], rtol=CRF_RTOL, atol=1e-6)
    if same.all():  # the selection rule is comparable when both sides scored the same hits
        for l in range(sp.L):
            for h in range(sp.H):
                for b in range(sp.B):
                    PT.check_keep(keep[l, h, moff[b]:moff[b + 1]], keep_orc[l, h, moff[b]:moff[b + 1]],
                                  v_orc[l, h, noff[b]:noff[b + 1]], int(moff[b + 1] - moff[b]),
                                  f"l={l} h={h} b={b}")
    # compaction driven by the oracle's keep sets, with a seeded per-slot state
    seeded = torch.rand(aux.shape, generator=g, device=DEV)
    aux.copy_(seeded)
    aux_before = seeded.cpu().numpy()
    pristine = PT.host_state(case)
    bt_before = pristine["bt"].copy()  # oracle_compaction below rewrites pristine in place
    cp.plan_compact(torch.from_numpy(np.ascontiguousarray(keep_orc)).to(DEV))
    cp.compact()
    cp.free_pages()
    torch.cuda.synchronize()
    PT.device_status_clean()
    PT.assert_state_equal(PT.host_state(case), PT.oracle_compaction(pristine, case, m, keep_orc),
                          "actkv chain")
    after = PT.host_state(case)
    aux_after = aux.cpu().numpy()
    P = sp.P
    for b in range(sp.B):
        X = -(-m[b] // P)
        for l in range(sp.L):
            for h in range(sp.H):
                for r in range(X * P):
                    pg = after["bt"][b, r // P]
                    tag = after["tags"][l, pg, h, r % P]
                    if tag < 0:
                        continue
                    src_pg = bt_before[b, tag // P]
                    assert aux_after[l, pg, h, r % P] == aux_before[l, src_pg, h, tag % P]
