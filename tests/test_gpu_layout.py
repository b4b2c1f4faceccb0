"""GPU parity of the layout variants of eviction (sentinel dead slots; order-preserving
compaction into fresh pages) with the oracle: the whole cache state, bit-exact.

Source: "IntentKV: Cross-Turn Intent-Aware KV Cache Pruning" (gist.science summary), section
on layout-preserving eviction (sentinel dead slot K = -10^4, V = 0; survivors keep their
slots) and its objection to in-place compaction (positions are renumbered), which the
fresh-page compaction answers by moving survivors in logical order into new pages.
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

SHAPES = [
    # d, P, sequence lengths
    (64, 8, (257, 64, 1023, 8)),
    (128, 16, (700, 260, 1, 33)),
    (128, 32, (4097, 96)),
    (64, 64, (300, 129, 2000)),
    (128, 16, tuple(17 + (7 * i) % 90 for i in range(130))),  # two launch chunks of sequences
]


@pytest.fixture(scope="module", autouse=True)
def built():
    from online_kv_cache_gb300 import build
    build.build()
    kvc.kvc_read_device_status(clear=True)


def oracle_sentinel(state, case, m, keep_np):
    oracle.evict_sentinel(state["k"], state["v"], state["tags"], 0, case.spec.L, state["bt"],
                          case.seg_start, case.seg_end, m, keep_np)
    return state


def oracle_fresh(state, case, m, keep_np):
    fresh = oracle.fresh_pages(state["free_ids"], int(state["free_top"][0]), case.spec.P,
                               case.seg_start, case.seg_end, m)
    oracle.compact_fresh(state["k"], state["v"], state["tags"], 0, case.spec.L, state["bt"],
                         case.seg_start, case.seg_end, m, keep_np, fresh)
    oracle.commit_fresh(state["bt"], state["nblocks"], state["free_ids"], state["free_top"],
                        case.spec.P, case.seg_start, case.seg_end, m, fresh)
    return state


def run_sentinel(case, m, keep):
    cp = PT.compactor(case, m)
    cp.evict_sentinel(keep.contiguous() if keep.numel() else None)
    return cp


def run_fresh(case, m, keep):
    cp = PT.compactor(case, m)
    plan = cp.plan_fresh(keep.contiguous() if keep.numel() else None)
    cp.compact(plan=plan)
    cp.commit_fresh()
    return cp


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("variant", ["sentinel", "fresh"])
def test_random_keeps(shape, variant):
    d, P, lengths = shape
    sp = workloads.custom(L=2, H=2, G=2, d=d, P=P, q=2, lengths=lengths, shuffle_pages=True,
                          headroom=1.1)
    case = workloads.build(sp, 11, DEV, with_q=False)
    for trial, ratio in enumerate((0.0, 0.05, 0.2, 0.7, 1.0)):
        m = [oracle.budget_ratio(x, ratio) for x in PT.seg_lengths(case)]
        snap = case.snapshot()
        pristine = PT.host_state(case)
        keep = workloads.random_keep(case, m, 200 + trial)
        (run_sentinel if variant == "sentinel" else run_fresh)(case, m, keep)
        torch.cuda.synchronize()
        PT.device_status_clean()
        want = (oracle_sentinel if variant == "sentinel" else oracle_fresh)(
            pristine, case, m, keep.cpu().numpy())
        PT.assert_state_equal(PT.host_state(case), want, f"{variant} d={d} P={P} ratio={ratio}")
        case.restore(snap)


@pytest.mark.parametrize("variant", ["sentinel", "fresh"])
def test_inner_segments_and_mixed_budgets(variant):
    """Segments that start and end inside sequences (later blocks shift down in the fresh
    variant), an empty segment, and budgets 0, partial and all in one call."""
    sp = workloads.custom(L=3, H=2, G=2, d=128, P=16, q=2, lengths=(1000, 200, 640, 90),
                          shuffle_pages=True, headroom=1.0)
    case = workloads.build(sp, 21, DEV, with_q=False)
    case.seg_start = [320, 0, 64, 0]
    case.seg_end = [800, 0, 640, 90]
    n = PT.seg_lengths(case)
    m = [150, 0, 0, 90]
    m = [min(a, b) for a, b in zip(m, n)]
    pristine = PT.host_state(case)
    keep = workloads.random_keep(case, m, 7)
    (run_sentinel if variant == "sentinel" else run_fresh)(case, m, keep)
    torch.cuda.synchronize()
    PT.device_status_clean()
    want = (oracle_sentinel if variant == "sentinel" else oracle_fresh)(pristine, case, m,
                                                                       keep.cpu().numpy())
    PT.assert_state_equal(PT.host_state(case), want, f"{variant} inner segments")


def test_fresh_physical_order_is_logical_order():
    """After the fresh-page compaction, walking each compacted segment's blocks in the block
    table visits the survivors in strictly ascending logical position (tags), then dead slots."""
    sp = workloads.custom(L=2, H=2, G=2, d=64, P=16, q=2, lengths=(900, 333), shuffle_pages=True,
                          headroom=1.0)
    case = workloads.build(sp, 3, DEV, with_q=False)
    m = [oracle.budget_ratio(x, 0.2) for x in PT.seg_lengths(case)]
    keep = workloads.random_keep(case, m, 9)
    run_fresh(case, m, keep)
    torch.cuda.synchronize()
    PT.device_status_clean()
    st = PT.host_state(case)
    k = keep.cpu().numpy()
    moff = np.concatenate([[0], np.cumsum(m)])
    P = sp.P
    for b, mb in enumerate(m):
        X = -(-mb // P)
        pages = st["bt"][b, :X]
        for l in range(sp.L):
            for h in range(sp.H):
                t = st["tags"][l, pages, h, :].reshape(-1)
                assert np.array_equal(t[:mb], k[l, h, moff[b]:moff[b + 1]])
                assert np.all(np.diff(t[:mb]) > 0) and np.all(t[mb:] == -1)


def test_fresh_stack_too_small_changes_nothing():
    """A free stack with fewer pages than the call pops: KVC_DEV_FREE_STACK, no byte changes."""
    sp = workloads.custom(L=1, H=2, G=2, d=64, P=16, q=2, lengths=(1024, 512), headroom=0.01)
    case = workloads.build(sp, 5, DEV, with_q=False)
    m = [400, 300]  # needs 25 + 19 fresh pages; the stack holds 1
    pristine = PT.host_state(case)
    keep = workloads.random_keep(case, m, 1)
    run_fresh(case, m, keep)
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status(clear=True) == kvc.KVC_DEV_FREE_STACK
    PT.assert_state_equal(PT.host_state(case), pristine, "fresh with an empty stack")


def test_sentinel_full_size_qwen3_shape():
    """The sentinel eviction on the full Qwen3-30B-A3B-shaped cache (48 layers, 4 KV heads,
    32768 keys, keep 20%), whole state bit-exact."""
    sp = workloads.spec("qwen3-30b-a3b")
    case = workloads.build(sp, 0, DEV, with_q=False)
    m = PT.lib_budgets(case)
    pristine = PT.host_state(case)
    keep = workloads.random_keep(case, m, 3)
    run_sentinel(case, m, keep)
    torch.cuda.synchronize()
    PT.device_status_clean()
    want = oracle_sentinel(pristine, case, m, keep.cpu().numpy())
    PT.assert_state_equal(PT.host_state(case), want, "sentinel qwen3 shape")


def test_fresh_qwen3_shape_8_layers():
    """The fresh-page compaction on 8 layers of the Qwen3-30B-A3B shape with 30% free pages."""
    sp = workloads.custom(L=8, H=4, G=8, d=128, P=16, q=1, lengths=(32768,), headroom=0.3)
    case = workloads.build(sp, 0, DEV, with_q=False)
    m = [oracle.budget_ratio(32768, 0.2)]
    pristine = PT.host_state(case)
    keep = workloads.random_keep(case, m, 4)
    run_fresh(case, m, keep)
    torch.cuda.synchronize()
    PT.device_status_clean()
    want = oracle_fresh(pristine, case, m, keep.cpu().numpy())
    PT.assert_state_equal(PT.host_state(case), want, "fresh qwen3 shape")
