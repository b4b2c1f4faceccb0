"""The KV-head split of one cache: under tensor parallelism over KV heads each rank holds the pools
and tags of its own heads, the whole block table and a copy of the allocator, and runs the
five calls on its heads alone.  Nothing is exchanged: the budgets and segment lengths are the
same on every rank, so the target region X, the freed blocks and the block-table rewrite are
too (ActKV 解剖, third component: the tail X logical blocks of a segment become the target, and
the emptied blocks go back to the scheduler).

One GPU stands in for the ranks: each head-half runs as a separate cache, one after the other,
from the same starting allocator state.  Checks:
* each half's scores and keep sets equal the whole-cache run's on its heads (keep sets up to the
  1e-4 selection band around the m-th oracle score);
* given the same selection, the halves' K, V and tag pools put side by side along the head axis
  equal the whole-cache run's bit for bit;
* both halves leave the block table, nblocks and free stack exactly as the whole-cache run does.
"""
import types

import numpy as np
import pytest
import torch

import online_kv_cache_gb300 as kvc
import oracle
import workloads
from tests import parity as PT

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from online_kv_cache_gb300 import build
    build.build()
    kvc.kvc_read_device_status(clear=True)


def head_slice(case, pristine, h0, h1):
    """A cache holding heads [h0, h1) of the pristine state, with its own copies of the block
    table and the allocator."""
    k, v, tags, bt, nb, fi, ft = [t.clone() for t in pristine]
    return types.SimpleNamespace(
        spec=case.spec, k_pool=k[:, :, h0:h1].contiguous(), v_pool=v[:, :, h0:h1].contiguous(),
        tags=tags[:, :, h0:h1].contiguous(), block_table=bt, nblocks=nb, free_ids=fi, free_top=ft,
        q=case.q[:, :, h0:h1].contiguous(), seg_start=case.seg_start, seg_end=case.seg_end,
        seq_len=case.seq_len)


@pytest.mark.parametrize("H,lengths,budget", [
    (4, (700, 300, 1), ("ratio", 0.2)),
    (8, (2048, 555, 4000), ("actkv", (0, 2, 1))),
])
def test_head_halves_compact_like_the_whole(H, lengths, budget):
    sp = workloads.custom(L=3, H=H, G=4, d=128, P=16, q=8, lengths=lengths, budget=budget,
                          kv="sinks", shuffle_pages=True)
    case = workloads.build(sp, 8, DEV)
    m = PT.lib_budgets(case)
    pristine = case.snapshot()

    whole = PT.run_chain(case, m, want_lse=False)
    torch.cuda.synchronize()
    PT.device_status_clean()
    keep_whole = whole.keep[:, :, :whole.Mtot].clone()
    s_whole = whole.scores[:, :, :whole.Ntot].cpu().numpy()
    s_orc, _ = PT.oracle_scores(types.SimpleNamespace(
        k_pool=pristine[0], block_table=pristine[3], nblocks=pristine[4], seg_start=case.seg_start,
        seg_end=case.seg_end, seq_len=case.seq_len, q=case.q, spec=sp))
    n = PT.seg_lengths(case)
    noff, moff = PT.unit_offsets(case, m)

    half = H // 2
    for h0, h1 in ((0, half), (half, H)):
        part = head_slice(case, pristine, h0, h1)
        cp = PT.compactor(part, m)
        cp.score(part.q, sp.scale, False)
        cp.select()
        torch.cuda.synchronize()
        s_part = cp.scores[:, :, :cp.Ntot].cpu().numpy()
        k_part = cp.keep[:, :, :cp.Mtot].cpu().numpy()
        for b in range(sp.B):
            for l in range(sp.L):
                for h in range(h1 - h0):
                    so = s_orc[l, h0 + h, noff[b]:noff[b + 1]]
                    PT.check_scores(s_part[l, h, noff[b]:noff[b + 1]], so, f"half {h0} unit {(b, l, h)}")
                    np.testing.assert_allclose(s_part[l, h, noff[b]:noff[b + 1]],
                                               s_whole[l, h0 + h, noff[b]:noff[b + 1]], rtol=2e-3)
                    PT.check_keep(k_part[l, h, moff[b]:moff[b + 1]],
                                  keep_whole[l, h0 + h, moff[b]:moff[b + 1]].cpu().numpy(), so,
                                  min(m[b], n[b]), f"half {h0} keep {(b, l, h)}")
        # the whole run's selection for these heads: the moved bytes are then fixed
        cp.plan_compact(keep_whole[:, h0:h1].contiguous())
        cp.compact()
        cp.free_pages()
        torch.cuda.synchronize()
        PT.device_status_clean()
        for name in ("k_pool", "v_pool", "tags"):
            got = getattr(part, name)
            want = getattr(case, name)[:, :, h0:h1]
            assert torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else got,
                               want.view(torch.int16) if want.dtype == torch.bfloat16 else want), \
                f"heads [{h0}, {h1}): {name} differs from the whole-cache run"
        for name in ("block_table", "nblocks", "free_ids", "free_top"):
            assert torch.equal(getattr(part, name), getattr(case, name)), \
                f"heads [{h0}, {h1}): {name} differs from the whole-cache run"
