"""Failure detection in the scoring kernels, driven without faulting the GPU.

Every wait between the roles of a scoring kernel (producer, MMA issuer, epilogue warpgroups) is
bounded.  When one runs out the kernel records KVC_DEV_WAIT_TIMEOUT in the device status word,
waits for the copies and MMAs it has already issued, frees its tensor memory and returns.  The
failure is made on the host: ``kvc_debug_stall_scoring`` makes the producer issue no proxy-row
load and shortens the waits, so the MMA issuer's first wait has nothing that can satisfy it and
runs out.  The tests check that the call returns, that the status bit (and only it) is set, and
that the next normal call on the same stream gives the oracle's scores and LSE: the context and
the SMs' tensor memory are usable again.
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
STALL_NS = 1_000_000  # 1 ms per wait


@pytest.fixture(scope="module", autouse=True)
def built():
    from online_kv_cache_gb300 import build
    build.build()
    kvc.kvc_read_device_status(clear=True)
    yield
    kvc.kvc_debug_stall_scoring(0)


@pytest.mark.parametrize("d,G,q,lengths,grid", [
    (64, 2, 8, (512,), None),            # the tiny shape: one row tile, both passes
    (128, 8, 64, (3000, 777), None),     # R = 512: four Q row tiles in pass 1, two pass-2 chunks
    (128, 8, 16, (9000,), "3"),          # many items per CTA: the abort reaches CTAs mid-loop
])
def test_wait_runs_out_then_next_call_is_clean(d, G, q, lengths, grid, monkeypatch):
    if grid is not None:
        monkeypatch.setenv("KVC_GRID_LIMIT", grid)
    sp = workloads.custom(L=2, H=2, G=G, d=d, P=16, q=q, lengths=lengths, shuffle_pages=True)
    case = workloads.build(sp, 4, DEV)
    m = PT.lib_budgets(case)
    cp = PT.compactor(case, m)
    kvc.kvc_read_device_status(clear=True)
    launches0 = kvc.kvc_launch_count()
    kvc.kvc_debug_stall_scoring(STALL_NS)
    try:
        cp.score(case.q, sp.scale, True)  # returns: every wait is bounded
        torch.cuda.synchronize()
    finally:
        kvc.kvc_debug_stall_scoring(0)
    assert kvc.kvc_launch_count() > launches0
    st = kvc.kvc_read_device_status(clear=True)
    assert st == kvc.KVC_DEV_WAIT_TIMEOUT, f"device status {st:#x}"

    # the same stream, the same buffers: a normal call gives the oracle's results
    cp.scores.fill_(float("nan"))
    cp.lse.fill_(float("nan"))
    cp.score(case.q, sp.scale, True)
    torch.cuda.synchronize()
    PT.device_status_clean()
    s_orc, lse_orc = PT.oracle_scores(case)
    PT.check_scores(cp.scores.cpu().numpy()[:, :, :cp.Ntot], s_orc, "after the timed-out call")
    PT.check_lse(cp.lse.cpu().numpy(), lse_orc, "after the timed-out call")


def test_stall_setting_is_validated():
    with pytest.raises(kvc.KvcError):
        kvc.kvc_debug_stall_scoring(-1)
    with pytest.raises(kvc.KvcError):
        kvc.kvc_debug_stall_scoring(10 ** 11)
    kvc.kvc_debug_stall_scoring(0)
