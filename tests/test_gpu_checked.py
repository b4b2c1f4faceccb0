"""Checked mode (KVC_CHECKED): a call that launched work synchronises and turns a set bit of the
device status word into KVC_ERR_DEVICE_CHECK; without it the call returns OK and the bit waits
in the status word.  The fault is made on the host: a keep position outside its segment, which
the plan kernel bounds-checks, reports and skips (nothing out of range is read or written)."""
import os

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


@pytest.fixture()
def checked(monkeypatch):
    monkeypatch.setenv("KVC_CHECKED", "1")
    yield
    kvc.kvc_read_device_status(clear=True)


def small_case():
    sp = workloads.custom(L=2, H=2, G=2, d=64, P=16, q=4, lengths=(300, 130), shuffle_pages=True)
    case = workloads.build(sp, 3, DEV)
    m = [oracle.budget_ratio(n, 0.2) for n in PT.seg_lengths(case)]
    cp = PT.compactor(case, m)
    return case, m, cp


def bad_keep(cp, case):
    """Ascending positions 0..m_b-1 for every unit, except that the last entry of unit (layer 0,
    head 0, sequence 0) is the segment length, one past its end."""
    row = torch.cat([torch.arange(int(mb), dtype=torch.int32, device=DEV) for mb in cp.m])
    keep = row.expand(case.spec.L, case.spec.H, -1).contiguous()
    keep[0, 0, int(cp.m[0]) - 1] = case.seg_end[0] - case.seg_start[0]
    return keep


def test_valid_chain_passes_in_checked_mode(checked):
    case, m, cp = small_case()
    cp.run(case.q, case.spec.scale)  # every call synchronises and finds the status word clean
    assert kvc.kvc_read_device_status(clear=True) == 0


def test_bad_keep_is_an_error_in_checked_mode(checked):
    case, m, cp = small_case()
    with pytest.raises(kvc.KvcError) as ei:
        cp.plan_compact(bad_keep(cp, case))
    assert ei.value.status == kvc.KVC_ERR_DEVICE_CHECK
    assert "checked mode" in kvc.kvc_last_error()
    assert kvc.kvc_read_device_status(clear=True) & kvc.KVC_DEV_BAD_KEEP


def test_bad_keep_without_checked_mode_sets_the_status_bit(monkeypatch):
    monkeypatch.delenv("KVC_CHECKED", raising=False)
    case, m, cp = small_case()
    cp.plan_compact(bad_keep(cp, case))  # returns OK: the launch is asynchronous
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status(clear=True) & kvc.KVC_DEV_BAD_KEEP
    assert kvc.kvc_read_device_status(clear=True) == 0  # cleared


def test_checked_mode_is_skipped_under_graph_capture(checked):
    """Capture cannot synchronise: the check stands aside and the replay still runs clean."""
    case, m, cp = small_case()
    snap = case.snapshot()
    cp.run(case.q, case.spec.scale)  # first calls (validation, attributes) outside the capture
    torch.cuda.synchronize()
    case.restore(snap)  # the run compacted the cache: back to the segments it describes
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cp.score(case.q, case.spec.scale, True)
        cp.select()
    case.restore(snap)
    g.replay()
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status(clear=True) == 0
