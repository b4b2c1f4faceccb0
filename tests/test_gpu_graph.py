"""The five C-ABI calls captured into a CUDA graph and replayed give the same result as the eager
calls, replay after replay (the bench times the step this way)."""
import numpy as np
import pytest
import torch

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


def chain(cp, case):
    cp.score(case.q, case.spec.scale, True)
    cp.select()
    cp.plan_compact()
    cp.compact()
    cp.free_pages()


@pytest.mark.parametrize("name", ["tiny", "multi-turn"])
def test_graph_replay_equals_eager(name):
    sp = workloads.spec(name)
    case = workloads.build(sp, 1, DEV)
    m = PT.lib_budgets(case)
    snap = case.snapshot()
    cp = PT.compactor(case, m)
    chain(cp, case)  # eager (also the first call of every kernel before capture)
    torch.cuda.synchronize()
    PT.device_status_clean()
    eager = PT.host_state(case)
    eager_scores = cp.scores.cpu().clone()
    eager_keep = cp.keep.cpu().clone()
    g = torch.cuda.CUDAGraph()
    case.restore(snap)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        chain(cp, case)
    for rep in range(3):
        case.restore(snap)
        cp.scores.zero_()
        cp.keep.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        PT.device_status_clean()
        assert torch.equal(cp.scores.cpu(), eager_scores), f"scores differ on replay {rep}"
        assert torch.equal(cp.keep.cpu(), eager_keep), f"keep differs on replay {rep}"
        PT.assert_state_equal(PT.host_state(case), eager, f"{name} replay {rep}")


@pytest.mark.parametrize("name", ["qwen3-30b-a3b", "batched-ragged"])
def test_graph_replay_equals_eager_full_size(name):
    """At full size, in the launch configuration the benchmark times (the five calls captured
    into one CUDA graph and replayed), the replay leaves scores, keep sets and the whole cache
    state bit-identical to the eager calls, whose parity with the oracle test_gpu_workloads
    checks at the same sizes.  Compared on the device."""
    sp = workloads.spec(name)
    case = workloads.build(sp, 0, DEV)
    m = PT.lib_budgets(case)
    snap = case.snapshot()
    cp = PT.compactor(case, m)
    chain(cp, case)
    torch.cuda.synchronize()
    PT.device_status_clean()
    eager_state = [t.clone() for t in case.state()]
    eager_scores, eager_keep = cp.scores.clone(), cp.keep.clone()
    g = torch.cuda.CUDAGraph()
    case.restore(snap)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        chain(cp, case)
    for rep in range(2):
        case.restore(snap)
        cp.scores.zero_()
        cp.keep.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        PT.device_status_clean()
        assert torch.equal(cp.scores, eager_scores), f"{name}: scores differ on replay {rep}"
        assert torch.equal(cp.keep, eager_keep), f"{name}: keep differs on replay {rep}"
        for i, (a, b) in enumerate(zip(case.state(), eager_state)):
            assert torch.equal(a, b), f"{name}: cache state tensor {i} differs on replay {rep}"
