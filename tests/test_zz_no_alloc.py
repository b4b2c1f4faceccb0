"""kvc_score_noalloc: scoring without a caller workspace.

Some callers cannot give the library a cudaMalloc'ed workspace (a serving engine whose allocator
already owns the device memory, code that must stay out of the CUDA allocator on its hot path).
This entry point keeps the workspace in a fixed device array inside the library.  The test calls
it twice in a row through the C ABI and compares both results with kvc_score's (caller workspace)
within the score tolerance of the other parity tests.  Between the two checked calls it runs one
on a different, larger cache, which leaves other contents in the shared array: nothing in the
array may need to start at zero or to hold the previous call's values.  It runs last (file
name) and passes both alone in a fresh process and after the other tests."""
import numpy as np
import pytest
import torch

import online_kv_cache_gb300 as kvc
import workloads
from tests import parity as PT

pytestmark = pytest.mark.gpu


def test_noalloc_scores_match_caller_workspace_twice():
    from online_kv_cache_gb300 import build
    build.build()
    sp = workloads.custom(L=2, H=2, G=8, d=128, P=16, q=64, lengths=(2048, 777), shuffle_pages=True)
    case = workloads.build(sp, 31, "cuda")
    m = PT.lib_budgets(case)
    cp = PT.compactor(case, m)
    assert kvc.kvc_score_workspace_size(cp.cache, cp.segs, sp.R) <= 16 << 20
    kvc.kvc_read_device_status(clear=True)
    cp.score(case.q, sp.scale, want_lse=True)
    torch.cuda.synchronize()
    ref_s = cp.scores[:, :, :cp.Ntot].double().cpu().numpy()
    ref_l = cp.lse.double().cpu().numpy()
    # a different, larger cache whose call fills more of the shared array
    sp2 = workloads.custom(L=3, H=4, G=8, d=128, P=16, q=32, lengths=(5000, 3001), shuffle_pages=True)
    case2 = workloads.build(sp2, 32, "cuda")
    cp2 = PT.compactor(case2, PT.lib_budgets(case2))
    need2 = kvc.kvc_score_workspace_size(cp2.cache, cp2.segs, sp2.R)
    assert kvc.kvc_score_workspace_size(cp.cache, cp.segs, sp.R) < need2 <= 16 << 20
    for call in range(2):
        scores = torch.full_like(cp.scores, float("nan"))
        lse = torch.full_like(cp.lse, float("nan"))
        kvc.kvc_score_noalloc(cp.cache, cp.segs, case.q, sp.R, sp.scale, scores, lse)
        torch.cuda.synchronize()
        PT.check_scores(scores[:, :, :cp.Ntot].cpu().numpy(), ref_s, f"no-alloc call {call}")
        PT.check_lse(lse.cpu().numpy(), ref_l, f"no-alloc call {call} lse")
        if call == 0:
            s2 = torch.empty_like(cp2.scores)
            l2 = torch.empty_like(cp2.lse)
            kvc.kvc_score_noalloc(cp2.cache, cp2.segs, case2.q, sp2.R, sp2.scale, s2, l2)
            torch.cuda.synchronize()
            cp2.score(case2.q, sp2.scale, want_lse=True)
            torch.cuda.synchronize()
            PT.check_scores(s2[:, :, :cp2.Ntot].cpu().numpy(), cp2.scores[:, :, :cp2.Ntot].double().cpu().numpy(),
                            "no-alloc call on the larger cache")
    assert kvc.kvc_read_device_status(clear=True) == 0
