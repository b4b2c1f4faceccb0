"""Host-side tests of the C ABI: the library loads, exports every symbol include/kvc.h
declares, validates arguments before any launch, and its host helpers agree with the oracle.
No test here needs a GPU or launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

import online_kv_cache_gb300 as kvc
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kvc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from online_kv_cache_gb300 import build
    build.build()
    return kvc.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(kvc.EXPORTED)


def test_version(lib):
    assert "sm_103a" in kvc.kvc_version()


def test_budget_helpers_agree_with_oracle(lib):
    rng = np.random.default_rng(0)
    for n in list(range(0, 200)) + list(rng.integers(1, 300000, 300)):
        for ratio in (0.0, 0.07, 0.1, 0.2, 0.25, 0.333, 0.5, 0.9, 1.0, 1.5, -0.1):
            assert kvc.kvc_budget_from_ratio(int(n), ratio) == oracle.budget_ratio(int(n), ratio)
    for k in range(-1, 25):
        want = oracle.budget_actkv(k)
        assert kvc.kvc_budget_actkv(k) == want
    assert [kvc.kvc_budget_actkv(k) for k in range(7)] == [512, 896, 1568, 2744, 4802, 8403, 14706]


def fake_cache(L=2, num_pages=64, H=2, P=16, d=128, max_blocks=8, batch=2):
    # 16-byte aligned fake device addresses: host validation never dereferences them
    return kvc.kvc_cache(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, L, num_pages, H, P, d,
                         max_blocks, batch)


def segs(s0, s1, sl):
    keep_alive = [np.asarray(x, np.int32) for x in (s0, s1, sl)]
    s = kvc.kvc_segments(*(a.ctypes.data for a in keep_alive), len(keep_alive[0]))
    return s, keep_alive


def ws_size(lib, cache, seg, R):
    out = ctypes.c_size_t(0)
    return lib.kvc_score_workspace_size(ctypes.byref(cache), ctypes.byref(seg), R, ctypes.byref(out)), out.value


def score_call(lib, cache, seg, R=16, scale=0.1, q=0x60000, scores=0x70000, ws=0x80000, ws_bytes=1 << 30):
    return lib.kvc_score(ctypes.byref(cache), ctypes.byref(seg), q, R, scale, scores, None, ws,
                         ws_bytes, None)


def test_score_argument_validation(lib):
    c = fake_cache()
    s, _ = segs([0, 16], [100, 64], [100, 80])
    assert ws_size(lib, c, s, 16)[0] == kvc.KVC_OK
    # bad head dim / page size / R
    for field, val, want in (("head_dim", 96, kvc.KVC_ERR_UNSUPPORTED),
                             ("page_size", 12, kvc.KVC_ERR_UNSUPPORTED),
                             ("page_size", 128, kvc.KVC_ERR_UNSUPPORTED),
                             ("num_layers", 0, kvc.KVC_ERR_INVALID_ARG)):
        bad = fake_cache()
        setattr(bad, field, val)
        assert score_call(lib, bad, s) == want, field
    assert score_call(lib, c, s, R=0) == kvc.KVC_ERR_UNSUPPORTED
    assert score_call(lib, c, s, R=4097) == kvc.KVC_ERR_UNSUPPORTED
    assert score_call(lib, c, s, scale=0.0) == kvc.KVC_ERR_INVALID_ARG
    assert score_call(lib, c, s, scale=float("nan")) == kvc.KVC_ERR_INVALID_ARG
    assert score_call(lib, c, s, q=0x60008) == kvc.KVC_ERR_INVALID_ARG  # misaligned q
    bad = fake_cache()
    bad.k_pool = 0x10008
    assert score_call(lib, bad, s) == kvc.KVC_ERR_INVALID_ARG
    # workspace too small or misaligned
    assert score_call(lib, c, s, ws_bytes=16) == kvc.KVC_ERR_WORKSPACE
    assert score_call(lib, c, s, ws=0x80010) == kvc.KVC_ERR_WORKSPACE
    assert "workspace" in kvc.kvc_last_error()


@pytest.mark.parametrize("s0,s1,sl,want", [
    ([8, 0], [100, 64], [100, 80], kvc.KVC_ERR_UNALIGNED_SEGMENT),   # start off a block boundary
    ([0, 0], [90, 64], [100, 80], kvc.KVC_ERR_UNALIGNED_SEGMENT),    # ragged end, not seq end
    ([0, 0], [101, 64], [100, 80], kvc.KVC_ERR_INVALID_ARG),         # past the sequence
    ([32, 0], [16, 64], [100, 80], kvc.KVC_ERR_INVALID_ARG),         # reversed
    ([0, 0], [100, 64], [100, 200], kvc.KVC_ERR_INVALID_ARG),        # seq_len > max_blocks*P
])
def test_segment_validation(lib, s0, s1, sl, want):
    c = fake_cache()
    s, _ = segs(s0, s1, sl)
    assert score_call(lib, c, s) == want


def test_batch_mismatch_and_null_segments(lib):
    c = fake_cache(batch=3)
    s, _ = segs([0, 0], [16, 16], [16, 16])
    assert score_call(lib, c, s) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_score(ctypes.byref(c), None, 0x60000, 16, 0.1, 0x70000, None, 0x80000, 1 << 30,
                         None) == kvc.KVC_ERR_INVALID_ARG


def test_budget_and_plan_validation(lib):
    c = fake_cache()
    s, _ = segs([0, 16], [100, 64], [100, 80])
    m = np.array([20, -1], np.int32)
    out = kvc.kvc_plan_sizes()
    assert lib.kvc_plan_buffer_sizes(ctypes.byref(c), ctypes.byref(s), m.ctypes.data,
                                     ctypes.byref(out)) == kvc.KVC_ERR_BUDGET
    m = np.array([20, 100], np.int32)  # clamped to n = 48
    assert lib.kvc_plan_buffer_sizes(ctypes.byref(c), ctypes.byref(s), m.ctypes.data,
                                     ctypes.byref(out)) == kvc.KVC_OK
    assert out.Mtot == 20 + 48 and out.Ntot == 100 + 48
    assert out.moves_len == 2 * 2 * 2 * 68
    assert out.freed_len == (7 - 2) + (3 - 3)
    assert out.units_len == 2 * 2 * 2 and out.dead_len == 2 * 2 * 2 * 16
    # an undersized plan is rejected before any launch
    plan = kvc.kvc_plan(0x100, 0x200, 0x300, 0x400, 0x500, 0x600, out.moves_len - 1, out.units_len,
                        out.dead_len, out.freed_len, out.new_rows_len)
    assert lib.kvc_plan_compact(ctypes.byref(c), ctypes.byref(s), m.ctypes.data, 0x700,
                                ctypes.byref(plan), None) == kvc.KVC_ERR_WORKSPACE
    assert lib.kvc_compact(ctypes.byref(c), ctypes.byref(s), m.ctypes.data, ctypes.byref(plan),
                           None) == kvc.KVC_ERR_WORKSPACE
    alloc = kvc.kvc_allocator(0x800, None, 10)
    plan.moves_len = out.moves_len
    assert lib.kvc_free_pages(ctypes.byref(c), ctypes.byref(s), m.ctypes.data, ctypes.byref(alloc),
                              ctypes.byref(plan), None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_select_topm(ctypes.byref(c), ctypes.byref(s), 0x100, None, 0x200, None, 0,
                               None) == kvc.KVC_ERR_INVALID_ARG


def test_select_rejects_overlong_segments_before_any_launch(lib):
    """Selection takes segments of at most 2^20 - 4096 positions (its per-warp 16-bit bin counts);
    one position more is KVC_ERR_UNSUPPORTED, decided on the host."""
    longest = (1 << 20) - 4096
    c = fake_cache(L=1, num_pages=16384, H=1, P=64, d=128, max_blocks=16384, batch=1)
    for n in (longest + 1, 1 << 20):
        s, keep_alive = segs([0], [n], [n])
        m = np.array([100], np.int32)
        st = lib.kvc_select_topm(ctypes.byref(c), ctypes.byref(s), 0x100, m.ctypes.data, 0x200, None, 0, None)
        assert st == kvc.KVC_ERR_UNSUPPORTED
        assert str(longest) in kvc.kvc_last_error()


def test_status_strings(lib):
    for st in range(-7, 1):
        assert kvc.kvc_status_string(st).startswith("KVC_")
    assert kvc.kvc_status_string(-99) == "KVC_ERR_UNKNOWN"


# ------------------------------------------------------------------ host validator

def good_state():
    bt = np.array([[3, 0, 5, -1], [1, 4, -1, -1]], np.int32)
    nb = np.array([3, 2], np.int32)
    free = np.array([7, 6, 2, 0, 0, 0, 0, 0], np.int32)
    return bt, nb, free


def test_validator_accepts_consistent_state(lib):
    bt, nb, free = good_state()
    kvc.kvc_validate_cache_host(bt, nb, [40, 20], 8, 16, free, 3)


@pytest.mark.parametrize("mutate,msg", [
    (lambda bt, nb, fr: bt.__setitem__((1, 1), 3), "mapped twice"),
    (lambda bt, nb, fr: bt.__setitem__((0, 0), 8), "outside the pool"),
    (lambda bt, nb, fr: bt.__setitem__((0, 3), 6), "not -1"),
    (lambda bt, nb, fr: fr.__setitem__(0, 5), "both mapped and free"),
    (lambda bt, nb, fr: fr.__setitem__(1, 7), "free twice"),
    (lambda bt, nb, fr: nb.__setitem__(1, 5), "out of range"),
])
def test_validator_rejects(lib, mutate, msg):
    bt, nb, free = good_state()
    mutate(bt, nb, free)
    with pytest.raises(kvc.KvcError) as ei:
        kvc.kvc_validate_cache_host(bt, nb, None, 8, 16, free, 3)
    assert msg in str(ei.value)


def test_validator_seq_len(lib):
    bt, nb, free = good_state()
    with pytest.raises(kvc.KvcError):
        kvc.kvc_validate_cache_host(bt, nb, [49, 20], 8, 16, free, 3)  # 49 slots need 4 blocks


def test_noalloc_rejects_workspace_beyond_its_scratch(lib):
    """kvc_score_noalloc refuses, before any launch, a call whose workspace exceeds its 16 MiB."""
    c = fake_cache(L=64, num_pages=40000, H=8, P=16, d=128, max_blocks=4096, batch=1)
    s, _ = segs([0], [65536], [65536])
    need = ctypes.c_size_t(0)
    assert lib.kvc_score_workspace_size(ctypes.byref(c), ctypes.byref(s), 4096, ctypes.byref(need)) == 0
    assert need.value > 16 << 20
    st = lib.kvc_score_noalloc(ctypes.byref(c), ctypes.byref(s), 0x60000, 4096, 0.1, 0x70000, None, None)
    assert st == kvc.KVC_ERR_WORKSPACE
    assert "scratch" in kvc.kvc_last_error()


def test_layout_variant_validation(lib):
    """The sentinel and fresh-page entry points validate before any launch; the fresh plan's
    return list holds every block of the segments that keep fewer than all positions."""
    c = fake_cache()
    s, _ = segs([0, 16], [100, 64], [100, 80])
    m = np.array([20, 48], np.int32)  # sequence 1 keeps all 48 of its positions
    assert lib.kvc_evict_sentinel(ctypes.byref(c), ctypes.byref(s), m.ctypes.data, None,
                                  None) == kvc.KVC_ERR_INVALID_ARG
    out = kvc.kvc_plan_sizes()
    assert lib.kvc_plan_fresh_buffer_sizes(ctypes.byref(c), ctypes.byref(s), m.ctypes.data,
                                           ctypes.byref(out)) == kvc.KVC_OK
    assert out.freed_len == 7  # ceil(100/16) blocks of sequence 0; sequence 1 is untouched
    assert out.moves_len == 2 * 2 * 2 * 68
    plan = kvc.kvc_plan(0x100, 0x200, 0x300, 0x400, 0x500, 0x600, out.moves_len, out.units_len,
                        out.dead_len, out.freed_len - 1, out.new_rows_len)
    alloc = kvc.kvc_allocator(0x800, 0x900, 10)
    assert lib.kvc_plan_fresh(ctypes.byref(c), ctypes.byref(s), m.ctypes.data, 0x700, None,
                              ctypes.byref(plan), None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_plan_fresh(ctypes.byref(c), ctypes.byref(s), m.ctypes.data, 0x700,
                              ctypes.byref(alloc), ctypes.byref(plan), None) == kvc.KVC_ERR_WORKSPACE
    assert "freed" in kvc.kvc_last_error()
    assert lib.kvc_commit_fresh(ctypes.byref(c), ctypes.byref(s), m.ctypes.data, ctypes.byref(alloc),
                                ctypes.byref(plan), None) == kvc.KVC_ERR_WORKSPACE
    bad = np.array([20, -1], np.int32)
    assert lib.kvc_evict_sentinel(ctypes.byref(c), ctypes.byref(s), bad.ctypes.data, 0x700,
                                  None) == kvc.KVC_ERR_BUDGET


def test_am_validation(lib):
    """kvc_am_fit checks its arguments before any launch: budget and row limits of the m x m
    fits, sweeps, pointers and the workspace; the workspace grows with R and is 0 when nothing is
    kept."""
    c = fake_cache()
    s, _ = segs([0, 16], [100, 64], [100, 80])
    m = np.array([20, 48], np.int32)

    def size(mm, R):
        out = ctypes.c_size_t(0)
        st = lib.kvc_am_workspace_size(ctypes.byref(c), ctypes.byref(s), mm.ctypes.data, R, ctypes.byref(out))
        return st, out.value

    st, b16 = size(m, 16)
    assert st == kvc.KVC_OK and b16 > 0 and b16 % 256 == 0
    # the header's count: per unit about 4 ((R + M)(M + 4) + R (d + 1) + M (5 d + 1)) bytes with M the
    # largest m launched together, plus the LSE pass's workspace and 4 B L H R bytes of row LSE
    for R in (16, 64, 200):
        M, d = int(m.max()), c.head_dim
        units = 2 * c.num_layers * c.num_kv_heads
        floats = (R + M) * (M + 4) + R * (d + 1) + M * (5 * d + 1)
        score = ctypes.c_size_t(0)
        assert lib.kvc_score_workspace_size(ctypes.byref(c), ctypes.byref(s), R, ctypes.byref(score)) == kvc.KVC_OK
        low = units * 4 * floats + score.value + 4 * c.batch * c.num_layers * c.num_kv_heads * R
        got = size(m, R)[1]
        assert low <= got <= low + units * (256 + 64) + 3 * 256, (R, got, low)
    assert size(m, 64)[1] > b16
    assert size(np.zeros(2, np.int32), 16) == (kvc.KVC_OK, 0)
    assert size(m, 4097)[0] == kvc.KVC_ERR_UNSUPPORTED
    assert size(m, 0)[0] == kvc.KVC_ERR_UNSUPPORTED

    def fit(mm=m, R=16, scale=0.1, q=0x60000, keep=0x70000, sweeps=4, ws=0x80000, ws_bytes=1 << 30, lse=None):
        return lib.kvc_am_fit(ctypes.byref(c), ctypes.byref(s), mm.ctypes.data, q, R, scale, lse, keep, sweeps,
                              None, None, ws, ws_bytes, None)

    assert fit(sweeps=-1) == kvc.KVC_ERR_INVALID_ARG
    assert fit(sweeps=1001) == kvc.KVC_ERR_INVALID_ARG
    assert fit(scale=float("inf")) == kvc.KVC_ERR_INVALID_ARG
    assert fit(q=0x60004) == kvc.KVC_ERR_INVALID_ARG
    assert fit(keep=None) == kvc.KVC_ERR_INVALID_ARG
    assert fit(lse=0x90002) == kvc.KVC_ERR_INVALID_ARG  # a caller's LSE must be 4-byte aligned
    assert fit(ws_bytes=b16 - 256) == kvc.KVC_ERR_WORKSPACE
    assert fit(ws=0x80010) == kvc.KVC_ERR_WORKSPACE
    assert fit(np.array([20, -1], np.int32)) == kvc.KVC_ERR_BUDGET
    big = fake_cache(max_blocks=256)
    sb, _ = segs([0, 0], [3000, 16], [3000, 16])
    out = ctypes.c_size_t(0)
    assert lib.kvc_am_workspace_size(ctypes.byref(big), ctypes.byref(sb), np.array([2049, 1], np.int32).ctypes.data,
                                     16, ctypes.byref(out)) == kvc.KVC_ERR_UNSUPPORTED
    assert "2048" in kvc.kvc_last_error()
