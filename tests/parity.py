"""Parity helpers shared by the GPU tests: run the CUDA path through the C ABI, run the oracle
on host copies of the same seeded inputs, compare with the documented rules.

Rules (the stated tolerances of the hot path; the score bound comes from fp32 logits of bf16
operands and fp32 exp/accumulation):
* scores: |s_gpu - s_orc| <= 2e-3 * s_orc where s_orc >= 1e-30, else s_gpu <= 1e-27;
* LSE: |lse_gpu - lse_orc| <= 1e-4 * max(1, |lse_orc|) (fp32 log-sum-exp of fp32 logits);
* keep sets: identical except positions whose oracle score lies within 1e-4 relative of the
  m-th oracle score; exactly m positions, ascending, unique;
* compaction (pools, tags, block table, nblocks, free stack): bit-exact given the selection.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import online_kv_cache_gb300 as kvc
import workloads

SCORE_RTOL = 2e-3
SCORE_FLOOR = 1e-30
SCORE_TINY = 1e-27
LSE_TOL = 1e-4
BAND = 1e-4


def seg_lengths(case):
    return [e - s for s, e in zip(case.seg_start, case.seg_end)]


def oracle_budgets(case):
    kind, arg = case.spec.budget
    n = seg_lengths(case)
    if kind == "ratio":
        return [oracle.budget_ratio(x, arg) for x in n]
    return [min(oracle.budget_actkv(k), x) for k, x in zip(arg, n)]


def lib_budgets(case):
    kind, arg = case.spec.budget
    n = seg_lengths(case)
    if kind == "ratio":
        return [kvc.kvc_budget_from_ratio(x, arg) for x in n]
    return [min(kvc.kvc_budget_actkv(k), x) for k, x in zip(arg, n)]


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def i32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().astype(np.int32)


def host_state(case, layers=None):
    sl = slice(None) if layers is None else slice(*layers)
    return dict(k=bits(case.k_pool[sl]), v=bits(case.v_pool[sl]), tags=i32(case.tags[sl]),
                bt=i32(case.block_table), nblocks=i32(case.nblocks), free_ids=i32(case.free_ids),
                free_top=i32(case.free_top))


def compactor(case, m):
    return kvc.Compactor(case.k_pool, case.v_pool, case.tags, case.block_table, case.nblocks,
                         case.free_ids, case.free_top, case.seg_start, case.seg_end, case.seq_len,
                         m, case.spec.R)


def oracle_scores(case, unit_mask=None):
    return oracle.score_cache(case.k_pool, case.block_table, case.nblocks, case.seg_start,
                              case.seg_end, case.seq_len, case.q, case.spec.scale, unit_mask)


def check_scores(s_gpu: np.ndarray, s_orc: np.ndarray, what=""):
    s_gpu = np.asarray(s_gpu, np.float64)
    big = s_orc >= SCORE_FLOOR
    rel = np.abs(s_gpu[big] - s_orc[big]) / s_orc[big]
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= SCORE_RTOL, f"{what}: max relative score error {worst:.3e}"
    assert np.all(s_gpu[~big] <= SCORE_TINY), f"{what}: tiny scores not tiny"
    assert np.all(np.isfinite(s_gpu)), f"{what}: non-finite score"
    return worst


def check_lse(l_gpu: np.ndarray, l_orc: np.ndarray, what=""):
    err = np.abs(np.asarray(l_gpu, np.float64) - l_orc) / np.maximum(1.0, np.abs(l_orc))
    worst = float(err.max()) if err.size else 0.0
    assert worst <= LSE_TOL, f"{what}: max LSE error {worst:.3e}"
    return worst


def check_keep(k_gpu: np.ndarray, k_orc: np.ndarray, s_orc: np.ndarray, m: int, what=""):
    """Keep-set rule; returns the number of in-band differences."""
    k_gpu = np.asarray(k_gpu)
    assert k_gpu.shape[0] == m, f"{what}: {k_gpu.shape[0]} kept, expected {m}"
    if m == 0:
        return 0
    assert np.all(np.diff(k_gpu) > 0), f"{what}: keep not strictly ascending"
    assert k_gpu[0] >= 0 and k_gpu[-1] < s_orc.shape[0], f"{what}: keep out of range"
    diff = np.setxor1d(k_gpu, k_orc)
    if diff.size == 0:
        return 0
    s_m = np.sort(s_orc)[::-1][m - 1]
    inband = np.abs(s_orc[diff] - s_m) <= BAND * s_m
    assert np.all(inband), (f"{what}: {int((~inband).sum())} selection differences outside the "
                            f"1e-4 band, e.g. positions {diff[~inband][:8]}")
    return int(diff.size)


def oracle_compaction(state, case, m, keep_np, layer_lo=0):
    """Oracle compaction of the host state (in place); keep_np [L][H][Mtot]."""
    L_total = case.spec.L
    oracle.compact_layers(state["k"], state["v"], state["tags"], layer_lo, L_total, state["bt"],
                          case.seg_start, case.seg_end, m, keep_np)
    oracle.free_blocks(state["bt"], state["nblocks"], state["free_ids"], state["free_top"],
                       case.spec.P, case.seg_start, case.seg_end, m)
    return state


def assert_state_equal(gpu_state, orc_state, what=""):
    for key in ("k", "v", "tags", "bt", "nblocks", "free_ids", "free_top"):
        a, b = gpu_state[key], orc_state[key]
        if not np.array_equal(a, b):
            bad = np.argwhere(a != b)
            raise AssertionError(f"{what}: {key} differs at {bad.shape[0]} positions, first "
                                 f"{bad[:4].tolist()}")


def run_chain(case, m, want_lse=True, keep_override=None):
    """Runs the five C-ABI calls on the current stream; returns the Compactor."""
    cp = compactor(case, m)
    cp.score(case.q, case.spec.scale, want_lse)
    cp.select()
    cp.plan_compact(keep_override)
    cp.compact()
    cp.free_pages()
    return cp


def device_status_clean():
    st = kvc.kvc_read_device_status(clear=True)
    assert st == 0, f"device status word = {st:#x}"


def host_state_from(snap):
    """Host copies of a Case.snapshot() list (k, v, tags, bt, nblocks, free_ids, free_top)."""
    k, v, tags, bt, nb, fi, ft = snap
    return dict(k=bits(k), v=bits(v), tags=i32(tags), bt=i32(bt), nblocks=i32(nb),
                free_ids=i32(fi), free_top=i32(ft))


def unit_offsets(case, m):
    n = seg_lengths(case)
    noff = np.concatenate([[0], np.cumsum(n)]).astype(np.int64)
    moff = np.concatenate([[0], np.cumsum([min(a, b) for a, b in zip(m, n)])]).astype(np.int64)
    return noff, moff
