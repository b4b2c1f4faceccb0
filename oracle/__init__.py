"""fp64 CPU oracle for online token-eviction compaction of a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA library (``online_kv_cache_gb300``)
and never imports it; the product path must not import this package.

The arithmetic lives in ``oracle.c`` (plain C, fp64, compiled with gcc); this
module only builds it, loads it with ctypes and marshals numpy arrays.  Each C
function cites the page passage it restates:

* scores  -- token-eviction score s_j = sqrt((1/q) sum_i alpha_ij^2) from
  "Practical Online KV Cache Compaction for LLM Agents" (section on the design
  space), with alpha = exp(logits - LSE) from the ActKV analysis page;
* select  -- top-m with ties to the lower position, ascending output;
* compact / free -- the ActKV conflict-free tail-region slot plan, simulated
  sequentially, and the return of the emptied blocks to the allocator;
* logical view -- the order-preserving out-of-place view (Chain Cache's
  logical-vs-physical split on the SparseEngine page);
* action attention / LRFU -- ActKV's action-critical entries (top 90% of the
  action attention mass) smoothed by LRFU (lambda = 0.5) into the eviction score;
* sentinel eviction / fresh-page compaction -- the layout-preserving dead
  slot (K = -10^4, V = 0) of the IntentKV page, and an order-preserving
  compaction into freshly allocated pages;
* Attention Matching (``oracle/am.py``, numpy fp64) -- the bias beta and the
  compact values V_C fitted on the survivors, from the tutorial page's section
  on the two compaction families.

Parity status: the score, selection and compaction functions are pinned by the
tests under ``tests/test_oracle_*.py`` (closed forms, invariants, brute force
over subsets and keep masks).  The readings the pages leave open (softmax
domain = segment, GQA pooling of all q*g rows, ascending-to-ascending pairing,
free-stack order) are fixed choices that no page value can confirm.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_budget_ratio.argtypes = [I64, D]
        lib.oracle_budget_ratio.restype = I64
        lib.oracle_budget_actkv.argtypes = [I]
        lib.oracle_budget_actkv.restype = I64
        lib.oracle_score_dense.argtypes = [P, P, I, I, I, D, P, P]
        lib.oracle_score_dense.restype = I
        lib.oracle_score_cache.argtypes = [P, P, P, I, I, I, I, I, I, P, P, P, I, P, I, D, P, P,
                                           P, I]
        lib.oracle_score_cache.restype = I
        lib.oracle_select.argtypes = [P, I, I, P]
        lib.oracle_select.restype = I
        lib.oracle_select_cache.argtypes = [P, I, I, P, P, I, P, P, I]
        lib.oracle_select_cache.restype = I
        lib.oracle_compact_layers.argtypes = [P, P, P, I, I, I, I, I, I, I, P, I, P, P, I, P, P]
        lib.oracle_compact_layers.restype = I
        lib.oracle_free_blocks.argtypes = [P, P, I, P, P, I, I, P, P, I, P]
        lib.oracle_free_blocks.restype = I
        lib.oracle_logical_view.argtypes = [P, P, P, I, I, I, I, I, I, P, I, P, I, P, P, P]
        lib.oracle_logical_view.restype = I
        lib.oracle_action_dense.argtypes = [P, P, I, I, I, D, P, P]
        lib.oracle_action_dense.restype = I
        lib.oracle_action_cache.argtypes = lib.oracle_score_cache.argtypes
        lib.oracle_action_cache.restype = I
        lib.oracle_action_hits.argtypes = [P, I, D, P]
        lib.oracle_action_hits.restype = I
        lib.oracle_lrfu_cache.argtypes = [P, I, I, I, I, P, I, P, P, I, P, D, D, P, P]
        lib.oracle_lrfu_cache.restype = I
        lib.oracle_sentinel_k_bits.argtypes = []
        lib.oracle_sentinel_k_bits.restype = ctypes.c_uint16
        lib.oracle_evict_sentinel.argtypes = [P, P, P, I, I, I, I, I, I, I, P, I, P, P, I, P, P]
        lib.oracle_evict_sentinel.restype = I
        lib.oracle_fresh_pages.argtypes = [P, ctypes.c_int32, I, P, P, I, P, P, P]
        lib.oracle_fresh_pages.restype = I
        lib.oracle_compact_fresh.argtypes = [P, P, P, I, I, I, I, I, I, I, P, I, P, P, I, P, P, P]
        lib.oracle_compact_fresh.restype = I
        lib.oracle_commit_fresh.argtypes = [P, P, I, P, P, I, I, P, P, I, P, P]
        lib.oracle_commit_fresh.restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(status: int, what: str):
    if status != OK:
        raise RuntimeError(f"oracle {what} failed with status {status}")


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else
               (os.cpu_count() or 1))


# --------------------------------------------------------------------------- budgets

def budget_ratio(n: int, ratio: float) -> int:
    return int(_load().oracle_budget_ratio(int(n), float(ratio)))


def budget_actkv(k: int) -> int:
    return int(_load().oracle_budget_actkv(int(k)))


# --------------------------------------------------------------------------- scores

def score_dense(Q: np.ndarray, K: np.ndarray, scale: float):
    """Scores of one unit from dense operands: returns (s[n], lse[R]) in fp64."""
    Q = _c(Q, np.float64)
    K = _c(K, np.float64)
    R, d = Q.shape
    n = K.shape[0]
    if K.ndim != 2 or (n and K.shape[1] != d):
        raise ValueError("Q is R x d and K is n x d")
    s = np.zeros(n, np.float64)
    lse = np.zeros(R, np.float64)
    _check(_load().oracle_score_dense(_ptr(Q), _ptr(K), R, n, d, float(scale), _ptr(s), _ptr(lse)),
           "score_dense")
    return s, lse


def _bits(a) -> np.ndarray:
    """bf16 array (torch tensor or uint16 numpy array) -> contiguous uint16 bits."""
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint16:
            raise TypeError("expected bf16 bits as uint16")
        return np.ascontiguousarray(a)
    import torch  # plumbing only: the oracle's arithmetic is in C
    t = a.detach().to("cpu").contiguous()
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return t.view(torch.int16).numpy().view(np.uint16)


def _i32(a) -> np.ndarray:
    if isinstance(a, np.ndarray):
        return _c(a, np.int32)
    if hasattr(a, "detach"):
        return _c(a.detach().to("cpu").numpy(), np.int32)
    return _c(np.asarray(a), np.int32)


def action_dense(Q: np.ndarray, K: np.ndarray, scale: float):
    """(a [n], lse [R]) in fp64: a_j = sum_i alpha_ij."""
    Q = _c(Q, np.float64)
    K = _c(K, np.float64)
    R, d = Q.shape
    n = K.shape[0]
    a = np.zeros(n, np.float64)
    lse = np.zeros(R, np.float64)
    _check(_load().oracle_action_dense(_ptr(Q), _ptr(K), R, n, d, float(scale), _ptr(a), _ptr(lse)),
           "action_dense")
    return a, lse


def action_hits(a: np.ndarray, frac: float = 0.9) -> np.ndarray:
    """0/1 flags of the action-critical entries of one unit."""
    a = _c(a, np.float64)
    hit = np.zeros(max(1, a.size), np.uint8)
    _check(_load().oracle_action_hits(_ptr(a), a.size, float(frac), _ptr(hit)), "action_hits")
    return hit[:a.size].astype(bool)


def lrfu_cache(crf_pool: np.ndarray, block_table, seg_start, seg_end, a: np.ndarray,
               frac: float = 0.9, lam: float = 0.5):
    """One LRFU step; crf_pool fp64 [L][num_pages][H][P] updated in place.  Returns (crf [L][H][Ntot],
    hits [L][H][Ntot] bool)."""
    if crf_pool.dtype != np.float64 or not crf_pool.flags.c_contiguous:
        raise TypeError("crf_pool must be a contiguous float64 array")
    L, num_pages, H, P = crf_pool.shape
    bt = _i32(block_table)
    s0, s1 = _i32(seg_start), _i32(seg_end)
    a = _c(a, np.float64)
    crf = np.zeros(a.shape, np.float64)
    hits = np.zeros(a.shape, np.uint8)
    _check(_load().oracle_lrfu_cache(_ptr(crf_pool), L, num_pages, H, P, _ptr(bt), bt.shape[1],
                                     _ptr(s0), _ptr(s1), len(s0), _ptr(a), float(frac), float(lam),
                                     _ptr(crf), _ptr(hits)), "lrfu_cache")
    return crf, hits.astype(bool)


def score_cache(k_pool, block_table, nblocks, seg_start, seg_end, seq_len, q, scale,
                unit_mask=None, threads=None, action=False):
    """Scores [L][H][Ntot] (fp64) and LSE [B][L][H][R] of every unit of a paged cache (with
    action=True the action attention a_j = sum_i alpha_ij instead of the score).

    k_pool: bf16 [L][num_pages][H][P][d]; q: bf16 [B][L][H][R][d]; the segment of
    sequence b is [seg_start[b], seg_end[b]) in its slot coordinates.  unit_mask
    [B][L][H] (bool) restricts the work to some units (others keep NaN)."""
    kb = _bits(k_pool)
    qb = _bits(q)
    L, num_pages, H, P, d = kb.shape
    B, Lq, Hq, R, dq = qb.shape
    if (Lq, Hq, dq) != (L, H, d):
        raise ValueError("q must be [B][L][H][R][d] matching the pool")
    bt = _i32(block_table)
    nbk = _i32(nblocks)
    s0 = _i32(seg_start)
    s1 = _i32(seg_end)
    sl = _i32(seq_len)
    Ntot = int((s1 - s0).sum())
    scores = np.full((L, H, Ntot), np.nan, np.float64)
    lse = np.full((B, L, H, R), np.nan, np.float64)
    mask = None if unit_mask is None else _c(np.asarray(unit_mask, dtype=bool).reshape(B, L, H),
                                             np.uint8)
    fn = _load().oracle_action_cache if action else _load().oracle_score_cache
    st = fn(_ptr(kb), _ptr(bt), _ptr(nbk), bt.shape[1], L, num_pages, H, P, d, _ptr(s0), _ptr(s1),
            _ptr(sl), B, _ptr(qb), R, float(scale), _ptr(mask), _ptr(scores), _ptr(lse),
            threads or default_threads())
    _check(st, "score_cache")
    return scores, lse


# --------------------------------------------------------------------------- selection

def select(s: np.ndarray, m: int) -> np.ndarray:
    """Top-m positions of one unit, ties to the lower position, ascending."""
    s = _c(s, np.float64)
    n = s.shape[0]
    keep = np.zeros(max(1, min(m, n)), np.int32)
    got = _load().oracle_select(_ptr(s), n, int(m), _ptr(keep))
    if got < 0:
        raise RuntimeError(f"oracle select failed with status {got}")
    return keep[:got].copy()


def select_cache(scores: np.ndarray, seg_start, seg_end, m, threads=None) -> np.ndarray:
    """Keep sets [L][H][Mtot] for scores [L][H][Ntot]."""
    scores = _c(scores, np.float64)
    L, H, _ = scores.shape
    s0, s1, mm = _i32(seg_start), _i32(seg_end), _i32(m)
    Mtot = int(np.minimum(mm, s1 - s0).sum())
    keep = np.full((L, H, max(Mtot, 1)), -1, np.int32)
    st = _load().oracle_select_cache(_ptr(scores), L, H, _ptr(s0), _ptr(s1), len(s0), _ptr(mm),
                                     _ptr(keep), threads or default_threads())
    _check(st, "select_cache")
    return keep[:, :, :Mtot].copy()


# --------------------------------------------------------------------------- compaction

def compact_layers(k_pool: np.ndarray, v_pool: np.ndarray, tags: np.ndarray, layer_lo: int,
                   L_total: int, block_table, seg_start, seg_end, m, keep: np.ndarray):
    """In-place compaction of pool slices holding layers [layer_lo, layer_lo + Lpart).

    k_pool / v_pool: uint16 bits [Lpart][num_pages][H][P][d] (modified in place),
    tags: int32 [Lpart][num_pages][H][P] (modified in place), keep [L_total][H][Mtot]."""
    for a, dt in ((k_pool, np.uint16), (v_pool, np.uint16), (tags, np.int32)):
        if a.dtype != dt or not a.flags.c_contiguous:
            raise TypeError("pool slices must be contiguous uint16 / int32 arrays")
    Lpart, num_pages, H, P, d = k_pool.shape
    bt = _i32(block_table)
    keep = _c(keep, np.int32)
    if keep.size == 0:
        keep = np.zeros(1, np.int32)
    s0, s1, mm = _i32(seg_start), _i32(seg_end), _i32(m)  # keep the buffers alive for the call
    st = _load().oracle_compact_layers(_ptr(k_pool), _ptr(v_pool), _ptr(tags), int(layer_lo), Lpart,
                                       int(L_total), num_pages, H, P, d, _ptr(bt), bt.shape[1],
                                       _ptr(s0), _ptr(s1), len(s0), _ptr(mm), _ptr(keep))
    _check(st, "compact_layers")


def free_blocks(block_table: np.ndarray, nblocks: np.ndarray, free_ids: np.ndarray,
                free_top: np.ndarray, P: int, seg_start, seg_end, m):
    """In-place update of the block table, block counts and free stack."""
    for a in (block_table, nblocks, free_ids, free_top):
        if a.dtype != np.int32 or not a.flags.c_contiguous:
            raise TypeError("allocator state must be contiguous int32 arrays")
    s0, s1, mm = _i32(seg_start), _i32(seg_end), _i32(m)
    st = _load().oracle_free_blocks(_ptr(block_table), _ptr(nblocks), block_table.shape[1],
                                    _ptr(free_ids), _ptr(free_top), free_ids.shape[0], int(P),
                                    _ptr(s0), _ptr(s1), len(s0), _ptr(mm))
    _check(st, "free_blocks")


def logical_view(k_pool: np.ndarray, v_pool: np.ndarray, tags: np.ndarray, layer: int, head: int,
                 bt_row, s0: int, keep: np.ndarray):
    """(Kc [m][d], Vc [m][d], pos [m]) of one unit before compaction, in keep order."""
    kb, vb, tg = _bits(k_pool), _bits(v_pool), _i32(tags)
    L, num_pages, H, P, d = kb.shape
    keep = _c(keep, np.int32)
    m = keep.shape[0]
    if m == 0:
        keep = np.zeros(1, np.int32)
    row = _i32(bt_row)
    Kc = np.zeros((max(m, 1), d), np.uint16)
    Vc = np.zeros((max(m, 1), d), np.uint16)
    pos = np.zeros(max(m, 1), np.int32)
    st = _load().oracle_logical_view(_ptr(kb), _ptr(vb), _ptr(tg), int(layer), int(head),
                                     num_pages, H, P, d, _ptr(row), int(s0), _ptr(keep), m,
                                     _ptr(Kc), _ptr(Vc), _ptr(pos))
    _check(st, "logical_view")
    return Kc[:m], Vc[:m], pos[:m]


# --------------------------------------------------------------------------- layout variants

def sentinel_k_bits() -> int:
    """bf16 bit pattern of the sentinel key element, bf16(-10^4)."""
    return int(_load().oracle_sentinel_k_bits())


def _pool_args(k_pool, v_pool, tags):
    for a, dt in ((k_pool, np.uint16), (v_pool, np.uint16), (tags, np.int32)):
        if a.dtype != dt or not a.flags.c_contiguous:
            raise TypeError("pool slices must be contiguous uint16 / int32 arrays")
    return k_pool.shape


def evict_sentinel(k_pool: np.ndarray, v_pool: np.ndarray, tags: np.ndarray, layer_lo: int,
                   L_total: int, block_table, seg_start, seg_end, m, keep: np.ndarray):
    """In place: every evicted position of every unit becomes a sentinel dead slot."""
    Lpart, num_pages, H, P, d = _pool_args(k_pool, v_pool, tags)
    bt = _i32(block_table)
    keep = _c(keep, np.int32)
    if keep.size == 0:
        keep = np.zeros(1, np.int32)
    s0, s1, mm = _i32(seg_start), _i32(seg_end), _i32(m)
    st = _load().oracle_evict_sentinel(_ptr(k_pool), _ptr(v_pool), _ptr(tags), int(layer_lo), Lpart,
                                       int(L_total), num_pages, H, P, d, _ptr(bt), bt.shape[1],
                                       _ptr(s0), _ptr(s1), len(s0), _ptr(mm), _ptr(keep))
    _check(st, "evict_sentinel")


def fresh_pages(free_ids: np.ndarray, free_top: int, P: int, seg_start, seg_end, m) -> np.ndarray:
    """Pages the fresh-page compaction pops, in pop order (sequences ascending)."""
    fi = _i32(free_ids)
    s0, s1, mm = _i32(seg_start), _i32(seg_end), _i32(m)
    count = np.zeros(1, np.int32)
    lib = _load()
    _check(lib.oracle_fresh_pages(_ptr(fi), int(free_top), int(P), _ptr(s0), _ptr(s1), len(s0),
                                  _ptr(mm), None, _ptr(count)), "fresh_pages")
    out = np.zeros(max(1, int(count[0])), np.int32)
    _check(lib.oracle_fresh_pages(_ptr(fi), int(free_top), int(P), _ptr(s0), _ptr(s1), len(s0),
                                  _ptr(mm), _ptr(out), _ptr(count)), "fresh_pages")
    return out[:int(count[0])]


def compact_fresh(k_pool: np.ndarray, v_pool: np.ndarray, tags: np.ndarray, layer_lo: int,
                  L_total: int, block_table, seg_start, seg_end, m, keep: np.ndarray,
                  fresh: np.ndarray):
    """In place: survivors of active sequences copied, in order, into their fresh pages."""
    Lpart, num_pages, H, P, d = _pool_args(k_pool, v_pool, tags)
    bt = _i32(block_table)
    keep = _c(keep, np.int32)
    if keep.size == 0:
        keep = np.zeros(1, np.int32)
    fr = _c(fresh, np.int32)
    if fr.size == 0:
        fr = np.zeros(1, np.int32)
    s0, s1, mm = _i32(seg_start), _i32(seg_end), _i32(m)
    st = _load().oracle_compact_fresh(_ptr(k_pool), _ptr(v_pool), _ptr(tags), int(layer_lo), Lpart,
                                      int(L_total), num_pages, H, P, d, _ptr(bt), bt.shape[1],
                                      _ptr(s0), _ptr(s1), len(s0), _ptr(mm), _ptr(keep), _ptr(fr))
    _check(st, "compact_fresh")


def commit_fresh(block_table: np.ndarray, nblocks: np.ndarray, free_ids: np.ndarray,
                 free_top: np.ndarray, P: int, seg_start, seg_end, m, fresh: np.ndarray):
    """In place: pops the fresh pages, returns the old ones, installs the new rows."""
    for a in (block_table, nblocks, free_ids, free_top):
        if a.dtype != np.int32 or not a.flags.c_contiguous:
            raise TypeError("allocator state must be contiguous int32 arrays")
    fr = _c(fresh, np.int32)
    if fr.size == 0:
        fr = np.zeros(1, np.int32)
    s0, s1, mm = _i32(seg_start), _i32(seg_end), _i32(m)
    st = _load().oracle_commit_fresh(_ptr(block_table), _ptr(nblocks), block_table.shape[1],
                                     _ptr(free_ids), _ptr(free_top), free_ids.shape[0], int(P),
                                     _ptr(s0), _ptr(s1), len(s0), _ptr(mm), _ptr(fr))
    _check(st, "commit_fresh")


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
