"""Python binding of libkvc: online token-eviction compaction of a paged KV cache on GB300.

Argument marshalling only.  Every step of the hot path runs in the CUDA kernels of
``libkvc.so`` behind the C ABI declared in ``include/kvc.h``; PyTorch provides device
memory and streams.  There is no CPU fallback: if the library has not been built (see
``online_kv_cache_gb300.build``), every call raises ``KvcLibraryMissing``.

The functions keep the C names:

    kvc_score -> kvc_select_topm -> kvc_plan_compact -> kvc_compact -> kvc_free_pages

``Compactor`` owns the workspace and plan buffers for one cache and issues the five calls
in order on the current stream.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")

KVC_OK = 0
KVC_ERR_INVALID_ARG = -1
KVC_ERR_UNALIGNED_SEGMENT = -2
KVC_ERR_BUDGET = -3
KVC_ERR_WORKSPACE = -4
KVC_ERR_UNSUPPORTED = -5
KVC_ERR_CUDA = -6
KVC_ERR_DEVICE_CHECK = -7

KVC_DEV_WAIT_TIMEOUT = 1
KVC_DEV_FREE_STACK = 2
KVC_DEV_BAD_PAGE = 4
KVC_DEV_BAD_KEEP = 8

EXPORTED = (
    "kvc_budget_from_ratio", "kvc_budget_actkv", "kvc_score_workspace_size", "kvc_score",
    "kvc_select_workspace_size", "kvc_select_topm", "kvc_plan_buffer_sizes", "kvc_plan_compact",
    "kvc_compact", "kvc_free_pages", "kvc_status_string", "kvc_last_error",
    "kvc_read_device_status", "kvc_validate_cache_host", "kvc_version", "kvc_score_lse",
    "kvc_score_alpha", "kvc_launch_count", "kvc_score_noalloc", "kvc_evict_sentinel",
    "kvc_plan_fresh_buffer_sizes", "kvc_plan_fresh", "kvc_commit_fresh", "kvc_score_action",
    "kvc_lrfu_update", "kvc_am_workspace_size", "kvc_am_fit", "kvc_debug_stall_scoring",
)


class KvcLibraryMissing(RuntimeError):
    pass


class KvcError(RuntimeError):
    def __init__(self, status: int, where: str, text: str):
        self.status = status
        super().__init__(f"{where}: {status_name(status)}: {text}")


class kvc_cache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("tags", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("nblocks", ctypes.c_void_p),
                ("num_layers", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("aux", ctypes.c_void_p)]


class kvc_segments(ctypes.Structure):
    _fields_ = [("seg_start", ctypes.c_void_p), ("seg_end", ctypes.c_void_p),
                ("seq_len", ctypes.c_void_p), ("batch", ctypes.c_int32)]


class kvc_allocator(ctypes.Structure):
    _fields_ = [("free_ids", ctypes.c_void_p), ("free_top", ctypes.c_void_p),
                ("capacity", ctypes.c_int32)]


class kvc_plan(ctypes.Structure):
    _fields_ = [("moves", ctypes.c_void_p), ("move_count", ctypes.c_void_p),
                ("dead", ctypes.c_void_p), ("dead_count", ctypes.c_void_p),
                ("freed", ctypes.c_void_p), ("new_rows", ctypes.c_void_p),
                ("moves_len", ctypes.c_int64), ("units_len", ctypes.c_int64),
                ("dead_len", ctypes.c_int64), ("freed_len", ctypes.c_int64),
                ("new_rows_len", ctypes.c_int64)]


class kvc_plan_sizes(ctypes.Structure):
    _fields_ = [("moves_len", ctypes.c_int64), ("units_len", ctypes.c_int64),
                ("dead_len", ctypes.c_int64), ("freed_len", ctypes.c_int64),
                ("new_rows_len", ctypes.c_int64), ("Mtot", ctypes.c_int64),
                ("Ntot", ctypes.c_int64)]


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libkvc.so (raises KvcLibraryMissing if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise KvcLibraryMissing(
                f"{LIB_PATH} is missing: build it with `python -m online_kv_cache_gb300.build` "
                "(nvcc, sm_103a); there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, D, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_float
        S = ctypes.c_size_t
        C, SG, A, PL = (ctypes.POINTER(kvc_cache), ctypes.POINTER(kvc_segments),
                        ctypes.POINTER(kvc_allocator), ctypes.POINTER(kvc_plan))
        sig = {
            "kvc_budget_from_ratio": (I64, [I64, D]),
            "kvc_budget_actkv": (I64, [I32]),
            "kvc_score_workspace_size": (I32, [C, SG, I32, ctypes.POINTER(S)]),
            "kvc_score": (I32, [C, SG, P, I32, F, P, P, P, S, P]),
            "kvc_select_workspace_size": (I32, [C, SG, P, ctypes.POINTER(S)]),
            "kvc_select_topm": (I32, [C, SG, P, P, P, P, S, P]),
            "kvc_plan_buffer_sizes": (I32, [C, SG, P, ctypes.POINTER(kvc_plan_sizes)]),
            "kvc_plan_compact": (I32, [C, SG, P, P, PL, P]),
            "kvc_compact": (I32, [C, SG, P, PL, P]),
            "kvc_free_pages": (I32, [C, SG, P, A, PL, P]),
            "kvc_status_string": (ctypes.c_char_p, [I32]),
            "kvc_last_error": (ctypes.c_char_p, []),
            "kvc_read_device_status": (I32, [ctypes.POINTER(ctypes.c_uint32), I32, P]),
            "kvc_validate_cache_host": (I32, [P, P, P, I32, I32, I32, I32, P, I32]),
            "kvc_version": (ctypes.c_char_p, []),
            "kvc_score_lse": (I32, [C, SG, P, I32, F, P, P, S, P]),
            "kvc_score_alpha": (I32, [C, SG, P, I32, F, P, P, P, S, P]),
            "kvc_launch_count": (ctypes.c_uint64, [I32]),
            "kvc_score_noalloc": (I32, [C, SG, P, I32, F, P, P, P]),
            "kvc_evict_sentinel": (I32, [C, SG, P, P, P]),
            "kvc_plan_fresh_buffer_sizes": (I32, [C, SG, P, ctypes.POINTER(kvc_plan_sizes)]),
            "kvc_plan_fresh": (I32, [C, SG, P, P, A, PL, P]),
            "kvc_commit_fresh": (I32, [C, SG, P, A, PL, P]),
            "kvc_score_action": (I32, [C, SG, P, I32, F, P, P, P, S, P]),
            "kvc_lrfu_update": (I32, [C, SG, P, F, F, P, P, P]),
            "kvc_am_workspace_size": (I32, [C, SG, P, I32, ctypes.POINTER(S)]),
            "kvc_am_fit": (I32, [C, SG, P, P, I32, F, P, P, I32, P, P, P, S, P]),
            "kvc_debug_stall_scoring": (I32, [I64]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def status_name(status: int) -> str:
    try:
        return lib().kvc_status_string(int(status)).decode()
    except KvcLibraryMissing:
        return str(status)


def _check(status: int, where: str):
    if status != KVC_OK:
        raise KvcError(status, where, lib().kvc_last_error().decode())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev_ptr(t: Optional[torch.Tensor], name: str, dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


class Cache:
    """kvc_cache over torch tensors (pools [L][num_pages][H][P][d] bf16, tags int32,
    block_table [B][max_blocks] int32, nblocks [B] int32)."""

    def __init__(self, k_pool, v_pool, tags, block_table, nblocks, aux=None):
        L, num_pages, H, P, d = k_pool.shape
        self.tensors = (k_pool, v_pool, tags, block_table, nblocks, aux)
        self.c = kvc_cache(
            _dev_ptr(k_pool, "k_pool", torch.bfloat16), _dev_ptr(v_pool, "v_pool", torch.bfloat16),
            _dev_ptr(tags, "tags", torch.int32), _dev_ptr(block_table, "block_table", torch.int32),
            _dev_ptr(nblocks, "nblocks", torch.int32), L, num_pages, H, P, d,
            block_table.shape[1], block_table.shape[0], _dev_ptr(aux, "aux", torch.float32))

    @property
    def ref(self):
        return ctypes.byref(self.c)


class Segments:
    """kvc_segments over host int32 arrays."""

    def __init__(self, seg_start: Sequence[int], seg_end: Sequence[int], seq_len: Sequence[int]):
        self.arrays = [np.ascontiguousarray(np.asarray(x, dtype=np.int32))
                       for x in (seg_start, seg_end, seq_len)]
        B = self.arrays[0].shape[0]
        self.s = kvc_segments(*(a.ctypes.data for a in self.arrays), B)

    @property
    def ref(self):
        return ctypes.byref(self.s)


class Allocator:
    def __init__(self, free_ids: torch.Tensor, free_top: torch.Tensor):
        self.tensors = (free_ids, free_top)
        self.a = kvc_allocator(_dev_ptr(free_ids, "free_ids", torch.int32),
                               _dev_ptr(free_top, "free_top", torch.int32), free_ids.numel())

    @property
    def ref(self):
        return ctypes.byref(self.a)


def _host_i32(m) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(m, dtype=np.int32))


# ----------------------------------------------------------------------------- C names

def kvc_version() -> str:
    return lib().kvc_version().decode()


def kvc_budget_from_ratio(n: int, ratio: float) -> int:
    return int(lib().kvc_budget_from_ratio(int(n), float(ratio)))


def kvc_budget_actkv(k: int) -> int:
    return int(lib().kvc_budget_actkv(int(k)))


def kvc_score_workspace_size(cache: Cache, segs: Segments, R: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().kvc_score_workspace_size(cache.ref, segs.ref, int(R), ctypes.byref(out)),
           "kvc_score_workspace_size")
    return int(out.value)


def kvc_score(cache: Cache, segs: Segments, q: torch.Tensor, R: int, scale: float,
              scores: torch.Tensor, lse: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
    _check(lib().kvc_score(cache.ref, segs.ref, _dev_ptr(q, "q", torch.bfloat16), int(R),
                           float(scale), _dev_ptr(scores, "scores", torch.float32),
                           _dev_ptr(lse, "lse", torch.float32), _dev_ptr(ws, "ws"),
                           ws.numel() * ws.element_size(), _stream(stream)), "kvc_score")


def kvc_score_lse(cache: Cache, segs: Segments, q: torch.Tensor, R: int, scale: float,
                  lse: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
    _check(lib().kvc_score_lse(cache.ref, segs.ref, _dev_ptr(q, "q", torch.bfloat16), int(R),
                               float(scale), _dev_ptr(lse, "lse", torch.float32), _dev_ptr(ws, "ws"),
                               ws.numel() * ws.element_size(), _stream(stream)), "kvc_score_lse")


def kvc_score_alpha(cache: Cache, segs: Segments, q: torch.Tensor, R: int, scale: float,
                    lse: Optional[torch.Tensor], scores: torch.Tensor, ws: torch.Tensor, stream=None):
    _check(lib().kvc_score_alpha(cache.ref, segs.ref, _dev_ptr(q, "q", torch.bfloat16), int(R),
                                 float(scale), _dev_ptr(lse, "lse", torch.float32),
                                 _dev_ptr(scores, "scores", torch.float32), _dev_ptr(ws, "ws"),
                                 ws.numel() * ws.element_size(), _stream(stream)), "kvc_score_alpha")


def kvc_score_noalloc(cache: Cache, segs: Segments, q: torch.Tensor, R: int, scale: float,
                      scores: torch.Tensor, lse: Optional[torch.Tensor] = None, stream=None):
    """kvc_score with the library's fixed device scratch instead of a caller workspace."""
    _check(lib().kvc_score_noalloc(cache.ref, segs.ref, _dev_ptr(q, "q", torch.bfloat16), int(R),
                                   float(scale), _dev_ptr(scores, "scores", torch.float32),
                                   _dev_ptr(lse, "lse", torch.float32), _stream(stream)),
           "kvc_score_noalloc")


def kvc_launch_count(reset: bool = False) -> int:
    return int(lib().kvc_launch_count(1 if reset else 0))


def kvc_debug_stall_scoring(stall_ns: int) -> None:
    """Failure-path test of the scoring kernels: stall_ns > 0 makes the scoring launches that follow
    withhold their proxy-row loads and give up their waits after stall_ns (KVC_DEV_WAIT_TIMEOUT);
    0 restores normal operation."""
    _check(lib().kvc_debug_stall_scoring(int(stall_ns)), "kvc_debug_stall_scoring")


def kvc_select_workspace_size(cache: Cache, segs: Segments, m) -> int:
    mm = _host_i32(m)
    out = ctypes.c_size_t(0)
    _check(lib().kvc_select_workspace_size(cache.ref, segs.ref, mm.ctypes.data, ctypes.byref(out)),
           "kvc_select_workspace_size")
    return int(out.value)


def kvc_select_topm(cache: Cache, segs: Segments, scores: torch.Tensor, m, keep: torch.Tensor,
                    ws: Optional[torch.Tensor] = None, stream=None):
    mm = _host_i32(m)
    _check(lib().kvc_select_topm(cache.ref, segs.ref, _dev_ptr(scores, "scores", torch.float32),
                                 mm.ctypes.data, _dev_ptr(keep, "keep", torch.int32),
                                 _dev_ptr(ws, "ws"),
                                 0 if ws is None else ws.numel() * ws.element_size(),
                                 _stream(stream)), "kvc_select_topm")


def kvc_plan_buffer_sizes(cache: Cache, segs: Segments, m) -> dict:
    mm = _host_i32(m)
    out = kvc_plan_sizes()
    _check(lib().kvc_plan_buffer_sizes(cache.ref, segs.ref, mm.ctypes.data, ctypes.byref(out)),
           "kvc_plan_buffer_sizes")
    return {name: int(getattr(out, name)) for name, _ in kvc_plan_sizes._fields_}


def kvc_plan_fresh_buffer_sizes(cache: Cache, segs: Segments, m) -> dict:
    mm = _host_i32(m)
    out = kvc_plan_sizes()
    _check(lib().kvc_plan_fresh_buffer_sizes(cache.ref, segs.ref, mm.ctypes.data, ctypes.byref(out)),
           "kvc_plan_fresh_buffer_sizes")
    return {name: int(getattr(out, name)) for name, _ in kvc_plan_sizes._fields_}


class Plan:
    """Caller-allocated plan buffers (device int32 tensors) for one (segments, budgets); with
    fresh=True sized for the fresh-page compaction."""

    def __init__(self, cache: Cache, segs: Segments, m, device=None, fresh: bool = False):
        sizes = (kvc_plan_fresh_buffer_sizes if fresh else kvc_plan_buffer_sizes)(cache, segs, m)
        device = device or cache.tensors[0].device
        mk = lambda n: torch.empty(max(1, n), dtype=torch.int32, device=device)
        self.sizes = sizes
        self.moves = mk(sizes["moves_len"])
        self.move_count = mk(sizes["units_len"])
        self.dead = mk(sizes["dead_len"])
        self.dead_count = mk(sizes["units_len"])
        self.freed = mk(sizes["freed_len"])
        self.new_rows = mk(sizes["new_rows_len"])
        self.p = kvc_plan(self.moves.data_ptr(), self.move_count.data_ptr(), self.dead.data_ptr(),
                          self.dead_count.data_ptr(), self.freed.data_ptr(),
                          self.new_rows.data_ptr(), self.moves.numel(), self.move_count.numel(),
                          self.dead.numel(), self.freed.numel(), self.new_rows.numel())

    @property
    def ref(self):
        return ctypes.byref(self.p)


def kvc_plan_compact(cache: Cache, segs: Segments, m, keep: torch.Tensor, plan: Plan, stream=None):
    mm = _host_i32(m)
    _check(lib().kvc_plan_compact(cache.ref, segs.ref, mm.ctypes.data,
                                  _dev_ptr(keep, "keep", torch.int32), plan.ref, _stream(stream)),
           "kvc_plan_compact")


def kvc_compact(cache: Cache, segs: Segments, m, plan: Plan, stream=None):
    mm = _host_i32(m)
    _check(lib().kvc_compact(cache.ref, segs.ref, mm.ctypes.data, plan.ref, _stream(stream)),
           "kvc_compact")


def kvc_free_pages(cache: Cache, segs: Segments, m, alloc: Allocator, plan: Plan, stream=None):
    mm = _host_i32(m)
    _check(lib().kvc_free_pages(cache.ref, segs.ref, mm.ctypes.data, alloc.ref, plan.ref,
                                _stream(stream)), "kvc_free_pages")


def kvc_evict_sentinel(cache: Cache, segs: Segments, m, keep: torch.Tensor, stream=None):
    mm = _host_i32(m)
    _check(lib().kvc_evict_sentinel(cache.ref, segs.ref, mm.ctypes.data,
                                    _dev_ptr(keep, "keep", torch.int32), _stream(stream)),
           "kvc_evict_sentinel")


def kvc_plan_fresh(cache: Cache, segs: Segments, m, keep: torch.Tensor, alloc: Allocator, plan: Plan,
                   stream=None):
    mm = _host_i32(m)
    _check(lib().kvc_plan_fresh(cache.ref, segs.ref, mm.ctypes.data, _dev_ptr(keep, "keep", torch.int32),
                                alloc.ref, plan.ref, _stream(stream)), "kvc_plan_fresh")


def kvc_commit_fresh(cache: Cache, segs: Segments, m, alloc: Allocator, plan: Plan, stream=None):
    mm = _host_i32(m)
    _check(lib().kvc_commit_fresh(cache.ref, segs.ref, mm.ctypes.data, alloc.ref, plan.ref,
                                  _stream(stream)), "kvc_commit_fresh")


def kvc_score_action(cache: Cache, segs: Segments, q: torch.Tensor, R: int, scale: float,
                     attn: torch.Tensor, lse: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
    _check(lib().kvc_score_action(cache.ref, segs.ref, _dev_ptr(q, "q", torch.bfloat16), int(R),
                                  float(scale), _dev_ptr(attn, "attn", torch.float32),
                                  _dev_ptr(lse, "lse", torch.float32), _dev_ptr(ws, "ws"),
                                  ws.numel() * ws.element_size(), _stream(stream)), "kvc_score_action")


def kvc_lrfu_update(cache: Cache, segs: Segments, attn: torch.Tensor, frac: float, lam: float,
                    crf_out: torch.Tensor, hits: Optional[torch.Tensor] = None, stream=None):
    _check(lib().kvc_lrfu_update(cache.ref, segs.ref, _dev_ptr(attn, "attn", torch.float32),
                                 float(frac), float(lam), _dev_ptr(crf_out, "crf_out", torch.float32),
                                 _dev_ptr(hits, "hits", torch.uint8), _stream(stream)),
           "kvc_lrfu_update")


def kvc_am_workspace_size(cache: Cache, segs: Segments, m, R: int) -> int:
    mm = _host_i32(m)
    out = ctypes.c_size_t(0)
    _check(lib().kvc_am_workspace_size(cache.ref, segs.ref, mm.ctypes.data, int(R), ctypes.byref(out)),
           "kvc_am_workspace_size")
    return int(out.value)


def kvc_am_fit(cache: Cache, segs: Segments, m, q: torch.Tensor, R: int, scale: float,
               keep: torch.Tensor, sweeps: int, beta: Optional[torch.Tensor], vc: Optional[torch.Tensor],
               ws: torch.Tensor, stream=None, lse: Optional[torch.Tensor] = None):
    mm = _host_i32(m)
    _check(lib().kvc_am_fit(cache.ref, segs.ref, mm.ctypes.data, _dev_ptr(q, "q", torch.bfloat16), int(R),
                            float(scale), _dev_ptr(lse, "lse", torch.float32),
                            _dev_ptr(keep, "keep", torch.int32), int(sweeps),
                            _dev_ptr(beta, "beta", torch.float32), _dev_ptr(vc, "vc", torch.float32),
                            _dev_ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)),
           "kvc_am_fit")


def kvc_status_string(status: int) -> str:
    return lib().kvc_status_string(int(status)).decode()


def kvc_last_error() -> str:
    return lib().kvc_last_error().decode()


def kvc_read_device_status(clear: bool = True, stream=None) -> int:
    out = ctypes.c_uint32(0)
    _check(lib().kvc_read_device_status(ctypes.byref(out), 1 if clear else 0, _stream(stream)),
           "kvc_read_device_status")
    return int(out.value)


def kvc_validate_cache_host(block_table, nblocks, seq_len, num_pages: int, page_size: int,
                            free_ids=None, free_top: int = 0) -> None:
    """Raises KvcError if the host copies of the cache bookkeeping are inconsistent."""
    bt = _host_i32(block_table.cpu() if isinstance(block_table, torch.Tensor) else block_table)
    nb = _host_i32(nblocks.cpu() if isinstance(nblocks, torch.Tensor) else nblocks)
    sl = None if seq_len is None else _host_i32(seq_len)
    fi = None if free_ids is None else _host_i32(
        free_ids.cpu() if isinstance(free_ids, torch.Tensor) else free_ids)
    _check(lib().kvc_validate_cache_host(bt.ctypes.data, nb.ctypes.data,
                                         None if sl is None else sl.ctypes.data, bt.shape[0],
                                         bt.shape[1], int(num_pages), int(page_size),
                                         None if fi is None else fi.ctypes.data, int(free_top)),
           "kvc_validate_cache_host")


# ----------------------------------------------------------------------------- driver

class Compactor:
    """Owns the workspace and plan buffers of one compaction and issues the five calls.

    cache tensors: k_pool, v_pool, tags, block_table, nblocks, free_ids, free_top (device);
    segments: host lists seg_start / seg_end / seq_len; m: host budgets per sequence."""

    def __init__(self, k_pool, v_pool, tags, block_table, nblocks, free_ids, free_top,
                 seg_start, seg_end, seq_len, m, R: int, aux=None):
        self.cache = Cache(k_pool, v_pool, tags, block_table, nblocks, aux)
        self.alloc = Allocator(free_ids, free_top)
        self.segs = Segments(seg_start, seg_end, seq_len)
        self.m = _host_i32(m)
        self.R = int(R)
        dev = k_pool.device
        L, _, H = k_pool.shape[:3]
        self.sizes = kvc_plan_buffer_sizes(self.cache, self.segs, self.m)
        self.Ntot, self.Mtot = self.sizes["Ntot"], self.sizes["Mtot"]
        self.scores = torch.empty((L, H, max(1, self.Ntot)), dtype=torch.float32, device=dev)
        self.keep = torch.empty((L, H, max(1, self.Mtot)), dtype=torch.int32, device=dev)
        B = block_table.shape[0]
        self.lse = torch.empty((B, L, H, self.R), dtype=torch.float32, device=dev)
        ws_bytes = kvc_score_workspace_size(self.cache, self.segs, self.R)
        self.ws = torch.empty(max(256, ws_bytes) + 256, dtype=torch.uint8, device=dev)
        off = (-self.ws.data_ptr()) % 256
        self.ws_view = self.ws[off:off + max(256, ws_bytes)]
        self.plan = Plan(self.cache, self.segs, self.m, dev)

    def score(self, q: torch.Tensor, scale: float, want_lse: bool = True, stream=None):
        kvc_score(self.cache, self.segs, q, self.R, scale, self.scores,
                  self.lse if want_lse else None, self.ws_view, stream)

    def score_lse(self, q: torch.Tensor, scale: float, want_lse: bool = False, stream=None):
        kvc_score_lse(self.cache, self.segs, q, self.R, scale, self.lse if want_lse else None,
                      self.ws_view, stream)

    def score_alpha(self, q: torch.Tensor, scale: float, lse: Optional[torch.Tensor] = None,
                    stream=None):
        kvc_score_alpha(self.cache, self.segs, q, self.R, scale, lse, self.scores, self.ws_view,
                        stream)

    def score_action(self, q: torch.Tensor, scale: float, stream=None):
        """Action attention a_j of every key into self.attn (ActKV's hit signal)."""
        if getattr(self, "attn", None) is None:
            self.attn = torch.empty_like(self.scores)
        kvc_score_action(self.cache, self.segs, q, self.R, scale, self.attn, None, self.ws_view, stream)

    def lrfu(self, frac: float = 0.9, lam: float = 0.5, hits: Optional[torch.Tensor] = None,
             stream=None):
        """One LRFU step on the cache's aux values; the new values become self.scores."""
        kvc_lrfu_update(self.cache, self.segs, self.attn, frac, lam, self.scores, hits, stream)

    def am_fit(self, q: torch.Tensor, scale: float, sweeps: int = 8, keep: Optional[torch.Tensor] = None,
               beta: Optional[torch.Tensor] = None, vc: Optional[torch.Tensor] = None, stream=None,
               lse: Optional[torch.Tensor] = None):
        """Attention Matching on the kept entries: beta into the cache's aux values (when it has
        them) and `beta`, V_C over the kept V rows and into `vc`.  `lse`: the rows' LSE from
        this compactor's scoring (self.lse after score(want_lse=True)), or None to recompute it."""
        if getattr(self, "am_ws", None) is None:
            nbytes = max(256, kvc_am_workspace_size(self.cache, self.segs, self.m, self.R))
            self.am_ws_raw = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.keep.device)
            off = (-self.am_ws_raw.data_ptr()) % 256
            self.am_ws = self.am_ws_raw[off:off + nbytes]
        kvc_am_fit(self.cache, self.segs, self.m, q, self.R, scale, self.keep if keep is None else keep,
                   sweeps, beta, vc, self.am_ws, stream, lse=lse)

    def select(self, stream=None):
        kvc_select_topm(self.cache, self.segs, self.scores, self.m, self.keep, None, stream)

    def plan_compact(self, keep: Optional[torch.Tensor] = None, stream=None):
        kvc_plan_compact(self.cache, self.segs, self.m, self.keep if keep is None else keep,
                         self.plan, stream)

    def compact(self, stream=None, plan: Optional[Plan] = None):
        kvc_compact(self.cache, self.segs, self.m, self.plan if plan is None else plan, stream)

    def evict_sentinel(self, keep: Optional[torch.Tensor] = None, stream=None):
        """Layout-preserving eviction: sentinel dead slots, nothing moves or is freed."""
        kvc_evict_sentinel(self.cache, self.segs, self.m, self.keep if keep is None else keep, stream)

    def plan_fresh(self, keep: Optional[torch.Tensor] = None, stream=None) -> Plan:
        """Plan of the order-preserving compaction into fresh pages (run it with compact(plan=...)
        and finish with commit_fresh)."""
        if getattr(self, "fresh_plan", None) is None:
            self.fresh_plan = Plan(self.cache, self.segs, self.m, self.keep.device, fresh=True)
        kvc_plan_fresh(self.cache, self.segs, self.m, self.keep if keep is None else keep, self.alloc,
                       self.fresh_plan, stream)
        return self.fresh_plan

    def commit_fresh(self, stream=None):
        kvc_commit_fresh(self.cache, self.segs, self.m, self.alloc, self.fresh_plan, stream)

    def free_pages(self, stream=None):
        kvc_free_pages(self.cache, self.segs, self.m, self.alloc, self.plan, stream)

    def run(self, q: torch.Tensor, scale: float, stream=None, want_lse: bool = False):
        """One full compaction: score, select, plan, copy, release."""
        self.score(q, scale, want_lse, stream)
        self.select(stream)
        self.plan_compact(None, stream)
        self.compact(stream)
        self.free_pages(stream)
