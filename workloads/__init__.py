"""Seeded synthetic inputs for online KV-cache compaction.

This module builds paged KV caches, proxy queries and budget requests with the
shapes and value distributions of the workloads the pages describe (agent
trajectories of 31-33K tokens, 128K contexts, keep ratio 0.2, delay-1
multi-turn compaction, ActKV's 512*1.75^k budgets).  No public benchmark or
dataset is available here; these synthetic caches stand in for them.

It is shared by the tests, the benchmark and the smoke check, and it holds
none of the method's arithmetic: no scores, no selection, no slot plan, no
budget rounding.  Budgets are passed on as requests (a keep ratio, or ActKV
growth steps k) that each side turns into entry counts with its own code.

Cache layout (all tensors on one device):
  k_pool, v_pool  bf16  [L][num_pages][H][P][d]
  tags            int32 [L][num_pages][H][P]   logical position, -1 = empty
  block_table     int32 [B][max_blocks]        page ids, -1 = unmapped
  nblocks         int32 [B]
  free_ids        int32 [num_pages]            free stack, top at free_top
  free_top        int32 [1]
  q               bf16  [B][L][H][R][d]        R = q * G proxy rows per KV head
Host-side: seq_len[b] (slots in use), seg_start[b], seg_end[b].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

ACTKV_STEPS = 7  # k = 0..6 for 512 * 1.75^k


@dataclasses.dataclass(frozen=True)
class Spec:
    """Shape and distribution recipe of one synthetic workload."""

    name: str
    L: int  # layers
    H: int  # KV heads
    G: int  # query heads per KV head (GQA group)
    d: int  # head dim
    P: int  # page size (slots per block)
    q: int  # proxy queries per query head
    lengths: tuple  # cached tokens per sequence
    budget: tuple  # ("ratio", r) or ("actkv", (k_0, k_1, ...))
    kv: str = "normal"  # "normal" | "sinks"
    qdist: str = "normal"  # "normal" | "planted4" | "aligned"
    shuffle_pages: bool = False
    headroom: float = 0.10

    @property
    def R(self) -> int:
        return self.q * self.G

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def B(self) -> int:
        return len(self.lengths)

    def entries(self) -> int:
        return self.L * self.H * int(sum(self.lengths))


def _ragged_draw(seed: int, B: int = 16, lo: int = 8192, hi: int = 131072):
    rng = np.random.default_rng([seed, 3])
    lengths = tuple(int(x) for x in rng.integers(lo, hi + 1, size=B))
    ks = tuple(int(x) for x in rng.integers(0, ACTKV_STEPS, size=B))
    return lengths, ks


def spec(name: str, seed: int = 0) -> Spec:
    """The named workloads.  Seeded draws (ragged lengths, budget steps) use ``seed``."""
    if name == "tiny":
        return Spec("tiny", L=1, H=2, G=2, d=64, P=16, q=8, lengths=(512,),
                    budget=("ratio", 0.2), kv="normal", qdist="planted4")
    if name == "qwen3-30b-a3b":
        return Spec("qwen3-30b-a3b", L=48, H=4, G=8, d=128, P=16, q=64, lengths=(32768,),
                    budget=("ratio", 0.2), kv="sinks", qdist="normal")
    if name == "batched-ragged":
        lengths, ks = _ragged_draw(seed)
        return Spec("batched-ragged", L=1, H=8, G=8, d=128, P=16, q=16, lengths=lengths,
                    budget=("actkv", ks), kv="normal", qdist="normal", shuffle_pages=True)
    if name == "batched-ragged-sinks":
        # The batched-ragged shape with the other reading of its K/V distribution: that of the
        # Qwen3-shaped cache (LogNormal token norms, the first 4 tokens x8 as attention sinks).
        lengths, ks = _ragged_draw(seed)
        return Spec("batched-ragged-sinks", L=1, H=8, G=8, d=128, P=16, q=16, lengths=lengths,
                    budget=("actkv", ks), kv="sinks", qdist="normal", shuffle_pages=True)
    if name == "long-context":
        return Spec("long-context", L=36, H=8, G=8, d=128, P=32, q=32, lengths=(131072,),
                    budget=("ratio", 0.2), kv="normal", qdist="aligned")
    if name == "multi-turn":
        # one compaction of the 20-turn schedule: segment of 1536 tokens, R = 16*... rows
        return Spec("multi-turn", L=28, H=2, G=8, d=128, P=16, q=256, lengths=(1536,),
                    budget=("ratio", 0.2), kv="normal", qdist="planted4")
    raise KeyError(name)


NAMES = ("tiny", "qwen3-30b-a3b", "batched-ragged", "batched-ragged-sinks", "long-context", "multi-turn")


def custom(name="custom", *, L=1, H=2, G=2, d=64, P=16, q=4, lengths=(100,), budget=("ratio", 0.2),
           kv="normal", qdist="normal", shuffle_pages=False, headroom=0.10) -> Spec:
    return Spec(name, L=L, H=H, G=G, d=d, P=P, q=q, lengths=tuple(int(x) for x in lengths),
                budget=budget, kv=kv, qdist=qdist, shuffle_pages=shuffle_pages, headroom=headroom)


@dataclasses.dataclass
class Case:
    spec: Spec
    seed: int
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    tags: torch.Tensor
    block_table: torch.Tensor
    nblocks: torch.Tensor
    free_ids: torch.Tensor
    free_top: torch.Tensor
    q: Optional[torch.Tensor]
    seq_len: list
    seg_start: list
    seg_end: list
    planted: Optional[list] = None  # per (b): LongTensor [L][H][k] planted segment positions

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[1])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    def budget_request(self):
        """("ratio", r) or ("actkv", ks) -- turned into entry counts by the caller's own code."""
        return self.spec.budget

    def state(self):
        """The mutable cache state, in a fixed order (for snapshots)."""
        return [self.k_pool, self.v_pool, self.tags, self.block_table, self.nblocks,
                self.free_ids, self.free_top]

    def snapshot(self):
        return [t.clone() for t in self.state()]

    def restore(self, snap):
        for dst, src in zip(self.state(), snap):
            dst.copy_(src)

    def to(self, device):
        f = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(
            self, k_pool=f(self.k_pool), v_pool=f(self.v_pool), tags=f(self.tags),
            block_table=f(self.block_table), nblocks=f(self.nblocks), free_ids=f(self.free_ids),
            free_top=f(self.free_top), q=f(self.q))


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + stream * 7919) % (2**63 - 1))
    return g


def _randn_bf16(shape, g, device, chunk_dim0=True) -> torch.Tensor:
    """N(0,1) bf16 tensor, generated in fp32 slices along dim 0 to bound temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for i in range(shape[0]):
        out[i] = torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32)
    return out


def _empty_allocator(num_pages: int, B: int, max_blocks: int, shuffle: bool, seed: int, device):
    if shuffle:
        ids = np.random.default_rng([seed, 11]).permutation(num_pages).astype(np.int32)
    else:
        ids = np.arange(num_pages - 1, -1, -1, dtype=np.int32)  # pops hand out 0, 1, 2, ...
    free_ids = torch.from_numpy(ids).to(device)
    free_top = torch.tensor([num_pages], dtype=torch.int32, device=device)
    block_table = torch.full((B, max_blocks), -1, dtype=torch.int32, device=device)
    nblocks = torch.zeros(B, dtype=torch.int32, device=device)
    return free_ids, free_top, block_table, nblocks


def pop_pages(free_ids: torch.Tensor, free_top: torch.Tensor, count: int) -> torch.Tensor:
    """Pop ``count`` page ids from the free stack (host-synchronous bookkeeping)."""
    top = int(free_top.item())
    if count > top:
        raise RuntimeError("page pool exhausted")
    ids = torch.flip(free_ids[top - count:top], dims=[0]).clone()  # free_ids[--top] order
    free_top.fill_(top - count)
    return ids


def write_tokens(case: Case, b: int, slot0: int, logical0: int, K: torch.Tensor, V: torch.Tensor):
    """Write K/V [L][H][T][d] for T tokens at slots [slot0, slot0+T) of sequence b."""
    P = case.spec.P
    T = K.shape[2]
    slots = torch.arange(slot0, slot0 + T, device=case.k_pool.device)
    pages = case.block_table[b].long()[slots // P]
    offs = slots % P
    kp = case.k_pool.permute(1, 3, 0, 2, 4)  # [page][slot][L][H][d] view
    vp = case.v_pool.permute(1, 3, 0, 2, 4)
    kp[pages, offs] = K.permute(2, 0, 1, 3).to(torch.bfloat16)
    vp[pages, offs] = V.permute(2, 0, 1, 3).to(torch.bfloat16)
    tg = case.tags.permute(1, 3, 0, 2)  # [page][slot][L][H]
    pos = torch.arange(logical0, logical0 + T, device=case.tags.device, dtype=torch.int32)
    tg[pages, offs] = pos.view(T, 1, 1).expand(T, case.spec.L, case.spec.H)


def gather_keys(case: Case, b: int, slot0: int, n: int) -> torch.Tensor:
    """K rows [L][H][n][d] (bf16) of slots [slot0, slot0+n) of sequence b."""
    P = case.spec.P
    slots = torch.arange(slot0, slot0 + n, device=case.k_pool.device)
    pages = case.block_table[b].long()[slots // P]
    offs = slots % P
    return case.k_pool.permute(1, 3, 0, 2, 4)[pages, offs].permute(1, 2, 0, 3)


def _planted4_q(case: Case, b: int, s0: int, n: int, R: int, g, rng) -> (torch.Tensor, torch.Tensor):
    """Q rows z_i + 3 * K_{p[i mod 4]} with 4 distinct planted positions per (layer, head)."""
    sp = case.spec
    dev = case.k_pool.device
    k = min(4, n)
    planted = np.stack([np.stack([np.sort(rng.choice(n, size=k, replace=False))
                                  for _ in range(sp.H)]) for _ in range(sp.L)])  # [L][H][k]
    planted_t = torch.from_numpy(planted).long().to(dev)
    Kseg = gather_keys(case, b, s0, n).float()  # [L][H][n][d]
    rows = torch.arange(R, device=dev) % k
    idx = planted_t[:, :, rows]  # [L][H][R]
    Kp = torch.gather(Kseg, 2, idx.unsqueeze(-1).expand(sp.L, sp.H, R, sp.d))
    z = torch.randn((sp.L, sp.H, R, sp.d), generator=g, device=dev, dtype=torch.float32)
    return (z + 3.0 * Kp).to(torch.bfloat16), planted_t


def _aligned_plant(case: Case, b: int, s0: int, n: int, q: torch.Tensor, g, rng) -> torch.Tensor:
    """Replace 1% of keys per (layer, head) by Q-aligned heavy hitters (cosine ~0.6).

    Planted key j (rank r among the planted positions) becomes
    ||z_j|| * (0.6 * qhat_{r mod R} + 0.8 * what), what a random unit vector
    orthogonal to qhat, z_j the key it replaces."""
    sp = case.spec
    dev = case.k_pool.device
    cnt = max(1, int(math.floor(0.01 * n)))
    R = q.shape[-2]
    planted = np.stack([np.stack([np.sort(rng.choice(n, size=cnt, replace=False))
                                  for _ in range(sp.H)]) for _ in range(sp.L)])  # [L][H][cnt]
    planted_t = torch.from_numpy(planted).long().to(dev)
    P = sp.P
    slots = s0 + planted_t  # [L][H][cnt]
    pages = case.block_table[b].long()[slots // P]
    offs = slots % P
    Lidx = torch.arange(sp.L, device=dev).view(-1, 1, 1).expand_as(pages)
    Hidx = torch.arange(sp.H, device=dev).view(1, -1, 1).expand_as(pages)
    z = case.k_pool[Lidx, pages, Hidx, offs].float()  # [L][H][cnt][d]
    qrows = torch.arange(cnt, device=dev) % R
    qhat = q[:, :, qrows].float()  # [L][H][cnt][d]
    qhat = qhat / qhat.norm(dim=-1, keepdim=True)
    w = torch.randn(z.shape, generator=g, device=dev, dtype=torch.float32)
    w = w - (w * qhat).sum(-1, keepdim=True) * qhat
    w = w / w.norm(dim=-1, keepdim=True)
    knew = z.norm(dim=-1, keepdim=True) * (0.6 * qhat + 0.8 * w)
    case.k_pool[Lidx, pages, Hidx, offs] = knew.to(torch.bfloat16)
    return planted_t


def build(sp: Spec, seed: int = 0, device="cpu", with_q: bool = True) -> Case:
    """A freshly filled paged cache for ``sp``: every sequence is one segment [0, n_b)."""
    device = torch.device(device)
    B, P, L, H, d = sp.B, sp.P, sp.L, sp.H, sp.d
    blocks = [math.ceil(n / P) for n in sp.lengths]
    used = sum(blocks)
    num_pages = max(used + 1, math.ceil(used * (1.0 + sp.headroom)))
    max_blocks = max(1, max(blocks))
    free_ids, free_top, block_table, nblocks = _empty_allocator(
        num_pages, B, max_blocks, sp.shuffle_pages, seed, device)
    g = _gen(device, seed, 1)
    k_pool = _randn_bf16((L, num_pages, H, P, d), g, device)
    v_pool = _randn_bf16((L, num_pages, H, P, d), g, device)
    tags = torch.full((L, num_pages, H, P), -1, dtype=torch.int32, device=device)
    case = Case(sp, seed, k_pool, v_pool, tags, block_table, nblocks, free_ids, free_top, None,
                list(sp.lengths), [0] * B, list(sp.lengths))
    for b in range(B):
        ids = pop_pages(free_ids, free_top, blocks[b])
        block_table[b, :blocks[b]] = ids
        nblocks[b] = blocks[b]
        slots = torch.arange(sp.lengths[b], device=device)
        pages = block_table[b].long()[slots // P]
        offs = slots % P
        case.tags.permute(1, 3, 0, 2)[pages, offs] = slots.to(torch.int32).view(-1, 1, 1).expand(
            -1, L, H)
    if sp.kv == "sinks":
        # per-(layer, head, slot) norm scale c ~ LogNormal(0, 0.5); the first 4 tokens of
        # every sequence get 8c (attention sinks).  Applied to K and V alike.
        c = torch.exp(0.5 * torch.randn((L, num_pages, H, P), generator=g, device=device))
        for b in range(B):
            first = torch.arange(min(4, sp.lengths[b]), device=device)
            pages = block_table[b].long()[first // P]
            c.permute(1, 3, 0, 2)[pages, first % P] *= 8.0
        for l in range(L):
            case.k_pool[l] = (case.k_pool[l].float() * c[l].unsqueeze(-1)).to(torch.bfloat16)
            case.v_pool[l] = (case.v_pool[l].float() * c[l].unsqueeze(-1)).to(torch.bfloat16)
    if with_q:
        make_q(case, seed)
    return case


def make_q(case: Case, seed: int, segments: Optional[Sequence[int]] = None):
    """Proxy queries [B][L][H][R][d] for the current segments (planted per spec.qdist)."""
    sp = case.spec
    dev = case.k_pool.device
    g = _gen(dev, seed, 2)
    rng = np.random.default_rng([seed, 5])
    R = sp.R
    q = torch.empty((sp.B, sp.L, sp.H, R, sp.d), dtype=torch.bfloat16, device=dev)
    planted = []
    for b in range(sp.B):
        s0, n = case.seg_start[b], case.seg_end[b] - case.seg_start[b]
        if sp.qdist == "planted4" and n > 0:
            qb, pl = _planted4_q(case, b, s0, n, R, g, rng)
            q[b] = qb
            planted.append(pl)
        else:
            for l in range(sp.L):
                q[b, l] = torch.randn((sp.H, R, sp.d), generator=g, device=dev,
                                      dtype=torch.float32).to(torch.bfloat16)
            if sp.qdist == "aligned" and n > 0:
                planted.append(_aligned_plant(case, b, s0, n, q[b], g, rng))
            else:
                planted.append(None)
    case.q = q
    case.planted = planted
    return q


# --------------------------------------------------------------------------- multi-turn

@dataclasses.dataclass(frozen=True)
class MultiTurnSpec:
    """Delay-1 online schedule: turn t appends ``tokens`` tokens; at the end of turn t >= 2
    the segment of turn t-1 is compacted with turn t's proxy queries."""

    L: int = 28
    H: int = 2
    G: int = 8
    d: int = 128
    P: int = 16
    q: int = 256
    tokens: int = 1536
    turns: int = 20
    ratio: float = 0.2
    headroom: float = 0.10

    def as_spec(self) -> Spec:
        return Spec("multi-turn", L=self.L, H=self.H, G=self.G, d=self.d, P=self.P, q=self.q,
                    lengths=(self.tokens,), budget=("ratio", self.ratio), kv="normal",
                    qdist="planted4")


class MultiTurn:
    """Drives the multi-turn schedule on a single-sequence cache.

    The caller compacts; this class only appends turns (popping pages from the
    free stack) and builds each compaction's proxy queries.  ``kept_blocks`` is
    the number of blocks a compacted segment keeps, which the caller reports
    back through :meth:`compacted` (it depends on the budget rule)."""

    def __init__(self, ms: MultiTurnSpec, seed: int, device, kept_blocks: int):
        self.ms = ms
        self.seed = seed
        self.device = torch.device(device)
        P = ms.P
        per_turn = math.ceil(ms.tokens / P)
        # peak mapped blocks: just after appending the last turn
        peak = per_turn * ms.turns - (per_turn - kept_blocks) * max(0, ms.turns - 2)
        self.num_pages = math.ceil(peak * (1.0 + ms.headroom))
        self.max_blocks = peak
        sp = ms.as_spec()
        free_ids, free_top, bt, nb = _empty_allocator(self.num_pages, 1, self.max_blocks, False,
                                                      seed, self.device)
        g = _gen(self.device, seed, 1)
        k_pool = _randn_bf16((ms.L, self.num_pages, ms.H, P, ms.d), g, self.device)
        v_pool = _randn_bf16((ms.L, self.num_pages, ms.H, P, ms.d), g, self.device)
        tags = torch.full((ms.L, self.num_pages, ms.H, P), -1, dtype=torch.int32,
                          device=self.device)
        self.case = Case(sp, seed, k_pool, v_pool, tags, bt, nb, free_ids, free_top, None,
                         [0], [0], [0])
        self.turn = 0
        self.logical_len = 0
        self.frozen_slots = 0  # slots held by compacted (frozen) segments
        self.turn_start_slot = {}

    def append_turn(self):
        ms, case = self.ms, self.case
        self.turn += 1
        t = self.turn
        P = ms.P
        nblk = math.ceil(ms.tokens / P)
        ids = pop_pages(case.free_ids, case.free_top, nblk)
        cur = int(case.nblocks[0].item())
        case.block_table[0, cur:cur + nblk] = ids
        case.nblocks[0] = cur + nblk
        slot0 = cur * P
        g = _gen(self.device, self.seed, 100 + t)
        K = torch.randn((ms.L, ms.H, ms.tokens, ms.d), generator=g, device=self.device)
        V = torch.randn((ms.L, ms.H, ms.tokens, ms.d), generator=g, device=self.device)
        write_tokens(case, 0, slot0, self.logical_len, K, V)
        self.turn_start_slot[t] = slot0
        self.logical_len += ms.tokens
        case.seq_len[0] = slot0 + ms.tokens

    def compaction_segment(self):
        """[s0, s1) of turn t-1's segment at the end of turn t (t >= 2)."""
        t = self.turn
        if t < 2:
            raise RuntimeError("nothing to compact before turn 2")
        s0 = self.turn_start_slot[t - 1]
        return s0, s0 + self.ms.tokens

    def prepare_compaction(self):
        """Sets the segment to turn t-1 and builds turn t's proxy queries for it."""
        s0, s1 = self.compaction_segment()
        self.case.seg_start[0], self.case.seg_end[0] = s0, s1
        make_q(self.case, self.seed * 1000 + self.turn)
        return s0, s1

    def compacted(self, kept_blocks: int):
        """Record that turn t-1's segment now holds ``kept_blocks`` blocks; later turns' slot
        starts shift down by the freed blocks."""
        t = self.turn
        s0, s1 = self.compaction_segment()
        freed = math.ceil(self.ms.tokens / self.ms.P) - kept_blocks
        shift = freed * self.ms.P
        self.turn_start_slot[t] -= shift
        self.case.seq_len[0] -= shift
        self.case.seg_start[0] = self.case.seg_end[0] = 0


def random_keep(case: Case, m: Sequence[int], seed: int) -> torch.Tensor:
    """A seeded keep set per unit, independent of any score: for every (layer, head, sequence)
    min(m_b, n_b) distinct segment positions in ascending order, laid out [L][H][Mtot]."""
    sp = case.spec
    dev = case.k_pool.device
    g = _gen(dev, seed, 7)
    n = [e - s for s, e in zip(case.seg_start, case.seg_end)]
    mm = [min(int(a), b) for a, b in zip(m, n)]
    Mtot = sum(mm)
    keep = torch.empty((sp.L, sp.H, max(1, Mtot)), dtype=torch.int32, device=dev)
    for l in range(sp.L):
        for h in range(sp.H):
            off = 0
            for b in range(len(n)):
                if mm[b] > 0:
                    pick = torch.randperm(n[b], generator=g, device=dev)[:mm[b]]
                    keep[l, h, off:off + mm[b]] = torch.sort(pick).values.to(torch.int32)
                off += mm[b]
    return keep[:, :, :Mtot]
