// layout.cu -- layout variants of eviction.
//
// Sentinel eviction ("IntentKV: Cross-Turn Intent-Aware KV Cache Pruning",
// section on layout-preserving eviction): an evicted position becomes a dead
// slot holding constants that remove its attention contribution (every key
// element bf16(-10^4), every value element 0, tag -1); no surviving entry
// moves and no page is freed.
//
// Fresh-page compaction (the same page's objection that in-place compaction
// renumbers positions, answered by moving every survivor in logical order):
// a sequence that keeps m < n positions takes X = ceil(m/P) pages from the
// free stack, its r-th survivor goes to slot r of those pages, and all nb old
// blocks of the segment go back to the stack.  The plan fills an ordinary
// kvc_plan (moves and dead slots), which kvc_compact executes; the commit
// pops the fresh pages, pushes the old ones and installs the new rows.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int kStackCluster = 8;  // CTAs of the fresh-page stack push (one cluster)
constexpr int kRowSplit = 8;      // CTAs per sequence for block-table rows (independent entries)


constexpr int kSentinelChunk = 4096;       // positions per sentinel block
constexpr uint32_t kSentinelPair = 0xC61CC61Cu;  // two bf16(-10^4) (= -9984)

// First index r in the ascending list a[0..n) with a[r] >= x.
__device__ __forceinline__ int lower_bound_i32(const int32_t* __restrict__ a, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// One block per (unit, 4096 positions): marks the unit's survivors of the
// chunk in a shared-memory bitmap, then writes the sentinel K row, a zero V
// row (16-byte stores, consecutive threads on consecutive chunks of a row)
// and tag -1 for every other position of the chunk.
template <int D>
__global__ void __launch_bounds__(256)
    sentinel_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ block_table,
                    const int32_t* __restrict__ keep, uint8_t* __restrict__ k_pool,
                    uint8_t* __restrict__ v_pool, int32_t* __restrict__ tags, unsigned* status) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  constexpr int64_t kRowBytes = (int64_t)D * 2;
  __shared__ uint32_t kept[kSentinelChunk / 32];
  const int64_t item = blockIdx.x;
  const SeqMeta& s = meta.seq[find_seq(meta, item)];
  const int per = max(1, (s.n + kSentinelChunk - 1) / kSentinelChunk);
  const int64_t local = item - s.item0;
  const int chunk = (int)(local % per);
  const int64_t lh = local / per;
  const int h = (int)(lh % meta.H), l = (int)(lh / meta.H);
  const int c0 = chunk * kSentinelChunk, c1 = min(c0 + kSentinelChunk, s.n);
  for (int i = threadIdx.x; i < kSentinelChunk / 32; i += blockDim.x) kept[i] = 0;
  __syncthreads();
  const int32_t* ku = keep + lh * meta.Mtot + s.moff;
  const int lo = lower_bound_i32(ku, s.m, c0), hi = lower_bound_i32(ku, s.m, c1);
  for (int r = lo + threadIdx.x; r < hi; r += blockDim.x) {
    const int32_t j = __ldg(ku + r);
    if (j < c0 || j >= c1) {  // the list is not ascending
      atomicOr(status, KVC_DEV_BAD_KEEP);
      continue;
    }
    atomicOr(&kept[(j - c0) >> 5], 1u << ((j - c0) & 31));
  }
  __syncthreads();
  const int P = meta.P, lp = meta.log2P;
  const int64_t HP = (int64_t)meta.H * P;
  const int64_t lbase = (int64_t)l * meta.num_pages * HP + (int64_t)h * P;
  const int32_t* bt = block_table + (int64_t)s.b * meta.max_blocks;
  const int np = c1 - c0;
  const int4 ksent = make_int4((int)kSentinelPair, (int)kSentinelPair, (int)kSentinelPair, (int)kSentinelPair);
  const int4 zero = make_int4(0, 0, 0, 0);
  for (int w = threadIdx.x; w < np * 2 * CH; w += blockDim.x) {
    const int p = w / (2 * CH), c = w % (2 * CH);
    if ((kept[p >> 5] >> (p & 31)) & 1u) continue;
    const int slot = s.s0 + c0 + p;
    const int32_t page = __ldg(bt + (slot >> lp));
    if (page < 0 || page >= meta.num_pages) {
      if (c == 0) atomicOr(status, KVC_DEV_BAD_PAGE);
      continue;
    }
    const int64_t row = lbase + (int64_t)page * HP + (slot & (P - 1));
    if (c < CH)
      *reinterpret_cast<int4*>(k_pool + row * kRowBytes + c * 16) = ksent;
    else
      *reinterpret_cast<int4*>(v_pool + row * kRowBytes + (c - CH) * 16) = zero;
    if (c == 0) tags[row] = -1;
  }
}

// Page handed out by pop number k of this call: the stack's top - 1 - k.
__device__ __forceinline__ int32_t fresh_page(const int32_t* __restrict__ free_ids, int top, int64_t k) {
  return free_ids[top - 1 - k];
}

// Fresh plan, one block per (unit, 1024 survivors): the r-th survivor moves
// from its slot (old block table) to slot r of the sequence's fresh pages;
// the unit's first block writes the counts and the dead slots m .. X*P-1 of
// the last fresh page.  Sequences that keep everything get no moves.  If the
// stack holds fewer than the call's pops, nothing is planned and the status
// word gets KVC_DEV_FREE_STACK.
__global__ void __launch_bounds__(256)
    fresh_moves_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ block_table,
                       const int32_t* __restrict__ keep, const int32_t* __restrict__ free_ids,
                       const int32_t* __restrict__ free_top, int32_t* __restrict__ moves,
                       int32_t* __restrict__ move_count, int32_t* __restrict__ dead,
                       int32_t* __restrict__ dead_count, unsigned* status) {
  const int64_t item = blockIdx.x;
  const SeqMeta& s = meta.seq[find_seq(meta, item)];
  const int per = max(1, (s.m + kFreshMovesPerBlock - 1) / kFreshMovesPerBlock);
  const int64_t local = item - s.item0;
  const int chunk = (int)(local % per);
  const int64_t lh = local / per;
  const int64_t u = lh * meta.B + s.b;
  const int P = meta.P, lp = meta.log2P;
  const bool active = s.m < s.n;
  const int top = *free_top;
  const bool ok = top >= meta.Xtot;
  if (chunk == 0 && threadIdx.x == 0) {
    if (active && !ok) atomicOr(status, KVC_DEV_FREE_STACK);
    move_count[u] = (active && ok) ? s.m : 0;
    dead_count[u] = (active && ok) ? s.X * P - s.m : 0;
  }
  if (!active || !ok) return;
  const int32_t* ku = keep + lh * meta.Mtot + s.moff;
  int2* mv = reinterpret_cast<int2*>(moves) + (lh * meta.Mtot + s.moff);
  const int32_t* bt = block_table + (int64_t)s.b * meta.max_blocks;
  const int k0 = chunk * kFreshMovesPerBlock, k1 = min(k0 + kFreshMovesPerBlock, s.m);
  for (int r = k0 + threadIdx.x; r < k1; r += blockDim.x) {
    const int32_t j = __ldg(ku + r);
    int2 m2 = make_int2(-1, -1);
    if (j < 0 || j >= s.n) {
      atomicOr(status, KVC_DEV_BAD_KEEP);
    } else {
      const int slot = s.s0 + j;
      const int32_t src_page = __ldg(bt + (slot >> lp));
      const int32_t dst_page = fresh_page(free_ids, top, (int64_t)s.xoff + (r >> lp));
      if (src_page < 0 || src_page >= meta.num_pages || dst_page < 0 || dst_page >= meta.num_pages)
        atomicOr(status, KVC_DEV_BAD_PAGE);
      else
        m2 = make_int2(src_page * P + (slot & (P - 1)), dst_page * P + (r & (P - 1)));
    }
    mv[r] = m2;
  }
  if (chunk == 0) {
    const int nd = s.X * P - s.m;
    const int32_t last = fresh_page(free_ids, top, (int64_t)s.xoff + s.X - 1);
    const bool last_ok = last >= 0 && last < meta.num_pages;
    for (int jd = threadIdx.x; jd < nd; jd += blockDim.x)
      dead[u * P + jd] = last_ok ? last * P + ((s.m + jd) & (P - 1)) : -1;
  }
}

// Fresh plan, kRowSplit blocks per sequence: the block-table row after the commit
// (the segment's nb entries replaced by the X fresh pages, later entries
// shifted down by nb - X, vacated entries -1) and the sequence's nb old
// pages at its offset of the call's return list.
__global__ void __launch_bounds__(256)
    fresh_rows_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ block_table,
                      const int32_t* __restrict__ nblocks, const int32_t* __restrict__ free_ids,
                      const int32_t* __restrict__ free_top, int32_t* __restrict__ freed,
                      int32_t* __restrict__ new_rows, unsigned* status) {
  const SeqMeta& s = meta.seq[blockIdx.x / kRowSplit];
  const int j0 = (int)(blockIdx.x % kRowSplit) * blockDim.x + threadIdx.x;
  const int js = kRowSplit * blockDim.x;
  const int P = meta.P;
  const int32_t* row = block_table + (int64_t)s.b * meta.max_blocks;
  int32_t* out = new_rows + (int64_t)s.b * meta.max_blocks;
  const int top = *free_top;
  const int nold = __ldg(nblocks + s.b);
  const int sb = s.s0 / P, f = s.nb - s.X;
  const bool active = s.m < s.n && top >= meta.Xtot;
  if (active && (nold < sb + s.nb || nold > meta.max_blocks)) {
    if (j0 == 0) atomicOr(status, KVC_DEV_BAD_PAGE);
  }
  const bool go = active && nold >= sb + s.nb && nold <= meta.max_blocks;
  for (int jb = j0; jb < meta.max_blocks; jb += js) {
    int32_t v = row[jb];
    if (go) {
      if (jb >= sb && jb < sb + s.X) v = fresh_page(free_ids, top, (int64_t)s.xoff + (jb - sb));
      else if (jb >= sb + s.X && jb < nold - f) v = row[jb + f];
      else if (jb >= nold - f && jb < nold) v = -1;
    }
    out[jb] = v;
  }
  if (go)
    for (int i = j0; i < s.nb; i += js) freed[s.foff + i] = row[sb + i];
}

// Fresh commit, one cluster of kStackCluster CTAs for the whole call: unless the
// status word already holds KVC_DEV_FREE_STACK, pops the call's Xtot pages and
// pushes the Ftot returned ones in their list order (rank 0 reads and checks the
// stack top, every rank pushes a slice, rank 0 moves the top after a cluster
// barrier); a stack that cannot take them sets KVC_DEV_FREE_STACK and changes
// nothing.
__global__ void __cluster_dims__(kStackCluster, 1, 1) __launch_bounds__(256)
    fresh_stack_kernel(int64_t Xtot, int64_t Ftot, const int32_t* __restrict__ freed,
                       int32_t* __restrict__ free_ids, int32_t* __restrict__ free_top, int32_t capacity,
                       unsigned* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  __shared__ int sh_base, sh_ok;
  if (rank == 0 && threadIdx.x == 0) {
    const unsigned st = *reinterpret_cast<volatile unsigned*>(status);
    const int top = *free_top;
    const int64_t base = (int64_t)top - Xtot;
    sh_ok = !(st & KVC_DEV_FREE_STACK) && base >= 0 && base + Ftot <= capacity;
    if (!(st & KVC_DEV_FREE_STACK) && !sh_ok) atomicOr(status, KVC_DEV_FREE_STACK);
    sh_base = (int)base;
  }
  cluster.sync();
  const int base = *cluster.map_shared_rank(&sh_base, 0);
  const int ok = *cluster.map_shared_rank(&sh_ok, 0);
  if (ok) {  // every rank pushes one slice
    const int64_t chunk = (Ftot + kStackCluster - 1) / kStackCluster;
    const int64_t lo = std::min<int64_t>(Ftot, rank * chunk), hi = std::min<int64_t>(Ftot, lo + chunk);
    copy_ints8(free_ids + base + lo, freed + lo, hi - lo);
  }
  cluster.sync();  // every slice is pushed and rank 0's values have been read
  if (rank == 0 && threadIdx.x == 0 && ok) *free_top = base + (int)Ftot;
}

// Fresh commit, kRowSplit blocks per sequence (after fresh_stack_kernel): installs
// the planned row and lowers nblocks by nb - X, unless the stack step failed.
__global__ void __launch_bounds__(256)
    fresh_install_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ new_rows,
                         int32_t* __restrict__ block_table, int32_t* __restrict__ nblocks,
                         const unsigned* status) {
  const SeqMeta& s = meta.seq[blockIdx.x / kRowSplit];
  const int j0 = (int)(blockIdx.x % kRowSplit) * blockDim.x + threadIdx.x;
  const int js = kRowSplit * blockDim.x;
  if (!(s.m < s.n)) return;
  if (*reinterpret_cast<const volatile unsigned*>(status) & KVC_DEV_FREE_STACK) return;
  const int64_t ro = (int64_t)s.b * meta.max_blocks;
  for (int jb = j0; jb < meta.max_blocks; jb += js) block_table[ro + jb] = new_rows[ro + jb];
  if (j0 == 0) nblocks[s.b] -= s.nb - s.X;
}

}  // namespace

cudaError_t launch_sentinel(const LayoutLaunch& ll, cudaStream_t stream) {
  for (size_t c = 0; c < ll.chunks; ++c) {
    const LaunchMeta& m = ll.meta[c];
    if (m.items <= 0) continue;
    if (m.d == 128)
      sentinel_kernel<128><<<(unsigned)m.items, 256, 0, stream>>>(
          m, ll.block_table, ll.keep, static_cast<uint8_t*>(ll.k_pool), static_cast<uint8_t*>(ll.v_pool),
          ll.tags, ll.status);
    else
      sentinel_kernel<64><<<(unsigned)m.items, 256, 0, stream>>>(
          m, ll.block_table, ll.keep, static_cast<uint8_t*>(ll.k_pool), static_cast<uint8_t*>(ll.v_pool),
          ll.tags, ll.status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
  }
  return cudaSuccess;
}

cudaError_t launch_fresh_plan(const LayoutLaunch& ll, cudaStream_t stream) {
  for (size_t c = 0; c < ll.chunks; ++c) {
    const LaunchMeta& m = ll.meta[c];
    if (m.items > 0) {
      fresh_moves_kernel<<<(unsigned)m.items, 256, 0, stream>>>(m, ll.block_table, ll.keep, ll.free_ids,
                                                                ll.free_top, ll.moves, ll.move_count,
                                                                ll.dead, ll.dead_count, ll.status);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      count_launch();
    }
    const LaunchMeta& r = ll.rows[c];
    if (r.nseq > 0) {
      fresh_rows_kernel<<<(unsigned)(r.nseq * kRowSplit), 256, 0, stream>>>(r, ll.block_table, ll.nblocks, ll.free_ids,
                                                              ll.free_top, ll.freed, ll.new_rows, ll.status);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      count_launch();
    }
  }
  return cudaSuccess;
}

cudaError_t launch_fresh_commit(const LayoutLaunch& ll, cudaStream_t stream) {
  if (ll.chunks == 0) return cudaSuccess;
  fresh_stack_kernel<<<kStackCluster, 256, 0, stream>>>(ll.rows[0].Xtot, ll.Ftot_all, ll.freed, ll.free_ids,
                                            ll.free_top, ll.capacity, ll.status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launch();
  for (size_t c = 0; c < ll.chunks; ++c) {
    const LaunchMeta& r = ll.rows[c];
    if (r.nseq <= 0) continue;
    fresh_install_kernel<<<(unsigned)(r.nseq * kRowSplit), 256, 0, stream>>>(r, ll.new_rows, ll.block_table_mut,
                                                               ll.nblocks, ll.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    count_launch();
  }
  return cudaSuccess;
}

}  // namespace kvc
