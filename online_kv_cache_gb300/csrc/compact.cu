// compact.cu -- conflict-free slot plan, one parallel copy, block release.
//
// The ActKV analysis page (zhichai.net, system-engineering paragraph) plans
// the compaction so that a single parallel copy suffices: the last X logical
// blocks of the segment form the target region T, each retained entry outside
// T is paired with one hole inside T, all pairs are copied at once, and the
// blocks emptied by the move go back to the scheduler.
//
// Pairing (per unit = layer l, KV head h, sequence b; segment-relative slots):
//   nb = ceil(n/P), X = ceil(m/P), Bs = (nb - X) P, T = [Bs, Bs + X P)
//   keep[0..c_out) lie before Bs (they move), keep[c_out..m) lie in T (stay)
//   r_i = keep[i] - Bs - (i - c_out)  = holes of T before keep[i] (non-decreasing)
//   hole k of T (ascending) sits at t_k = Bs + k + #{i >= c_out : r_i <= k}
//   move k (k < c_out): keep[k] -> t_k;  holes k in [c_out, c_out + X P - m): dead
// Every move is computed independently (two binary searches), so the planner
// is one thread per hole with no scan.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int kPlanThreads = 512;
constexpr int kEmitWords = 4;  // plan: bitmap words a warp emits at once

// Block-wide exclusive prefix sum of one value per thread (kPlanThreads threads);
// returns the exclusive prefix and writes the block total to *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = lane < kPlanThreads / 32 ? warp_sums[lane] : 0u;
    uint32_t y = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += t;
    }
    if (lane < kPlanThreads / 32) warp_sums[lane] = y - w;
    if (lane == 31) *total = y;
  }
  __syncthreads();
  const uint32_t r = warp_sums[warp] + x - v;
  __syncthreads();
  return r;
}

// One CTA per unit (sequence, layer, head).  Inside survivors keep[c_out..m)
// are marked in a shared-memory bitmap of the target region T; a block scan over
// the bitmap words numbers the holes of T in ascending slot order; hole k takes
// the k-th outside survivor (k < c_out) or is dead.
__device__ __forceinline__ void plan_block(const LaunchMeta& meta, int64_t item, const int32_t* __restrict__ block_table,
                                           const int32_t* __restrict__ keep, int32_t* __restrict__ moves,
                                           int32_t* __restrict__ move_count, int32_t* __restrict__ dead,
                                           int32_t* __restrict__ dead_count, unsigned* status) {
  extern __shared__ uint32_t bitmap[];  // meta.words words
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t sh_total;
  __shared__ uint32_t word_holes[kPlanThreads], word_first[kPlanThreads];
  const int si = find_seq(meta, item);
  const SeqMeta& s = meta.seq[si];
  const int P = meta.P;
  const int64_t local = item - s.item0;
  const int h = (int)(local % meta.H);
  const int l = (int)(local / meta.H);
  const int64_t lh = (int64_t)l * meta.H + h;
  const int64_t u = lh * meta.B + s.b;
  const int32_t* ku = keep + lh * meta.Mtot + s.moff;
  const int m = s.m;
  const int XP = s.X * P;
  const int Bs = (s.nb - s.X) * P;
  const int tid = threadIdx.x;

  // c_out = #{keep < Bs}.  keep is ascending, so probes below Bs form a prefix:
  // each round narrows [lo, hi] (which holds the answer) by a factor of the
  // block size; every thread takes the same branches.
  int lo = 0, hi = m;
  while (lo < hi) {
    const int step = (hi - lo + kPlanThreads - 1) / kPlanThreads;
    const int i = lo + tid * step;
    const int below = __syncthreads_count((i < hi) && (__ldg(ku + i) < Bs));
    if (below == 0) {
      hi = lo;
    } else {
      const int last = lo + (below - 1) * step;  // last probe below Bs
      hi = min(hi, last + step);
      lo = last + 1;
    }
  }
  const int c_out = lo;
  if (tid == 0) {
    move_count[u] = c_out;
    dead_count[u] = XP - m;
  }
  if (XP == 0) return;

  // bitmap of inside survivors
  const int words = (XP + 31) >> 5;
  for (int w = tid; w < words; w += kPlanThreads) bitmap[w] = 0u;
  __syncthreads();
#pragma unroll 4
  for (int i = c_out + tid; i < m; i += kPlanThreads) {
    const int32_t pos = __ldg(ku + i);
    const int rel = pos - Bs;
    if (rel < 0 || rel >= XP || pos >= s.n) {
      atomicOr(status, KVC_DEV_BAD_KEEP);
      continue;
    }
    atomicOr(&bitmap[rel >> 5], 1u << (rel & 31));
  }
  __syncthreads();

  // number the holes and emit moves / dead slots: kPlanThreads bitmap words at a
  // time, a block scan numbers each word's first hole.  A full round of words
  // keeps every thread busy on its own word's holes; a partial one (few words:
  // most threads would idle) hands each word to a warp, lane b taking bit b, so
  // a word's holes need one round of loads rather than one per hole
  const int32_t* bt_row = block_table + (int64_t)s.b * meta.max_blocks;
  const int ndead = XP - m;
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t base = 0;
  for (int w0 = 0; w0 < words; w0 += kPlanThreads) {
    const int w = w0 + tid;
    uint32_t holes = 0u;
    if (w < words) {
      holes = ~bitmap[w];
      const int valid = XP - (w << 5);
      if (valid < 32) holes &= (1u << valid) - 1u;
    }
    const uint32_t before = block_exclusive_scan(__popc(holes), warp_sums, &sh_total);
    const uint32_t total = sh_total;
    word_holes[tid] = holes;
    word_first[tid] = base + before;
    __syncthreads();
    const int nw = min(kPlanThreads, words - w0);
    if (nw == kPlanThreads) {  // a full round: every thread emits its own word's holes in turn
      uint32_t k = base + before;
      while (holes != 0u) {
        const int bit = __ffs(holes) - 1;
        holes &= holes - 1u;
        if ((int)k < c_out + ndead) {
          const int t = s.s0 + Bs + (w << 5) + bit;
          const int32_t dpage = __ldg(bt_row + t / P);
          int32_t dst = -1;
          if (dpage < 0 || dpage >= meta.num_pages) atomicOr(status, KVC_DEV_BAD_PAGE);
          else dst = dpage * P + t % P;
          if ((int)k < c_out) {
            const int32_t pos = __ldg(ku + k);
            int32_t src = -1;
            if (pos < 0 || pos >= s.n) {
              atomicOr(status, KVC_DEV_BAD_KEEP);
            } else {
              const int32_t spage = __ldg(bt_row + (s.s0 + pos) / P);
              if (spage < 0 || spage >= meta.num_pages) atomicOr(status, KVC_DEV_BAD_PAGE);
              else src = spage * P + (s.s0 + pos) % P;
            }
            reinterpret_cast<int2*>(moves)[lh * meta.Mtot + s.moff + k] = make_int2(src, dst);
          } else {
            dead[u * P + (k - c_out)] = dst;
          }
        }
        ++k;
      }
    }
    // a partial round: each warp takes kEmitWords words at once, their loads issued together
    for (int i0 = warp; nw < kPlanThreads && i0 < nw; i0 += kEmitWords * (kPlanThreads / 32)) {
      int k[kEmitWords], t[kEmitWords], pos[kEmitWords];
      int32_t dpage[kEmitWords], spage[kEmitWords];
#pragma unroll
      for (int q = 0; q < kEmitWords; ++q) {
        const int i = i0 + q * (kPlanThreads / 32);
        const uint32_t hw = i < nw ? word_holes[i] : 0u;
        k[q] = -1;
        if ((hw >> lane) & 1u) {
          const int kk = (int)(word_first[i] + __popc(hw & ((1u << lane) - 1u)));
          if (kk < c_out + ndead) k[q] = kk;
        }
        t[q] = s.s0 + Bs + ((w0 + i) << 5) + lane;
        dpage[q] = k[q] >= 0 ? __ldg(bt_row + t[q] / P) : -1;
        pos[q] = (k[q] >= 0 && k[q] < c_out) ? __ldg(ku + k[q]) : -1;
      }
#pragma unroll
      for (int q = 0; q < kEmitWords; ++q) {
        spage[q] = -1;
        if (k[q] >= 0 && k[q] < c_out && pos[q] >= 0 && pos[q] < s.n) spage[q] = __ldg(bt_row + (s.s0 + pos[q]) / P);
      }
#pragma unroll
      for (int q = 0; q < kEmitWords; ++q) {
        if (k[q] < 0) continue;
        int32_t dst = -1;
        if (dpage[q] < 0 || dpage[q] >= meta.num_pages) atomicOr(status, KVC_DEV_BAD_PAGE);
        else dst = dpage[q] * P + t[q] % P;
        if (k[q] < c_out) {
          int32_t src = -1;
          if (pos[q] < 0 || pos[q] >= s.n) {
            atomicOr(status, KVC_DEV_BAD_KEEP);
          } else if (spage[q] < 0 || spage[q] >= meta.num_pages) {
            atomicOr(status, KVC_DEV_BAD_PAGE);
          } else {
            src = spage[q] * P + (s.s0 + pos[q]) % P;
          }
          reinterpret_cast<int2*>(moves)[lh * meta.Mtot + s.moff + k[q]] = make_int2(src, dst);
        } else {
          dead[u * P + (k[q] - c_out)] = dst;
        }
      }
    }
    base += total;
    __syncthreads();  // word_holes / word_first are rewritten for the next 512 words
  }
}

// Block-table rows after the release and the list of freed pages (sequence
// order, ascending block order).  kRowSplit CTAs per sequence, each taking every
// kRowSplit-th stretch of 256 entries (every entry is independent).
constexpr int kRowSplit = 8;

__device__ __forceinline__ void rows_block(const LaunchMeta& meta, int blk, const int32_t* __restrict__ block_table,
                                           const int32_t* __restrict__ nblocks, int32_t* __restrict__ freed,
                                           int32_t* __restrict__ new_rows, unsigned* status) {
  const SeqMeta& s = meta.seq[blk / kRowSplit];
  const int j0 = (blk % kRowSplit) * blockDim.x + threadIdx.x;
  const int js = kRowSplit * blockDim.x;
  const int P = meta.P;
  const int f = s.nb - s.X;
  const int sb = s.s0 / P;
  const int32_t* row = block_table + (int64_t)s.b * meta.max_blocks;
  int32_t* out = new_rows + (int64_t)s.b * meta.max_blocks;
  const int nold = __ldg(nblocks + s.b);
  if (nold < sb + s.nb || nold > meta.max_blocks) {
    if (j0 == 0) atomicOr(status, KVC_DEV_BAD_PAGE);
    for (int j = j0; j < meta.max_blocks; j += js) out[j] = row[j];
    return;
  }
  for (int j = j0; j < meta.max_blocks; j += js) {
    int32_t v = row[j];
    if (j >= sb && j < nold - f) v = row[j + f];
    else if (j >= nold - f && j < nold) v = -1;
    out[j] = v;
  }
  for (int i = j0; i < f; i += js) freed[s.foff + i] = row[sb + i];
}

// The slot plan and the block-table rows in one launch: blocks [0, plan.items)
// plan one unit each, the next rows.nseq * kRowSplit blocks build the new
// block-table rows and the freed lists (the two read the same block table and
// write disjoint buffers).
__global__ void __launch_bounds__(kPlanThreads)
    plan_rows_kernel(const __grid_constant__ LaunchMeta plan, const __grid_constant__ LaunchMeta rows,
                     const int32_t* __restrict__ block_table, const int32_t* __restrict__ nblocks,
                     const int32_t* __restrict__ keep, int32_t* __restrict__ moves,
                     int32_t* __restrict__ move_count, int32_t* __restrict__ dead,
                     int32_t* __restrict__ dead_count, int32_t* __restrict__ freed,
                     int32_t* __restrict__ new_rows, unsigned* status) {
  if ((int64_t)blockIdx.x < plan.items)
    plan_block(plan, blockIdx.x, block_table, keep, moves, move_count, dead, dead_count, status);
  else
    rows_block(rows, (int)(blockIdx.x - plan.items), block_table, nblocks, freed, new_rows, status);
}

// One parallel copy.  A block copies up to meta.mpb moves of one unit
// (the unit is decoded once per block): each move moves a K row and a V row
// (d bf16 each, 16-byte vectors, D/4 lanes per move), the tag and, when the
// cache has one, the per-slot aux value; U moves are
// in flight per lane group.  The unit's first block also writes tag -1 to its
// dead holes.
template <int D>
__global__ void __launch_bounds__(256)
    copy_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ moves,
                const int32_t* __restrict__ move_count, const int32_t* __restrict__ dead,
                const int32_t* __restrict__ dead_count, uint8_t* __restrict__ k_pool,
                uint8_t* __restrict__ v_pool, int32_t* __restrict__ tags, float* __restrict__ aux) {
  constexpr int LPM = D / 4;     // lanes per move
  constexpr int MPW = 32 / LPM;  // moves per warp step
  constexpr int CH = D / 8;      // 16-byte chunks per row
  constexpr int U = 1;           // moves in flight per lane group (more resident warps beat more per thread)
  constexpr int64_t kRowBytes = (int64_t)D * 2;
  const int64_t item = blockIdx.x;
  const int si = find_seq(meta, item);
  const SeqMeta& s = meta.seq[si];
  const int per = max(1, (s.m + meta.mpb - 1) / meta.mpb);
  const int64_t local = item - s.item0;
  const int chunk = (int)(local % per);
  const int64_t lh = local / per;
  const int h = (int)(lh % meta.H), l = (int)(lh / meta.H);
  const int64_t u = lh * meta.B + s.b;
  const int P = meta.P, lp = meta.log2P;
  const int64_t HP = (int64_t)meta.H * P;
  const int64_t lbase = (int64_t)l * meta.num_pages * HP + (int64_t)h * P;
  const int cnt = __ldg(move_count + u);
  const int k0 = chunk * meta.mpb, k1 = min(k0 + meta.mpb, cnt);
  const int2* mv = reinterpret_cast<const int2*>(moves) + (lh * meta.Mtot + s.moff);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane / LPM, c = lane % LPM;
  const int which = c / CH, ch = c % CH;
  uint8_t* pool = which ? v_pool : k_pool;
  constexpr int kStride = 8 * MPW;  // moves per block step (8 warps)
  for (int kb = k0 + warp * MPW + grp; kb < k1; kb += U * kStride) {
    int4 val[U];
    int64_t drow[U];
    int32_t tag[U];
    float ax[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int k = kb + q * kStride;
      drow[q] = -1;
      if (k < k1) {
        const int2 m2 = __ldg(mv + k);
        if (m2.x >= 0 && m2.y >= 0) {
          const int64_t srow = lbase + (int64_t)(m2.x >> lp) * HP + (m2.x & (P - 1));
          drow[q] = lbase + (int64_t)(m2.y >> lp) * HP + (m2.y & (P - 1));
          val[q] = *reinterpret_cast<const int4*>(pool + srow * kRowBytes + ch * 16);
          if (c == 0) {
            tag[q] = tags[srow];
            if (aux) ax[q] = aux[srow];
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < U; ++q) {
      if (drow[q] < 0) continue;
      *reinterpret_cast<int4*>(pool + drow[q] * kRowBytes + ch * 16) = val[q];
      if (c == 0) {
        tags[drow[q]] = tag[q];
        if (aux) aux[drow[q]] = ax[q];
      }
    }
  }
  if (chunk == 0) {
    const int nd = __ldg(dead_count + u);
    for (int j = threadIdx.x; j < nd; j += blockDim.x) {
      const int32_t dst = __ldg(dead + u * P + j);
      if (dst >= 0) tags[lbase + (int64_t)(dst >> lp) * HP + (dst & (P - 1))] = -1;
    }
  }
}

// Installs the new block-table rows and lowers nblocks (one CTA per sequence),
// and pushes the freed pages onto the free stack (the last cluster of
// kPushCluster CTAs: rank 0 reads the stack top and checks the capacity, every
// rank pushes a slice, rank 0 moves the top once all have).  A push that would
// overflow the stack's capacity sets KVC_DEV_FREE_STACK and pushes nothing.
constexpr int kPushCluster = 8;

__global__ void __cluster_dims__(kPushCluster, 1, 1) __launch_bounds__(256)
    free_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ new_rows,
                const int32_t* __restrict__ freed, int32_t* __restrict__ block_table,
                int32_t* __restrict__ nblocks, int32_t* __restrict__ free_ids,
                int32_t* __restrict__ free_top, int32_t capacity, unsigned* status) {
  const int seq_ctas = (meta.nseq + kPushCluster - 1) / kPushCluster * kPushCluster;
  if ((int)blockIdx.x < seq_ctas) {
    if ((int)blockIdx.x >= meta.nseq) return;
    const SeqMeta& s = meta.seq[blockIdx.x];
    const int f = s.nb - s.X;
    if (f <= 0) return;
    const int64_t ro = (int64_t)s.b * meta.max_blocks;
    copy_ints8(block_table + ro, new_rows + ro, meta.max_blocks);
    if (threadIdx.x == 0) nblocks[s.b] -= f;
    return;
  }
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  __shared__ int sh_top;
  __shared__ int sh_ok;
  const int64_t f0 = meta.seq[0].foff;
  const int64_t count = meta.Ftot;  // pages freed by this launch's sequences
  if (rank == 0 && threadIdx.x == 0) {
    const int top = *free_top;
    sh_top = top;
    sh_ok = (top >= 0 && (int64_t)top + count <= capacity) ? 1 : 0;
    if (!sh_ok) atomicOr(status, KVC_DEV_FREE_STACK);
  }
  cluster.sync();
  const int top = *cluster.map_shared_rank(&sh_top, 0);
  const int ok = *cluster.map_shared_rank(&sh_ok, 0);
  if (ok) {
    const int64_t chunk = (count + kPushCluster - 1) / kPushCluster;
    const int64_t lo = std::min<int64_t>(count, rank * chunk), hi = std::min<int64_t>(count, lo + chunk);
    copy_ints8(free_ids + top + lo, freed + f0 + lo, hi - lo);
  }
  cluster.sync();  // every slice is pushed and rank 0's top has been read
  if (rank == 0 && threadIdx.x == 0 && ok) *free_top = top + (int)count;
}

}  // namespace

cudaError_t launch_plan(const CompactLaunch& cl, cudaStream_t stream) {
  for (size_t c = 0; c < cl.chunks; ++c) {
    const LaunchMeta& m = cl.plan_meta[c];
    const LaunchMeta& r = cl.rows_meta[c];
    const int64_t blocks = m.items + (int64_t)r.nseq * kRowSplit;
    if (blocks <= 0) continue;
    const size_t smem = (size_t)std::max(1, m.words) * sizeof(uint32_t);
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(plan_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    plan_rows_kernel<<<(unsigned)blocks, kPlanThreads, smem, stream>>>(
        m, r, cl.block_table, cl.nblocks, cl.keep, cl.moves, cl.move_count, cl.dead, cl.dead_count, cl.freed,
        cl.new_rows, cl.status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
  }
  return cudaSuccess;
}

cudaError_t launch_compact(const CompactLaunch& cl, cudaStream_t stream) {
  for (size_t c = 0; c < cl.chunks; ++c) {
    const LaunchMeta& m = cl.copy_meta[c];
    if (m.items <= 0) continue;
    if (m.d == 128)
      copy_kernel<128><<<(unsigned)m.items, 256, 0, stream>>>(
          m, cl.moves, cl.move_count, cl.dead, cl.dead_count, static_cast<uint8_t*>(cl.k_pool),
          static_cast<uint8_t*>(cl.v_pool), cl.tags, cl.aux);
    else
      copy_kernel<64><<<(unsigned)m.items, 256, 0, stream>>>(
          m, cl.moves, cl.move_count, cl.dead, cl.dead_count, static_cast<uint8_t*>(cl.k_pool),
          static_cast<uint8_t*>(cl.v_pool), cl.tags, cl.aux);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
  }
  return cudaSuccess;
}

cudaError_t launch_free(const CompactLaunch& cl, cudaStream_t stream) {
  for (size_t c = 0; c < cl.chunks; ++c) {
    const LaunchMeta& m = cl.free_meta[c];
    if (m.nseq <= 0) continue;
    const int seq_ctas = (m.nseq + kPushCluster - 1) / kPushCluster * kPushCluster;
    free_kernel<<<(unsigned)(seq_ctas + kPushCluster), 256, 0, stream>>>(m, cl.new_rows, cl.freed, cl.block_table_mut,
                                                            cl.nblocks, cl.free_ids, cl.free_top,
                                                            cl.capacity, cl.status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
  }
  return cudaSuccess;
}

}  // namespace kvc
