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
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

constexpr int kPlanThreads = 256;

__device__ __forceinline__ int32_t phys_slot(const int32_t* bt_row, int slot, int P, int num_pages,
                                             unsigned* status) {
  const int32_t page = __ldg(bt_row + slot / P);
  if (page < 0 || page >= num_pages) {
    atomicOr(status, KVC_DEV_BAD_PAGE);
    return -1;
  }
  return page * P + slot % P;
}

__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ block_table,
                const int32_t* __restrict__ keep, int32_t* __restrict__ moves,
                int32_t* __restrict__ move_count, int32_t* __restrict__ dead,
                int32_t* __restrict__ dead_count, unsigned* status) {
  __shared__ int sh_cout;
  const int64_t item = blockIdx.x;
  const int si = find_seq(meta, item);
  const SeqMeta& s = meta.seq[si];
  const int P = meta.P;
  const int per = max(1, (s.X * P + kPlanThreads - 1) / kPlanThreads);
  int64_t local = item - s.item0;
  const int chunk = (int)(local % per);
  local /= per;
  const int h = (int)(local % meta.H);
  const int l = (int)(local / meta.H);
  const int64_t lh = (int64_t)l * meta.H + h;
  const int64_t u = lh * meta.B + s.b;
  const int32_t* ku = keep + lh * meta.Mtot + s.moff;
  const int m = s.m;
  const int Bs = (s.nb - s.X) * P;
  if (threadIdx.x == 0) {
    int lo = 0, hi = m;  // first index with keep >= Bs
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(ku + mid) < Bs) lo = mid + 1; else hi = mid;
    }
    sh_cout = lo;
    if (chunk == 0) {
      move_count[u] = lo;
      dead_count[u] = s.X * P - m;
    }
  }
  __syncthreads();
  const int c_out = sh_cout;
  const int k = chunk * kPlanThreads + threadIdx.x;
  if (k >= c_out + (s.X * P - m)) return;
  // number of retained entries of T that precede hole k
  int lo = c_out, hi = m;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(ku + mid) - Bs - (mid - c_out) <= k) lo = mid + 1; else hi = mid;
  }
  const int t = Bs + k + (lo - c_out);
  const int32_t* bt_row = block_table + (int64_t)s.b * meta.max_blocks;
  const int32_t dst = phys_slot(bt_row, s.s0 + t, P, meta.num_pages, status);
  if (k < c_out) {
    const int32_t pos = __ldg(ku + k);
    int32_t src = -1;
    if (pos < 0 || pos >= s.n) atomicOr(status, KVC_DEV_BAD_KEEP);
    else src = phys_slot(bt_row, s.s0 + pos, P, meta.num_pages, status);
    const int64_t mi = lh * meta.Mtot + s.moff + k;
    moves[2 * mi] = src;
    moves[2 * mi + 1] = dst;
  } else {
    dead[u * P + (k - c_out)] = dst;
  }
}

// Block-table rows after the release and the list of freed pages (sequence
// order, ascending block order).  One CTA per sequence.
__global__ void __launch_bounds__(kPlanThreads)
    rows_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ block_table,
                const int32_t* __restrict__ nblocks, int32_t* __restrict__ freed,
                int32_t* __restrict__ new_rows, unsigned* status) {
  const SeqMeta& s = meta.seq[blockIdx.x];
  const int P = meta.P;
  const int f = s.nb - s.X;
  const int sb = s.s0 / P;
  const int32_t* row = block_table + (int64_t)s.b * meta.max_blocks;
  int32_t* out = new_rows + (int64_t)s.b * meta.max_blocks;
  const int nold = __ldg(nblocks + s.b);
  if (nold < sb + s.nb || nold > meta.max_blocks) {
    if (threadIdx.x == 0) atomicOr(status, KVC_DEV_BAD_PAGE);
    for (int j = threadIdx.x; j < meta.max_blocks; j += blockDim.x) out[j] = row[j];
    return;
  }
  for (int j = threadIdx.x; j < meta.max_blocks; j += blockDim.x) {
    int32_t v = row[j];
    if (j >= sb && j < nold - f) v = row[j + f];
    else if (j >= nold - f && j < nold) v = -1;
    out[j] = v;
  }
  for (int i = threadIdx.x; i < f; i += blockDim.x) freed[s.foff + i] = row[sb + i];
}

// One parallel copy: each move copies a K row, a V row (d bf16 each, 16-byte
// vectors, D/4 lanes per move) and the tag; then dead holes get tag -1.
template <int D>
__global__ void __launch_bounds__(256)
    copy_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ moves,
                const int32_t* __restrict__ move_count, const int32_t* __restrict__ dead,
                const int32_t* __restrict__ dead_count, uint8_t* __restrict__ k_pool,
                uint8_t* __restrict__ v_pool, int32_t* __restrict__ tags) {
  constexpr int LPM = D / 4;        // lanes per move (16 B each, K and V rows)
  constexpr int MPW = 32 / LPM;     // moves per warp per step
  constexpr int CH = D / 8;         // 16-byte chunks per row
  constexpr int U = 4;              // moves in flight per lane group
  constexpr int64_t kRowBytes = (int64_t)D * 2;
  const int lane = threadIdx.x & 31;
  const int grp = lane / LPM, c = lane % LPM;
  const int which = c / CH, ch = c % CH;
  uint8_t* pool = which ? v_pool : k_pool;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t Mc = meta.items / ((int64_t)meta.L * meta.H);  // moves per (l, h) in this launch
  const int P = meta.P;
  const int64_t layer_rows = (int64_t)meta.num_pages * meta.H * P;

  for (int64_t base = gw * (MPW * U); base < meta.items; base += nw * (MPW * U)) {
    int4 val[U];
    int64_t dst_row[U];
    int32_t tag[U];
    bool act[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int64_t g = base + q * MPW + grp;
      act[q] = false;
      dst_row[q] = 0;
      tag[q] = 0;
      if (g < meta.items) {
        const int64_t lh = g / Mc;
        const int64_t rem = g - lh * Mc;
        const int si = find_seq(meta, rem);
        const SeqMeta& s = meta.seq[si];
        const int k = (int)(rem - s.item0);
        const int h = (int)(lh % meta.H), l = (int)(lh / meta.H);
        if (k < __ldg(move_count + lh * meta.B + s.b)) {
          const int64_t mi = lh * meta.Mtot + s.moff + k;
          const int32_t src = __ldg(moves + 2 * mi), dst = __ldg(moves + 2 * mi + 1);
          if (src >= 0 && dst >= 0) {
            const int64_t lbase = l * layer_rows + h * P;
            const int64_t src_row = lbase + (int64_t)(src / P) * meta.H * P + src % P;
            dst_row[q] = lbase + (int64_t)(dst / P) * meta.H * P + dst % P;
            val[q] = *reinterpret_cast<const int4*>(pool + src_row * kRowBytes + ch * 16);
            if (c == 0) tag[q] = tags[src_row];
            act[q] = true;
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < U; ++q) {
      if (!act[q]) continue;
      *reinterpret_cast<int4*>(pool + dst_row[q] * kRowBytes + ch * 16) = val[q];
      if (c == 0) tags[dst_row[q]] = tag[q];
    }
  }

  // dead holes of every unit of this launch: tag -1, bytes untouched
  const int64_t ndead = (int64_t)meta.L * meta.H * meta.nseq * P;
  for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < ndead;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(g % P);
    const int64_t r2 = g / P;
    const int si = (int)(r2 % meta.nseq);
    const int64_t lh = r2 / meta.nseq;
    const SeqMeta& s = meta.seq[si];
    const int64_t u = lh * meta.B + s.b;
    if (j >= __ldg(dead_count + u)) continue;
    const int32_t dst = __ldg(dead + u * P + j);
    if (dst < 0) continue;
    const int h = (int)(lh % meta.H), l = (int)(lh / meta.H);
    tags[l * layer_rows + h * P + (int64_t)(dst / P) * meta.H * P + dst % P] = -1;
  }
}

// Installs the new block-table rows, lowers nblocks, and pushes the freed
// pages onto the free stack (CTA nseq).  A push that would overflow the
// stack's capacity sets KVC_DEV_FREE_STACK and pushes nothing.
__global__ void __launch_bounds__(256)
    free_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ new_rows,
                const int32_t* __restrict__ freed, int32_t* __restrict__ block_table,
                int32_t* __restrict__ nblocks, int32_t* __restrict__ free_ids,
                int32_t* __restrict__ free_top, int32_t capacity, unsigned* status) {
  if ((int)blockIdx.x < meta.nseq) {
    const SeqMeta& s = meta.seq[blockIdx.x];
    const int f = s.nb - s.X;
    if (f <= 0) return;
    const int64_t ro = (int64_t)s.b * meta.max_blocks;
    for (int j = threadIdx.x; j < meta.max_blocks; j += blockDim.x) block_table[ro + j] = new_rows[ro + j];
    if (threadIdx.x == 0) nblocks[s.b] -= f;
    return;
  }
  __shared__ int sh_top;
  __shared__ int sh_ok;
  const int64_t f0 = meta.seq[0].foff;
  const int64_t count = meta.Ftot;  // pages freed by this launch's sequences
  if (threadIdx.x == 0) {
    const int top = *free_top;
    sh_top = top;
    sh_ok = (top >= 0 && (int64_t)top + count <= capacity) ? 1 : 0;
    if (!sh_ok) atomicOr(status, KVC_DEV_FREE_STACK);
  }
  __syncthreads();
  if (!sh_ok) return;
  for (int64_t i = threadIdx.x; i < count; i += blockDim.x) free_ids[sh_top + i] = freed[f0 + i];
  __syncthreads();
  if (threadIdx.x == 0) *free_top = sh_top + (int)count;
}

}  // namespace

cudaError_t launch_plan(const CompactLaunch& cl, cudaStream_t stream) {
  for (size_t c = 0; c < cl.chunks; ++c) {
    const LaunchMeta& m = cl.plan_meta[c];
    if (m.items > 0) {
      plan_kernel<<<(unsigned)m.items, kPlanThreads, 0, stream>>>(
          m, cl.block_table, cl.keep, cl.moves, cl.move_count, cl.dead, cl.dead_count, cl.status);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      count_launch();
    }
    const LaunchMeta& r = cl.rows_meta[c];
    if (r.nseq > 0) {
      rows_kernel<<<(unsigned)r.nseq, kPlanThreads, 0, stream>>>(r, cl.block_table, cl.nblocks,
                                                                 cl.freed, cl.new_rows, cl.status);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      count_launch();
    }
  }
  return cudaSuccess;
}

cudaError_t launch_compact(const CompactLaunch& cl, cudaStream_t stream) {
  for (size_t c = 0; c < cl.chunks; ++c) {
    const LaunchMeta& m = cl.copy_meta[c];
    if (m.nseq <= 0) continue;
    const int64_t warps_needed = (m.items + 3) / 4 + 1;
    const int64_t dead_threads = (int64_t)m.L * m.H * m.nseq * m.P;
    int64_t blocks = std::max<int64_t>((warps_needed + 7) / 8, (dead_threads + 255) / 256);
    blocks = std::min<int64_t>(std::max<int64_t>(blocks, 1), (int64_t)cl.num_sms * 8);
    if (m.d == 128)
      copy_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(
          m, cl.moves, cl.move_count, cl.dead, cl.dead_count, static_cast<uint8_t*>(cl.k_pool),
          static_cast<uint8_t*>(cl.v_pool), cl.tags);
    else
      copy_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(
          m, cl.moves, cl.move_count, cl.dead, cl.dead_count, static_cast<uint8_t*>(cl.k_pool),
          static_cast<uint8_t*>(cl.v_pool), cl.tags);
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
    free_kernel<<<(unsigned)(m.nseq + 1), 256, 0, stream>>>(m, cl.new_rows, cl.freed, cl.block_table_mut,
                                                            cl.nblocks, cl.free_ids, cl.free_top,
                                                            cl.capacity, cl.status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
  }
  return cudaSuccess;
}

}  // namespace kvc
