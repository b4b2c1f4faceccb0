// select.cu -- top-m position selection per (layer, KV head, sequence).
//
// Token eviction keeps the m positions with the highest score s_j and drops
// the rest ("Practical Online KV Cache Compaction for LLM Agents", design-space
// section).  Equal scores go to the lower position; the kept positions are
// written in ascending order (the order the slot plan consumes them).
//
// A thread-block cluster of CS 512-thread CTAs per unit (CS > 1 only when the
// units are too few to fill the GPU and long enough to split, up to 8); CTA r
// of the cluster owns the r-th contiguous slice of the unit's positions.  Scores are >= 0, so their fp32
// bit patterns order like the values.  Three radix passes over the bits (11,
// 11, 10 from the top) find the exact bit pattern T of the m-th largest score
// and how many elements equal to T are kept (k_eq); each pass counts into
// warp-private histograms with plain shared atomics (scores bunch into few
// bins, and per-warp bins keep those updates from queueing across the block),
// then every CTA adds up the cluster's histograms through distributed shared
// memory and picks the same digit.  The same histograms give each CTA how many
// of its elements are > T and == T, so a CTA's ranks start after its
// lower-ranked peers' counts.  A final pass keeps every element > T and the
// first k_eq elements == T (in position order across the cluster), and writes
// each kept position at its rank (warp ballots + a block scan of the warp
// counts).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

constexpr int kSelThreads = 512;
constexpr int kWarps = kSelThreads / 32;
constexpr int kU = 8;                         // elements per thread per tile
constexpr int kTileElems = kSelThreads * kU;  // element e of a tile: q * kSelThreads + tid
constexpr int kV = 4;                         // 16-byte loads per thread in flight (counting passes)
constexpr int kBins = 2048;
// warp-private count histograms: two 16-bit bin counts per 32-bit word (a warp
// sees at most 2^16 - 1 elements of a unit per pass for n < 2^20)
constexpr int kWarpWords = kBins / 2;
constexpr size_t kSelSmem = (size_t)kWarps * kWarpWords * sizeof(uint32_t);
constexpr int kSelSlice = 16384;  // fewest positions per CTA of a cluster

// Element i of a tile sits at tile + q * kSelThreads + tid, so every load
// instruction is coalesced and the (q, warp, lane) order is the index order
// used for ranks.
template <int CS>
__global__ void __cluster_dims__(CS, 1, 1) __launch_bounds__(kSelThreads)
    select_topm_kernel(const __grid_constant__ LaunchMeta meta, const float* __restrict__ scores,
                       int32_t* __restrict__ keep) {
  namespace cg = cooperative_groups;
  __shared__ uint32_t hist[kBins];   // this CTA's counts (read by the peers)
  __shared__ uint32_t ghist[kBins];  // the cluster's counts
  extern __shared__ uint32_t whist[];  // [kWarps][kWarpWords]
  __shared__ uint32_t pre_gt[kU * kWarps], pre_eq[kU * kWarps];
  __shared__ uint32_t sh_digit, sh_k, sh_tot_gt, sh_tot_eq, sh_above;
  __shared__ uint32_t sh_cnt[2];     // this CTA's elements > T and == T (read by the peers)
  __shared__ uint32_t wsum[kWarps];  // per-warp totals of the digit search's scan

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = CS > 1 ? (int)cg::this_cluster().block_rank() : 0;
  const int64_t item = blockIdx.x / CS;
  const int si = find_seq(meta, item);
  const SeqMeta& s = meta.seq[si];
  const int64_t local = item - s.item0;
  const int h = (int)(local % meta.H);
  const int l = (int)(local / meta.H);
  const int n = s.n, m = s.m;
  const int chunk = (n + CS - 1) / CS;
  const int lo = min(n, rank * chunk), hi = min(n, lo + chunk);
  const uint32_t* key =
      reinterpret_cast<const uint32_t*>(scores + ((int64_t)l * meta.H + h) * meta.Ntot + s.off);
  int32_t* out = keep + ((int64_t)l * meta.H + h) * meta.Mtot + s.moff;
  if (m <= 0) return;  // (the same for every CTA of the cluster)
  if (m >= n) {
    for (int i = lo + tid; i < hi; i += kSelThreads) out[i] = i;
    return;
  }

  // ---- radix select of the m-th largest bit pattern (11, 11, 10 bits)
  uint32_t prefix = 0, pmask = 0, k = (uint32_t)m, my_gt = 0, my_eq = 0;
  bool crowded = false;  // the previous pass's chosen bin held over a quarter of this slice
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int width = pass == 2 ? 10 : 11;
    const uint32_t dmask = (1u << width) - 1u;
    const int nbins = 1 << width;
    uint32_t* wh = whist + warp * kWarpWords;
    for (int i = lane; i < kWarpWords / 4; i += 32) reinterpret_cast<uint4*>(wh)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    // counting ignores order: 16-byte loads over the aligned body (kV in flight per
    // thread), single elements over the unaligned head and tail
    auto count = [&](uint32_t x) {
      if ((x & pmask) == prefix) {
        const uint32_t d = (x >> sh) & dmask;
        atomicAdd(&wh[d >> 1], (d & 1u) ? 0x10000u : 1u);
      }
    };
    const int lo_al = min(hi, lo + (int)((4u - (uint32_t)((reinterpret_cast<uintptr_t>(key + lo) >> 2) & 3u)) & 3u));
    const int hi_al = lo_al + ((hi - lo_al) & ~3);
    if (lo + tid < lo_al) count(__ldg(key + lo + tid));
    if (hi_al + tid < hi) count(__ldg(key + hi_al + tid));
    const uint4* kv = reinterpret_cast<const uint4*>(key + lo_al);
    const int nv = (hi_al - lo_al) >> 2;
#pragma unroll 1
    for (int v0 = 0; v0 < nv; v0 += kSelThreads * kV) {
      uint4 u[kV];
#pragma unroll
      for (int q = 0; q < kV; ++q) {
        const int v = v0 + q * kSelThreads + tid;
        u[q] = (v < nv) ? __ldg(kv + v) : make_uint4(0u, 0u, 0u, 0u);
      }
      if (crowded) {
        // most of the filtered elements share few digits (e.g. scores with a handful of
        // values): one atomic adds the lanes that share the first hitting lane's digit
        auto count_shared = [&](uint32_t x, bool ok) {
          const bool hit = ok && (x & pmask) == prefix;
          const uint32_t d = (x >> sh) & dmask;
          const unsigned hits = __ballot_sync(0xffffffffu, hit);
          if (hits == 0u) return;
          const int src = __ffs(hits) - 1;
          const uint32_t dl = __shfl_sync(0xffffffffu, d, src);
          const unsigned same = __ballot_sync(0xffffffffu, hit && d == dl);
          if (lane == src) atomicAdd(&wh[dl >> 1], (uint32_t)__popc(same) << ((dl & 1u) * 16));
          if (hit && d != dl) atomicAdd(&wh[d >> 1], (d & 1u) ? 0x10000u : 1u);
        };
#pragma unroll
        for (int q = 0; q < kV; ++q) {
          const bool ok = v0 + q * kSelThreads + tid < nv;
          count_shared(u[q].x, ok);
          count_shared(u[q].y, ok);
          count_shared(u[q].z, ok);
          count_shared(u[q].w, ok);
        }
      } else {
#pragma unroll
        for (int q = 0; q < kV; ++q) {
          if (v0 + q * kSelThreads + tid < nv) {
            count(u[q].x);
            count(u[q].y);
            count(u[q].z);
            count(u[q].w);
          }
        }
      }
    }
    __syncthreads();
    // thread t owns the bpt bins (hi_b - bpt, hi_b], counted from the top: it merges
    // them (over the warps, then over the cluster), and a block scan of the owners'
    // sums in thread order finds the digit where the count from the top reaches k
    const int bpt = nbins / kSelThreads;
    const int hi_b = nbins - 1 - tid * bpt;
    uint32_t own[kBins / kSelThreads];
#pragma unroll
    for (int j = 0; j < kBins / kSelThreads; ++j) {
      own[j] = 0;
      if (j < bpt) {
        const int b = hi_b - j;
#pragma unroll 4
        for (int w = 0; w < kWarps; ++w) own[j] += (whist[w * kWarpWords + (b >> 1)] >> ((b & 1) * 16)) & 0xFFFFu;
        hist[b] = own[j];
      }
    }
    if constexpr (CS > 1) {
      cg::this_cluster().sync();  // every CTA's counts are in place
#pragma unroll
      for (int j = 0; j < kBins / kSelThreads; ++j) {
        if (j < bpt) {
          uint32_t c = 0;
#pragma unroll
          for (int r = 0; r < CS; ++r) c += cg::this_cluster().map_shared_rank(hist, r)[hi_b - j];
          ghist[hi_b - j] = c;
          own[j] = c;
        }
      }
    }
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < kBins / kSelThreads; ++j) sum += own[j];
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();  // also: every bin of hist (and ghist) is in place
    uint32_t excl = incl - sum;
    for (int w = 0; w < warp; ++w) excl += wsum[w];
    if (excl < k && excl + sum >= k) {
      uint32_t acc = excl;
#pragma unroll
      for (int j = 0; j < kBins / kSelThreads; ++j) {
        if (j < bpt && acc < k) {
          if (acc + own[j] >= k) {
            sh_digit = (uint32_t)(hi_b - j);
            sh_k = k - acc;
          }
          acc += own[j];
        }
      }
    }
    __syncthreads();
    const uint32_t digit = sh_digit;
    crowded = 4u * hist[digit] > (uint32_t)(hi - lo);  // block-uniform: every thread reads the same count
    if constexpr (CS > 1) {
      // this CTA's elements above the chosen digit are > T; at the last digit, == T
      uint32_t above = 0;
      for (int b = (int)digit + 1 + tid; b < nbins; b += kSelThreads) above += hist[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
      if (tid == 0) sh_above = 0;
      __syncthreads();
      if (lane == 0 && above) atomicAdd(&sh_above, above);
      __syncthreads();
      my_gt += sh_above;
      if (pass == 2) my_eq = hist[digit];
      cg::this_cluster().sync();  // no CTA rewrites its counts while a peer reads them
    }
    prefix |= digit << sh;
    pmask |= dmask << sh;
    k = sh_k;
    __syncthreads();
  }
  const uint32_t T = prefix;   // bit pattern of the m-th largest score
  const uint32_t k_eq = k;     // elements equal to T that are kept (lowest positions first)

  // ---- order-preserving compaction: rank = #(> T before) + min(#(== T before), k_eq)
  uint32_t base_gt = 0, base_eq = 0;
  if constexpr (CS > 1) {
    if (tid == 0) {
      sh_cnt[0] = my_gt;
      sh_cnt[1] = my_eq;
    }
    cg::this_cluster().sync();
    for (int r = 0; r < rank; ++r) {
      const uint32_t* pc = cg::this_cluster().map_shared_rank(sh_cnt, r);
      base_gt += pc[0];
      base_eq += pc[1];
    }
    cg::this_cluster().sync();  // peers may exit once every CTA has read their counts
  }
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll 1
  for (int tile = lo; tile < hi; tile += kTileElems) {
    uint32_t u[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int i = tile + q * kSelThreads + tid;
      u[q] = (i < hi) ? __ldg(key + i) : 0u;
    }
    unsigned bg[kU], be[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int i = tile + q * kSelThreads + tid;
      bg[q] = __ballot_sync(0xffffffffu, i < hi && u[q] > T);
      be[q] = __ballot_sync(0xffffffffu, i < hi && u[q] == T);
      if (lane == 0) {
        pre_gt[q * kWarps + warp] = __popc(bg[q]);
        pre_eq[q * kWarps + warp] = __popc(be[q]);
      }
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scan of the kU * kWarps counts in (q, warp) order
      constexpr int per = kU * kWarps / 32;
      uint32_t g[per], e[per], sg = 0, se = 0;
#pragma unroll
      for (int j = 0; j < per; ++j) {
        g[j] = pre_gt[lane * per + j];
        e[j] = pre_eq[lane * per + j];
        sg += g[j];
        se += e[j];
      }
      uint32_t ig = sg, ie = se;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t tg = __shfl_up_sync(0xffffffffu, ig, o);
        const uint32_t te = __shfl_up_sync(0xffffffffu, ie, o);
        if (lane >= o) { ig += tg; ie += te; }
      }
      uint32_t rg = ig - sg, re = ie - se;
#pragma unroll
      for (int j = 0; j < per; ++j) {
        pre_gt[lane * per + j] = rg;
        pre_eq[lane * per + j] = re;
        rg += g[j];
        re += e[j];
      }
      if (lane == 31) { sh_tot_gt = ig; sh_tot_eq = ie; }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int i = tile + q * kSelThreads + tid;
      const uint32_t gt_before = base_gt + pre_gt[q * kWarps + warp] + __popc(bg[q] & lt_mask);
      const uint32_t eq_before = base_eq + pre_eq[q * kWarps + warp] + __popc(be[q] & lt_mask);
      const bool gt = (bg[q] >> lane) & 1u, eq = (be[q] >> lane) & 1u;
      const uint32_t rnk = gt_before + min(eq_before, k_eq);
      if ((gt || (eq && eq_before < k_eq)) && rnk < (uint32_t)m) out[rnk] = i;
    }
    base_gt += sh_tot_gt;
    base_eq += sh_tot_eq;
    __syncthreads();
  }
}

}  // namespace

// Units of at most kSmallSel positions: one CTA sorts the unit whole in shared
// memory.  Key of position i: its score's bit pattern above (2^32 - 1 - i), so
// that a descending sort puts higher scores first and, among equal scores,
// lower positions first (scores are >= 0: their bit patterns order like the
// values).  A bitonic network over the keys padded with zeros (below every
// real key) to a power of two, then the first m keys mark their positions and
// a block scan writes the marked positions in ascending order.  The result is
// the radix path's exactly: the same total order, without its per-pass
// histogram clearing and merging, which dominates on short units.  Measured
// (one select call, 20 in a row): 512 positions 20.3 -> 16.1 us; at 1536 the
// network's 66 barrier-separated stages cost more than the radix passes
// (21.3 -> 23.2 us), hence the limit.
constexpr int kSmallSel = 1024;
constexpr int kSmallPer = kSmallSel / kSelThreads;  // positions per thread in the final scan

__global__ void __launch_bounds__(kSelThreads)
    select_small_kernel(const __grid_constant__ LaunchMeta meta, const float* __restrict__ scores,
                        int32_t* __restrict__ keep) {
  __shared__ unsigned long long sk[kSmallSel];
  __shared__ uint8_t mark[kSmallSel];
  __shared__ uint32_t warp_tot[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t item = blockIdx.x;
  const int si = find_seq(meta, item);
  const SeqMeta& s = meta.seq[si];
  const int64_t local = item - s.item0;
  const int h = (int)(local % meta.H);
  const int l = (int)(local / meta.H);
  const int n = s.n, m = s.m;
  const uint32_t* key =
      reinterpret_cast<const uint32_t*>(scores + ((int64_t)l * meta.H + h) * meta.Ntot + s.off);
  int32_t* out = keep + ((int64_t)l * meta.H + h) * meta.Mtot + s.moff;
  if (m <= 0) return;
  if (m >= n) {
    for (int i = tid; i < n; i += kSelThreads) out[i] = i;
    return;
  }
  int n2 = 2;
  while (n2 < n) n2 <<= 1;
  for (int i = tid; i < n2; i += kSelThreads)
    sk[i] = i < n ? ((unsigned long long)__ldg(key + i) << 32) | (0xFFFFFFFFu - (uint32_t)i) : 0ull;
  for (int i = tid; i < kSmallSel; i += kSelThreads) mark[i] = 0;  // the final scan reads all of it
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      // pair q compares positions i (bit j clear: q with a zero bit inserted at j) and i + j
      for (int q = tid; q < (n2 >> 1); q += kSelThreads) {
        const int i = ((q & ~(j - 1)) << 1) | (q & (j - 1));
        const unsigned long long a = sk[i], b = sk[i + j];
        if (((i & k) == 0) ? (a < b) : (a > b)) {  // descending runs where bit k of i is clear
          sk[i] = b;
          sk[i + j] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int r = tid; r < m; r += kSelThreads) mark[0xFFFFFFFFu - (uint32_t)sk[r]] = 1;
  __syncthreads();
  // ascending output: thread t owns positions [t * kSmallPer, (t + 1) * kSmallPer)
  const int p0 = tid * kSmallPer;
  uint32_t cnt = 0;
#pragma unroll
  for (int e = 0; e < kSmallPer; ++e) cnt += mark[p0 + e];
  uint32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  uint32_t base = incl - cnt;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
#pragma unroll
  for (int e = 0; e < kSmallPer; ++e)
    if (mark[p0 + e]) out[base++] = p0 + e;
}

cudaError_t launch_select(const SelectLaunch& sl, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 != cudaSuccess) return e0;
  if (dev >= 64 || !attr_set[dev]) {
    for (const void* k : {reinterpret_cast<const void*>(select_topm_kernel<1>),
                          reinterpret_cast<const void*>(select_topm_kernel<2>),
                          reinterpret_cast<const void*>(select_topm_kernel<4>),
                          reinterpret_cast<const void*>(select_topm_kernel<8>)}) {
      e0 = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSelSmem);
      if (e0 != cudaSuccess) return e0;
    }
    if (dev < 64) attr_set[dev] = true;
  }
  for (size_t c = 0; c < sl.chunks; ++c) {
    const LaunchMeta& m = sl.meta[c];
    if (m.items <= 0) continue;
    // CTAs per unit: a cluster only when the units are too few to fill the GPU twice
    // over (each CTA pays a fixed histogram cost per pass), with at least kSelSlice
    // positions per CTA, at most 8 (a portable cluster)
    int max_n = 0;
    for (int i = 0; i < m.nseq; ++i) max_n = max(max_n, m.seq[i].n);
    if (max_n <= kSmallSel) {  // short units: sorted whole, one CTA each
      select_small_kernel<<<(unsigned)m.items, kSelThreads, 0, stream>>>(m, sl.scores, sl.keep);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      count_launch();
      continue;
    }
    const int by_size = (max_n + kSelSlice - 1) / kSelSlice;
    const int by_fill = (int)std::max<int64_t>(1, (2 * (int64_t)sl.num_sms) / std::max<int64_t>(1, m.items));
    const int want = min(by_size, by_fill);
    const int cs = want >= 8 ? 8 : (want >= 4 ? 4 : (want >= 2 ? 2 : 1));
    const unsigned grid = (unsigned)(m.items * cs);
    if (cs == 8)
      select_topm_kernel<8><<<grid, kSelThreads, kSelSmem, stream>>>(m, sl.scores, sl.keep);
    else if (cs == 4)
      select_topm_kernel<4><<<grid, kSelThreads, kSelSmem, stream>>>(m, sl.scores, sl.keep);
    else if (cs == 2)
      select_topm_kernel<2><<<grid, kSelThreads, kSelSmem, stream>>>(m, sl.scores, sl.keep);
    else
      select_topm_kernel<1><<<grid, kSelThreads, kSelSmem, stream>>>(m, sl.scores, sl.keep);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
  }
  return cudaSuccess;
}

}  // namespace kvc
