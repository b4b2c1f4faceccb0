// actkv.cu -- ActKV's eviction score: action-critical entries smoothed by LRFU.
//
// "ActKV 解剖" (zhichai.net analysis of ActKV), first component: for every KV
// entry the attention of all action tokens is gathered (kvc_score_action);
// entries within the top 90% count as action-critical; LRFU, the page-cache
// policy that scores entries by recency and frequency, takes "hit by action
// attention" as its reference signal, with decay lambda = 0.5.
//
// One block per unit (layer, KV head, sequence):
//   1. total action mass T of the segment, in 2^-40 fixed point (64-bit
//      integers: exact, order-independent sums, so the result does not
//      depend on thread scheduling);
//   2. three radix passes over the fp32 bit patterns (non-negative values
//      order like their bit patterns), 11/11/10 bits, each a mass histogram,
//      find the largest value tau with mass(a >= tau) >= ceil(frac * T):
//      the action-critical entries are those with a >= tau (boundary ties
//      included; nothing when T = 0 or frac = 0);
//   3. every slot of the segment: crf <- 2^-lambda crf + hit, in the per-slot
//      state (cache->aux) and in the eviction score row.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace kvc {

namespace {

constexpr int kLrfuThreads = 512;
constexpr double kFix = 1099511627776.0;  // 2^40: fixed-point scale of the action mass

__device__ __forceinline__ unsigned long long fix_mass(float a) {
  return (unsigned long long)((double)a * kFix);
}

// Largest digit d (scanning from the top) whose bins d..top hold >= need; returns
// d and writes the mass of the bins above d.  One warp; `hist` in shared memory.
__device__ int pick_digit(const unsigned long long* hist, int nbins, unsigned long long need,
                          unsigned long long* above) {
  const int lane = threadIdx.x & 31;
  const int per = nbins / 32;
  // lane 0 holds the top bins
  const int hi = nbins - 1 - lane * per;
  unsigned long long mine = 0;
  for (int k = 0; k < per; ++k) mine += hist[hi - k];
  unsigned long long incl = mine;  // inclusive prefix from the top
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const unsigned ballot = __ballot_sync(0xffffffffu, incl >= need);
  int digit = 0;
  unsigned long long ab = 0;
  if (ballot != 0) {
    const int src = __ffs(ballot) - 1;
    unsigned long long before = __shfl_sync(0xffffffffu, incl - mine, src);
    if (lane == src) {
      const int top = nbins - 1 - src * per;
      for (int k = 0; k < per; ++k) {
        const unsigned long long h = hist[top - k];
        if (before + h >= need) {
          digit = top - k;
          break;
        }
        before += h;
      }
      ab = before;
    }
    digit = __shfl_sync(0xffffffffu, digit, src);
    ab = __shfl_sync(0xffffffffu, ab, src);
  }
  *above = ab;
  return digit;
}

__global__ void __launch_bounds__(kLrfuThreads)
    lrfu_kernel(const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ block_table,
                const float* __restrict__ attn, float* __restrict__ crf_pool, float* __restrict__ crf_out,
                uint8_t* __restrict__ hits_out, float frac, float decay, unsigned* status) {
  __shared__ unsigned long long hist[2048];
  __shared__ unsigned long long sh_total, sh_need;
  __shared__ uint32_t sh_prefix, sh_mask;
  __shared__ int sh_any;
  const int64_t item = blockIdx.x;
  const SeqMeta& s = meta.seq[find_seq(meta, item)];
  const int64_t lh = item - s.item0;
  const int h = (int)(lh % meta.H), l = (int)(lh / meta.H);
  const float* au = attn + lh * meta.Ntot + s.off;
  const int n = s.n;

  // 1. total mass
  if (threadIdx.x == 0) sh_total = 0;
  __syncthreads();
  unsigned long long mine = 0;
  for (int j = threadIdx.x; j < n; j += blockDim.x) mine += fix_mass(fmaxf(au[j], 0.0f));
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_down_sync(0xffffffffu, mine, o);
  if ((threadIdx.x & 31) == 0) atomicAdd(&sh_total, mine);
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long T = sh_total;
    sh_any = (T > 0 && frac > 0.0f) ? 1 : 0;
    sh_need = (unsigned long long)ceil((double)T * (double)frac);
    if (sh_need == 0) sh_need = 1;
    sh_prefix = 0;
    sh_mask = 0;
  }
  __syncthreads();

  // 2. radix passes: 11, 11, 10 bits from the top
  if (sh_any) {
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
      const int nb = 1 << widths[pass];
      for (int k = threadIdx.x; k < nb; k += blockDim.x) hist[k] = 0;
      __syncthreads();
      const uint32_t prefix = sh_prefix, mask = sh_mask;
      for (int j = threadIdx.x; j < n; j += blockDim.x) {
        const float v = fmaxf(au[j], 0.0f);
        const uint32_t bits = __float_as_uint(v);
        if ((bits & mask) == prefix)
          atomicAdd(&hist[(bits >> shifts[pass]) & (nb - 1)], fix_mass(v));
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        unsigned long long above = 0;
        const int d = pick_digit(hist, nb, sh_need, &above);
        if (threadIdx.x == 0) {
          sh_need -= above;
          sh_prefix = prefix | ((uint32_t)d << shifts[pass]);
          sh_mask = mask | ((uint32_t)(nb - 1) << shifts[pass]);
        }
      }
      __syncthreads();
    }
  }
  const bool any = sh_any != 0;
  const uint32_t tau = sh_prefix;

  // 3. LRFU step on every slot of the segment
  const int P = meta.P, lp = meta.log2P;
  const int32_t* bt = block_table + (int64_t)s.b * meta.max_blocks;
  const int64_t HP = (int64_t)meta.H * P;
  const int64_t lbase = (int64_t)l * meta.num_pages * HP + (int64_t)h * P;
  float* co = crf_out + lh * meta.Ntot + s.off;
  uint8_t* ho = hits_out ? hits_out + lh * meta.Ntot + s.off : nullptr;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const bool hit = any && __float_as_uint(fmaxf(au[j], 0.0f)) >= tau;
    const int slot = s.s0 + j;
    const int32_t page = __ldg(bt + (slot >> lp));
    float v = 0.0f;
    if (page < 0 || page >= meta.num_pages) {
      atomicOr(status, KVC_DEV_BAD_PAGE);
    } else {
      const int64_t e = lbase + (int64_t)page * HP + (slot & (P - 1));
      v = fmaf(decay, crf_pool[e], hit ? 1.0f : 0.0f);
      crf_pool[e] = v;
    }
    co[j] = v;
    if (ho) ho[j] = hit ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_lrfu(const LrfuLaunch& ll, cudaStream_t stream) {
  for (size_t c = 0; c < ll.chunks; ++c) {
    const LaunchMeta& m = ll.meta[c];
    if (m.items <= 0) continue;
    lrfu_kernel<<<(unsigned)m.items, kLrfuThreads, 0, stream>>>(m, ll.block_table, ll.attn, ll.crf_pool,
                                                                ll.crf_out, ll.hits, ll.frac, ll.decay,
                                                                ll.status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
  }
  return cudaSuccess;
}

}  // namespace kvc
