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
//   2. four radix passes over the fp32 bit patterns (non-negative values
//      order like their bit patterns), 8 bits each, each a mass histogram
//      (warp-private bins, the 64-bit mass added as four 16-bit parts with
//      32-bit shared atomics),
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
constexpr int kU = 4;  // elements in flight per thread in every pass
constexpr int kBins = 256;   // 8-bit radix digits, four passes
constexpr int kParts = 4;    // 16-bit parts of a fixed-point mass (< 2^64)
constexpr size_t kLrfuSmem = (size_t)(kLrfuThreads / 32) * kParts * kBins * sizeof(uint32_t);
constexpr int kFixBits = 40;  // action mass in units of 2^-40

// floor(a * 2^40) for a finite a >= 0, from the float's exponent and mantissa
// with integer shifts (no floating-point conversion: this runs on every
// element of every pass).  a <= 4096 keeps the result below 2^53.
__device__ __forceinline__ unsigned long long fix_mass(float a) {
  const uint32_t bits = __float_as_uint(a);
  const int e = (int)((bits >> 23) & 0xFFu);
  if (e == 0) return 0ull;  // zero and subnormals: below 2^-126
  const unsigned long long m = (unsigned long long)((bits & 0x7FFFFFu) | 0x800000u);
  const int sh = e - 127 - 23 + kFixBits;  // a = m * 2^(e - 150)
  if (sh >= 0) return m << sh;
  return (-sh >= 64) ? 0ull : (m >> (-sh));
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
  constexpr int kWarps = kLrfuThreads / 32;
  // warp-private mass histograms: four 16-bit parts of each element's fixed-point
  // mass, each added with a 32-bit shared atomic into its own bin (a warp sees at
  // most 2^16 elements per pass, so no part sum overflows)
  extern __shared__ uint32_t whist_raw[];
  uint32_t(*whist)[kParts][kBins] = reinterpret_cast<uint32_t(*)[kParts][kBins]>(whist_raw);
  __shared__ unsigned long long hist[kBins];
  __shared__ unsigned long long sh_total, sh_need;
  __shared__ uint32_t sh_prefix, sh_mask;
  __shared__ int sh_any;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  for (int base = threadIdx.x; base < n; base += kU * kLrfuThreads) {
    float v[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int j = base + k * kLrfuThreads;
      v[k] = j < n ? __ldg(au + j) : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < kU; ++k) mine += fix_mass(fmaxf(v[k], 0.0f));
  }
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_down_sync(0xffffffffu, mine, o);
  if (lane == 0) atomicAdd(&sh_total, mine);
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

  // 2. radix passes over the fp32 bit patterns, 8 bits at a time from the top
  if (sh_any) {
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int k = lane; k < kParts * kBins; k += 32) (&whist[warp][0][0])[k] = 0;
      __syncwarp();
      const uint32_t prefix = sh_prefix, mask = sh_mask;
      // warp-uniform trip count; kU coalesced loads in flight per thread
      for (int base = warp * 32 * kU; base < n; base += kLrfuThreads * kU) {
        float vk[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int j = base + k * 32 + lane;
          vk[k] = j < n ? fmaxf(__ldg(au + j), 0.0f) : -1.0f;  // -1: past the end
        }
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const uint32_t bits = __float_as_uint(vk[k]);
          const bool in = vk[k] >= 0.0f && (bits & mask) == prefix;
          const unsigned digit = in ? ((bits >> shift) & (kBins - 1)) : (unsigned)kBins;
          if (in) {
            const unsigned long long fm = fix_mass(vk[k]);
#pragma unroll
            for (int q = 0; q < kParts; ++q) {
              const uint32_t part = (uint32_t)((fm >> (16 * q)) & 0xFFFFu);
              if (part) atomicAdd(&whist[warp][q][digit], part);
            }
          }
        }
      }
      __syncthreads();
      for (int k = threadIdx.x; k < kBins; k += blockDim.x) {
        unsigned long long t = 0;
        for (int w = 0; w < kWarps; ++w)
#pragma unroll
          for (int q = 0; q < kParts; ++q) t += (unsigned long long)whist[w][q][k] << (16 * q);
        hist[k] = t;
      }
      __syncthreads();
      if (warp == 0) {
        unsigned long long above = 0;
        const int d = pick_digit(hist, kBins, sh_need, &above);
        if (lane == 0) {
          sh_need -= above;
          sh_prefix = prefix | ((uint32_t)d << shift);
          sh_mask = mask | ((uint32_t)(kBins - 1) << shift);
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
  for (int base = threadIdx.x; base < n; base += kU * kLrfuThreads) {
    float av[kU], old[kU];
    int64_t e[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k) {  // loads of kU positions first
      const int j = base + k * kLrfuThreads;
      e[k] = -1;
      av[k] = 0.0f;
      old[k] = 0.0f;
      if (j < n) {
        av[k] = __ldg(au + j);
        const int slot = s.s0 + j;
        const int32_t page = __ldg(bt + (slot >> lp));
        if (page < 0 || page >= meta.num_pages) {
          atomicOr(status, KVC_DEV_BAD_PAGE);
        } else {
          e[k] = lbase + (int64_t)page * HP + (slot & (P - 1));
          old[k] = crf_pool[e[k]];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int j = base + k * kLrfuThreads;
      if (j >= n) continue;
      const bool hit = any && __float_as_uint(fmaxf(av[k], 0.0f)) >= tau;
      float v = 0.0f;
      if (e[k] >= 0) {
        v = fmaf(decay, old[k], hit ? 1.0f : 0.0f);
        crf_pool[e[k]] = v;
      }
      co[j] = v;
      if (ho) ho[j] = hit ? 1 : 0;
    }
  }
}

}  // namespace

cudaError_t launch_lrfu(const LrfuLaunch& ll, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 != cudaSuccess) return e0;
  if (dev >= 64 || !attr_set[dev]) {
    e0 = cudaFuncSetAttribute(lrfu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLrfuSmem);
    if (e0 != cudaSuccess) return e0;
    if (dev < 64) attr_set[dev] = true;
  }
  for (size_t c = 0; c < ll.chunks; ++c) {
    const LaunchMeta& m = ll.meta[c];
    if (m.items <= 0) continue;
    lrfu_kernel<<<(unsigned)m.items, kLrfuThreads, kLrfuSmem, stream>>>(m, ll.block_table, ll.attn, ll.crf_pool,
                                                                ll.crf_out, ll.hits, ll.frac, ll.decay,
                                                                ll.status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
  }
  return cudaSuccess;
}

}  // namespace kvc
