// score.cu -- two-pass proxy-query attention-mass scoring on tcgen05 tensor cores.
//
// What it computes (token-eviction score of "Practical Online KV Cache
// Compaction for LLM Agents", design-space section; LSE recovery of the ActKV
// analysis page, system-engineering paragraph), per unit (sequence b, layer l,
// KV head h) with proxy rows q_i (i < R) and segment keys k_j (j < n):
//   LSE_i = log sum_j exp(scale q_i.k_j)
//   s_j   = sqrt((1/R) sum_i exp(2 (scale q_i.k_j - LSE_i)))
//
// Pass 1 (lse_pass):   D[128 rows x 128 keys] = Q_tile * K_tile^T per job; the
//                      epilogue keeps an online (max, sum) per row in the log2
//                      domain; each item (unit, row tile, key split) writes one
//                      partial per row.
// Combine (lse_combine): merges the partials of a row into
//                      o_i = 2 log2(sum_j 2^(c q_i.k_j)) - kBias  (c = scale*log2 e).
// Pass 2 (alpha_pass): D[128 keys x W rows] = K_tile * Q_chunk^T per job; every
//                      TMEM lane is one key, so sum_i 2^(2c L_ij - o_i) is a
//                      per-thread running sum; s_j = sqrt(sum / R) * 2^(-kBias/2).
//
// Both passes are persistent kernels (one CTA per SM) with the same roles:
//   warp 0      TMA producer (one elected lane): paged K tiles, Q tiles
//   warp 1      TMEM allocator + MMA issuer (one lane)
//   warps 2..5  epilogue: tcgen05.ld from TMEM, exponentials, reductions
// K tiles are gathered page by page through the block table (one 2-D TMA box
// of P rows x 64 columns per page and 128-byte k-block) straight into the
// 128-byte-swizzled K-major layout the MMA descriptors read.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int kTile = 128;          // keys per K tile, rows per Q tile
constexpr float kBias = 100.0f;     // alpha^2 is accumulated as alpha^2 * 2^kBias
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kEpiWarp0 = 2;        // first epilogue warp
constexpr int kThreads = 192;       // 6 warps

template <int D>
struct Cfg {
  static constexpr int KB = D / 64;                   // 128-byte k-blocks per row
  static constexpr int kTileBytes = kTile * D * 2;    // one 128-row operand tile
  static constexpr int kKbBytes = kTile * 128;        // one k-block of a 128-row tile
  // pass 1
  static constexpr int kP1QStages = 2;
  static constexpr int kP1KStages = (D == 128) ? 4 : 8;
  static constexpr int kP1Bars = 2 * kP1QStages + 2 * kP1KStages + 4;
  static constexpr int kP1Smem =
      1024 + (kP1QStages + kP1KStages) * kTileBytes + kP1Bars * 8 + 16;
  // pass 2
  static constexpr int kMaxW = 256;
  static constexpr int kChunkBytes = kMaxW * D * 2;
  static constexpr int kP2KStages = 2;
  static constexpr int kP2QStages = 2;
  static constexpr int kP2Bars = 2 * kP2QStages + 2 * kP2KStages + 4;
  static constexpr int kP2Smem =
      1024 + kP2KStages * kTileBytes + kP2QStages * kChunkBytes + kP2Bars * 8 + 16;
};

struct Unit {
  int si, b, l, h;
  int s0, n;
  int64_t off;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Issues the TMA loads of key tile `kt` of a unit into `dst` (layout:
// [k-block][128 rows][128 B], 128-byte swizzle), completing on `bar`.  Pages
// past the segment end are not loaded; their rows are masked by the consumer.
template <int D>
__device__ __forceinline__ void load_key_tile(const CUtensorMap* tmK, uint8_t* dst, uint64_t* bar,
                                              const int32_t* bt_row, const Unit& u, int kt,
                                              const LaunchMeta& meta, unsigned* status) {
  const int P = meta.P;
  const int ppt = kTile / P;  // pages per tile (2..16)
  int32_t rows[16];
  uint32_t bytes = 0;
  for (int p = 0; p < ppt; ++p) {
    const int slot = kt * kTile + p * P;
    int32_t row = -1;
    if (slot < u.n) {
      const int32_t page = __ldg(bt_row + (u.s0 + slot) / P);
      if (page < 0 || page >= meta.num_pages) {
        atomicOr(status, KVC_DEV_BAD_PAGE);
      } else {
        row = ((u.l * meta.num_pages + page) * meta.H + u.h) * P;
        bytes += Cfg<D>::KB * P * 128;
      }
    }
    rows[p] = row;
  }
  mbar_arrive_expect_tx(bar, bytes);
  for (int p = 0; p < ppt; ++p) {
    if (rows[p] < 0) continue;
#pragma unroll
    for (int kb = 0; kb < Cfg<D>::KB; ++kb)
      tma_load_2d(dst + kb * Cfg<D>::kKbBytes + p * P * 128, tmK, bar, kb * 64, rows[p]);
  }
}

// ============================================================== pass 1

struct P1Item {
  Unit u;
  int rt, t0, t1;
};

__device__ __forceinline__ P1Item decode_p1(const LaunchMeta& meta, int64_t item) {
  P1Item it;
  const int si = find_seq(meta, item);
  const SeqMeta& s = meta.seq[si];
  int64_t local = item - s.item0;
  it.rt = (int)(local % meta.rowtiles);
  local /= meta.rowtiles;
  const int sp = (int)(local % s.split);
  local /= s.split;
  it.u.h = (int)(local % meta.H);
  it.u.l = (int)(local / meta.H);
  it.u.si = si;
  it.u.b = s.b;
  it.u.s0 = s.s0;
  it.u.n = s.n;
  it.u.off = s.off;
  const int T = (s.n + kTile - 1) / kTile;
  it.t0 = (int)((int64_t)sp * T / s.split);
  it.t1 = (int)((int64_t)(sp + 1) * T / s.split);
  return it;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    lse_pass_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ block_table,
                    float2* __restrict__ part, unsigned* status) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::kP1QStages * C::kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sK + C::kP1KStages * C::kTileBytes);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + C::kP1QStages;
  uint64_t* k_full = q_empty + C::kP1QStages;
  uint64_t* k_empty = k_full + C::kP1KStages;
  uint64_t* t_full = k_empty + C::kP1KStages;
  uint64_t* t_empty = t_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kP1QStages; ++i) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1); }
    for (int i = 0; i < C::kP1KStages; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&t_full[i], 1); mbar_init(&t_empty[i], 128); }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmQ);
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(tmem_slot, 256);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t qit = 0, kit = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < meta.items && ok; item += gridDim.x) {
        const P1Item it = decode_p1(meta, item);
        const int qs = qit % C::kP1QStages;
        if (!(ok = mbar_wait(&q_empty[qs], ((qit / C::kP1QStages) & 1) ^ 1, abort_flag, status))) break;
        const int qrow = ((it.u.b * meta.L + it.u.l) * meta.H + it.u.h) * meta.R + it.rt * kTile;
        mbar_arrive_expect_tx(&q_full[qs], C::KB * C::kKbBytes);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_2d(sQ + qs * C::kTileBytes + kb * C::kKbBytes, &tmQ, &q_full[qs], kb * 64, qrow);
        ++qit;
        const int32_t* bt_row = block_table + (int64_t)it.u.b * meta.max_blocks;
        for (int kt = it.t0; kt < it.t1; ++kt) {
          const int ks = kit % C::kP1KStages;
          if (!(ok = mbar_wait(&k_empty[ks], ((kit / C::kP1KStages) & 1) ^ 1, abort_flag, status))) break;
          load_key_tile<D>(&tmK, sK + ks * C::kTileBytes, &k_full[ks], bt_row, it.u, kt, meta, status);
          ++kit;
        }
      }
      if (!ok) {  // let issued copies land before the CTA exits
        for (uint32_t j = (kit > C::kP1KStages ? kit - C::kP1KStages : 0); j < kit; ++j)
          mbar_wait(&k_full[j % C::kP1KStages], (j / C::kP1KStages) & 1, nullptr, status);
        for (uint32_t j = (qit > C::kP1QStages ? qit - C::kP1QStages : 0); j < qit; ++j)
          mbar_wait(&q_full[j % C::kP1QStages], (j / C::kP1QStages) & 1, nullptr, status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTile, kTile);
      uint32_t qit = 0, kit = 0, jt = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < meta.items && ok; item += gridDim.x) {
        const P1Item it = decode_p1(meta, item);
        const int qs = qit % C::kP1QStages;
        if (!(ok = mbar_wait(&q_full[qs], (qit / C::kP1QStages) & 1, abort_flag, status))) break;
        const uint32_t a_base = smem_u32(sQ + qs * C::kTileBytes);
        for (int kt = it.t0; kt < it.t1; ++kt) {
          const int ks = kit % C::kP1KStages;
          const int tb = jt & 1;
          if (!(ok = mbar_wait(&k_full[ks], (kit / C::kP1KStages) & 1, abort_flag, status))) break;
          if (!(ok = mbar_wait(&t_empty[tb], ((jt >> 1) & 1) ^ 1, abort_flag, status))) break;
          tc_fence_after_sync();
          const uint32_t b_base = smem_u32(sK + ks * C::kTileBytes);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t koff = (k >> 2) * C::kKbBytes + (k & 3) * 32;
            mma_bf16(tmem + tb * kTile, sdesc_k_sw128(a_base + koff), sdesc_k_sw128(b_base + koff),
                     idesc, k > 0);
          }
          mma_commit(&k_empty[ks]);
          mma_commit(&t_full[tb]);
          ++kit;
          ++jt;
        }
        if (!ok) break;
        mma_commit(&q_empty[qs]);
        ++qit;
      }
      if (!ok && jt > 0)  // the last commit covers every MMA issued
        mbar_wait(&t_full[(jt - 1) & 1], ((jt - 1) >> 1) & 1, nullptr, status);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int sub = warp & 3;
    const int r = sub * 32 + lane;  // TMEM lane = Q row of the tile
    const uint32_t t_lane = tmem + ((uint32_t)(sub * 32) << 16);
    const float c = meta.scale * kLog2e;
    uint32_t jt = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < meta.items && ok; item += gridDim.x) {
      const P1Item it = decode_p1(meta, item);
      float m_run = -INFINITY, s_run = 0.0f;
      for (int kt = it.t0; kt < it.t1; ++kt) {
        const int tb = jt & 1;
        ok = mbar_wait(&t_full[tb], (jt >> 1) & 1, abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }  // warp-uniform, converged
        tc_fence_after_sync();
        float v[kTile];
#pragma unroll
        for (int q = 0; q < kTile / 32; ++q) tmem_ld32(t_lane + tb * kTile + q * 32, v + q * 32);
        tc_fence_before_sync();
        mbar_arrive(&t_empty[tb]);
        ++jt;
        const int valid = min(kTile, it.u.n - kt * kTile);
        float tmax = -INFINITY;
        if (valid == kTile) {
#pragma unroll
          for (int j = 0; j < kTile; ++j) tmax = fmaxf(tmax, v[j]);
        } else {
#pragma unroll
          for (int j = 0; j < kTile; ++j)
            if (j < valid) tmax = fmaxf(tmax, v[j]);
        }
        const float mnew = fmaxf(m_run, tmax * c);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        if (valid == kTile) {
#pragma unroll
          for (int j = 0; j < kTile; j += 4) {
            a0 += ex2_approx(fmaf(v[j + 0], c, -mnew));
            a1 += ex2_approx(fmaf(v[j + 1], c, -mnew));
            a2 += ex2_approx(fmaf(v[j + 2], c, -mnew));
            a3 += ex2_approx(fmaf(v[j + 3], c, -mnew));
          }
        } else {
#pragma unroll
          for (int j = 0; j < kTile; ++j)
            if (j < valid) a0 += ex2_approx(fmaf(v[j], c, -mnew));
        }
        s_run = fmaf(s_run, ex2_approx(m_run - mnew), (a0 + a1) + (a2 + a3));
        m_run = mnew;
      }
      if (!ok) break;
      part[item * kTile + r] = make_float2(m_run, s_run);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, 256);
  }
}

// ============================================================== combine

__global__ void lse_combine_kernel(const __grid_constant__ LaunchMeta meta,
                                   const float2* __restrict__ part, float* __restrict__ obias,
                                   float* __restrict__ lse_out) {
  const float ln2 = 0.6931471805599453f;
  for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < meta.items;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int si = find_seq(meta, g);
    const SeqMeta& s = meta.seq[si];
    int64_t local = g - s.item0;
    const int i = (int)(local % meta.R_pad);
    local /= meta.R_pad;
    const int h = (int)(local % meta.H);
    const int l = (int)(local / meta.H);
    const int64_t u = ((int64_t)s.b * meta.L + l) * meta.H + h;
    if (i >= meta.R) {
      obias[u * meta.R_pad + i] = INFINITY;  // padded rows contribute exp2(-inf) = 0
      continue;
    }
    const int rt = i / kTile, rr = i % kTile;
    const int64_t base = s.item1 + ((int64_t)(l * meta.H + h) * s.split) * meta.rowtiles + rt;
    float M = -INFINITY;
    for (int sp = 0; sp < s.split; ++sp) M = fmaxf(M, part[(base + (int64_t)sp * meta.rowtiles) * kTile + rr].x);
    float S = 0.0f;
    for (int sp = 0; sp < s.split; ++sp) {
      const float2 p = part[(base + (int64_t)sp * meta.rowtiles) * kTile + rr];
      S += p.y * exp2f(p.x - M);
    }
    const float lg = M + log2f(S);  // log2 sum_j 2^(c L_ij)
    obias[u * meta.R_pad + i] = 2.0f * lg - kBias;
    if (lse_out != nullptr) lse_out[u * meta.R + i] = lg * ln2;
  }
}

// Pass-2 offsets from a caller-supplied natural-log LSE (for instance the
// log-sum-exp the attention kernel produced for the same proxy queries).
__global__ void obias_from_lse_kernel(const __grid_constant__ LaunchMeta meta,
                                      const float* __restrict__ lse_in, float* __restrict__ obias) {
  for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < meta.items;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int si = find_seq(meta, g);
    const SeqMeta& s = meta.seq[si];
    int64_t local = g - s.item0;
    const int i = (int)(local % meta.R_pad);
    local /= meta.R_pad;
    const int h = (int)(local % meta.H);
    const int l = (int)(local / meta.H);
    const int64_t u = ((int64_t)s.b * meta.L + l) * meta.H + h;
    obias[u * meta.R_pad + i] =
        (i < meta.R) ? 2.0f * kLog2e * lse_in[u * meta.R + i] - kBias : INFINITY;
  }
}

// ============================================================== pass 2

struct P2Item {
  Unit u;
  int kt;
};

__device__ __forceinline__ P2Item decode_p2(const LaunchMeta& meta, int64_t item) {
  P2Item it;
  const int si = find_seq(meta, item);
  const SeqMeta& s = meta.seq[si];
  const int T = (s.n + kTile - 1) / kTile;
  int64_t local = item - s.item0;
  it.kt = (int)(local % T);
  local /= T;
  it.u.h = (int)(local % meta.H);
  it.u.l = (int)(local / meta.H);
  it.u.si = si;
  it.u.b = s.b;
  it.u.s0 = s.s0;
  it.u.n = s.n;
  it.u.off = s.off;
  return it;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    alpha_pass_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ LaunchMeta meta,
                      const int32_t* __restrict__ block_table, const float* __restrict__ obias,
                      float* __restrict__ scores, unsigned* status) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sK = smem;
  uint8_t* sQ = sK + C::kP2KStages * C::kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sQ + C::kP2QStages * C::kChunkBytes);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + C::kP2KStages;
  uint64_t* q_full = k_empty + C::kP2KStages;
  uint64_t* q_empty = q_full + C::kP2QStages;
  uint64_t* t_full = q_empty + C::kP2QStages;
  uint64_t* t_empty = t_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int W = meta.W;
  const int nchunks = meta.nchunks;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kP2KStages; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    for (int i = 0; i < C::kP2QStages; ++i) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&t_full[i], 1); mbar_init(&t_empty[i], 128); }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmQ);
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(tmem_slot, 512);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t kit = 0, qit = 0;
      bool ok = true;
      const uint32_t chunk_bytes = (uint32_t)(C::KB * W * 128);
      for (int64_t item = blockIdx.x; item < meta.items && ok; item += gridDim.x) {
        const P2Item it = decode_p2(meta, item);
        const int ks = kit % C::kP2KStages;
        if (!(ok = mbar_wait(&k_empty[ks], ((kit / C::kP2KStages) & 1) ^ 1, abort_flag, status))) break;
        load_key_tile<D>(&tmK, sK + ks * C::kTileBytes, &k_full[ks],
                         block_table + (int64_t)it.u.b * meta.max_blocks, it.u, it.kt, meta, status);
        ++kit;
        const int qrow0 = ((it.u.b * meta.L + it.u.l) * meta.H + it.u.h) * meta.R;
        for (int cidx = 0; cidx < nchunks; ++cidx) {
          const int qs = qit % C::kP2QStages;
          if (!(ok = mbar_wait(&q_empty[qs], ((qit / C::kP2QStages) & 1) ^ 1, abort_flag, status))) break;
          mbar_arrive_expect_tx(&q_full[qs], chunk_bytes);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_2d(sQ + qs * C::kChunkBytes + kb * W * 128, &tmQ, &q_full[qs], kb * 64,
                        qrow0 + cidx * W);
          ++qit;
        }
      }
      if (!ok) {
        for (uint32_t j = (kit > C::kP2KStages ? kit - C::kP2KStages : 0); j < kit; ++j)
          mbar_wait(&k_full[j % C::kP2KStages], (j / C::kP2KStages) & 1, nullptr, status);
        for (uint32_t j = (qit > C::kP2QStages ? qit - C::kP2QStages : 0); j < qit; ++j)
          mbar_wait(&q_full[j % C::kP2QStages], (j / C::kP2QStages) & 1, nullptr, status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTile, W);
      uint32_t kit = 0, qit = 0, jt = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < meta.items && ok; item += gridDim.x) {
        const int ks = kit % C::kP2KStages;
        if (!(ok = mbar_wait(&k_full[ks], (kit / C::kP2KStages) & 1, abort_flag, status))) break;
        const uint32_t a_base = smem_u32(sK + ks * C::kTileBytes);
        for (int cidx = 0; cidx < nchunks; ++cidx) {
          const int qs = qit % C::kP2QStages;
          const int tb = jt & 1;
          if (!(ok = mbar_wait(&q_full[qs], (qit / C::kP2QStages) & 1, abort_flag, status))) break;
          if (!(ok = mbar_wait(&t_empty[tb], ((jt >> 1) & 1) ^ 1, abort_flag, status))) break;
          tc_fence_after_sync();
          const uint32_t b_base = smem_u32(sQ + qs * C::kChunkBytes);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t aoff = (k >> 2) * C::kKbBytes + (k & 3) * 32;
            const uint32_t boff = (k >> 2) * (uint32_t)(W * 128) + (k & 3) * 32;
            mma_bf16(tmem + tb * C::kMaxW, sdesc_k_sw128(a_base + aoff),
                     sdesc_k_sw128(b_base + boff), idesc, k > 0);
          }
          mma_commit(&q_empty[qs]);
          mma_commit(&t_full[tb]);
          ++qit;
          ++jt;
        }
        if (!ok) break;
        mma_commit(&k_empty[ks]);
        ++kit;
      }
      if (!ok && jt > 0)
        mbar_wait(&t_full[(jt - 1) & 1], ((jt - 1) >> 1) & 1, nullptr, status);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int sub = warp & 3;
    const int r = sub * 32 + lane;  // TMEM lane = key of the tile
    const uint32_t t_lane = tmem + ((uint32_t)(sub * 32) << 16);
    const float c2 = 2.0f * meta.scale * kLog2e;
    const float inv_r = 1.0f / (float)meta.R;
    const float unbias = exp2f(-0.5f * kBias);
    uint32_t jt = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < meta.items && ok; item += gridDim.x) {
      const P2Item it = decode_p2(meta, item);
      const int64_t u = ((int64_t)it.u.b * meta.L + it.u.l) * meta.H + it.u.h;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      for (int cidx = 0; cidx < nchunks; ++cidx) {
        const int tb = jt & 1;
        ok = mbar_wait(&t_full[tb], (jt >> 1) & 1, abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }  // warp-uniform, converged
        tc_fence_after_sync();
        const float* ob = obias + u * meta.R_pad + cidx * W;
        for (int col0 = 0; col0 < W; col0 += 32) {
          float v[32];
          tmem_ld32(t_lane + tb * C::kMaxW + col0, v);
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 o = __ldg(reinterpret_cast<const float4*>(ob + col0 + j));
            a0 += ex2_approx(fmaf(v[j + 0], c2, -o.x));
            a1 += ex2_approx(fmaf(v[j + 1], c2, -o.y));
            a2 += ex2_approx(fmaf(v[j + 2], c2, -o.z));
            a3 += ex2_approx(fmaf(v[j + 3], c2, -o.w));
          }
        }
        tc_fence_before_sync();
        mbar_arrive(&t_empty[tb]);
        ++jt;
      }
      if (!ok) break;
      const int key = it.kt * kTile + r;
      if (key < it.u.n) {
        const float acc = (a0 + a1) + (a2 + a3);
        scores[((int64_t)it.u.l * meta.H + it.u.h) * meta.Ntot + it.u.off + key] =
            sqrtf(acc * inv_r) * unbias;
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_score_d(const ScoreLaunch& sl, cudaStream_t stream) {
  using C = Cfg<D>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(lse_pass_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kP1Smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(alpha_pass_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kP2Smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  for (size_t c = 0; c < sl.chunks; ++c) {
    if (sl.phases & kPhaseLse) {
      const LaunchMeta& m1 = sl.pass1[c];
      if (m1.items > 0) {
        const int grid = (int)std::min<int64_t>(m1.items, sl.num_sms);
        lse_pass_kernel<D><<<grid, kThreads, C::kP1Smem, stream>>>(*sl.tmK, *sl.tmQ1, m1, sl.block_table,
                                                                   sl.part, sl.status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
      }
      const LaunchMeta& mc = sl.combine[c];
      if (mc.items > 0) {
        const int grid = (int)std::min<int64_t>((mc.items + 255) / 256, (int64_t)sl.num_sms * 8);
        lse_combine_kernel<<<grid, 256, 0, stream>>>(mc, sl.part, sl.obias, sl.lse_out);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
      }
    }
    if (sl.phases & kPhaseLseIn) {
      const LaunchMeta& mc = sl.combine[c];
      if (mc.items > 0) {
        const int grid = (int)std::min<int64_t>((mc.items + 255) / 256, (int64_t)sl.num_sms * 8);
        obias_from_lse_kernel<<<grid, 256, 0, stream>>>(mc, sl.lse_in, sl.obias);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
      }
    }
    if (sl.phases & kPhaseAlpha) {
      const LaunchMeta& m2 = sl.pass2[c];
      if (m2.items > 0) {
        const int grid = (int)std::min<int64_t>(m2.items, sl.num_sms);
        alpha_pass_kernel<D><<<grid, kThreads, C::kP2Smem, stream>>>(*sl.tmK, *sl.tmQ2, m2, sl.block_table,
                                                                     sl.obias, sl.scores, sl.status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
      }
    }
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_score(const ScoreLaunch& sl, cudaStream_t stream) {
  if (sl.d == 128) return launch_score_d<128>(sl, stream);
  if (sl.d == 64) return launch_score_d<64>(sl, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvc
