// am.cu -- Attention Matching on the token-eviction survivors.
//
// Source: "Practical Online KV Cache Compaction for LLM Agents: An Empirical
// Study" (agifrontier tutorial page), section on the two compaction families:
// after the top-m keys K_C are chosen, AM fits an additive attention bias beta
// (one value per kept key) and compact values V_C so that, on the proxy
// queries Q, the compacted attention reproduces the full one:
//   min_beta || exp(Q K_C^T + beta) 1_m - exp(Q K^T) 1_n ||^2      (mass fit)
//   min_V_C  || A_hat(Q; K_C, beta, V_C) - A(Q; K, V) ||_F^2        (value fit)
//
// With w = exp(beta) >= 0 the mass fit is non-negative least squares in w.
// Both fits run as cyclic coordinate descent on their normal equations,
// starting from token eviction's own answer (w = 1, V_C = the kept values),
// T sweeps over the kept keys in ascending position order; every logit of a
// unit is shifted by c = max_i LSE_i, which changes neither minimiser.
//
// The contractions run on the tensor cores: the targets (the full attention
// output over all n keys) with bf16 Q, K and V exactly as stored and the
// probabilities split into two bf16 parts; the Gram products, which the
// ill-conditioned fits need to fp32 accuracy (a single bf16 or tf32 rounding
// would put ~1e-3 into them), with every fp32 operand split into three bf16
// parts.  The coordinate descents are fp32 on the CUDA cores.  Per unit, after
// the rows' log-sum-exp LSE_i over all n keys (the scoring LSE pass, the
// caller's or run by the entry point), the kernels run in launch order
//   am_targets_tc_kernel  Y = softmax(L) V over all n keys on the tensor cores
//                      and E = exp(L_C - c) over the kept keys, s = exp(LSE - c)
//   am_x0_kernel       X0 = the kept values (fp32)
//   am_atb_tc_kernel   G = E^T [E | s]              (mode 0, tensor cores)
//   am_mass_kernel     w by projected coordinate descent; beta = ln w
//   am_probs_kernel    Ph = rows of E diag(w), normalised (in place)
//   am_atb_tc_kernel   H = Ph^T Ph, Bm = Ph^T Y     (modes 1 and 2, one launch)
//   am_atb_tc_kernel   H X0 - Bm, the value fit's starting gradient (mode 3)
//   am_value_kernel    V_C by coordinate descent; written to the pool (bf16)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int kAmThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
// A coordinate moves only when its gradient exceeds 2^-17 of the scale of the
// gradient's own terms.  E and s come from fp32 logits (128-term fp32 dot
// products), whose relative error reaches ~2e-5 where the logits are large
// (concentrated attention); the normal equations square cond(E), up to 1e16
// there, so the gradient of a key with almost no attention is that error
// alone, and a step on it (w_j to 1e8, V_C rows to 1e9) wrecks the value fit.
// Measured on this kernel against the plain fp64 descent: at 2^-20 such units
// diverge (value residual 9e-2 of |Y| above the plain descent's); at 2^-14
// real steps of well-conditioned fits are frozen (residuals up to 2e-3 of the
// target norm above); from 2^-16 to 2^-18 both stay within 6e-6.  2^-17 keeps
// a factor of 8 from the level that diverges.
constexpr float kAmGuard = 7.62939453125e-06f;  // 2^-17

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

struct AmUnit {
  int k;        // sequence index within the launch
  int l, h;
  int b, s0, n, m, ldE;
  int64_t moff;
  float* base;  // the unit's workspace
};

__device__ __forceinline__ AmUnit am_unit(const AmMeta& meta, int64_t unit, float* ws) {
  int lo = 0, hi = meta.nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (meta.seq[mid].unit0 <= unit) lo = mid; else hi = mid - 1;
  }
  const AmSeq& q = meta.seq[lo];
  const int r = (int)(unit - q.unit0);
  AmUnit u;
  u.k = lo;
  u.l = r / meta.H;
  u.h = r % meta.H;
  u.b = q.b;
  u.s0 = q.s0;
  u.n = q.n;
  u.m = q.m;
  u.ldE = q.ldE;
  u.moff = q.moff;
  u.base = ws + q.ws + (int64_t)r * q.unit_floats;  // regions laid out for the launch's largest m
  return u;
}

// Pool row of segment position `pos` of the unit, or -1 (bad page, reported).
__device__ __forceinline__ int64_t am_row(const AmMeta& meta, const AmUnit& u, const int32_t* bt, int pos,
                                          unsigned* status) {
  const int slot = u.s0 + pos;
  const int32_t page = bt[(int64_t)u.b * meta.max_blocks + slot / meta.P];
  if (page < 0 || page >= meta.num_pages) {
    atomicOr(status, KVC_DEV_BAD_PAGE);
    return -1;
  }
  return (((int64_t)u.l * meta.num_pages + page) * meta.H + u.h) * meta.P + slot % meta.P;
}

// Kept position j of the unit, or -1 (outside the segment, reported).
__device__ __forceinline__ int am_kept(const AmMeta& meta, const AmUnit& u, const int32_t* keep, int j,
                                       unsigned* status) {
  const int pos = keep[((int64_t)u.l * meta.H + u.h) * meta.Mtot + u.moff + j];
  if (pos < 0 || pos >= u.n) {
    atomicOr(status, KVC_DEV_BAD_KEEP);
    return -1;
  }
  return pos;
}

// ------------------------------------------------------------------ targets (tensor cores)
// Block = (unit, 128 proxy rows), 352 threads:
//   warp 0      producer: the block's Q rows (two-dimensional TMA, once), then
//               the K tiles of 128 keys, page by page (four-dimensional TMA: one
//               copy per page lands as 1024-byte atoms of 8 keys x 64 head-dim
//               elements), through a ring of kTcStages whose stages free up as
//               soon as a tile's logits are formed; the block-table entries of
//               the next tile are loaded while this tile is issued
//   warp 10     producer of the V tiles the same way, through a second ring
//               whose stages free up when a tile's output MMAs are done
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer
//   warps 2..9  epilogue, two per TMEM lane quarter (32 rows), each with 64 of a
//               tile's 128 columns
// Per key tile t the issuer forms S = Q K_t^T (bf16 operands, fp32 in TMEM; two
// S buffers, so tile t+1's logits form while tile t's probabilities are made).
// The epilogue turns row i of S into p_ij = 2^(c L_ij - lse2_i) with the row's
// log-sum-exp from the scoring LSE pass, so p <= 1 and no running maximum or
// rescaling of the output is needed; it splits p into its bf16 rounding and
// the bf16 of the remainder (16 bits of mantissa together) and stores both into
// TMEM.  The issuer then accumulates Y += P_hi V_t + P_lo V_t with A read from
// TMEM and V_t as an MN-major B operand (the pool stores V key by key).  At the
// end Y = softmax(L) V and the LSE rows go to the unit's workspace.  E over the
// kept keys is formed from the same logits after P's hand-off, read back from the
// S buffer column by column (a kept key's column is the same for the whole warp).
// TMEM columns: S0 [0, 128), S1 [128, 256), P_hi [256, 320), P_lo [320, 384),
// Y [384, 384 + D).
constexpr int kTcThreads = 352;
constexpr int kTcWarpV = 10;   // the V producer
constexpr int kTcEpi = 8;      // epilogue warps
constexpr int kTcStages = 2;
constexpr int kTcRows = 128;   // proxy rows per block = MMA M
constexpr int kTcKeys = 128;   // keys per tile
constexpr int kTcHead = 1024;  // barriers, TMEM address, abort flag

template <int D>
constexpr int tc_tile_bytes() { return kTcKeys * D * 2; }
template <int D>
constexpr int tc_smem_bytes() {  // head, slack, Q rows, the K and V rings, keep list, turn-arounds
  return kTcHead + 1024 + kTcRows * D * 2 + kTcStages * 2 * tc_tile_bytes<D>() + kAmMaxM * 4 + kTcEpi * 32 * 33 * 4;
}
static_assert(tc_smem_bytes<128>() <= 227 * 1024, "targets working set fits one CTA's shared memory");


template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    am_targets_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmQ, const AmMeta meta,
                         const int32_t* __restrict__ bt, const int32_t* __restrict__ keep,
                         const float* __restrict__ lse_rows, float* ws, unsigned* status) {
  constexpr int KB = D / 64;                     // 128-byte k-blocks per row
  constexpr int kTile = tc_tile_bytes<D>();
  constexpr uint32_t kColP = 256, kColPlo = 320, kColY = 384;
  extern __shared__ __align__(16) uint8_t tc_smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(tc_smem);
  uint64_t* q_full = bars;                        // [1]
  uint64_t* k_full = bars + 1;                    // [kTcStages] K tile landed
  uint64_t* k_empty = k_full + kTcStages;         // [kTcStages] its logits are formed
  uint64_t* v_full = k_empty + kTcStages;         // [kTcStages] V tile landed
  uint64_t* v_empty = v_full + kTcStages;         // [kTcStages] its output MMAs are done
  uint64_t* s_full = v_empty + kTcStages;         // [2] S buffer formed
  uint64_t* s_empty = s_full + 2;                 // [2] S buffer read (every epilogue warp)
  uint64_t* p_full = s_empty + 2;                 // P stored (every epilogue warp)
  uint64_t* p_empty = p_full + 1;                 // P read by the output MMAs
  uint64_t* y_full = p_empty + 1;                 // all output MMAs done
  uint64_t* drain = y_full + 1;                   // abort: every MMA issued is done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tc_smem + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* sQ = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem) + kTcHead + 1023) &
                                           ~uintptr_t(1023));
  uint8_t* sK = sQ + kTcRows * D * 2;             // K ring: stage s at s * kTile
  uint8_t* sV = sK + kTcStages * kTile;           // V ring
  int32_t* sKeep = reinterpret_cast<int32_t*>(sV + kTcStages * kTile);  // the unit's kept positions
  float* sTr = reinterpret_cast<float*>(sKeep + kAmMaxM);  // [kTcEpi][32][33] turn-around
  float* red = reinterpret_cast<float*>(tc_smem + 576);  // [kTcEpi] epilogue warps' maxima of the rows' LSE

  const int rb = (meta.R + kTcRows - 1) / kTcRows;
  const AmUnit u = am_unit(meta, blockIdx.x / rb, ws);
  const int r0 = (int)(blockIdx.x % rb) * kTcRows;
  const int T = (u.n + kTcKeys - 1) / kTcKeys;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // zero the K/V ring: rows of pages past the segment are never loaded and
  // must hold finite values (their probabilities are 0)
  for (int i = threadIdx.x; i < kTcStages * 2 * kTile / 16; i += kTcThreads)
    reinterpret_cast<uint4*>(sK)[i] = make_uint4(0u, 0u, 0u, 0u);
  const int64_t lrow = (((int64_t)u.b * meta.L + u.l) * meta.H + u.h) * meta.R;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) { mbar_init(&s_full[i], 1); mbar_init(&s_empty[i], kTcEpi); }
    mbar_init(p_full, kTcEpi);
    mbar_init(p_empty, 1);
    mbar_init(y_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmQ);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the zeroed ring, for the tensor cores
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(tmem_slot, 512);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == kTcWarpV) {
    // ---------------------------------------------------------- producers
    // warp 0: the Q rows (once) and the K tiles; warp kTcWarpV: the V tiles.  A K
    // stage is free again once its logits are formed, a V stage once its output
    // MMAs are done, so K runs a tile further ahead than a shared ring allows.
    const bool is_k = warp == 0;
    uint8_t* ring = is_k ? sK : sV;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    bool ok = true;
    uint32_t issued = 0;  // tiles whose copies were issued
    if (is_k) {
      const int64_t qrow = (((int64_t)u.b * meta.L + u.l) * meta.H + u.h) * meta.R + r0;
      if (lane == 0) mbar_arrive_expect_tx(q_full, KB * kTcRows * 128);
      __syncwarp();
      if (lane < KB) tma_load_2d(sQ + lane * kTcRows * 128, &tmQ, q_full, lane * 64, (int32_t)qrow);
    }
    const int ppt = kTcKeys / meta.P;  // pages per tile (<= 16)
    const int32_t* bt_row = bt + (int64_t)u.b * meta.max_blocks;
    auto page_of = [&](int t) -> int32_t {
      const int slot = t * kTcKeys + lane * meta.P;
      if (lane >= ppt || slot >= u.n) return -1;
      const int32_t pg = __ldg(bt_row + (u.s0 + slot) / meta.P);
      if (pg < 0 || pg >= meta.num_pages) {
        if (is_k) atomicOr(status, KVC_DEV_BAD_PAGE);  // outside the pool: reported (once), not read
        return -1;
      }
      return pg;
    };
    int32_t pg_next = page_of(0);
    for (int t = 0; t < T && ok; ++t) {
      const int32_t pg = pg_next;
      if (t + 1 < T) pg_next = page_of(t + 1);
      const int st = t % kTcStages;
      if (lane == 0) ok = mbar_wait(&empty[st], ((t / kTcStages) & 1) ^ 1, abort_flag, status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const unsigned valid = __ballot_sync(0xffffffffu, pg >= 0);
      if (lane == 0) mbar_arrive_expect_tx(&full[st], __popc(valid) * KB * meta.P * 128u);
      __syncwarp();
      if (pg >= 0) {
        const int32_t prow = (int32_t)((((int64_t)u.l * meta.num_pages + pg) * meta.H + u.h) * meta.P);
        uint8_t* dst = ring + st * kTile + lane * meta.P * D * 2;
        if (is_k)
          tma_load_4d(dst, &tmK, &full[st], 0, 0, 0, prow >> 3);
        else
          tma_load_4d(dst, &tmV, &full[st], 0, 0, 0, prow >> 3);
      }
      ++issued;
    }
    // let the copies issued land before the CTA exits, whichever role gave up
    if (lane == 0) {
      if (is_k) mbar_wait(q_full, 0, nullptr, status);
      for (uint32_t t = issued > (uint32_t)kTcStages ? issued - kTcStages : 0; t < issued; ++t)
        mbar_wait(&full[t % kTcStages], (t / kTcStages) & 1, nullptr, status);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, abort_flag, status);
      bool issued = false;
      const uint32_t idesc_s = idesc_bf16_f32(kTcRows, kTcKeys);
      const uint32_t idesc_y = idesc_bf16_f32(kTcRows, D) | (1u << 16);  // B (V) MN-major
      const uint64_t q_desc = sdesc_k_sw128(smem_u32(sQ));
      auto issue_s = [&](int t) {  // S[t & 1] = Q K_t^T
        const int st = t % kTcStages;
        const uint64_t k_desc = sdesc_k_sw128(smem_u32(sK + st * kTile), KB * 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_bf16(tmem + (uint32_t)(t & 1) * 128u,
                   q_desc + ((uint64_t)((k >> 2) * (kTcRows * 128) + (k & 3) * 32) >> 4),
                   k_desc + ((uint64_t)((k >> 2) * 1024 + (k & 3) * 32) >> 4), idesc_s, k > 0);
        mma_commit(&s_full[t & 1]);
        mma_commit(&k_empty[st]);  // the K stage is free once the logits are formed
        issued = true;
      };
      for (int t = 0; t <= T && ok; ++t) {
        // S of tile t (ahead of tile t - 1's output MMAs)
        if (t < T) {
          if (!(ok = mbar_wait(&k_full[t % kTcStages], (t / kTcStages) & 1, abort_flag, status))) break;
          if (!(ok = mbar_wait(&s_empty[t & 1], ((t >> 1) & 1) ^ 1, abort_flag, status))) break;
          tc_fence_after_sync();
          issue_s(t);
        }
        if (t == 0) continue;
        // output of tile t - 1: Y += P_hi V + P_lo V
        const int tp = t - 1;
        if (!(ok = mbar_wait(p_full, tp & 1, abort_flag, status))) break;
        if (!(ok = mbar_wait(&v_full[tp % kTcStages], (tp / kTcStages) & 1, abort_flag, status))) break;
        tc_fence_after_sync();
        const uint32_t v_base = smem_u32(sV + (tp % kTcStages) * kTile);
#pragma unroll
        for (int k = 0; k < kTcKeys / 16; ++k) {  // 16 keys = two 8-key atoms per step
          const uint64_t v_desc = sdesc_mn_sw128(v_base + k * 2 * KB * 1024, 1024, KB * 1024);
          mma_bf16_tmem_a(tmem + kColY, tmem + kColP + 8 * k, v_desc, idesc_y, (tp > 0 || k > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < kTcKeys / 16; ++k) {
          const uint64_t v_desc = sdesc_mn_sw128(v_base + k * 2 * KB * 1024, 1024, KB * 1024);
          mma_bf16_tmem_a(tmem + kColY, tmem + kColPlo + 8 * k, v_desc, idesc_y, 1u);
        }
        mma_commit(p_empty);
        mma_commit(&v_empty[tp % kTcStages]);
      }
      if (ok) {
        mma_commit(y_full);
      } else if (issued) {  // one more commit covers every MMA issued
        mma_commit(drain);
        mbar_wait(drain, 0, nullptr, status);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q4 = warp & 3;               // TMEM lane quarter of this warp
    const int hf = (warp - 2) >> 2;        // which 64 of a tile's 128 columns
    const int r = q4 * 32 + lane;          // row within the tile
    const int i = r0 + r;                  // proxy row
    const uint32_t t_lane = tmem + ((uint32_t)(q4 * 32) << 16);
    const float c2 = meta.scale * kLog2e;
    // the unit's kept positions (ascending) and the shift c = max_i LSE_i of its
    // rows, loaded by the epilogue warps alone while the producers already stream
    const int et = threadIdx.x - 64;  // 0 .. 32 kTcEpi - 1
    const int64_t krow0 = ((int64_t)u.l * meta.H + u.h) * meta.Mtot + u.moff;
    for (int k = et; k < u.m; k += 32 * kTcEpi) {
      const int32_t pos = __ldg(keep + krow0 + k);
      // the tile walk below needs the positions inside the segment and strictly ascending
      if (pos < 0 || pos >= u.n || (k > 0 && pos <= __ldg(keep + krow0 + k - 1))) atomicOr(status, KVC_DEV_BAD_KEEP);
      sKeep[k] = pos;
    }
    float cmax = -INFINITY;
    for (int k = et; k < meta.R; k += 32 * kTcEpi) cmax = fmaxf(cmax, __ldg(lse_rows + lrow + k));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    if (lane == 0) red[warp - 2] = cmax;
    bar_sync_n(1, 32 * kTcEpi);  // sKeep and red complete
    const float lse = i < meta.R ? lse_rows[lrow + i] : INFINITY;
    const float lse2 = lse * kLog2e;
    float c = red[0];
#pragma unroll
    for (int w = 1; w < kTcEpi; ++w) c = fmaxf(c, red[w]);
    const float cc = c * kLog2e;
    // stores of E and Y go through the warp's 32 x 33 turn-around, so that each
    // runs along one row (lane = column) instead of down 32 rows (lane = row)
    float* tr = sTr + (warp - 2) * 32 * 33;
    const int iw = r0 + q4 * 32;                // the warp's first proxy row
    float* Ew = u.base + (int64_t)iw * u.ldE;   // E[i][k] = exp(L_i,keep[k] - c), column m = s_i
    int kk = 0;                                 // first kept position not yet passed
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      ok = mbar_wait(&s_full[t & 1], (t >> 1) & 1, abort_flag, status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after_sync();
      const uint32_t s_col = t_lane + (uint32_t)(t & 1) * 128u;
      float v0[32], v1[32];  // this warp's 64 logits of the row
      tmem_ld32(s_col + 64 * hf, v0);
      tmem_ld32(s_col + 64 * hf + 32, v1);
      const int nvalid = u.n - t * kTcKeys - 64 * hf;
      if (nvalid < 64) {  // keys past the segment: p = 0
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          if (jj >= nvalid) v0[jj] = -INFINITY;
          if (jj + 32 >= nvalid) v1[jj] = -INFINITY;
        }
      }
      // the probabilities first (while the previous tile's output MMAs still read P),
      // then the wait for P's buffer, then the stores
      const float2 cc2 = make_float2(c2, c2), nl2 = make_float2(-lse2, -lse2), neg = make_float2(-1.0f, -1.0f);
      uint32_t hi[2][16], lo[2][16];  // 32 keys per chunk: 16 packed pairs into each of P_hi and P_lo
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const float* vv = ch ? v1 : v0;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 x = __ffma2_rn(make_float2(vv[2 * e], vv[2 * e + 1]), cc2, nl2);
          const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          const __nv_bfloat162 h = __float22bfloat162_rn(p);  // .x (the low half) is the even key
          const uint32_t hb = *reinterpret_cast<const uint32_t*>(&h);
          const float2 hfl = make_float2(__uint_as_float(hb << 16), __uint_as_float(hb & 0xFFFF0000u));
          const __nv_bfloat162 l = __float22bfloat162_rn(__ffma2_rn(hfl, neg, p));  // p - hi, rounded
          hi[ch][e] = hb;
          lo[ch][e] = *reinterpret_cast<const uint32_t*>(&l);
        }
      }
      ok = mbar_wait(p_empty, (t & 1) ^ 1, abort_flag, status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after_sync();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int cg = 2 * hf + ch;  // keys 32 cg .. 32 cg + 31 of the tile
        tmem_st16(t_lane + kColP + cg * 16, hi[ch]);
        tmem_st16(t_lane + kColPlo + cg * 16, lo[ch]);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      // E after the hand-off of P, so that its loads and stores overlap the output
      // MMAs instead of delaying them; S's buffer is released once E is read
      {  // E over the kept keys of this warp's 64 columns of the tile, from the same logits as
         // the LSE pass: a kept key's column is the same for the whole warp, so it is read
         // straight from TMEM, eight columns per load-and-wait
        // the kept keys of the tile's two halves: positions ascend, so 32 of them
        // at a time and two ballots count them (one round unless more than 32
        // keys of the tile are kept)
        int n_lo = 0, n_all = 0;
        for (int base = kk;; base += 32) {
          const int pos = base + lane < u.m ? sKeep[base + lane] : INT_MAX;
          const unsigned in_lo = __ballot_sync(0xffffffffu, pos < t * kTcKeys + 64);
          const unsigned in_all = __ballot_sync(0xffffffffu, pos < (t + 1) * kTcKeys);
          n_lo += __popc(in_lo);
          n_all += __popc(in_all);
          if (in_all != 0xffffffffu) break;
        }
        const int k_mid = kk + n_lo, k_end = kk + n_all;
        const int ka = hf ? k_mid : kk, kb = hf ? k_end : k_mid;
        for (int kc = ka; kc < kb; kc += 32) {  // 32 kept columns at a time
          const int nk = min(32, kb - kc);
          for (int k0 = kc; k0 < kc + nk; k0 += 8) {
            uint32_t a[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int k = min(k0 + e, kb - 1);
              a[e] = s_col + (uint32_t)max(0, sKeep[k] - t * kTcKeys);
            }
            float ev[8];
            tmem_ld1x8(a, ev);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (k0 + e < kc + nk) tr[lane * 33 + (k0 - kc) + e] = exp2f(fmaf(ev[e], c2, -cc));
          }
          __syncwarp();
          if (lane < nk) {
#pragma unroll 4
            for (int rr = 0; rr < 32; ++rr)
              if (iw + rr < meta.R) Ew[(int64_t)rr * u.ldE + kc + lane] = tr[rr * 33 + lane];
          }
          __syncwarp();
        }
        kk = k_end;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[t & 1]);
    }
    if (ok) {
      ok = mbar_wait(y_full, 0, abort_flag, status);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after_sync();
      float* Yw = u.base + am_off_Y(meta.R, meta.max_m, u.ldE) + (int64_t)iw * D;
#pragma unroll 1
      for (int col = 64 * hf; col < min(D, 64 * hf + 64); col += 32) {  // this warp's half of Y's columns
        float y[32];
        tmem_ld32(t_lane + kColY + col, y);
#pragma unroll
        for (int e = 0; e < 32; ++e) tr[lane * 33 + e] = y[e];
        __syncwarp();
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr)
          if (iw + rr < meta.R) Yw[(int64_t)rr * D + col + lane] = tr[rr * 33 + lane];
        __syncwarp();
      }
      if (hf == 0 && i < meta.R) {
        u.base[am_off_lse(meta.R, meta.max_m, u.ldE, D) + i] = lse;
        u.base[(int64_t)i * u.ldE + u.m] = exp2f((lse - c) * kLog2e);
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

// ------------------------------------------------------------------ A^T B on the tensor cores
// C[p][q] = sum_i A[i][p] B[i][q] over the R proxy rows, for the three Gram
// products of the fits:
//   mode 0: A = E (m columns), B = [E | s] (m + 1), C = G        (stride ldE)
//   mode 1: A = B = Ph (m columns),                 C = H in G's place
//   mode 2: A = Ph, B = Y (d columns, stride d),    C = Bm       (stride d),
//           summed over up to kAmBmParts ranges of the rows by separate blocks
//           (range p > 0 into Bp part p - 1); it runs in the same launch as
//           mode 1, whose blocks come first and never read B
//   mode 3: A = H (m rows), B = X0 (the kept values), C = H X0 - Bm in Bm's
//           place, Bm's first row range only (the value fit's starting
//           gradient once the value fit subtracts the others; H is symmetric)
// on tcgen05 with fp32-level accuracy: every fp32 value
// x is split into three bf16 parts (x0 = bf16(x), x1 = bf16(x - x0),
// x2 = bf16(x - x0 - x1): 8 + 8 + 8 significant bits, x0 + x1 + x2 = x to the
// last bit of x's significand), and the six part products whose weight is
// above 2^-24 are accumulated in fp32 in TMEM: a0b0 + a0b1 + a1b0 + a1b1 +
// a0b2 + a2b0 (each product of two 8-bit significands is exact).
//
// C is cut into 128 x 128 tiles.  G's first m columns and H are symmetric:
// only tiles with p0 <= q0 are computed, and each also writes its transpose
// (a diagonal tile writes its upper triangle and mirrors it), so both
// triangles hold the same numbers.  A block takes up to three consecutive
// tiles of the unit (row-major over the computed ones), one 128-column TMEM
// accumulator each, and the distinct 128-column strips they read (at most
// four: modes 0 and 1 read both operands from the same matrix, E's strips
// taken over the m + 1 columns of [E | s]), so a strip shared by its tiles is
// loaded and split once.  Per chunk of 16 proxy rows, warp 16 loads each strip
// as one TMA box of the launch's 3-D tensor map (every unit of a launch is laid
// out for the launch's largest m: rows past R and columns past the map read as
// zeros) into a ring of two stages (full / empty mbarriers); warps 1-15 split
// 8 consecutive values at a time with the packed fp32->bf16x2 conversion
// (values past the unit's own columns become zeros) and write the parts as
// MN-major operands (1024-byte atoms of 8 rows x 64 elements along p or q:
// LBO = 1024 B along p/q, SBO = 2048 B along the rows) into one of three
// operand buffers, then arrive on its "ready" mbarrier; one thread of warp 0
// only issues the six MMAs per tile (M = N = 128, K = 16, both operands
// MN-major) and commits them to the buffer's "done" mbarrier.  The epilogue
// turns each warp's 32 x 32 block of C around in shared memory so that its
// stores run along rows.
constexpr int kTbThreads = 544;                             // warp 0 issues, warps 1-15 split, warp 16 loads
constexpr int kTbRows = 16;                                 // proxy rows per chunk (one K step)
constexpr int kTbTiles = 3;                                 // output tiles per block
constexpr int kTbStrips = 4;                                // distinct strips per block, at most
constexpr int kTbPart = kTbRows * 128 * 2;                  // one bf16 part of one strip: 4 KB
constexpr int kTbBuf = kTbStrips * 3 * kTbPart;             // every strip's three parts
constexpr int kTbStripFloats = kTbRows * 128;               // one strip's fp32 rows of a chunk (one box)
constexpr int kTbStageFloats = kTbStrips * kTbStripFloats;  // one ring stage
constexpr int kTbStages = 2;
constexpr int kTbBufs = 3;                                  // operand buffers: the split runs up to two chunks ahead
constexpr int kTbWorkers = 15 * 32;                         // the splitting warps
constexpr int kTbItems = (kTbStageFloats / 8 + kTbWorkers - 1) / kTbWorkers;  // 8-value splits per worker
constexpr int kTbSmem = 1024 + 1024 + kTbBufs * kTbBuf + kTbStages * kTbStageFloats * 4;  // head, slack, buffers, ring
static_assert(kTbSmem <= 227 * 1024, "operand buffers and the fp32 ring fit one CTA's shared memory");
constexpr int kAtbTile = 128;  // output tile of the A^T B products

// The computed tiles of one unit: rows mt = ceil(m / 128) of p, nt columns of
// q; the symmetric modes take mi <= ni only.
struct TileGrid {
  int mt, nt;
  bool sym;
  __host__ __device__ int count() const { return sym ? mt * nt - mt * (mt - 1) / 2 : mt * nt; }
  // tile number t (row-major over the computed tiles) -> (mi, ni)
  __host__ __device__ void tile(int t, int& mi, int& ni) const {
    for (mi = 0;; ++mi) {
      const int in_row = sym ? nt - mi : nt;
      if (t < in_row) break;
      t -= in_row;
    }
    ni = (sym ? mi : 0) + t;
  }
};
__host__ __device__ inline TileGrid tile_grid(int mode, int m, int d) {
  TileGrid g;
  g.mt = (m + kAtbTile - 1) / kAtbTile;
  g.nt = mode >= 2 ? (d + kAtbTile - 1) / kAtbTile : (mode == 0 ? m + 1 + kAtbTile - 1 : m + kAtbTile - 1) / kAtbTile;
  g.sym = mode < 2;
  return g;
}
// blocks per unit for the largest m of a launch
inline int atb_blocks_per_unit(int mode, int max_m, int d) {
  return (tile_grid(mode, max_m, d).count() + kTbTiles - 1) / kTbTiles;
}

__device__ __forceinline__ uint32_t bf2_bits(float a, float b) {
  const __nv_bfloat162 h = __float22bfloat162_rn(make_float2(a, b));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kTbThreads, 1)
    am_atb_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const AmMeta meta, float* ws, int mode_lo, int bpu_lo, int64_t blocks_lo, int bpu2,
                     unsigned* status) {
  extern __shared__ __align__(16) uint8_t tb_smem[];
  uint64_t* done = reinterpret_cast<uint64_t*>(tb_smem);  // [kTbBufs] an operand buffer's MMAs are done
  uint64_t* ready = done + kTbBufs;                        // [kTbBufs] an operand buffer is split
  uint64_t* full = ready + kTbBufs;                              // [kTbStages] a ring stage's rows are in
  uint64_t* empty = full + kTbStages;                      // [kTbStages] a ring stage is split
  uint64_t* fin = empty + kTbStages;                       // every MMA is done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tb_smem + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* bufs = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tb_smem) + 1024 + 1023) &
                                             ~uintptr_t(1023));
  float* ring = reinterpret_cast<float*>(bufs + kTbBufs * kTbBuf);
  // blocks [0, blocks_lo) run mode_lo over all K rows; the others (modes 1 and 2
  // in one launch) run mode 2 over one of meta.bm_parts ranges of the rows
  int mode = mode_lo, blocks_per_unit = bpu_lo, part = 0, nparts = 1;
  int64_t lb = blockIdx.x;
  if (lb >= blocks_lo) {
    lb -= blocks_lo;
    mode = 2;
    blocks_per_unit = bpu2;
    nparts = meta.bm_parts;
    part = (int)(lb % nparts);
    lb /= nparts;
  }
  const int64_t unit = lb / blocks_per_unit;
  const AmUnit u = am_unit(meta, unit, ws);
  const int M = u.m;
  const int N = mode == 0 ? u.m + 1 : (mode == 1 ? u.m : meta.d);
  const int K = mode == 3 ? u.m : meta.R;  // the rows summed over
  const TileGrid tg = tile_grid(mode, M, meta.d);
  const int t0 = (int)(lb % blocks_per_unit) * kTbTiles;
  const int ntiles = min(kTbTiles, tg.count() - t0);
  if (ntiles <= 0) return;
  // the block's tiles and strips: strip slot k holds the 128 columns from
  // scol[k] of A, or (modes 2 and 3, slots from ybase on) of B; tile k reads
  // slots sa[k] and sb[k]
  int tmi[kTbTiles], tni[kTbTiles], sa[kTbTiles], sb[kTbTiles];
  int scol[kTbStrips];
  int nstr = 0;
#pragma unroll
  for (int k = 0; k < kTbTiles; ++k) {
    tmi[k] = tni[k] = sa[k] = sb[k] = 0;
    if (k < ntiles) tg.tile(t0 + k, tmi[k], tni[k]);
  }
  auto find_or_add = [&](int col) {
    for (int k = 0; k < nstr; ++k)
      if (scol[k] == col) return k;
    scol[nstr] = col;
    return nstr++;
  };
#pragma unroll
  for (int k = 0; k < kTbTiles; ++k)
    if (k < ntiles) sa[k] = find_or_add(tmi[k] * 128);
  const int ybase = nstr;
#pragma unroll
  for (int k = 0; k < kTbTiles; ++k) {
    if (k >= ntiles) continue;
    if (mode >= 2) {
      const int col = tni[k] * 128;
      int found = -1;
      for (int st = ybase; st < nstr; ++st)
        if (scol[st] == col) found = st;
      if (found < 0) {
        scol[nstr] = col;
        found = nstr++;
      }
      sb[k] = found;
    } else {
      sb[k] = find_or_add(tni[k] * 128);
    }
  }
  // columns of an A strip inside the unit's matrix (the maps run to the
  // launch's row stride): mode 0 takes E over the m + 1 columns of [E | s]
  // (row m of C is not kept), so that one strip serves both operands of a
  // diagonal tile; B's maps (Y, X0) end at d
  const int ncolX = mode == 0 ? N : M;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this block's chunks of kTbRows rows: [c_lo, c_lo + nchunks)
  const int nchunks_all = (K + kTbRows - 1) / kTbRows;
  const int c_lo = (int)((int64_t)part * nchunks_all / nparts);
  const int nchunks = (int)((int64_t)(part + 1) * nchunks_all / nparts) - c_lo;
  if (threadIdx.x == 0) {
    for (int b = 0; b < kTbBufs; ++b) {
      mbar_init(&done[b], 1);
      mbar_init(&ready[b], kTbWorkers);
    }
    for (int st = 0; st < kTbStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kTbWorkers);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_slot, 512);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {  // the MMA issuer: one chunk's MMAs once its operands are split
      // both operands MN-major (transpose bits), bf16 x bf16 -> fp32, M = N = 128
      const uint32_t idesc = idesc_bf16_f32(128, 128) | (1u << 15) | (1u << 16);
      const uint64_t dbase = sdesc_mn_sw128(smem_u32(bufs), 1024, 2048);  // + (byte offset >> 4)
      const int pa[6] = {0, 0, 1, 1, 0, 2}, pb[6] = {0, 1, 0, 1, 2, 0};
      for (int c = 0; c < nchunks; ++c) {
        if (!mbar_wait(&ready[c % kTbBufs], (uint32_t)(c / kTbBufs) & 1u, abort_flag, status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t boff = (uint32_t)(c % kTbBufs) * kTbBuf;
#pragma unroll
        for (int k = 0; k < kTbTiles; ++k) {
          if (k >= ntiles) break;
          const uint32_t a = boff + sa[k] * 3 * kTbPart, b = boff + sb[k] * 3 * kTbPart;
#pragma unroll
          for (int pr = 0; pr < 6; ++pr)
            mma_bf16(tmem + k * 128, dbase + ((a + pa[pr] * kTbPart) >> 4), dbase + ((b + pb[pr] * kTbPart) >> 4),
                     idesc, (c > 0 || pr > 0) ? 1u : 0u);
        }
        mma_commit(&done[c % kTbBufs]);
      }
    }
    __syncwarp();
  } else if (warp == kTbThreads / 32 - 1) {  // the producer: one box per strip and chunk
    if (lane == 0) {
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        const int st = c % kTbStages;
        if (c >= kTbStages &&  // the workers have split the stage's previous chunk
            !mbar_wait(&empty[st], (uint32_t)(c / kTbStages - 1) & 1u, abort_flag, status)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[st], (uint32_t)nstr * kTbStripFloats * 4);
        float* stg = ring + st * kTbStageFloats;
        for (int k = 0; k < nstr; ++k) {
          const bool fromB = mode >= 2 && k >= ybase;
          tma_load_3d(stg + k * kTbStripFloats, fromB ? &tmB : &tmA, &full[st], scol[k], (c_lo + c) * kTbRows,
                      (int)unit);
        }
        issued = c + 1;
      }
      // the copies in flight land before the block leaves (bounded waits)
      for (int c = max(0, issued - kTbStages); c < issued; ++c)
        mbar_wait(&full[c % kTbStages], (uint32_t)(c / kTbStages) & 1u, nullptr, status);
    }
    __syncwarp();
  } else {  // workers: split the staged rows, hand the operand buffer over
    const int wt = threadIdx.x - 32;
    for (int c = 0; c < nchunks; ++c) {
      const int st0 = c % kTbStages;
      bool w_ok = mbar_wait(&full[st0], (uint32_t)(c / kTbStages) & 1u, abort_flag, status);
      if (w_ok && c >= kTbBufs)  // the MMAs of chunk c - kTbBufs have read this operand buffer
        w_ok = mbar_wait(&done[c % kTbBufs], (uint32_t)(c / kTbBufs - 1) & 1u, abort_flag, status);
      if (!w_ok) {
        ok = false;
        break;
      }
      uint8_t* buf = bufs + (c % kTbBufs) * kTbBuf;
      const float* stg = ring + st0 * kTbStageFloats;
#pragma unroll
      for (int k = 0; k < kTbItems; ++k) {  // 8 values per item
        const int e = wt + k * kTbWorkers;
        const int st = e >> 8, r = (e >> 4) & (kTbRows - 1), g = e & 15;
        if (st >= nstr) continue;
        const float* sp = stg + st * kTbStripFloats + r * 128 + g * 8;
        const float4 v0 = *reinterpret_cast<const float4*>(sp);
        const float4 v1 = *reinterpret_cast<const float4*>(sp + 4);
        float x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        // A's columns past this unit's, and (mode 3: the maps run to the launch's
        // largest m) rows past it, are not its own
        const int nv = (c_lo + c) * kTbRows + r >= K ? 0 : (mode >= 2 && st >= ybase ? 8 : ncolX - scol[st] - g * 8);
        if (nv < 8) {
#pragma unroll
          for (int t = 0; t < 8; ++t)
            if (t >= nv) x[t] = 0.0f;
        }
        uint32_t h0[4], h1[4], h2[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float a = x[2 * t], b = x[2 * t + 1];
          h0[t] = bf2_bits(a, b);
          const float ra = a - __uint_as_float(h0[t] << 16), rb = b - __uint_as_float(h0[t] & 0xFFFF0000u);
          h1[t] = bf2_bits(ra, rb);
          h2[t] = bf2_bits(ra - __uint_as_float(h1[t] << 16), rb - __uint_as_float(h1[t] & 0xFFFF0000u));
        }
        // MN-major atom layout: row r, 8 elements at g * 8 along p / q
        const int off = (r >> 3) * 2048 + (g >> 3) * 1024 + (r & 7) * 128 + (((g & 7) ^ (r & 7)) << 4);
        uint8_t* base = buf + st * 3 * kTbPart + off;
        *reinterpret_cast<uint4*>(base) = make_uint4(h0[0], h0[1], h0[2], h0[3]);
        *reinterpret_cast<uint4*>(base + kTbPart) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
        *reinterpret_cast<uint4*>(base + 2 * kTbPart) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the parts, for the tensor cores
      mbar_arrive(&ready[c % kTbBufs]);
      mbar_arrive(&empty[st0]);
    }
  }
  if (!ok) *abort_flag = 1;
  if (threadIdx.x == 0) mma_commit(fin);  // covers every MMA issued (also after an abort)
  const bool fin_ok = mbar_wait(fin, 0, nullptr, status);
  if (__syncthreads_and(ok && fin_ok && !*abort_flag)) {
    tc_fence_after_sync();
    const int q4 = warp & 3, cq = (warp >> 2) & 3;  // TMEM lane quarter; columns [32 cq, 32 cq + 32) of a tile
    // The operand buffers are free now: each warp turns its 32 x 32 block
    // around in shared memory, so that a store (and mode 3's load) covers 32
    // consecutive columns of one row.
    float* tr = reinterpret_cast<float*>(bufs) + warp * 32 * 33;
    // C: G or H (stride ldE), Bm (stride d), or (mode 2, row range p > 0) Bp part p - 1
    float* C = mode >= 2 ? u.base + am_off_Bm(meta.R, meta.max_m, u.ldE, meta.d) : u.base + am_off_G(meta.R, u.ldE);
    if (mode == 2 && part > 0)
      C = u.base + am_off_Bp(meta.R, meta.max_m, u.ldE, meta.d) + (part - 1) * (int64_t)meta.max_m * meta.d;
    const int ldc = mode >= 2 ? meta.d : u.ldE;
#pragma unroll 1
    for (int k = 0; k < ntiles && warp < 16; ++k) {
      const bool dg = tg.sym && tmi[k] == tni[k];
      const int p0w = tmi[k] * 128 + q4 * 32, pr = p0w + lane;
      float y[32];
      if (nchunks > 0) {
        tmem_ld32(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(k * 128 + cq * 32), y);
      } else {  // a row range without rows adds nothing
#pragma unroll
        for (int t = 0; t < 32; ++t) y[t] = 0.0f;
      }
      const int qb = tni[k] * 128 + cq * 32;
      if (tg.sym) {  // the transpose: C[q][p] for q < m (not G's column m), lanes along p coalesced
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (pr < M && qb + t < M && qb + t > pr) C[(int64_t)(qb + t) * ldc + pr] = y[t];
      }
#pragma unroll
      for (int t = 0; t < 32; ++t) tr[lane * 33 + t] = y[t];
      __syncwarp();
      const int q = qb + lane;  // this lane's column; rows p0w .. p0w + 31
      if (mode == 3) {  // C = H X0 - (Bm's first row range), 16 rows at a time: their Bm values first
#pragma unroll
        for (int r0 = 0; r0 < 32; r0 += 16) {
          float bm[16];
#pragma unroll
          for (int r = 0; r < 16; ++r)
            bm[r] = (p0w + r0 + r < M && q < N) ? C[(int64_t)(p0w + r0 + r) * ldc + q] : 0.0f;
#pragma unroll
          for (int r = 0; r < 16; ++r)
            if (p0w + r0 + r < M && q < N) C[(int64_t)(p0w + r0 + r) * ldc + q] = tr[(r0 + r) * 33 + lane] - bm[r];
        }
      } else {
#pragma unroll
        for (int r = 0; r < 32; ++r)
          if (p0w + r < M && q < N && (!dg || q >= p0w + r)) C[(int64_t)(p0w + r) * ldc + q] = tr[r * 33 + lane];
      }
      __syncwarp();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ blocked descents
// Both fits are cyclic coordinate descents on normal equations: a step on
// coordinate j reads gradient row j, moves x_j, and adds the move times row j
// of the Gram matrix (its column j) to every gradient row.  The kernels take
// the coordinates 32 at a time, in the same order, and split each block of 32
// steps between the warps:
//   * warp 0 runs the 32 steps, keeping the block's own 32 gradient rows
//     current after every step from the block's 32 x 32 diagonal tile;
//   * meanwhile warps 1-7 add the previous block's moves to the other rows,
//     g_i += sum_t M[jp + t][i] dx_t in step order (one pass over the previous
//     block's 32 rows of M, coalesced along i; none when nothing moved), and
//     stage the next block's tiles with cp.async.  The current block's own
//     rows get the previous block's moves first, from a staged 32 x 32 cross
//     tile, and a named barrier then releases warp 0.
// Every step sees the gradient of the one-coordinate-at-a-time descent, and
// every gradient entry receives the same fused multiply-adds in the same order.
constexpr int kDb = 32;                    // coordinates per block: one warp's lanes
constexpr int kTileLd = 36;                // row stride of a staged tile (floats, 16-byte rows)
constexpr int kTile = kDb * kTileLd;       // one staged tile
constexpr int kHelpers = kAmThreads - 32;  // warps 1-7

// tile[t][k] = M[r0 + t][c0 + k] for t < nr, k < nc, zero elsewhere (16-byte
// cp.async; rows of M 16-byte aligned), spread over threads tid of nthr.
__device__ __forceinline__ void stage_tile(float* tile, const float* M, int64_t ld, int r0, int nr, int c0, int nc,
                                           int tid, int nthr) {
  for (int e = tid; e < kDb * (kDb / 4); e += nthr) {
    const int t = e >> 3, q = e & 7;
    const int valid = t < nr ? max(0, min(4, nc - 4 * q)) : 0;
    const float* src = valid > 0 ? M + (int64_t)(r0 + t) * ld + c0 + 4 * q : M;
    cp_async_16z(tile + t * kTileLd + 4 * q, src, valid * 4);
  }
}

// Sums of rows i0 .. i0 + 3 of M over its first m columns, in every lane of
// the warp (lanes take every 32nd column; four rows at a time keep four loads
// in flight per column step).  Rows at or past m get 0.
__device__ __forceinline__ void row_sums4(const float* __restrict__ M, int64_t ld, int m, int i0, float (&sum)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < 4; ++r) sum[r] = 0.0f;
  for (int k = lane; k < m; k += 32) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
      if (i0 + r < m) sum[r] += M[(int64_t)(i0 + r) * ld + k];
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], o);
}

// ------------------------------------------------------------------ mass fit
// Block = unit.  Projected cyclic coordinate descent on min_{w >= 0} ||E w - s||^2
// from w = 1: with g = G w - b, coordinate j moves to max(0, w_j - g_j / G_jj)
// and g follows by the change times row j of G (G symmetric).  Coordinate j
// moves only when |g_j| > 2^-17 b_j (every term of G w and of b = E^T s is
// >= 0, so b_j is their scale).  In a block's steps lane k of warp 0 holds
// coordinate j0 + k; the coordinate of step t broadcasts its gradient by
// shuffle.  Writes w (workspace), beta = ln w (-inf at 0) to `beta` and to the
// per-slot state of each kept entry.
constexpr int kMassHead = 2 * kDb + 4 * kTile + 4;  // moves [2][32], tiles [2][diag, cross], flags
__host__ __device__ constexpr int mass_smem_bytes(int m) { return (kMassHead + 4 * m) * 4; }

__global__ void __launch_bounds__(kAmThreads) am_mass_kernel(const AmMeta meta, const int32_t* __restrict__ bt,
                                                             const int32_t* __restrict__ keep, float* ws,
                                                             float* aux, float* beta, unsigned* status) {
  extern __shared__ __align__(16) float am_smem[];
  const AmUnit u = am_unit(meta, blockIdx.x, ws);
  const int m = u.m;
  if (m <= 0) return;
  float* dws = am_smem;                                       // [2][32] moves of the last two blocks
  float* tiles = dws + 2 * kDb;                               // [2][2][kTile]
  int* moved = reinterpret_cast<int*>(tiles + 4 * kTile);     // [2] did that block move; [2] did this sweep
  float* g = am_smem + kMassHead;                             // [m] gradient G w - b
  float* w = g + m;                                           // [m]
  float* thr = w + m;                                         // [m] 2^-17 b_j; +inf where G_jj <= 0
  float* diag = thr + m;                                      // [m] G_jj
  const float* G = u.base + am_off_G(meta.R, u.ldE);
  const int64_t ld = u.ldE;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i0 = warp * 4; i0 < m; i0 += kAmThreads / 8) {  // g = G 1 - b, four rows per warp at a time
    float acc[4];
    row_sums4(G, ld, m, i0, acc);
    if (lane < 4 && i0 + lane < m) {
      const int i = i0 + lane;
      const float* gr = G + (int64_t)i * ld;
      const float b = gr[m], d = gr[i];
      const float a = lane == 0 ? acc[0] : lane == 1 ? acc[1] : lane == 2 ? acc[2] : acc[3];
      g[i] = a - b;
      w[i] = 1.0f;
      thr[i] = d > 0.0f ? kAmGuard * b : INFINITY;
      diag[i] = d;
    }
  }
  if (threadIdx.x < 3) moved[threadIdx.x] = 0;
  const int nb = (m + kDb - 1) / kDb;
  stage_tile(tiles, G, ld, 0, min(kDb, m), 0, min(kDb, m), threadIdx.x, kAmThreads);  // block 0's diagonal
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  const int64_t iters = (int64_t)meta.sweeps * nb;
  int jp = 0, cntp = 0;  // the previous block
  for (int64_t it = 0; it < iters; ++it) {
    const int cur = (int)(it & 1), prev = cur ^ 1;
    const int j0 = (int)(it % nb) * kDb, cnt = min(kDb, m - j0);
    const float* dtile = tiles + cur * 2 * kTile;  // diag[t][k] = G[j0 + t][j0 + k]
    const float* ctile = dtile + kTile;            // cross[t][k] = G[jp + t][j0 + k]
    // A sweep in which no coordinate moved left g and w as they were, so the
    // next one would repeat it: the descent has reached its fixed point.
    if (j0 == 0 && it > 0 && moved[2] == 0) break;
    if (warp == 0) {
      bar_sync_n(1, kAmThreads);  // the block's rows have the previous block's moves
      const bool v = lane < cnt;
      const int j = j0 + lane;
      float gk = v ? g[j] : 0.0f;
      const float w0 = v ? w[j] : 0.0f, tk = v ? thr[j] : INFINITY, dk = v ? 1.0f / diag[j] : 1.0f;
      float wk = w0, dwk = 0.0f;
      // If no coordinate of the block would move on the gradient as it stands,
      // none moves at all (a step that does not move changes nothing): skip.
      const bool would = v && (fabsf(gk) > tk ? fmaxf(0.0f, w0 - gk * dk) : w0) != w0;
      const bool steps = __any_sync(0xffffffffu, would);
#pragma unroll
      for (int t = 0; t < kDb; ++t) {
        if (t >= cnt || !steps) break;
        const float gt = __shfl_sync(0xffffffffu, gk, t);
        const float wt = __shfl_sync(0xffffffffu, w0, t);  // w of coordinate t before its own step
        const float tt = __shfl_sync(0xffffffffu, tk, t);
        const float dt = __shfl_sync(0xffffffffu, dk, t);  // 1 / G_tt
        const float nw = fabsf(gt) > tt ? fmaxf(0.0f, wt - gt * dt) : wt;
        const float dl = nw - wt;
        if (dl != 0.0f) {
          gk = fmaf(dl, dtile[t * kTileLd + lane], gk);
          if (lane == t) {
            wk = nw;
            dwk = dl;
          }
        }
      }
      if (v && steps) {
        g[j] = gk;
        w[j] = wk;
      }
      dws[cur * kDb + lane] = dwk;
      const bool any = __any_sync(0xffffffffu, dwk != 0.0f);
      if (lane == 0) {
        moved[cur] = any ? 1 : 0;
        moved[2] = (j0 == 0 ? 0 : moved[2]) | (any ? 1 : 0);  // read by every thread before bar_sync
      }
    } else {
      const int tid = threadIdx.x - 32;
      const float* dwp = dws + prev * kDb;
      const bool apply = moved[prev] != 0 && nb > 1;
      if (apply && warp == 1 && lane < cnt) {  // the block's own rows, from the cross tile
        float acc = g[j0 + lane];
        for (int t = 0; t < cntp; ++t) acc = fmaf(dwp[t], ctile[t * kTileLd + lane], acc);
        g[j0 + lane] = acc;
      }
      bar_arrive_n(1, kAmThreads);
      if (apply) {  // every other row, from the previous block's rows of G
        for (int i = tid; i < m; i += kHelpers) {
          if ((i >= jp && i < jp + cntp) || (i >= j0 && i < j0 + cnt)) continue;
          float h[kDb];
#pragma unroll
          for (int t = 0; t < kDb; ++t) h[t] = t < cntp ? G[(int64_t)(jp + t) * ld + i] : 0.0f;
          float acc = g[i];
#pragma unroll
          for (int t = 0; t < kDb; ++t)
            if (t < cntp) acc = fmaf(dwp[t], h[t], acc);
          g[i] = acc;
        }
      }
      if (it + 1 < iters) {  // the next block's tiles
        const int jn = (int)((it + 1) % nb) * kDb, cntn = min(kDb, m - jn);
        float* nt = tiles + prev * 2 * kTile;
        stage_tile(nt, G, ld, jn, cntn, jn, cntn, tid, kHelpers);
        stage_tile(nt + kTile, G, ld, j0, cnt, jn, cntn, tid, kHelpers);
        cp_async_commit();
        cp_async_wait_all();
      }
    }
    jp = j0;
    cntp = cnt;
    __syncthreads();
  }
  float* wout = u.base + am_off_w(meta.R, meta.max_m, u.ldE, meta.d);
  const int64_t orow = ((int64_t)u.l * meta.H + u.h) * meta.Mtot + u.moff;
  for (int j = threadIdx.x; j < m; j += kAmThreads) {
    const float wj = w[j];
    wout[j] = wj;
    const float bj = wj > 0.0f ? logf(wj) : -INFINITY;
    if (beta != nullptr) beta[orow + j] = bj;
    if (aux != nullptr) {
      const int pos = am_kept(meta, u, keep, j, status);
      const int64_t row = pos < 0 ? -1 : am_row(meta, u, bt, pos, status);
      if (row >= 0) aux[row] = bj;
    }
  }
}

// ------------------------------------------------------------------ compact probabilities
// Block = (unit, 8 proxy rows), one warp per row: z_i = sum_j E_ij w_j, then
// Ph_ij = E_ij w_j / z_i in place (a row without mass stays zero); the first
// 512 products stay in registers between the two, so E is read once.
__global__ void __launch_bounds__(kAmThreads) am_probs_kernel(const AmMeta meta, float* ws) {
  const int rb = (meta.R + 7) / 8;
  const AmUnit u = am_unit(meta, blockIdx.x / rb, ws);
  const int i = (int)(blockIdx.x % rb) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= meta.R) return;
  float* E = u.base + (int64_t)i * u.ldE;
  const float* w = u.base + am_off_w(meta.R, meta.max_m, u.ldE, meta.d);
  constexpr int kHeld = 16;  // E_ij w_j held in registers for the first 32 x kHeld columns
  float ew[kHeld];
  float z = 0.0f;
#pragma unroll
  for (int t = 0; t < kHeld; ++t) {
    const int j = lane + 32 * t;
    ew[t] = j < u.m ? E[j] * w[j] : 0.0f;
  }
#pragma unroll
  for (int t = 0; t < kHeld; ++t) z += ew[t];
  for (int j = lane + 32 * kHeld; j < u.m; j += 32) z += E[j] * w[j];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  const float inv = z > 0.0f ? 1.0f / z : 0.0f;
#pragma unroll
  for (int t = 0; t < kHeld; ++t) {
    const int j = lane + 32 * t;
    if (j < u.m) E[j] = ew[t] * inv;
  }
  for (int j = lane + 32 * kHeld; j < u.m; j += 32) E[j] = E[j] * w[j] * inv;
}

// ------------------------------------------------------------------ kept values
// Block = (unit, 8 kept entries), one warp per entry: X0[j] = the kept entry's
// V row (bf16 -> fp32) into the unit's X region (zero for a bad page or
// position, which is reported).
template <int D>
__global__ void __launch_bounds__(kAmThreads) am_x0_kernel(const AmMeta meta, const int32_t* __restrict__ bt,
                                                           const int32_t* __restrict__ keep,
                                                           const uint16_t* __restrict__ vp, float* ws,
                                                           unsigned* status) {
  const int jb = (meta.max_m + 7) / 8;
  const AmUnit u = am_unit(meta, blockIdx.x / jb, ws);
  const int j = (int)(blockIdx.x % jb) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= u.m) return;
  int64_t row = -1;
  if (lane == 0) {
    const int pos = am_kept(meta, u, keep, j, status);
    row = pos < 0 ? -1 : am_row(meta, u, bt, pos, status);
  }
  row = __shfl_sync(0xffffffffu, row, 0);
  float* X = u.base + am_off_X(meta.R, meta.max_m, u.ldE, D) + (int64_t)j * D;
  for (int e = lane * 2; e < D; e += 64) {
    float2 v = make_float2(0.0f, 0.0f);
    if (row >= 0) {
      const uint32_t b2 = *reinterpret_cast<const uint32_t*>(vp + row * D + e);
      v = make_float2(bf16_bits_to_float(b2 & 0xffffu), bf16_bits_to_float(b2 >> 16));
    }
    *reinterpret_cast<float2*>(X + e) = v;
  }
}

// ------------------------------------------------------------------ value fit
// Block = (unit, 16 of the d value columns).  The columns are independent
// least-squares problems sharing H = Ph^T Ph: cyclic coordinate descent from
// X = the kept values with gradient Gv = H X - Bm (shared memory, column-major
// with an odd stride); row j of X moves by -Gv_j / H_jj when |Gv_jc| > 2^-17
// pi_j S_c (pi_j = sum_k H_jk, S_c = max_i |Y_ic| + max_k |X0_kc|: the scale
// of the gradient's terms in column c).  In a block's steps lane c of warp 0
// holds column c of the block's 32 gradient rows; the diagonal tile's row t
// is read as a broadcast.  The starting gradient H X0 - Bm comes from the
// tensor-core Gram kernel (mode 3, in Bm's place) and X0 from am_x0_kernel;
// X lives in its own workspace region.  At the end V_C is written to `vc`
// (fp32) and over the kept entries' V rows (bf16, round to nearest even).
constexpr int kVc = 16;  // value columns per block
__host__ __device__ constexpr int value_ld(int m) { return m | 1; }
constexpr int kValueHead = 2 * kDb * kVc + 4 * kTile + 2 * kVc + 4;  // moves, tiles, scales, flags
__host__ __device__ constexpr int value_smem_bytes(int m) { return (kValueHead + kVc * value_ld(m) + 2 * m) * 4; }
static_assert(value_smem_bytes(kAmMaxM) <= 227 * 1024 && mass_smem_bytes(kAmMaxM) <= 227 * 1024,
              "descent working sets fit one CTA's shared memory at the largest m");
static_assert(kValueHead % 4 == 0 && kMassHead % 4 == 0, "the per-row arrays start 16-byte aligned");

// Gs[c][i] += sum_{t < cnt} M[j0 + t][i] dxs[t][c], t in step order, for the
// rows i outside [e0, e1) and [f0, f1); one thread (tid of nthr) per row.
__device__ __forceinline__ void value_update(const float* __restrict__ M, int64_t ld, int m, int ldv, int j0, int cnt,
                                             const float* dxs, float* Gs, int e0, int e1, int f0, int f1, int tid,
                                             int nthr) {
  for (int i = tid; i < m; i += nthr) {
    if ((i >= e0 && i < e1) || (i >= f0 && i < f1)) continue;
    float h[kDb];
#pragma unroll
    for (int t = 0; t < kDb; ++t) h[t] = t < cnt ? M[(int64_t)(j0 + t) * ld + i] : 0.0f;
    float acc[kVc];
#pragma unroll
    for (int c = 0; c < kVc; ++c) acc[c] = Gs[c * ldv + i];
#pragma unroll
    for (int t = 0; t < kDb; ++t) {
      if (t >= cnt) break;
      const float4* d4 = reinterpret_cast<const float4*>(dxs + t * kVc);
#pragma unroll
      for (int q = 0; q < kVc / 4; ++q) {
        const float4 d = d4[q];
        acc[4 * q + 0] = fmaf(h[t], d.x, acc[4 * q + 0]);
        acc[4 * q + 1] = fmaf(h[t], d.y, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(h[t], d.z, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(h[t], d.w, acc[4 * q + 3]);
      }
    }
#pragma unroll
    for (int c = 0; c < kVc; ++c) Gs[c * ldv + i] = acc[c];
  }
}

// X[j0 + t][col0 + c] += dxs[t][c]: the moves of a block's steps into X.
__device__ __forceinline__ void value_moves(float* X, int ld, int col0, int j0, int cnt, const float* dxs, int tid,
                                            int nthr) {
  for (int e = tid; e < cnt * kVc; e += nthr) {
    const int t = e / kVc, c = e % kVc;
    X[(int64_t)(j0 + t) * ld + col0 + c] += dxs[e];
  }
}

template <int D>
__global__ void __launch_bounds__(kAmThreads, 3) am_value_kernel(const AmMeta meta, const int32_t* __restrict__ bt,
                                                                 const int32_t* __restrict__ keep, uint16_t* vp,
                                                                 float* ws, float* vc, unsigned* status) {
  extern __shared__ __align__(16) float am_smem[];
  constexpr int kCb = D / kVc;
  const AmUnit u = am_unit(meta, blockIdx.x / kCb, ws);
  const int col0 = (int)(blockIdx.x % kCb) * kVc;
  const int m = u.m;
  if (m <= 0) return;
  const int ldv = value_ld(m);
  float* dxs = am_smem;                                    // [2][32][kVc] moves of the last two blocks
  float* tiles = dxs + 2 * kDb * kVc;                      // [2][2][kTile]
  float* S = tiles + 4 * kTile;                            // [kVc] column scales
  float* Sx = S + kVc;                                     // [kVc] max |X0| (bits)
  int* moved = reinterpret_cast<int*>(Sx + kVc);           // [2] did that block move
  float* Gs = am_smem + kValueHead;                        // [kVc][ldv] gradient, column-major
  float* hdiag = Gs + kVc * ldv;                           // [m] 1 / H_jj (0 where H_jj <= 0)
  float* thrb = hdiag + m;                                 // [m] 2^-17 pi_j; +inf where H_jj <= 0
  const float* Hm = u.base + am_off_G(meta.R, u.ldE);
  const int64_t ld = u.ldE;
  const float* G0 = u.base + am_off_Bm(meta.R, meta.max_m, u.ldE, D);  // H X0 - Bm (row stride D)
  float* Xg = u.base + am_off_X(meta.R, meta.max_m, u.ldE, D);           // X, from X0 (row stride D)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i0 = warp * 4; i0 < m; i0 += kAmThreads / 8) {  // H_jj and pi_j, four rows per warp at a time
    float ps[4];
    row_sums4(Hm, ld, m, i0, ps);
    if (lane < 4 && i0 + lane < m) {
      const int i = i0 + lane;
      const float d = Hm[(int64_t)i * ld + i];
      const float p = lane == 0 ? ps[0] : lane == 1 ? ps[1] : lane == 2 ? ps[2] : ps[3];
      hdiag[i] = d > 0.0f ? 1.0f / d : 0.0f;
      thrb[i] = d > 0.0f ? kAmGuard * p : INFINITY;
    }
  }
  {  // the starting gradient: H X0 - (Bm's first row range) in Bm's place, minus its other ranges in order
    const float* Bp = u.base + am_off_Bp(meta.R, meta.max_m, u.ldE, D);
    const int64_t bp_stride = (int64_t)meta.max_m * D;
    static_assert(kAmBmParts == 4, "three more row ranges at most, loaded side by side below");
    const int np = meta.bm_parts;
    for (int e = threadIdx.x; e < m * kVc; e += kAmThreads) {
      const int i = e / kVc, c = e % kVc;
      const int64_t o = (int64_t)i * D + col0 + c;
      const float g0 = G0[o];
      const float b1 = np > 1 ? Bp[o] : 0.0f;
      const float b2 = np > 2 ? Bp[bp_stride + o] : 0.0f;
      const float b3 = np > 3 ? Bp[2 * bp_stride + o] : 0.0f;
      Gs[c * ldv + i] = ((g0 - b1) - b2) - b3;
    }
  }
  if (threadIdx.x < 2 * kVc) S[threadIdx.x] = 0.0f;  // S: max |Y| bits, Sx: max |X0| bits
  if (threadIdx.x < 2) moved[threadIdx.x] = 0;
  __syncthreads();
  {
    const int c = threadIdx.x % kVc;
    const float* Y = u.base + am_off_Y(meta.R, meta.max_m, u.ldE);
    float ym = 0.0f, xm = 0.0f;
    for (int i = threadIdx.x / kVc; i < meta.R; i += kAmThreads / kVc)
      ym = fmaxf(ym, fabsf(Y[(int64_t)i * D + col0 + c]));
    for (int j = threadIdx.x / kVc; j < m; j += kAmThreads / kVc)
      xm = fmaxf(xm, fabsf(Xg[(int64_t)j * D + col0 + c]));
    atomicMax(reinterpret_cast<int*>(S) + c, __float_as_int(ym));  // non-negative floats order as ints
    atomicMax(reinterpret_cast<int*>(Sx) + c, __float_as_int(xm));
  }
  __syncthreads();
  if (threadIdx.x < kVc) S[threadIdx.x] += Sx[threadIdx.x];
  const int nb = (m + kDb - 1) / kDb;
  stage_tile(tiles, Hm, ld, 0, min(kDb, m), 0, min(kDb, m), threadIdx.x, kAmThreads);  // block 0's diagonal
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  const int64_t iters = (int64_t)meta.sweeps * nb;
  int jp = 0, cntp = 0;  // the previous block
  int64_t it = 0;
  for (; it < iters; ++it) {
    const int cur = (int)(it & 1), prev = cur ^ 1;
    const int j0 = (int)(it % nb) * kDb, cnt = min(kDb, m - j0);
    const float* dtile = tiles + cur * 2 * kTile;  // diag[t][k] = H[j0 + t][j0 + k]
    const float* ctile = dtile + kTile;            // cross[t][k] = H[jp + t][j0 + k]
    if (j0 == 0 && moved[prev] == 0) {
      // A sweep starts with every gradient entry current.  If no coordinate
      // would move in any column, none ever will: the fixed point is reached.
      bool would = false;
      for (int e = threadIdx.x; e < m * kVc; e += kAmThreads) {
        const int i = e % m, c = e / m;
        const float gi = Gs[c * ldv + i];
        would |= fabsf(gi) > thrb[i] * S[c] && -gi * hdiag[i] != 0.0f;
      }
      if (!__syncthreads_or(would)) break;
    }
    float* dxc = dxs + cur * kDb * kVc;
    const float* dxp = dxs + prev * kDb * kVc;
    if (warp == 0) {
      bar_sync_n(1, kAmThreads);  // the block's rows have the previous block's moves
      const int c = lane & (kVc - 1);
      const float Sc = S[c];
      float gv[kDb];
#pragma unroll
      for (int t = 0; t < kDb; ++t) gv[t] = t < cnt ? Gs[c * ldv + j0 + t] : 0.0f;
      // If no step of the block would move any column on the gradient as it
      // stands, none moves at all (a step that does not move changes nothing).
      bool would = false;
#pragma unroll
      for (int t = 0; t < kDb; ++t)
        if (t < cnt) would |= fabsf(gv[t]) > thrb[j0 + t] * Sc && -gv[t] * hdiag[j0 + t] != 0.0f;
      const bool steps = __any_sync(0xffffffffu, would);
      bool mv = false;
#pragma unroll
      for (int t = 0; t < kDb; ++t) {
        if (!steps) break;
        float dl = 0.0f;
        if (t < cnt) {
          const float gt = gv[t];
          dl = fabsf(gt) > thrb[j0 + t] * Sc ? -gt * hdiag[j0 + t] : 0.0f;
          if (__any_sync(0xffffffffu, dl != 0.0f)) {
            mv = true;
            const float4* t4 = reinterpret_cast<const float4*>(dtile + t * kTileLd);
#pragma unroll
            for (int q = 0; q < kDb / 4; ++q) {
              const float4 h = t4[q];
              gv[4 * q + 0] = fmaf(h.x, dl, gv[4 * q + 0]);
              gv[4 * q + 1] = fmaf(h.y, dl, gv[4 * q + 1]);
              gv[4 * q + 2] = fmaf(h.z, dl, gv[4 * q + 2]);
              gv[4 * q + 3] = fmaf(h.w, dl, gv[4 * q + 3]);
            }
          }
        }
        if (lane < kVc) dxc[t * kVc + c] = dl;
      }
      if (lane < kVc && steps) {
#pragma unroll
        for (int t = 0; t < kDb; ++t)
          if (t < cnt) Gs[c * ldv + j0 + t] = gv[t];
      }
      if (lane == 0) moved[cur] = mv ? 1 : 0;
    } else {
      const int tid = threadIdx.x - 32;
      const bool mvp = moved[prev] != 0;
      const bool apply = mvp && nb > 1;
      if (apply && warp <= kVc / 4 && lane < cnt) {  // the block's own rows, four columns per warp
        const int c0 = (warp - 1) * 4;
        float acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = Gs[(c0 + q) * ldv + j0 + lane];
        for (int t = 0; t < cntp; ++t) {
          const float h = ctile[t * kTileLd + lane];
          const float4 d = *reinterpret_cast<const float4*>(dxp + t * kVc + c0);
          acc[0] = fmaf(h, d.x, acc[0]);
          acc[1] = fmaf(h, d.y, acc[1]);
          acc[2] = fmaf(h, d.z, acc[2]);
          acc[3] = fmaf(h, d.w, acc[3]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) Gs[(c0 + q) * ldv + j0 + lane] = acc[q];
      }
      bar_arrive_n(1, kAmThreads);
      if (mvp) value_moves(Xg, D, col0, jp, cntp, dxp, tid, kHelpers);
      if (apply) value_update(Hm, ld, m, ldv, jp, cntp, dxp, Gs, jp, jp + cntp, j0, j0 + cnt, tid, kHelpers);
      if (it + 1 < iters) {  // the next block's tiles
        const int jn = (int)((it + 1) % nb) * kDb, cntn = min(kDb, m - jn);
        float* nt = tiles + prev * 2 * kTile;
        stage_tile(nt, Hm, ld, jn, cntn, jn, cntn, tid, kHelpers);
        stage_tile(nt + kTile, Hm, ld, j0, cnt, jn, cntn, tid, kHelpers);
        cp_async_commit();
        cp_async_wait_all();
      }
    }
    jp = j0;
    cntp = cnt;
    __syncthreads();
  }
  if (it > 0 && moved[(it - 1) & 1])  // the last block's moves into X
    value_moves(Xg, D, col0, jp, cntp, dxs + ((it - 1) & 1) * kDb * kVc, threadIdx.x, kAmThreads);
  __syncthreads();
  const int64_t orow = ((int64_t)u.l * meta.H + u.h) * meta.Mtot + u.moff;
  for (int j = threadIdx.x; j < m; j += kAmThreads) {  // one kept entry (its 16 columns) per thread
    const int pos = am_kept(meta, u, keep, j, status);
    const int64_t row = pos < 0 ? -1 : am_row(meta, u, bt, pos, status);
    float x[kVc];
#pragma unroll
    for (int q = 0; q < kVc / 4; ++q) {  // X rows are 16-byte aligned (region and stride)
      const float4 v = *reinterpret_cast<const float4*>(Xg + (int64_t)j * D + col0 + 4 * q);
      x[4 * q] = v.x;
      x[4 * q + 1] = v.y;
      x[4 * q + 2] = v.z;
      x[4 * q + 3] = v.w;
    }
    if (vc != nullptr) {
#pragma unroll
      for (int c = 0; c < kVc; ++c) vc[(orow + j) * D + col0 + c] = x[c];
    }
    if (row >= 0) {  // bf16, round to nearest even; 32 bytes at a 32-byte boundary of the V row
      uint32_t b[kVc / 2];
#pragma unroll
      for (int c = 0; c < kVc / 2; ++c) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * c], x[2 * c + 1]);
        b[c] = *reinterpret_cast<const uint32_t*>(&h);
      }
      uint4* dst = reinterpret_cast<uint4*>(vp + row * D + col0);
      dst[0] = make_uint4(b[0], b[1], b[2], b[3]);
      dst[1] = make_uint4(b[4], b[5], b[6], b[7]);
    }
  }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D>
cudaError_t launch_am_d(const AmLaunch& al, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !attr_set[dev]) {
    if ((e = set_smem(am_targets_tc_kernel<D>, tc_smem_bytes<D>())) != cudaSuccess) return e;
    if ((e = set_smem(am_atb_tc_kernel, kTbSmem)) != cudaSuccess) return e;
    if ((e = set_smem(am_mass_kernel, mass_smem_bytes(kAmMaxM))) != cudaSuccess) return e;
    if ((e = set_smem(am_value_kernel<D>, value_smem_bytes(kAmMaxM))) != cudaSuccess) return e;
    if (dev < 64) attr_set[dev] = true;
  }
  uint16_t* vp = static_cast<uint16_t*>(al.v_pool);
  auto check = [&]() {
    count_launch();
    return cudaGetLastError();
  };
  for (size_t ci = 0; ci < al.chunks; ++ci) {
    const AmMeta& m = al.meta[ci];
    if (m.units <= 0) continue;
    const int rbt = (m.R + kTcRows - 1) / kTcRows;
    am_targets_tc_kernel<D><<<(unsigned)(m.units * rbt), kTcThreads, tc_smem_bytes<D>(), stream>>>(
        *al.tmK, *al.tmVpool, *al.tmQ, m, al.block_table, al.keep, al.lse_rows, al.ws, al.status);
    if ((e = check()) != cudaSuccess) return e;
    am_x0_kernel<D><<<(unsigned)(m.units * ((m.max_m + 7) / 8)), kAmThreads, 0, stream>>>(
        m, al.block_table, al.keep, vp, al.ws, al.status);
    if ((e = check()) != cudaSuccess) return e;
    const int g0 = atb_blocks_per_unit(0, m.max_m, D), g1 = atb_blocks_per_unit(1, m.max_m, D);
    const int g2 = atb_blocks_per_unit(2, m.max_m, D), g3 = atb_blocks_per_unit(3, m.max_m, D);
    const int64_t nb0 = m.units * g0, nb1 = m.units * g1, nb2 = m.units * g2 * m.bm_parts, nb3 = m.units * g3;
    am_atb_tc_kernel<<<(unsigned)nb0, kTbThreads, kTbSmem, stream>>>(al.tmX[ci], al.tmX[ci], m, al.ws, 0, g0, nb0,
                                                                     0, al.status);
    if ((e = check()) != cudaSuccess) return e;
    am_mass_kernel<<<(unsigned)m.units, kAmThreads, mass_smem_bytes(m.max_m), stream>>>(
        m, al.block_table, al.keep, al.ws, al.aux, al.beta, al.status);
    if ((e = check()) != cudaSuccess) return e;
    am_probs_kernel<<<(unsigned)(m.units * ((m.R + 7) / 8)), kAmThreads, 0, stream>>>(m, al.ws);
    if ((e = check()) != cudaSuccess) return e;
    // H = Ph^T Ph and Bm = Ph^T Y in one launch (mode 1 never reads B): Bm's
    // row-range blocks fill the SMs the blocks of H leave idle
    am_atb_tc_kernel<<<(unsigned)(nb1 + nb2), kTbThreads, kTbSmem, stream>>>(al.tmX[ci], al.tmY[ci], m, al.ws, 1,
                                                                             g1, nb1, g2, al.status);
    if ((e = check()) != cudaSuccess) return e;
    am_atb_tc_kernel<<<(unsigned)nb3, kTbThreads, kTbSmem, stream>>>(al.tmH[ci], al.tmX0[ci], m, al.ws, 3, g3, nb3,
                                                                     0, al.status);
    if ((e = check()) != cudaSuccess) return e;
    am_value_kernel<D><<<(unsigned)(m.units * (D / kVc)), kAmThreads, value_smem_bytes(m.max_m), stream>>>(
        m, al.block_table, al.keep, vp, al.ws, al.vc, al.status);
    if ((e = check()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_am(const AmLaunch& al, cudaStream_t stream) {
  if (al.chunks == 0) return cudaSuccess;
  return al.meta[0].d == 64 ? launch_am_d<64>(al, stream) : launch_am_d<128>(al, stream);
}

}  // namespace kvc
