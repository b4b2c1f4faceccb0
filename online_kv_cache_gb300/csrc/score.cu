// score.cu -- two-pass proxy-query attention-mass scoring on tcgen05 tensor cores.
//
// What it computes (token-eviction score of "Practical Online KV Cache
// Compaction for LLM Agents", design-space section; LSE recovery of the ActKV
// analysis page, system-engineering paragraph), per unit (sequence b, layer l,
// KV head h) with proxy rows q_i (i < R) and segment keys k_j (j < n):
//   LSE_i = log sum_j exp(scale q_i.k_j)
//   s_j   = sqrt((1/R) sum_i exp(2 (scale q_i.k_j - LSE_i)))
//
// Both passes share one persistent, warp-specialised skeleton (one CTA per SM):
//   warp 0      producer: loads the row group of Q and streams 128-key K
//               tiles through a ring, gathered page by page through the block
//               table with 2-D TMA (the block-table entries arrive kPageRing - 1
//               tiles ahead through cp.async)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2, 3  idle (they complete warpgroup 0, which hands its registers to
//               the epilogue through setmaxnreg)
//   warps 4..11 two epilogue warpgroups; they take the MMA jobs alternately
//               and drain the TMEM accumulator slots round robin
// A work item is (unit, row group, key range).  Each K tile yields one MMA job
// per 128-row tile (pass 1) or per W-row chunk (pass 2) of the group.
//
// Pass 1 (lse pass):   D[128 rows x 128 keys] = Q_tile K_tile^T; per row a
//                      running (offset, sum) in the log2 domain, the offset
//                      raised only when a tile would overflow the sum; each
//                      warpgroup writes one partial per (item, row).
// Combine:             merges the partials of a row into the pass-2 offset
//                      nob_i = kBias - pw log2 sum_j 2^(c q_i.k_j)  (c = scale log2 e).
// Pass 2 (alpha pass): D[128 keys x W rows] = K_tile Q_chunk^T; every TMEM lane
//                      is one key, so sum_i 2^(pw c L_ij + nob_i) = 2^kBias sum_i
//                      alpha_ij^pw is a per-thread running sum; with pw = 2 the
//                      score s_j = sqrt(sum/R) 2^(-kBias/2), with pw = 1 the
//                      action attention a_j = sum 2^(-kBias) (the attention all
//                      rows pay to key j, "ActKV 解剖", first component); or a
//                      per-group partial sum when R spans several row groups
//                      (finished by score_finalize).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int kTile = 128;          // keys per K tile, rows per Q tile
constexpr float kBias = 100.0f;     // alpha^2 is accumulated as alpha^2 * 2^kBias
constexpr float kLog2e = 1.4426950408889634f;
// 12 warps: warpgroup 0 = producer, MMA issuer and two idle warps; warpgroups
// 1 and 2 = epilogue.  After the start-up barrier warpgroup 0 gives registers
// to the epilogue: 4 x 32 x kRegsControl + 8 x 32 x kRegsEpilogue equals the
// launch allocation of 384 threads x kRegsLaunch (the host checks the kernel
// was built with kRegsLaunch registers before the first launch).
constexpr int kThreads = 384;
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 72;
constexpr int kRegsEpilogue = 216;
static_assert(128 * kRegsControl + 256 * kRegsEpilogue == kThreads * kRegsLaunch, "register split");
constexpr int kMaxKStages = 8;
constexpr int kPageRing = 8;        // key tiles whose block-table entries are in flight
constexpr int kPagesPerTileMax = 16; // 128 keys in pages of >= 8 slots

template <int D>
struct Cfg {
  static constexpr int KB = D / 64;                 // 128-byte k-blocks per row
  static constexpr int kTileBytes = kTile * D * 2;  // one 128-row operand tile
  static constexpr int kKbBytes = kTile * 128;      // one k-block of a 128-row Q tile
  // K tiles: 1024-byte atoms (8 rows x one k-block) ordered (row group, k-block)
  static constexpr int kKGroup = KB * 1024;          // stride between 8-key row groups
  static constexpr int kKPageBytesPerRow = D * 2;    // a page of P keys fills P * D * 2 bytes
};

struct Unit {
  int b, l, h, g;
  int s0, n;
  int64_t off;
};

struct Item {
  Unit u;
  int t0, t1;  // key tiles [t0, t1)
  int J;       // jobs per K tile (row tiles or chunks of this row group)
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// item -> (unit, row group, key range).  Order: split fastest, then group, head, layer.
// `rev`: items are taken from the end of the launch's list (the alpha pass
// does this: the companion LSE pass ended on the last units, so their keys
// are still in L2 when the alpha pass starts on them).
__device__ __forceinline__ Item decode_item(const LaunchMeta& meta, int64_t item, int total_sub, bool rev) {
  Item it;
  if (rev) item = meta.items - 1 - item;
  const int si = find_seq(meta, item);
  const SeqMeta& s = meta.seq[si];
  // 32-bit arithmetic: a sequence owns fewer than 2^32 items of a launch, and the
  // 64-bit divisions cost the MMA issuer ~0.5 us at every item boundary
  uint32_t local = (uint32_t)(item - s.item0);
  const uint32_t split = (uint32_t)s.split;
  const uint32_t sp = local % split;
  local /= split;
  it.u.g = (int)(local % (uint32_t)meta.ngroups);
  local /= (uint32_t)meta.ngroups;
  it.u.h = (int)(local % (uint32_t)meta.H);
  it.u.l = (int)(local / (uint32_t)meta.H);
  it.u.b = s.b;
  it.u.s0 = s.s0;
  it.u.n = s.n;
  it.u.off = s.off;
  const uint32_t T = ((uint32_t)s.n + kTile - 1) / kTile;
  if (T < 46341u) {  // (sp + 1) * T < 2^31
    it.t0 = (int)(sp * T / split);
    it.t1 = (int)((sp + 1) * T / split);
  } else {
    it.t0 = (int)((uint64_t)sp * T / split);
    it.t1 = (int)((uint64_t)(sp + 1) * T / split);
  }
  it.J = min(meta.gsub, total_sub - it.u.g * meta.gsub);
  return it;
}

// sum_jj 2^(c v_jj - m) over one TMEM row of a key tile (masked keys hold -inf).
__device__ __forceinline__ float tile_exp2_sum(const float (&v)[kTile], float c, float m) {
  const float2 cc = make_float2(c, c), nm = make_float2(-m, -m);
  float2 a0 = make_float2(0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
#pragma unroll
  for (int jj = 0; jj < kTile; jj += 8) {
    const float2 x0 = __ffma2_rn(make_float2(v[jj + 0], v[jj + 1]), cc, nm);
    const float2 x1 = __ffma2_rn(make_float2(v[jj + 2], v[jj + 3]), cc, nm);
    const float2 x2 = __ffma2_rn(make_float2(v[jj + 4], v[jj + 5]), cc, nm);
    const float2 x3 = __ffma2_rn(make_float2(v[jj + 6], v[jj + 7]), cc, nm);
    a0 = __fadd2_rn(a0, make_float2(ex2_approx(x0.x), ex2_approx(x0.y)));
    a1 = __fadd2_rn(a1, make_float2(ex2_approx(x1.x), ex2_approx(x1.y)));
    a2 = __fadd2_rn(a2, make_float2(ex2_approx(x2.x), ex2_approx(x2.y)));
    a3 = __fadd2_rn(a3, make_float2(ex2_approx(x3.x), ex2_approx(x3.y)));
  }
  const float2 s01 = __fadd2_rn(a0, a1), s23 = __fadd2_rn(a2, a3);
  return (s01.x + s01.y) + (s23.x + s23.y);
}

// Pass-2 accumulation over up to 128 columns of a key's TMEM row:
// acc += sum_col 2^(2c L_col + nob_col) for the first min(ncol, 128) columns
// (ncol a multiple of 8; ob 32-byte aligned, read 8 offsets per load).
__device__ __forceinline__ void alpha2_cols(const float (&v)[128], const float* __restrict__ ob, int ncol,
                                            float2 c2, float2 (&acc2)[2]) {
#pragma unroll
  for (int jj = 0; jj < 128; jj += 8) {
    if (ncol >= 128 || jj < ncol) {
      float o[8];
      ldg_nc_v8(ob + jj, o);
      const float2 x0 = __ffma2_rn(make_float2(v[jj + 0], v[jj + 1]), c2, make_float2(o[0], o[1]));
      const float2 x1 = __ffma2_rn(make_float2(v[jj + 2], v[jj + 3]), c2, make_float2(o[2], o[3]));
      const float2 x2 = __ffma2_rn(make_float2(v[jj + 4], v[jj + 5]), c2, make_float2(o[4], o[5]));
      const float2 x3 = __ffma2_rn(make_float2(v[jj + 6], v[jj + 7]), c2, make_float2(o[6], o[7]));
      acc2[0] = __fadd2_rn(acc2[0], make_float2(ex2_approx(x0.x), ex2_approx(x0.y)));
      acc2[1] = __fadd2_rn(acc2[1], make_float2(ex2_approx(x1.x), ex2_approx(x1.y)));
      acc2[0] = __fadd2_rn(acc2[0], make_float2(ex2_approx(x2.x), ex2_approx(x2.y)));
      acc2[1] = __fadd2_rn(acc2[1], make_float2(ex2_approx(x3.x), ex2_approx(x3.y)));
    }
  }
}

// ============================================================== skeleton

// PASS 1: A = Q row tile (M = 128 rows) read from TMEM, B = K tile (N = 128
//         keys).  At the start of each item the group's row tiles pass through
//         a two-buffer shared-memory staging ring and tcgen05.cp copies them
//         into TMEM columns 256..511, so the MMAs fetch only B from shared memory.
// PASS 2: A = K tile (M = 128 keys), B = Q chunk (N = W rows), both from shared
//         memory (the Q group stays resident there).
// Jobs run tile by tile: for each K tile, one job per row tile / chunk of the
// group; job number jc (counted over the CTA's whole run) goes to warpgroup
// jc & 1 and to TMEM accumulator slot jc % nslots.  Slots are 128 columns wide
// (256 in pass 2 when W > 128) and fill the columns pass 1's resident Q leaves
// free, so small row groups get three or four slots and a deeper
// MMA -> epilogue pipeline.  Only one K tile is in use at a time, so a ring of
// kst tiles keeps kst - 1 tiles in flight.  The block-table entries of the
// next kPageRing - 1 tiles travel ahead of the K ring through cp.async into a
// shared-memory ring, so no TMA issue waits on a global load.
// PW (pass 2): the power of alpha summed per key -- 2 for the eviction score,
// 1 for the action attention (a compile-time constant: the pass-2 epilogue
// is sensitive to every instruction of its inner loop).
template <int D, int PASS, int PW = 2>
__global__ void __launch_bounds__(kThreads, 1)
    score_pass_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ LaunchMeta meta, const int32_t* __restrict__ block_table,
                      float2* __restrict__ part1, const float* __restrict__ nob,
                      float* __restrict__ out2, unsigned* status) {
  using C = Cfg<D>;
  constexpr uint32_t kQTmemCols = D / 2;          // TMEM columns per 128-row Q tile
  // TMEM: accumulator slots from column 0; pass 1 keeps its Q row tiles at the top
  const uint32_t slot_cols = (PASS == 1 || meta.W <= 128) ? 128u : 256u;
  const uint32_t q_col0 = (PASS == 1) ? 512u - (uint32_t)meta.gsub * kQTmemCols : 512u;
  const uint32_t nslots = min(4u, q_col0 / slot_cols);
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // [barriers | TMEM address, abort flag | reduction buffer | page ring][pad to 1024][Q group][K ring]
  const int kst = meta.kst;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
  uint8_t* sQ = align1024(smem_raw + kScoreSmemHead);
  uint8_t* sK = sQ + meta.qbytes;
  uint64_t* q_full = bars;               // [4] one per row tile / chunk of the group
  uint64_t* q_empty = bars + 4;          // [4]
  uint64_t* k_full = bars + 8;           // [kMaxKStages]
  uint64_t* k_empty = k_full + kMaxKStages;
  uint64_t* t_full = k_empty + kMaxKStages;  // [4] TMEM slots
  uint64_t* t_empty = t_full + 4;
  uint64_t* drain = t_empty + 4;         // pass 1: all MMAs of the previous item done
  uint64_t* red_full = drain + 1;        // [2] pass 2: a tile's other share is in `red`
  uint64_t* red_empty = red_full + 2;    // [2] pass 2: `red` may be written again
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + 384);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // limit of every wait between the roles (the abort drains keep the default)
  const unsigned long long wait_ns = meta.stall_ns > 0 ? (unsigned long long)meta.stall_ns : kWaitLimitNs;
  float* red = reinterpret_cast<float*>(smem_raw + 512);           // [2 parity][128] (pass 2)
  int32_t* page_ring = reinterpret_cast<int32_t*>(smem_raw + 1536);  // [kPageRing][16]

  const int total_sub = (PASS == 1) ? meta.rowtiles : meta.nchunks;
  const int sub_rows = (PASS == 1) ? kTile : meta.W;  // Q rows per job
  const uint32_t sub_bytes = (uint32_t)(C::KB * sub_rows * 128);
  // pass 1: staging buffers for Q sub-tiles on their way to TMEM (2, or 4 when
  // items are short and a whole row group is prefetched during the previous item)
  const uint32_t qst = (PASS == 1) ? (uint32_t)meta.qbytes / sub_bytes : 4u;
  const uint32_t qsh = qst == 4u ? 2u : 1u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1); }
    for (int i = 0; i < kMaxKStages; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    for (int i = 0; i < 4; ++i) { mbar_init(&t_full[i], 1); mbar_init(&t_empty[i], 4); }  // 4 warps
    mbar_init(drain, 1);
    for (int i = 0; i < 2; ++i) { mbar_init(&red_full[i], 4); mbar_init(&red_empty[i], 4); }  // 4 warps
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

  if (warp < 4) {
    setmaxnreg_dec<kRegsControl>();
  if (warp == 0) {
    // ---------------------------------------------------------- producer (whole warp)
    // Load order per item: its first min(kst-1, tiles) K tiles, then its Q group
    // (sub-tile by sub-tile as the previous item releases them), then the rest.
    uint32_t kcount = 0, q_use[4] = {0, 0, 0, 0}, qc = 0;
    int pks = 0;        // K ring stage of the next tile and its phase parity
    uint32_t pkph = 0;
    bool ok = true;
    const int ppt = kTile / meta.P;  // pages per key tile (<= kPagesPerTileMax)
    // Page-ring cursor: one commit group per key tile of this CTA, in K order;
    // lane p < ppt copies the block-table entry of page p of the tile.
    int64_t pf_item = blockIdx.x;
    Item pf = pf_item < meta.items ? decode_item(meta, pf_item, total_sub, PASS == 2) : Item{};
    int pf_t = pf.t0;
    uint32_t pf_count = 0;
    auto page_prefetch = [&]() {
      if (pf_item < meta.items) {
        const int slot = pf_t * kTile + lane * meta.P;
        if (lane < ppt && slot < pf.u.n)
          cp_async_4(page_ring + (pf_count % kPageRing) * kPagesPerTileMax + lane,
                     block_table + (int64_t)pf.u.b * meta.max_blocks + (pf.u.s0 + slot) / meta.P);
        if (++pf_t >= pf.t1) {
          pf_item += gridDim.x;
          if (pf_item < meta.items) {
            pf = decode_item(meta, pf_item, total_sub, PASS == 2);
            pf_t = pf.t0;
          }
        }
      }
      cp_async_commit();
      ++pf_count;
    };
    for (int i = 0; i < kPageRing - 1; ++i) page_prefetch();

    int64_t k_item = blockIdx.x, q_item = blockIdx.x;
    Item kit_ = k_item < meta.items ? decode_item(meta, k_item, total_sub, PASS == 2) : Item{};
    int kt = kit_.t0;

    while (ok && (k_item < meta.items || q_item < meta.items)) {
      const int pre = min(kst - 1, kit_.t1 - kit_.t0);
      // Q of item q_item goes after that item's first `pre` K tiles (or at once
      // when the K cursor has already passed them)
      bool do_q = q_item < meta.items &&
                  (q_item < k_item || k_item >= meta.items ||
                   (q_item == k_item && kt >= kit_.t0 + pre));
      if (PASS == 1 && qst == 4u && !do_q && q_item == k_item + gridDim.x) {
        // a whole row group is staged: the next item's Q goes as soon as its
        // buffers are free (tested, not waited for, so K keeps flowing)
        unsigned fr = 0;
        if (lane == 0) fr = mbar_try_wait(&q_empty[qc & 3u], ((qc >> 2) & 1u) ^ 1u) ? 1u : 0u;
        do_q = __shfl_sync(0xffffffffu, fr, 0) != 0u;
      }
      if (do_q) {
        const Item qi = decode_item(meta, q_item, total_sub, PASS == 2);
        const int qrow = ((qi.u.b * meta.L + qi.u.l) * meta.H + qi.u.h) * meta.R +
                         qi.u.g * meta.gsub * sub_rows;
        // stall_ns > 0 (failure-path test): no proxy-row load is issued, so the
        // MMA role's wait for them can only run out
        for (int j = 0; j < qi.J && ok && meta.stall_ns == 0; ++j) {
          // pass 1: staging buffer qc % 2; pass 2: the group's own sub-tile slot j
          const int qs = (PASS == 1) ? (int)(qc & (qst - 1)) : j;
          const uint32_t qpar = (PASS == 1) ? ((qc >> qsh) & 1) : (q_use[j] & 1);
          if (lane == 0) {
            ok = mbar_wait(&q_empty[qs], qpar ^ 1, abort_flag, status, wait_ns);
            if (ok) mbar_arrive_expect_tx(&q_full[qs], sub_bytes);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;  // only issued loads are counted: the abort drain waits for them
          if (lane < C::KB)  // lane kb: k-block kb of the sub-tile
            tma_load_2d(sQ + (qs * C::KB + lane) * sub_rows * 128, &tmQ, &q_full[qs], lane * 64,
                        qrow + j * sub_rows);
          ++q_use[j];
          ++qc;
        }
        q_item += gridDim.x;
        continue;
      }
      // page rows of key tile kt (its ring entry was committed kPageRing - 1 groups ago)
      page_prefetch();
      cp_async_wait_group<kPageRing - 1>();
      int32_t prow = -1;
      if (lane < ppt && kt * kTile + lane * meta.P < kit_.u.n) {
        const int32_t page = page_ring[(kcount % kPageRing) * kPagesPerTileMax + lane];
        if (page < 0 || page >= meta.num_pages)
          atomicOr(status, KVC_DEV_BAD_PAGE);  // outside the pool: reported, not read
        else
          prow = ((kit_.u.l * meta.num_pages + page) * meta.H + kit_.u.h) * meta.P;
      }

      const int ks = pks;
      if (lane == 0) ok = mbar_wait(&k_empty[ks], pkph ^ 1u, abort_flag, status, wait_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const unsigned valid = __ballot_sync(0xffffffffu, prow >= 0);
      if (lane == 0) mbar_arrive_expect_tx(&k_full[ks], __popc(valid) * C::KB * meta.P * 128);
      __syncwarp();
      // Lane p copies page p of the tile (its P keys, every k-block) and all the
      // lanes issue in one instruction: a single issuing lane tops out near
      // 2.6 TB/s of 4 KB pages on the whole GPU, one page per lane near 5.5 TB/s.
      if (prow >= 0)
        tma_load_4d(sK + ks * C::kTileBytes + lane * meta.P * C::kKPageBytesPerRow, &tmK, &k_full[ks], 0, 0, 0,
                    prow >> 3);
      ++kcount;
      if (++pks == kst) {
        pks = 0;
        pkph ^= 1u;
      }
      if (++kt >= kit_.t1) {
        k_item += gridDim.x;
        if (k_item < meta.items) {
          kit_ = decode_item(meta, k_item, total_sub, PASS == 2);
          kt = kit_.t0;
        }
      }
    }
    cp_async_wait_all();  // no page copy outlives the CTA
    // Let the last copies issued land before the CTA exits, whether this role
    // or another gave up (in a normal run they have landed or are about to:
    // completion does not depend on any consumer).
    if (lane == 0) {
      for (uint32_t j = (kcount > (uint32_t)kst ? kcount - kst : 0); j < kcount; ++j)
        mbar_wait(&k_full[j % kst], (j / kst) & 1, nullptr, status);
      if (PASS == 1) {
        for (uint32_t j = (qc > qst ? qc - qst : 0); j < qc; ++j)
          mbar_wait(&q_full[j & (qst - 1)], (j >> qsh) & 1, nullptr, status);
      } else {
        for (int j = 0; j < 4; ++j)
          if (q_use[j] > 0) mbar_wait(&q_full[j], (q_use[j] - 1) & 1, nullptr, status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // One thread issues every MMA; its loop is on the critical path for short
    // jobs, so descriptors are built once per tile and stepped along K by adding
    // the 16-byte-unit offset of each k-step to the start-address field.
    if (lane == 0) {
      const uint32_t idesc = (PASS == 1) ? idesc_bf16_f32(kTile, kTile) : idesc_bf16_f32(kTile, meta.W);
      uint32_t q_use[4] = {0, 0, 0, 0};
      uint32_t slot = 0, use = 0;  // accumulator slot of the next job and its use count
      int ks = 0;                  // K ring stage of the next tile and its phase parity
      uint32_t kph = 0;
      uint32_t qc = 0, dc = 0;
      bool issued = false, ok = true;
      const uint32_t q_base = smem_u32(sQ);
      const uint64_t q_desc = sdesc_k_sw128(q_base);
      const uint32_t q_kb_step = (uint32_t)(sub_rows * 128) >> 4;  // one k-block of a Q sub-tile
      for (int64_t item = blockIdx.x; item < meta.items && ok; item += gridDim.x) {
        const Item it = decode_item(meta, item, total_sub, PASS == 2);
        if (PASS == 1) {
          // the previous item's MMAs read the TMEM copy of Q: let them finish
          if (issued) {
            mma_commit(drain);
            if (!(ok = mbar_wait(drain, dc & 1, abort_flag, status, wait_ns))) break;
            ++dc;
            tc_fence_after_sync();
          }
          // the group's Q sub-tiles into TMEM; the tensor pipe runs the copies and the
          // MMAs in issue order.  (Copying each sub-tile just before its first job was
          // measured slower: a copy then waits behind the epilogue's slot release.)
          for (int j = 0; j < it.J && ok; ++j) {
            const uint32_t qs = qc & (qst - 1);
            if (!(ok = mbar_wait(&q_full[qs], (qc >> qsh) & 1, abort_flag, status, wait_ns))) break;
            const uint64_t stage = q_desc + ((qs * sub_bytes) >> 4);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              tmem_cp_128x256b(tmem + q_col0 + j * kQTmemCols + k * 8,
                               stage + (((k >> 2) * C::kKbBytes + (k & 3) * 32) >> 4));
            mma_commit(&q_empty[qs]);  // staging buffer free once the copy is done
            issued = true;
            ++qc;
          }
        } else {
          for (int j = 0; j < it.J && ok; ++j) ok = mbar_wait(&q_full[j], q_use[j] & 1, abort_flag, status, wait_ns);
        }
        if (!ok) break;
        for (int t = it.t0; t < it.t1 && ok; ++t) {
          if (!(ok = mbar_wait(&k_full[ks], kph, abort_flag, status, wait_ns))) break;
          const uint64_t k_desc = sdesc_k_sw128(smem_u32(sK + ks * C::kTileBytes), C::kKGroup);
          for (int j = 0; j < it.J; ++j) {
            if (!(ok = mbar_wait(&t_empty[slot], (use & 1) ^ 1, abort_flag, status, wait_ns))) break;
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem + slot * slot_cols;
            if (PASS == 1) {
              const uint32_t a_tmem = tmem + q_col0 + j * kQTmemCols;
#pragma unroll
              for (int k = 0; k < D / 16; ++k)
                mma_bf16_tmem_a(d_tmem, a_tmem + k * 8, k_desc + (((k >> 2) * 1024 + (k & 3) * 32) >> 4),
                                idesc, k > 0);
            } else {
              const uint64_t qj = q_desc + ((j * sub_bytes) >> 4);
#pragma unroll
              for (int k = 0; k < D / 16; ++k)
                mma_bf16(d_tmem, k_desc + (((k >> 2) * 1024 + (k & 3) * 32) >> 4),
                         qj + (k >> 2) * q_kb_step + (k & 3) * 2, idesc, k > 0);
            }
            mma_commit(&t_full[slot]);
            if (PASS == 2 && t == it.t1 - 1) mma_commit(&q_empty[j]);  // last use of this Q sub-tile
            issued = true;
            if (++slot == nslots) {
              slot = 0;
              ++use;
            }
          }
          if (!ok) break;
          mma_commit(&k_empty[ks]);
          if (++ks == kst) {
            ks = 0;
            kph ^= 1u;
          }
        }
        for (int j = 0; j < it.J; ++j) ++q_use[j];
      }
      if (!ok && issued) {  // one more commit covers every copy and MMA issued
        mma_commit(drain);
        mbar_wait(drain, dc & 1, nullptr, status);
      }
    }
  }  // warps 2 and 3: nothing to do
  } else {
    setmaxnreg_inc<kRegsEpilogue>();
    // ---------------------------------------------------------- epilogue warpgroups
    const int wg = (warp - 4) >> 2;
    const int sub = warp & 3;  // TMEM lane quarter this warp may access
    const int r = sub * 32 + lane;  // TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(sub * 32) << 16);
    const float c = meta.scale * kLog2e;
    uint32_t jc = 0, red_count = 0;
    uint32_t slot = 0, use = 0;  // accumulator slot of job jc and its use count
    bool ok = true;
    for (int64_t item = blockIdx.x; item < meta.items && ok; item += gridDim.x) {
      const Item it = decode_item(meta, item, total_sub, PASS == 2);
      float m_run[4], s_run[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        m_run[j] = -INFINITY;
        s_run[j] = 0.0f;
      }
      const int64_t u = ((int64_t)it.u.b * meta.L + it.u.l) * meta.H + it.u.h;
      for (int t = it.t0; t < it.t1 && ok; ++t) {
        const int valid = min(kTile, it.u.n - t * kTile);
        float2 acc2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        bool mine = false;
#pragma unroll 1
        for (int j = 0; j < it.J; ++j, ++jc, slot = (slot + 1 == nslots) ? 0 : slot + 1,
                 use += (slot == 0)) {
          if ((int)(jc & 1) != wg) continue;
          mine = true;
          ok = mbar_wait(&t_full[slot], use & 1, abort_flag, status, wait_ns);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t taddr = t_lane + slot * slot_cols;
          float v[128];
          if (PASS == 1) {
            tmem_ld128(taddr, v);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&t_empty[slot]);  // the warp's 32 TMEM lanes are read
            if (valid < kTile) {
#pragma unroll
              for (int jj = 0; jj < kTile; ++jj)
                if (jj >= valid) v[jj] = -INFINITY;
            }
            float mprev = m_run[0], sprev = s_run[0];
#pragma unroll
            for (int q = 1; q < 4; ++q)
              if (j == q) {
                mprev = m_run[q];
                sprev = s_run[q];
              }
            // The row's offset need not be its running maximum: any finite offset
            // m gives the same sum * 2^m as long as no term overflows.  The first
            // tile of the item takes its first key's logit (never masked); a tile
            // whose sum stays at or below 2^64 (every logit at most ~64 above the
            // offset, ~500 q.k units at scale 1/sqrt(128)) adds to the row as it
            // stands, and only a tile above that (or inf/NaN) takes its exact
            // maximum and rescales.  The row's sum then stays below 2^77 over
            // 2^20 keys, and (offset, sum) merge like any pair in the combine.
            if (mprev == -INFINITY) mprev = v[0] * c;
            float mnew = mprev, snew;
            const float tile_sum = tile_exp2_sum(v, c, mprev);
            if (tile_sum <= 0x1p64f) {
              snew = sprev + tile_sum;
            } else {
              float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
              for (int jj = 0; jj < kTile; jj += 8) {
                mx0 = max3f(mx0, v[jj + 0], v[jj + 1]);
                mx1 = max3f(mx1, v[jj + 2], v[jj + 3]);
                mx2 = max3f(mx2, v[jj + 4], v[jj + 5]);
                mx3 = max3f(mx3, v[jj + 6], v[jj + 7]);
              }
              mnew = fmaxf(mprev, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c);
              snew = fmaf(sprev, ex2_approx(mprev - mnew), tile_exp2_sum(v, c, mnew));
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (j == q) {
                m_run[q] = mnew;
                s_run[q] = snew;
              }
          } else {
            const float2 c2 = make_float2((float)PW * c, (float)PW * c);
            const float* ob = nob + u * meta.R_pad + (it.u.g * meta.gsub + j) * meta.W;
            for (int col0 = 0; col0 < meta.W; col0 += 128) {
              tmem_ld128(taddr + col0, v);
              if (col0 + 128 >= meta.W) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&t_empty[slot]);
              }
              alpha2_cols(v, ob + col0, meta.W - col0, c2, acc2);
            }
          }
        }
        if (!ok) break;
        if (PASS == 2) {
          const float2 s2 = __fadd2_rn(acc2[0], acc2[1]);
          float acc = s2.x + s2.y;
          bool writer = mine;
          if (it.J > 1) {
            // Both warpgroups hold a share of this tile's rows.  The one that
            // drained the tile's last job (usually the later one) adds the
            // other's share from `red` and writes the score; the other never
            // waits except for `red` to be free again, two tiles later.
            const uint32_t par = red_count & 1, use = red_count >> 1;
            ++red_count;
            float* rb = red + par * kTile;
            writer = (wg == (int)((jc - 1) & 1));
            if (!writer) {
              ok = mbar_wait(&red_empty[par], (use & 1) ^ 1, abort_flag, status, wait_ns);
              if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
              }
              rb[r] = acc;
              __syncwarp();
              if (lane == 0) mbar_arrive(&red_full[par]);
            } else {
              ok = mbar_wait(&red_full[par], use & 1, abort_flag, status, wait_ns);
              if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
              }
              acc += rb[r];
              __syncwarp();
              if (lane == 0) mbar_arrive(&red_empty[par]);
            }
          }
          const int key = t * kTile + r;
          if (writer && key < it.u.n) {
            const int64_t o = ((int64_t)it.u.l * meta.H + it.u.h) * meta.Ntot + it.u.off + key;
            if (meta.ngroups == 1)
              out2[o] = (PW == 2) ? sqrtf(acc / (float)meta.R) * exp2f(-0.5f * kBias)
                                  : acc * exp2f(-kBias);
            else
              out2[(int64_t)it.u.g * meta.L * meta.H * meta.Ntot + o] = acc;
          }
        }
      }
      if (!ok) break;
      if (PASS == 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < it.J) part1[((item * 2 + wg) * 4 + j) * kTile + r] = make_float2(m_run[j], s_run[j]);
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

// ============================================================== combine / offsets

// Merges the pass-1 partials of each row into the pass-2 offset
// nob_i = kBias - pw log2 sum_j 2^(c L_ij) (rows >= R: -inf) and the natural-log
// LSE.  One thread per (unit, row); the items of the companion pass-1 launch
// start at seq.item1.
__global__ void lse_combine_kernel(const __grid_constant__ LaunchMeta meta,
                                   const float2* __restrict__ part, float* __restrict__ nob,
                                   float* __restrict__ lse_out, int ngroups1, int gsub1) {
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
      nob[u * meta.R_pad + i] = -INFINITY;  // padded rows contribute 2^-inf = 0
      continue;
    }
    const int rt = i / kTile, rr = i % kTile;
    const int grp = rt / gsub1, jj = rt % gsub1;
    const int64_t base = s.item1 + ((int64_t)(l * meta.H + h) * ngroups1 + grp) * s.split;
    float M = -INFINITY;
    for (int sp = 0; sp < s.split; ++sp)
      for (int w = 0; w < 2; ++w) M = fmaxf(M, part[(((base + sp) * 2 + w) * 4 + jj) * kTile + rr].x);
    float S = 0.0f;
    for (int sp = 0; sp < s.split; ++sp)
      for (int w = 0; w < 2; ++w) {
        const float2 p = part[(((base + sp) * 2 + w) * 4 + jj) * kTile + rr];
        if (p.y > 0.0f) S += p.y * exp2f(p.x - M);
      }
    const float lg = M + log2f(S);  // log2 sum_j 2^(c L_ij)
    nob[u * meta.R_pad + i] = kBias - meta.pw * lg;
    if (lse_out != nullptr) lse_out[u * meta.R + i] = lg * ln2;
  }
}

// Pass-2 offsets from a caller-supplied natural-log LSE (for instance the
// log-sum-exp the attention kernel produced for the same proxy queries).
__global__ void nob_from_lse_kernel(const __grid_constant__ LaunchMeta meta,
                                    const float* __restrict__ lse_in, float* __restrict__ nob) {
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
    nob[u * meta.R_pad + i] =
        (i < meta.R) ? kBias - meta.pw * kLog2e * lse_in[u * meta.R + i] : -INFINITY;
  }
}

// Scores from the per-row-group partial sums of pass 2 (R spanning several
// groups): s = sqrt(sum_g part_g / R) 2^(-kBias/2) (pw = 2) or the action
// attention sum_g part_g 2^(-kBias) (pw = 1).
__global__ void score_finalize_kernel(const __grid_constant__ LaunchMeta meta,
                                      const float* __restrict__ part2, float* __restrict__ scores) {
  const int64_t LHN = (int64_t)meta.L * meta.H * meta.Ntot;
  const float unbias = exp2f(-0.5f * kBias);
  const bool te = meta.pw == 2.0f;
  for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < LHN;
       g += (int64_t)gridDim.x * blockDim.x) {
    float acc = 0.0f;
    for (int q = 0; q < meta.ngroups; ++q) acc += part2[q * LHN + g];
    scores[g] = te ? sqrtf(acc / (float)meta.R) * unbias : acc * unbias * unbias;
  }
}

template <int D>
cudaError_t launch_score_d(const ScoreLaunch& sl, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    // the register split inside the kernel assumes this launch allocation; a
    // build with any other count is refused rather than launched
    const void* kernels[3] = {reinterpret_cast<const void*>(score_pass_kernel<D, 1>),
                              reinterpret_cast<const void*>(score_pass_kernel<D, 2, 2>),
                              reinterpret_cast<const void*>(score_pass_kernel<D, 2, 1>)};
    for (const void* k : kernels) {
      cudaFuncAttributes fa;
      if ((e = cudaFuncGetAttributes(&fa, k)) != cudaSuccess) return e;
      if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidKernelImage;
      if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kScoreSmemLimit)) !=
          cudaSuccess)
        return e;
    }
    attr_set[dev] = true;
  }
  for (size_t c = 0; c < sl.chunks; ++c) {
    const LaunchMeta& m1 = sl.pass1[c];
    if (sl.phases & kPhaseLse) {
      if (m1.items > 0) {
        const int grid = (int)std::min<int64_t>(m1.items, sl.grid_limit);
        const int smem = score_smem_bytes(m1.qbytes, m1.kst, D);
        score_pass_kernel<D, 1><<<grid, kThreads, smem, stream>>>(*sl.tmK, *sl.tmQ1, m1, sl.block_table,
                                                                  sl.part, nullptr, nullptr, sl.status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
      }
      const LaunchMeta& mc = sl.combine[c];
      if (mc.items > 0) {
        const int grid = (int)std::min<int64_t>((mc.items + 255) / 256, (int64_t)sl.num_sms * 8);
        lse_combine_kernel<<<grid, 256, 0, stream>>>(mc, sl.part, sl.obias, sl.lse_out, m1.ngroups,
                                                     m1.gsub);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
      }
    }
    if (sl.phases & kPhaseLseIn) {
      const LaunchMeta& mc = sl.combine[c];
      if (mc.items > 0) {
        const int grid = (int)std::min<int64_t>((mc.items + 255) / 256, (int64_t)sl.num_sms * 8);
        nob_from_lse_kernel<<<grid, 256, 0, stream>>>(mc, sl.lse_in, sl.obias);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
      }
    }
    if (sl.phases & kPhaseAlpha) {
      const LaunchMeta& m2 = sl.pass2[c];
      if (m2.items > 0) {
        const int grid = (int)std::min<int64_t>(m2.items, sl.grid_limit);
        const int smem = score_smem_bytes(m2.qbytes, m2.kst, D);
        float* out = (m2.ngroups == 1) ? sl.scores : sl.part2;
        if (m2.pw == 1.0f)
          score_pass_kernel<D, 2, 1><<<grid, kThreads, smem, stream>>>(*sl.tmK, *sl.tmQ2, m2, sl.block_table,
                                                                       nullptr, sl.obias, out, sl.status);
        else
          score_pass_kernel<D, 2, 2><<<grid, kThreads, smem, stream>>>(*sl.tmK, *sl.tmQ2, m2, sl.block_table,
                                                                       nullptr, sl.obias, out, sl.status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launch();
      }
    }
  }
  if ((sl.phases & kPhaseAlpha) && sl.chunks > 0 && sl.pass2[0].ngroups > 1) {
    const LaunchMeta& mf = sl.pass2[0];
    const int64_t n = (int64_t)mf.L * mf.H * mf.Ntot;
    const int grid = (int)std::min<int64_t>((n + 255) / 256, (int64_t)sl.num_sms * 8);
    score_finalize_kernel<<<grid, 256, 0, stream>>>(mf, sl.part2, sl.scores);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    count_launch();
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
