// internal.h -- host-side launch descriptions passed from the C-ABI front end
// (api.cu) to the kernel launchers (score.cu, select.cu, compact.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <vector>

#include "common.cuh"

namespace kvc {

// Counts kernel launches issued by the library (read by kvc_launch_count).
void count_launch();

enum ScorePhase : unsigned {
  kPhaseLse = 1,      // pass 1 + combine: per-row LSE -> pass-2 offsets (and lse_out)
  kPhaseLseIn = 2,    // pass-2 offsets from a caller-supplied LSE
  kPhaseAlpha = 4,    // pass 2: scores
};

// Dynamic shared memory of a scoring pass: the barrier block, up to 1024 B of
// alignment padding, the resident row group of Q and `kst` K tiles of 128 keys.
constexpr int kScoreSmemLimit = 232448;  // 227 KB per block on sm_103a
constexpr int kScoreSmemHead = 2048;     // barriers, TMEM address, reduction buffer, page ring
__host__ __device__ constexpr int score_smem_bytes(int qbytes, int kst, int d) {
  return kScoreSmemHead + 1024 + qbytes + kst * 128 * d * 2;
}

struct ScoreLaunch {
  unsigned phases = kPhaseLse | kPhaseAlpha;
  const float* lse_in = nullptr;       // [B][L][H][R] natural-log LSE (kPhaseLseIn)
  int d = 0;
  int num_sms = 0;
  int grid_limit = 0;                  // persistent CTAs per pass (<= num_sms)
  size_t chunks = 0;
  const LaunchMeta* pass1 = nullptr;   // [chunks]
  const LaunchMeta* combine = nullptr; // [chunks]
  const LaunchMeta* pass2 = nullptr;   // [chunks]
  const CUtensorMap* tmK = nullptr;    // K pool, box {64, P}
  const CUtensorMap* tmQ1 = nullptr;   // Q, box {64, 128}
  const CUtensorMap* tmQ2 = nullptr;   // Q, box {64, W}
  const int32_t* block_table = nullptr;
  float2* part = nullptr;              // pass-1 partials (workspace)
  float* part2 = nullptr;              // pass-2 per-row-group partial sums (workspace)
  float* obias = nullptr;              // per-row pass-2 offsets (workspace)
  float* lse_out = nullptr;
  float* scores = nullptr;
  unsigned* status = nullptr;
};

cudaError_t launch_score(const ScoreLaunch& sl, cudaStream_t stream);

struct SelectLaunch {
  int num_sms = 0;
  size_t chunks = 0;
  const LaunchMeta* meta = nullptr;    // [chunks]; one item per (seq, l, h)
  const float* scores = nullptr;
  int32_t* keep = nullptr;
  unsigned* status = nullptr;
};

cudaError_t launch_select(const SelectLaunch& sl, cudaStream_t stream);

struct CompactLaunch {
  int num_sms = 0;
  size_t chunks = 0;
  const LaunchMeta* plan_meta = nullptr;  // [chunks]; items: (seq, l, h, hole block)
  const LaunchMeta* rows_meta = nullptr;  // [chunks]; items: (seq, block-table block)
  const LaunchMeta* copy_meta = nullptr;  // [chunks]; items: (l, h, seq, move)
  const LaunchMeta* free_meta = nullptr;  // [chunks]
  const int32_t* block_table = nullptr;
  int32_t* block_table_mut = nullptr;
  int32_t* nblocks = nullptr;
  const int32_t* keep = nullptr;
  void* k_pool = nullptr;
  void* v_pool = nullptr;
  int32_t* tags = nullptr;
  float* aux = nullptr;  // per-slot state moved with the tags, or null
  int32_t* moves = nullptr;
  int32_t* move_count = nullptr;
  int32_t* dead = nullptr;
  int32_t* dead_count = nullptr;
  int32_t* freed = nullptr;
  int32_t* new_rows = nullptr;
  int32_t* free_ids = nullptr;
  int32_t* free_top = nullptr;
  int32_t capacity = 0;
  unsigned* status = nullptr;
};

// Layout variants of eviction (layout.cu): sentinel dead slots, and the plan
// and commit of the order-preserving compaction into fresh pages.
struct LayoutLaunch {
  size_t chunks = 0;
  const LaunchMeta* meta = nullptr;  // [chunks]
  const LaunchMeta* rows = nullptr;  // [chunks] one item per sequence (fresh plan / commit)
  const int32_t* block_table = nullptr;
  int32_t* block_table_mut = nullptr;
  int32_t* nblocks = nullptr;
  const int32_t* keep = nullptr;
  void* k_pool = nullptr;
  void* v_pool = nullptr;
  int32_t* tags = nullptr;
  int32_t* moves = nullptr;
  int32_t* move_count = nullptr;
  int32_t* dead = nullptr;
  int32_t* dead_count = nullptr;
  int32_t* freed = nullptr;
  int32_t* new_rows = nullptr;
  int32_t* free_ids = nullptr;
  int32_t* free_top = nullptr;
  int32_t capacity = 0;
  int64_t Ftot_all = 0;  // pages returned by the whole call (fresh commit)
  unsigned* status = nullptr;
};

// ActKV's LRFU step (actkv.cu): one block per unit.
struct LrfuLaunch {
  size_t chunks = 0;
  const LaunchMeta* meta = nullptr;  // [chunks], one item per unit
  const int32_t* block_table = nullptr;
  const float* attn = nullptr;       // [L][H][Ntot] action attention
  float* crf_pool = nullptr;         // [L][num_pages][H][P] per-slot LRFU values
  float* crf_out = nullptr;          // [L][H][Ntot] eviction scores
  uint8_t* hits = nullptr;           // [L][H][Ntot] or null
  float frac = 0.9f;
  float decay = 0.70710678f;
  unsigned* status = nullptr;
};

// Longest segment the selection kernel takes.  Its per-warp 16-bit bin counts
// must stay below 2^16: with 16-byte loads a warp of the 16 counts 32 of every
// 512 vectors (128 of every 2048 positions) plus at most 6 unaligned head and
// tail positions, 510 * 128 + 6 = 65286 for n = 2^20 - 4096.
constexpr int kSelectMaxSegment = (1 << 20) - 4096;

// Survivors per block of the fresh-page move kernel (the host sizes its grid
// with the same count).
constexpr int kFreshMovesPerBlock = 1024;

// Longest segment the LRFU kernel takes: its per-warp 16-bit mass parts stay
// below 2^32 for up to 2^16 elements per warp (16 warps).
constexpr int kLrfuMaxSegment = 1 << 20;

// Attention Matching on the survivors (am.cu).  Units are (sequence, layer,
// head) with m > 0; every unit owns `unit_floats` floats of the workspace:
//   E   [R][ldE]   exp(L_C - c) in columns [0, m), s = exp(LSE - c) in column m;
//                  overwritten by the compact probabilities Ph after the mass fit
//   G   [m][ldE]   E^T [E | s] (the mass fit's Gram matrix and E^T s in column m);
//                  overwritten by H = Ph^T Ph for the value fit
//   Y   [R][d]     full attention output softmax(L) V
//   lse [R]        natural-log row mass of the full attention
//   Bm  [m][d]     Ph^T Y over the first of its row ranges (H X0 minus it
//                  replaces it; the value fit subtracts the other ranges)
//   w   [m4]       fitted exp(beta)
//   X   [m][d]     the value fit's unknowns (from the kept values X0)
//   Bp  [kAmBmParts - 1][m][d]  Ph^T Y over the other row ranges
struct AmSeq {
  int32_t b, s0, n, m;
  int32_t ldE;          // row stride of E and G: the launch's largest m + 1, rounded up to a multiple of 4
  int32_t pad;
  int64_t moff;         // offset of the sequence in [L][H][Mtot]
  int64_t unit0;        // first unit of the sequence in this launch
  int64_t ws;           // float offset of the sequence's first unit in the workspace
  int64_t unit_floats;  // workspace floats per unit (every unit of a launch laid out for its largest m)
};

struct AmMeta {
  int32_t nseq, L, H, P, d, num_pages, max_blocks, R;
  int32_t max_m;   // largest m of the launch (grid sizing)
  int32_t sweeps;  // coordinate-descent sweeps of each fit
  float scale;
  int32_t bm_parts;  // row ranges Bm = Ph^T Y is summed over (1 .. kAmBmParts)
  int64_t Mtot;
  int64_t units;   // units of this launch
  AmSeq seq[kMaxSeqPerLaunch];
};

// Unit workspace offsets (floats, from the unit's base).
__host__ __device__ inline int64_t am_off_G(int R, int ldE) { return (int64_t)R * ldE; }
__host__ __device__ inline int64_t am_off_Y(int R, int m, int ldE) { return (int64_t)(R + m) * ldE; }
__host__ __device__ inline int64_t am_off_lse(int R, int m, int ldE, int d) {
  return am_off_Y(R, m, ldE) + (int64_t)R * d;
}
__host__ __device__ inline int64_t am_off_Bm(int R, int m, int ldE, int d) { return am_off_lse(R, m, ldE, d) + R; }
__host__ __device__ inline int64_t am_off_w(int R, int m, int ldE, int d) {
  return am_off_Bm(R, m, ldE, d) + (int64_t)m * d;
}
// X: the value fit's unknowns [m][d] (16-byte aligned: a tensor map reads it)
__host__ __device__ inline int64_t am_off_X(int R, int m, int ldE, int d) {
  return (am_off_w(R, m, ldE, d) + ((m + 3) & ~3) + 3) & ~int64_t(3);
}
// Bm = Ph^T Y is summed over up to kAmBmParts row ranges by separate blocks
// (they fill the SMs the blocks of H = Ph^T Ph leave idle); range p > 0 lands
// in Bp part p - 1.  The starting-gradient product leaves H X0 - (range 0) in
// Bm's place and the value fit subtracts ranges 1, 2, .. in order as it loads it.
constexpr int kAmBmParts = 4;
__host__ __device__ inline int64_t am_off_Bp(int R, int m, int ldE, int d) {
  return am_off_X(R, m, ldE, d) + (int64_t)m * d;
}
__host__ __device__ inline int64_t am_unit_floats(int R, int m, int ldE, int d) {
  const int64_t x = am_off_Bp(R, m, ldE, d) + (int64_t)(kAmBmParts - 1) * m * d;
  return (x + 63) & ~int64_t(63);  // 256-byte aligned units
}

// Largest budget and proxy-row count the fits take (the Gram matrices are m x m).
constexpr int kAmMaxM = 2048;
constexpr int kAmMaxR = 4096;

struct AmLaunch {
  size_t chunks = 0;
  const AmMeta* meta = nullptr;  // [chunks]
  const CUtensorMap* tmK = nullptr;  // K pool, one page per box (as the scoring passes)
  const CUtensorMap* tmVpool = nullptr;  // V pool, same geometry
  const CUtensorMap* tmQ = nullptr;  // Q, box {64, 128}
  // [chunks] fp32 operands of the Gram products, [unit][row][column] with a {128, 16, 1} box
  const CUtensorMap* tmX = nullptr;  // E / Ph: [unit][R][ldE]
  const CUtensorMap* tmY = nullptr;  // Y: [unit][R][d]
  const CUtensorMap* tmH = nullptr;  // H (in G's place): [unit][largest m][ldE]
  const CUtensorMap* tmX0 = nullptr;  // X0: [unit][largest m][d]
  const float* lse_rows = nullptr;   // [B][L][H][R] natural-log LSE of every proxy row
  const int32_t* block_table = nullptr;
  const void* k_pool = nullptr;
  void* v_pool = nullptr;
  const uint16_t* q = nullptr;   // [B][L][H][R][d]
  const int32_t* keep = nullptr; // [L][H][Mtot]
  float* ws = nullptr;
  float* aux = nullptr;          // per-slot beta, or null
  float* beta = nullptr;         // [L][H][Mtot] or null
  float* vc = nullptr;           // [L][H][Mtot][d] or null
  unsigned* status = nullptr;
};

cudaError_t launch_am(const AmLaunch& al, cudaStream_t stream);

cudaError_t launch_lrfu(const LrfuLaunch& ll, cudaStream_t stream);
cudaError_t launch_sentinel(const LayoutLaunch& ll, cudaStream_t stream);
cudaError_t launch_fresh_plan(const LayoutLaunch& ll, cudaStream_t stream);
cudaError_t launch_fresh_commit(const LayoutLaunch& ll, cudaStream_t stream);

cudaError_t launch_plan(const CompactLaunch& cl, cudaStream_t stream);
cudaError_t launch_compact(const CompactLaunch& cl, cudaStream_t stream);
cudaError_t launch_free(const CompactLaunch& cl, cudaStream_t stream);

}  // namespace kvc
