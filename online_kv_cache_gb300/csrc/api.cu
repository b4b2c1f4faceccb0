// api.cu -- the C ABI of libkvc (declared in include/kvc.h).
//
// Host side only: argument validation (before any launch), launch metadata
// (every grid and offset is derived from the host-known segment lengths and
// budgets, so the hot path needs no device->host read), TMA descriptors for
// the paged K pool and the proxy queries, and the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "kvc.h"

namespace kvc {

__device__ unsigned int g_device_status;

namespace {

thread_local std::string g_last_error;

kvc_status fail(kvc_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

kvc_status cuda_fail(cudaError_t e, const char* where) {
  return fail(KVC_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

kvc_status ok() {
  g_last_error.clear();
  return KVC_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The planner keeps a bitmap of the target region in shared memory (<= 192 KB).
constexpr int kMaxTargetSlots = 192 * 1024 * 8;
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
  int num_sms = 0;
  unsigned* status = nullptr;
};

kvc_status device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(KVC_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& di = cache[dev];
  if (di.status == nullptr) {
    e = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    di.status = static_cast<unsigned*>(p);
  }
  *out = di;
  return KVC_OK;
}

// Like device_info, but without a usable device reports the GB300's 152 SMs (the
// work split, and so the workspace size, depends on the SM count).
kvc_status device_info_or_default(DeviceInfo* out) {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
    cudaGetLastError();
    out->num_sms = 152;
    out->status = nullptr;
    return KVC_OK;
  }
  return device_info(out);
}

// Persistent-grid size of the scoring passes: one CTA per SM, or fewer when
// the KVC_GRID_LIMIT environment variable asks for it (a test knob that makes
// every CTA walk many work items).
int grid_limit(int num_sms) {
  const char* e = std::getenv("KVC_GRID_LIMIT");
  if (e != nullptr) {
    const int v = std::atoi(e);
    if (v > 0) return std::min(v, num_sms);
  }
  return num_sms;
}

// ------------------------------------------------------------- validation

enum Need : unsigned {
  kNeedK = 1, kNeedV = 2, kNeedTags = 4, kNeedBT = 8, kNeedNB = 16,
};

// NVTX range around each C-ABI call (seen by nsys / ncu; a no-op without a tool).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

// Checked mode (environment KVC_CHECKED set and not "0"): a call that launched work
// waits for its stream and turns a set bit of the device status word (a bad page, a
// bad keep position, an expired wait, a stack overflow) into KVC_ERR_DEVICE_CHECK.
// Skipped while the stream is being captured into a graph.
kvc_status launched(kvc_stream_t stream, const char* where) {
  const char* env = std::getenv("KVC_CHECKED");
  if (env == nullptr || env[0] == '\0' || (env[0] == '0' && env[1] == '\0')) return ok();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return ok();
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, where);
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e, where);
  if (v != 0) return fail(KVC_ERR_DEVICE_CHECK, "%s: device status word 0x%x (checked mode)", where, v);
  return ok();
}

kvc_status check_cache(const kvc_cache* c, unsigned need) {
  if (c == nullptr) return fail(KVC_ERR_INVALID_ARG, "cache is NULL");
  if (c->num_layers <= 0 || c->num_pages <= 0 || c->num_kv_heads <= 0 || c->page_size <= 0 ||
      c->head_dim <= 0 || c->max_blocks <= 0 || c->batch <= 0)
    return fail(KVC_ERR_INVALID_ARG, "cache dimensions must be positive");
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(KVC_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", c->head_dim);
  const int P = c->page_size;
  if (P < 8 || P > 64 || (P & (P - 1)) != 0)
    return fail(KVC_ERR_UNSUPPORTED, "page_size %d (supported: 8, 16, 32, 64)", P);
  const int64_t rows = (int64_t)c->num_layers * c->num_pages * c->num_kv_heads * P;
  if (rows >= (int64_t(1) << 31))
    return fail(KVC_ERR_UNSUPPORTED, "L*num_pages*H*P = %lld exceeds 2^31", (long long)rows);
  if ((need & kNeedK) && (c->k_pool == nullptr || !aligned16(c->k_pool)))
    return fail(KVC_ERR_INVALID_ARG, "k_pool is NULL or not 16-byte aligned");
  if ((need & kNeedV) && (c->v_pool == nullptr || !aligned16(c->v_pool)))
    return fail(KVC_ERR_INVALID_ARG, "v_pool is NULL or not 16-byte aligned");
  if ((need & kNeedTags) && c->tags == nullptr) return fail(KVC_ERR_INVALID_ARG, "tags is NULL");
  if ((need & kNeedBT) && c->block_table == nullptr)
    return fail(KVC_ERR_INVALID_ARG, "block_table is NULL");
  if ((need & kNeedNB) && c->nblocks == nullptr) return fail(KVC_ERR_INVALID_ARG, "nblocks is NULL");
  return KVC_OK;
}

// One active sequence (n > 0) of a call.
struct Seq {
  int32_t b, s0, n, m, nb, X;
};

struct Plan {
  std::vector<Seq> seqs;  // active sequences, ascending b
  int64_t Ntot = 0, Mtot = 0, Ftot = 0;
  std::vector<int64_t> off, moff, foff;  // per active sequence
};

kvc_status build_plan(const kvc_cache* c, const kvc_segments* s, const int32_t* m, Plan* out) {
  if (s == nullptr || s->seg_start == nullptr || s->seg_end == nullptr || s->seq_len == nullptr)
    return fail(KVC_ERR_INVALID_ARG, "segments or one of its arrays is NULL");
  if (s->batch != c->batch)
    return fail(KVC_ERR_INVALID_ARG, "segments batch %d != cache batch %d", s->batch, c->batch);
  const int P = c->page_size;
  Plan p;
  for (int b = 0; b < s->batch; ++b) {
    const int32_t s0 = s->seg_start[b], s1 = s->seg_end[b], len = s->seq_len[b];
    if (len < 0 || ceil_div(len, P) > c->max_blocks)
      return fail(KVC_ERR_INVALID_ARG, "seq_len[%d] = %d does not fit max_blocks", b, len);
    if (s0 < 0 || s1 < s0 || s1 > len)
      return fail(KVC_ERR_INVALID_ARG, "segment %d = [%d, %d) outside [0, %d]", b, s0, s1, len);
    if (s0 % P != 0 || (s1 % P != 0 && s1 != len))
      return fail(KVC_ERR_UNALIGNED_SEGMENT,
                  "segment %d = [%d, %d) must start on a block boundary and end on one or at the "
                  "sequence end (%d)",
                  b, s0, s1, len);
    int32_t mb = 0;
    if (m != nullptr) {
      if (m[b] < 0) return fail(KVC_ERR_BUDGET, "m[%d] = %d < 0", b, m[b]);
      mb = std::min(m[b], s1 - s0);
    }
    const int32_t n = s1 - s0;
    if (n == 0) continue;
    Seq q{b, s0, n, mb, (int32_t)ceil_div(n, P), (int32_t)ceil_div(mb, P)};
    p.seqs.push_back(q);
    p.off.push_back(p.Ntot);
    p.moff.push_back(p.Mtot);
    p.foff.push_back(p.Ftot);
    p.Ntot += n;
    p.Mtot += mb;
    p.Ftot += q.nb - q.X;
  }
  // rows before an active sequence's offsets in the ragged [L][H][Ntot] layout
  if (p.Ntot >= (int64_t(1) << 31)) return fail(KVC_ERR_UNSUPPORTED, "sum of segment lengths >= 2^31");
  // offsets of inactive sequences are not needed: they own no entries
  *out = std::move(p);
  return KVC_OK;
}

LaunchMeta base_meta(const kvc_cache* c, const Plan& p) {
  LaunchMeta lm;
  std::memset(&lm, 0, sizeof lm);
  lm.L = c->num_layers;
  lm.H = c->num_kv_heads;
  lm.P = c->page_size;
  lm.d = c->head_dim;
  lm.num_pages = c->num_pages;
  lm.max_blocks = c->max_blocks;
  lm.B = c->batch;
  lm.Ntot = p.Ntot;
  lm.Mtot = p.Mtot;
  lm.Ftot = p.Ftot;
  int lp = 0;
  while ((1 << lp) < c->page_size) ++lp;
  lm.log2P = lp;
  return lm;
}

void fill_seq(SeqMeta* sm, const Plan& p, size_t i) {
  const Seq& q = p.seqs[i];
  sm->b = q.b;
  sm->s0 = q.s0;
  sm->n = q.n;
  sm->m = q.m;
  sm->nb = q.nb;
  sm->X = q.X;
  sm->split = 1;
  sm->off = p.off[i];
  sm->moff = p.moff[i];
  sm->foff = p.foff[i];
}

// Splits the active sequences into launch chunks of at most kMaxSeqPerLaunch.
std::vector<std::pair<size_t, size_t>> chunks_of(const Plan& p) {
  std::vector<std::pair<size_t, size_t>> ch;
  for (size_t i = 0; i < p.seqs.size(); i += kMaxSeqPerLaunch)
    ch.emplace_back(i, std::min(p.seqs.size(), i + (size_t)kMaxSeqPerLaunch));
  return ch;
}

// ------------------------------------------------------------- scoring

struct ScoreGeom {
  int R, R_pad, W, nchunks, rowtiles;
  int gsub1, ngroups1, qbytes1, kst1;  // pass 1: row tiles per group, groups, smem
  int gsub2, ngroups2, qbytes2, kst2;  // pass 2: chunks per group, groups, smem
};

ScoreGeom score_geom(int R, int d) {
  ScoreGeom g;
  g.R = R;
  const int R32 = (int)ceil_div(R, 32) * 32;
  g.nchunks = (int)ceil_div(R32, 256);
  g.W = (int)ceil_div(ceil_div(R, g.nchunks), 32) * 32;
  g.R_pad = g.W * g.nchunks;
  g.rowtiles = (int)ceil_div(R, kScoreTile);
  const int tile_bytes = kScoreTile * d * 2;
  const int fixed = score_smem_bytes(0, 0, d);
  g.gsub1 = std::min(4, g.rowtiles);
  g.ngroups1 = (int)ceil_div(g.rowtiles, g.gsub1);
  // pass 1 keeps Q in TMEM; its sub-tiles pass through staging buffers: a whole row
  // group (4) when it has more than two, so the next item's Q is in shared memory
  // before this item's MMAs drain (measured: -3.6% on short items, -0.8% on long
  // ones, although fewer K stages remain), else two
  g.qbytes1 = (g.gsub1 > 2 ? 4 : 2) * kScoreTile * d * 2;
  g.kst1 = std::min(8, (kScoreSmemLimit - fixed - g.qbytes1) / tile_bytes);
  g.gsub2 = std::min(g.nchunks, std::max(1, 512 / g.W));
  g.ngroups2 = (int)ceil_div(g.nchunks, g.gsub2);
  g.qbytes2 = g.gsub2 * g.W * d * 2;
  g.kst2 = std::min(8, (kScoreSmemLimit - fixed - g.qbytes2) / tile_bytes);
  return g;
}

// Key tiles per work item.  Items are dealt round-robin to one persistent CTA
// per SM, so the pass ends when the busiest CTA does: choose the item size that
// minimises (items per CTA, rounded up) x (tiles per item) + a per-item cost.
int tiles_per_item(const kvc_cache* c, const Plan& p, int ngroups, int num_sms) {
  const int64_t LHg = (int64_t)c->num_layers * c->num_kv_heads * ngroups;
  double best = 1e300;
  int best_tpi = 2;
  for (int tpi = 2; tpi <= 48; ++tpi) {
    int64_t items = 0, max_tiles = 0;
    for (const Seq& q : p.seqs) {
      const int64_t T = ceil_div(q.n, kScoreTile);
      const int64_t split = std::min<int64_t>(T, ceil_div(T, tpi));
      items += LHg * split;
      max_tiles = std::max<int64_t>(max_tiles, ceil_div(T, split));
    }
    const double per_cta = (double)ceil_div(items, num_sms);
    const double cost = per_cta * ((double)max_tiles + 1.0);
    if (cost < best - 1e-9) {
      best = cost;
      best_tpi = tpi;
    }
  }
  return best_tpi;
}

// Failure-path test of the scoring kernels: > 0 withholds their proxy-row
// loads and limits the waits between their roles (kvc_debug_stall_scoring).
std::atomic<int64_t> g_stall_ns{0};

struct ScorePlan {
  std::vector<LaunchMeta> p1, comb, p2;
  size_t part_bytes = 0, obias_bytes = 0, part2_bytes = 0;
};

void build_score_plan(const kvc_cache* c, const Plan& p, const ScoreGeom& g, float scale, float pw, int num_sms,
                      ScorePlan* sp) {
  const int64_t LH = (int64_t)c->num_layers * c->num_kv_heads;
  const int tpi1 = tiles_per_item(c, p, g.ngroups1, num_sms);
  const int tpi2 = tiles_per_item(c, p, g.ngroups2, num_sms);
  int64_t max_p1 = 0;
  for (auto [lo, hi] : chunks_of(p)) {
    LaunchMeta a = base_meta(c, p), k = base_meta(c, p), z = base_meta(c, p);
    for (LaunchMeta* lm : {&a, &k, &z}) {
      lm->nseq = (int)(hi - lo);
      lm->R = g.R;
      lm->R_pad = g.R_pad;
      lm->W = g.W;
      lm->nchunks = g.nchunks;
      lm->rowtiles = g.rowtiles;
      lm->scale = scale;
      lm->pw = pw;
      lm->stall_ns = g_stall_ns.load(std::memory_order_relaxed);
    }
    a.ngroups = g.ngroups1;
    a.gsub = g.gsub1;
    a.qbytes = g.qbytes1;
    a.kst = g.kst1;

    z.ngroups = g.ngroups2;
    z.gsub = g.gsub2;
    z.qbytes = g.qbytes2;
    z.kst = g.kst2;
    int64_t i1 = 0, ic = 0, i2 = 0;
    for (size_t i = lo; i < hi; ++i) {
      const size_t j = i - lo;
      for (LaunchMeta* lm : {&a, &k, &z}) fill_seq(&lm->seq[j], p, i);
      const int T = (int)ceil_div(p.seqs[i].n, kScoreTile);
      const int split1 = (int)std::min<int64_t>(T, ceil_div(T, tpi1));
      const int split2 = (int)std::min<int64_t>(T, ceil_div(T, tpi2));
      a.seq[j].split = split1;
      k.seq[j].split = split1;
      z.seq[j].split = split2;
      a.seq[j].item0 = i1;
      k.seq[j].item0 = ic;
      k.seq[j].item1 = i1;
      z.seq[j].item0 = i2;
      i1 += LH * g.ngroups1 * split1;
      ic += LH * g.R_pad;
      i2 += LH * g.ngroups2 * split2;
    }
    a.items = i1;
    k.items = ic;
    z.items = i2;
    max_p1 = std::max(max_p1, i1);
    sp->p1.push_back(a);
    sp->comb.push_back(k);
    sp->p2.push_back(z);
  }
  sp->part_bytes = (size_t)max_p1 * 2 * 4 * kScoreTile * sizeof(float2);
  sp->obias_bytes = (size_t)c->batch * LH * g.R_pad * sizeof(float);
  sp->part2_bytes = g.ngroups2 > 1 ? (size_t)g.ngroups2 * LH * p.Ntot * sizeof(float) : 0;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor [rows][d] with a {64, box_rows} box and 128-byte swizzle.
kvc_status make_tmap(CUtensorMap* map, const void* base, int64_t rows, int d, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return KVC_OK;
}

// A launch's per-unit fp32 matrices as a 3-D tensor [unit][row][column]
// (row stride ld floats, unit stride unit_floats floats) with a {128, 16, 1}
// box and no swizzle: one box is 16 rows of a 128-column strip, dense in
// shared memory; rows past `rows` and columns past `cols` read as zeros.
kvc_status make_amap(CUtensorMap* map, const float* base, int64_t cols, int64_t rows, int64_t units, int64_t ld,
                     int64_t unit_floats) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)units};
  const cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)unit_floats * 4};
  const cuuint32_t box[3] = {128, 16, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled (AM operands) failed (%d)", (int)r);
  return KVC_OK;
}

// The K pool as a 4-D tensor [row group][k-block][row in group][64 elements]
// (k-blocks of 64 head-dim elements = 128 B, groups of 8 rows): one box of
// {64, 8, d/64, P/8} fetches a whole page of one head in one copy and lands in
// shared memory as 1024-byte swizzle atoms ordered (row group, k-block), the
// layout the MMA reads with a group stride of (d/64) x 1024 B.
kvc_status make_kmap(CUtensorMap* map, const void* base, int64_t rows, int d, int P) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[4] = {64, 8, (cuuint64_t)(d / 64), (cuuint64_t)(rows / 8)};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, 128, (cuuint64_t)d * 2 * 8};
  const cuuint32_t box[4] = {64, 8, (cuuint32_t)(d / 64), (cuuint32_t)(P / 8)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled (K pages) failed (%d)", (int)r);
  return KVC_OK;
}

}  // namespace
}  // namespace kvc

using namespace kvc;

extern "C" {

const char* kvc_version(void) { return "kvc 0.1 (sm_103a)"; }

const char* kvc_last_error(void) { return g_last_error.c_str(); }

const char* kvc_status_string(kvc_status st) {
  switch (st) {
    case KVC_OK: return "KVC_OK";
    case KVC_ERR_INVALID_ARG: return "KVC_ERR_INVALID_ARG";
    case KVC_ERR_UNALIGNED_SEGMENT: return "KVC_ERR_UNALIGNED_SEGMENT";
    case KVC_ERR_BUDGET: return "KVC_ERR_BUDGET";
    case KVC_ERR_WORKSPACE: return "KVC_ERR_WORKSPACE";
    case KVC_ERR_UNSUPPORTED: return "KVC_ERR_UNSUPPORTED";
    case KVC_ERR_CUDA: return "KVC_ERR_CUDA";
    case KVC_ERR_DEVICE_CHECK: return "KVC_ERR_DEVICE_CHECK";
    default: return "KVC_ERR_UNKNOWN";
  }
}

int64_t kvc_budget_from_ratio(int64_t n, double ratio) {
  if (n <= 0 || !std::isfinite(ratio)) return 0;
  const double x = ratio * (double)n - 1e-9 * (double)n;
  int64_t m = (int64_t)std::ceil(x);
  return std::max<int64_t>(0, std::min<int64_t>(m, n));
}

int64_t kvc_budget_actkv(int32_t k) {
  if (k < 0) return -1;
  // 512 * (7/4)^k = 7^k * 2^(9 - 2k), floored, capped at 30000
  int64_t num = 512;
  int64_t den = 1;
  for (int i = 0; i < k; ++i) {
    if (num / den >= 30000) return 30000;
    num *= 7;
    den *= 4;
  }
  return std::min<int64_t>(30000, num / den);
}

kvc_status kvc_score_workspace_size(const kvc_cache* cache, const kvc_segments* segs, int32_t R,
                                    size_t* bytes) {
  kvc_status st = check_cache(cache, 0);
  if (st != KVC_OK) return st;
  if (bytes == nullptr) return fail(KVC_ERR_INVALID_ARG, "bytes is NULL");
  if (R < 1 || R > 4096) return fail(KVC_ERR_UNSUPPORTED, "R = %d (supported: 1..4096)", R);
  Plan p;
  if ((st = build_plan(cache, segs, nullptr, &p)) != KVC_OK) return st;
  DeviceInfo di;
  if ((st = device_info_or_default(&di)) != KVC_OK) return st;
  ScorePlan sp;
  build_score_plan(cache, p, score_geom(R, cache->head_dim), 1.0f, 2.0f, di.num_sms, &sp);
  *bytes = align256(sp.part_bytes) + align256(sp.obias_bytes) + align256(sp.part2_bytes);
  return ok();
}

}  // extern "C"

namespace kvc {
namespace {

// Validation, descriptors and launches shared by kvc_score, kvc_score_lse and kvc_score_alpha.
kvc_status score_common(const char* where, unsigned phases, float pw, const kvc_cache* cache,
                        const kvc_segments* segs, const uint16_t* q, int32_t R, float scale,
                        const float* lse_in, float* lse_out, float* scores, void* ws, size_t ws_bytes,
                        kvc_stream_t stream) {
  const NvtxRange nvtx_range(where);
  kvc_status st = check_cache(cache, kNeedK | kNeedBT);
  if (st != KVC_OK) return st;
  if (R < 1 || R > 4096) return fail(KVC_ERR_UNSUPPORTED, "R = %d (supported: 1..4096)", R);
  if (!std::isfinite(scale) || !(scale > 0.0f)) return fail(KVC_ERR_INVALID_ARG, "scale must be finite and > 0");
  Plan p;
  if ((st = build_plan(cache, segs, nullptr, &p)) != KVC_OK) return st;
  if (p.seqs.empty()) return ok();
  if (q == nullptr || !aligned16(q)) return fail(KVC_ERR_INVALID_ARG, "q is NULL or not 16-byte aligned");
  if ((phases & kPhaseAlpha) && scores == nullptr) return fail(KVC_ERR_INVALID_ARG, "scores is NULL");
  if ((phases & kPhaseLseIn) && lse_in == nullptr) return fail(KVC_ERR_INVALID_ARG, "lse is NULL");
  DeviceInfo di;
  if ((st = device_info_or_default(&di)) != KVC_OK) return st;
  const ScoreGeom g = score_geom(R, cache->head_dim);
  ScorePlan sp;
  build_score_plan(cache, p, g, scale, pw, di.num_sms, &sp);
  const size_t need = align256(sp.part_bytes) + align256(sp.obias_bytes) + align256(sp.part2_bytes);
  if (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(KVC_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  if ((st = device_info(&di)) != KVC_OK) return st;

  const int64_t krows = (int64_t)cache->num_layers * cache->num_pages * cache->num_kv_heads * cache->page_size;
  const int64_t qrows = (int64_t)cache->batch * cache->num_layers * cache->num_kv_heads * R;
  if (qrows >= (int64_t(1) << 31)) return fail(KVC_ERR_UNSUPPORTED, "B*L*H*R >= 2^31");
  CUtensorMap tmK, tmQ1, tmQ2;
  if ((st = make_kmap(&tmK, cache->k_pool, krows, cache->head_dim, cache->page_size)) != KVC_OK) return st;
  if ((st = make_tmap(&tmQ1, q, qrows, cache->head_dim, kScoreTile)) != KVC_OK) return st;
  if ((st = make_tmap(&tmQ2, q, qrows, cache->head_dim, g.W)) != KVC_OK) return st;

  ScoreLaunch sl;
  sl.phases = phases;
  sl.lse_in = lse_in;
  sl.d = cache->head_dim;
  sl.num_sms = di.num_sms;
  sl.grid_limit = grid_limit(di.num_sms);
  sl.chunks = sp.p1.size();
  sl.pass1 = sp.p1.data();
  sl.combine = sp.comb.data();
  sl.pass2 = sp.p2.data();
  sl.tmK = &tmK;
  sl.tmQ1 = &tmQ1;
  sl.tmQ2 = &tmQ2;
  sl.block_table = cache->block_table;
  sl.part = static_cast<float2*>(ws);
  sl.obias = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align256(sp.part_bytes));
  sl.part2 = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align256(sp.part_bytes) +
                                      align256(sp.obias_bytes));
  sl.lse_out = lse_out;
  sl.scores = scores;
  sl.status = di.status;
  const cudaError_t e = launch_score(sl, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, where);
  return launched(stream, where);
}

std::atomic<uint64_t> g_launches{0};

}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace kvc

extern "C" {

kvc_status kvc_score(const kvc_cache* cache, const kvc_segments* segs, const uint16_t* q, int32_t R,
                     float scale, float* scores, float* lse, void* ws, size_t ws_bytes,
                     kvc_stream_t stream) {
  return score_common("kvc_score", kPhaseLse | kPhaseAlpha, 2.0f, cache, segs, q, R, scale, nullptr, lse,
                      scores, ws, ws_bytes, stream);
}

kvc_status kvc_score_lse(const kvc_cache* cache, const kvc_segments* segs, const uint16_t* q, int32_t R,
                         float scale, float* lse, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  return score_common("kvc_score_lse", kPhaseLse, 2.0f, cache, segs, q, R, scale, nullptr, lse, nullptr, ws,
                      ws_bytes, stream);
}

kvc_status kvc_score_alpha(const kvc_cache* cache, const kvc_segments* segs, const uint16_t* q, int32_t R,
                           float scale, const float* lse, float* scores, void* ws, size_t ws_bytes,
                           kvc_stream_t stream) {
  const unsigned phases = kPhaseAlpha | (lse != nullptr ? kPhaseLseIn : 0u);
  return score_common("kvc_score_alpha", phases, 2.0f, cache, segs, q, R, scale, lse, nullptr, scores, ws,
                      ws_bytes, stream);
}

kvc_status kvc_score_action(const kvc_cache* cache, const kvc_segments* segs, const uint16_t* q, int32_t R,
                            float scale, float* attn, float* lse, void* ws, size_t ws_bytes,
                            kvc_stream_t stream) {
  return score_common("kvc_score_action", kPhaseLse | kPhaseAlpha, 1.0f, cache, segs, q, R, scale, nullptr,
                      lse, attn, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- no-alloc scoring
//
// kvc_score with its workspace in a fixed device array owned by the library,
// for callers that cannot hand the library a cudaMalloc'ed workspace.

}  // extern "C"

namespace kvc {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device (cudaGetSymbolAddress must run with that device current; in host code
// the symbol itself is only a host-side stand-in).
kvc_status noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(KVC_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    addr[dev] = p;
  }
  *out = addr[dev];
  return KVC_OK;
}

}  // namespace
}  // namespace kvc

extern "C" {

kvc_status kvc_score_noalloc(const kvc_cache* cache, const kvc_segments* segs, const uint16_t* q,
                             int32_t R, float scale, float* scores, float* lse, kvc_stream_t stream) {
  size_t need = 0;
  kvc_status st = kvc_score_workspace_size(cache, segs, R, &need);
  if (st != KVC_OK) return st;
  if (need > kNoAllocScratchBytes)
    return fail(KVC_ERR_WORKSPACE,
                "kvc_score_noalloc: this call needs %zu bytes of workspace; the library's fixed "
                "scratch holds %zu (use kvc_score with a caller workspace)",
                need, kNoAllocScratchBytes);
  void* ws = nullptr;
  if ((st = noalloc_scratch(&ws)) != KVC_OK) return st;
  return kvc_score(cache, segs, q, R, scale, scores, lse, ws, kNoAllocScratchBytes, stream);
}

uint64_t kvc_launch_count(int32_t reset) {
  return reset ? g_launches.exchange(0) : g_launches.load();
}

kvc_status kvc_debug_stall_scoring(int64_t stall_ns) {
  if (stall_ns < 0 || stall_ns > 10000000000ll)
    return fail(KVC_ERR_INVALID_ARG, "kvc_debug_stall_scoring: stall_ns must be in [0, 1e10], got %lld",
                (long long)stall_ns);
  g_stall_ns.store(stall_ns, std::memory_order_relaxed);
  return KVC_OK;
}

kvc_status kvc_select_workspace_size(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m,
                                     size_t* bytes) {
  kvc_status st = check_cache(cache, 0);
  if (st != KVC_OK) return st;
  if (bytes == nullptr) return fail(KVC_ERR_INVALID_ARG, "bytes is NULL");
  Plan p;
  if ((st = build_plan(cache, segs, m, &p)) != KVC_OK) return st;
  *bytes = 0;
  return ok();
}

kvc_status kvc_select_topm(const kvc_cache* cache, const kvc_segments* segs, const float* scores,
                           const int32_t* m, int32_t* keep, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  const NvtxRange nvtx_range("kvc_select_topm");
  (void)ws;
  (void)ws_bytes;
  kvc_status st = check_cache(cache, 0);
  if (st != KVC_OK) return st;
  if (m == nullptr) return fail(KVC_ERR_INVALID_ARG, "m is NULL");
  Plan p;
  if ((st = build_plan(cache, segs, m, &p)) != KVC_OK) return st;
  if (p.seqs.empty() || p.Mtot == 0) return ok();
  if (scores == nullptr || keep == nullptr) return fail(KVC_ERR_INVALID_ARG, "scores or keep is NULL");
  for (const Seq& q : p.seqs)
    if (q.n > kSelectMaxSegment)
      return fail(KVC_ERR_UNSUPPORTED, "segment of %d positions: selection takes at most %d", q.n,
                  kSelectMaxSegment);
  DeviceInfo di;
  if ((st = device_info(&di)) != KVC_OK) return st;
  const int64_t LH = (int64_t)cache->num_layers * cache->num_kv_heads;
  std::vector<LaunchMeta> metas;
  for (auto [lo, hi] : chunks_of(p)) {
    LaunchMeta lm = base_meta(cache, p);
    lm.nseq = (int)(hi - lo);
    int64_t it = 0;
    for (size_t i = lo; i < hi; ++i) {
      fill_seq(&lm.seq[i - lo], p, i);
      lm.seq[i - lo].item0 = it;
      it += LH;
    }
    lm.items = it;
    metas.push_back(lm);
  }
  SelectLaunch sl;
  sl.num_sms = di.num_sms;
  sl.chunks = metas.size();
  sl.meta = metas.data();
  sl.scores = scores;
  sl.keep = keep;
  sl.status = di.status;
  const cudaError_t e = launch_select(sl, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvc_select_topm launch");
  return launched(stream, "kvc_select_topm");
}

kvc_status kvc_plan_buffer_sizes(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m,
                                 kvc_plan_sizes* out) {
  kvc_status st = check_cache(cache, 0);
  if (st != KVC_OK) return st;
  if (m == nullptr || out == nullptr) return fail(KVC_ERR_INVALID_ARG, "m or out is NULL");
  Plan p;
  if ((st = build_plan(cache, segs, m, &p)) != KVC_OK) return st;
  const int64_t LH = (int64_t)cache->num_layers * cache->num_kv_heads;
  out->moves_len = 2 * LH * p.Mtot;
  out->units_len = LH * cache->batch;
  out->dead_len = LH * cache->batch * cache->page_size;
  out->freed_len = p.Ftot;
  out->new_rows_len = (int64_t)cache->batch * cache->max_blocks;
  out->Mtot = p.Mtot;
  out->Ntot = p.Ntot;
  return ok();
}

namespace {

kvc_status check_plan(const kvc_cache* cache, const Plan& p, const kvc_plan* plan) {
  if (plan == nullptr) return fail(KVC_ERR_INVALID_ARG, "plan is NULL");
  const int64_t LH = (int64_t)cache->num_layers * cache->num_kv_heads;
  struct { const int32_t* ptr; int64_t have, need; const char* name; } bufs[] = {
      {plan->moves, plan->moves_len, 2 * LH * p.Mtot, "moves"},
      {plan->move_count, plan->units_len, LH * cache->batch, "move_count"},
      {plan->dead, plan->dead_len, LH * cache->batch * cache->page_size, "dead"},
      {plan->dead_count, plan->units_len, LH * cache->batch, "dead_count"},
      {plan->freed, plan->freed_len, p.Ftot, "freed"},
      {plan->new_rows, plan->new_rows_len, (int64_t)cache->batch * cache->max_blocks, "new_rows"},
  };
  for (const auto& b : bufs) {
    if (b.need > 0 && (b.ptr == nullptr || b.have < b.need))
      return fail(KVC_ERR_WORKSPACE, "plan buffer %s needs %lld elements (have %lld)", b.name,
                  (long long)b.need, (long long)b.have);
  }
  return KVC_OK;
}

// Moves per copy block: 128, or fewer (down to 16) when the launch moves too
// little to give every SM 16 blocks: a small compaction is bound by the latency
// of each warp's chain of dependent loads, not by bandwidth.
int copy_moves_per_block(int64_t moves, int num_sms) {
  int mpb = 128;
  while (mpb > 16 && ceil_div(moves, mpb) < (int64_t)num_sms * 16) mpb >>= 1;
  return mpb;
}

void compact_metas(const kvc_cache* cache, const Plan& p, int num_sms, std::vector<LaunchMeta>* plan_m,
                   std::vector<LaunchMeta>* rows_m, std::vector<LaunchMeta>* copy_m,
                   std::vector<LaunchMeta>* free_m) {
  const int64_t LH = (int64_t)cache->num_layers * cache->num_kv_heads;
  const int P = cache->page_size;
  for (auto [lo, hi] : chunks_of(p)) {
    LaunchMeta a = base_meta(cache, p), r = base_meta(cache, p), c = base_meta(cache, p),
               f = base_meta(cache, p);
    const int nseq = (int)(hi - lo);
    a.nseq = r.nseq = c.nseq = f.nseq = nseq;
    int64_t moves = 0;
    for (size_t i = lo; i < hi; ++i) moves += LH * p.seqs[i].m;
    c.mpb = copy_moves_per_block(moves, num_sms);
    int64_t ia = 0, ic = 0, fc = 0;
    for (size_t i = lo; i < hi; ++i) {
      const size_t j = i - lo;
      for (LaunchMeta* lm : {&a, &r, &c, &f}) fill_seq(&lm->seq[j], p, i);
      const Seq& q = p.seqs[i];
      a.seq[j].item0 = ia;
      ia += LH;  // one planning CTA per unit
      a.words = std::max<int32_t>(a.words, (int32_t)ceil_div((int64_t)q.X * P, 32));
      c.seq[j].item0 = ic;  // copy blocks: one per (unit, mpb moves)
      ic += LH * std::max<int64_t>(1, ceil_div(q.m, c.mpb));
      fc += q.nb - q.X;
    }
    a.items = ia;
    c.items = ic;
    f.Ftot = fc;
    plan_m->push_back(a);
    rows_m->push_back(r);
    copy_m->push_back(c);
    free_m->push_back(f);
  }
}

}  // namespace

kvc_status kvc_plan_compact(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m,
                            const int32_t* keep, const kvc_plan* plan, kvc_stream_t stream) {
  const NvtxRange nvtx_range("kvc_plan_compact");
  kvc_status st = check_cache(cache, kNeedBT | kNeedNB);
  if (st != KVC_OK) return st;
  if (m == nullptr) return fail(KVC_ERR_INVALID_ARG, "m is NULL");
  Plan p;
  if ((st = build_plan(cache, segs, m, &p)) != KVC_OK) return st;
  for (const Seq& q : p.seqs)
    if ((int64_t)q.X * cache->page_size > kMaxTargetSlots)
      return fail(KVC_ERR_UNSUPPORTED, "target region of %lld slots exceeds %d (budget too large)",
                  (long long)q.X * cache->page_size, kMaxTargetSlots);
  if ((st = check_plan(cache, p, plan)) != KVC_OK) return st;
  if (p.seqs.empty()) return ok();
  if (p.Mtot > 0 && keep == nullptr) return fail(KVC_ERR_INVALID_ARG, "keep is NULL");
  DeviceInfo di;
  if ((st = device_info(&di)) != KVC_OK) return st;
  std::vector<LaunchMeta> pm, rm, cm, fm;
  compact_metas(cache, p, di.num_sms, &pm, &rm, &cm, &fm);
  CompactLaunch cl;
  cl.num_sms = di.num_sms;
  cl.chunks = pm.size();
  cl.plan_meta = pm.data();
  cl.rows_meta = rm.data();
  cl.block_table = cache->block_table;
  cl.nblocks = cache->nblocks;
  cl.keep = keep;
  cl.moves = plan->moves;
  cl.move_count = plan->move_count;
  cl.dead = plan->dead;
  cl.dead_count = plan->dead_count;
  cl.freed = plan->freed;
  cl.new_rows = plan->new_rows;
  cl.status = di.status;
  const cudaError_t e = launch_plan(cl, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvc_plan_compact launch");
  return launched(stream, "kvc_plan_compact");
}

kvc_status kvc_compact(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m,
                       const kvc_plan* plan, kvc_stream_t stream) {
  const NvtxRange nvtx_range("kvc_compact");
  kvc_status st = check_cache(cache, kNeedK | kNeedV | kNeedTags);
  if (st != KVC_OK) return st;
  if (m == nullptr) return fail(KVC_ERR_INVALID_ARG, "m is NULL");
  Plan p;
  if ((st = build_plan(cache, segs, m, &p)) != KVC_OK) return st;
  if ((st = check_plan(cache, p, plan)) != KVC_OK) return st;
  if (p.seqs.empty()) return ok();
  DeviceInfo di;
  if ((st = device_info(&di)) != KVC_OK) return st;
  std::vector<LaunchMeta> pm, rm, cm, fm;
  compact_metas(cache, p, di.num_sms, &pm, &rm, &cm, &fm);
  CompactLaunch cl;
  cl.num_sms = di.num_sms;
  cl.chunks = cm.size();
  cl.copy_meta = cm.data();
  cl.k_pool = cache->k_pool;
  cl.v_pool = cache->v_pool;
  cl.tags = cache->tags;
  cl.aux = cache->aux;
  cl.moves = plan->moves;
  cl.move_count = plan->move_count;
  cl.dead = plan->dead;
  cl.dead_count = plan->dead_count;
  cl.status = di.status;
  const cudaError_t e = launch_compact(cl, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvc_compact launch");
  return launched(stream, "kvc_compact");
}

kvc_status kvc_free_pages(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m,
                          const kvc_allocator* alloc, const kvc_plan* plan, kvc_stream_t stream) {
  const NvtxRange nvtx_range("kvc_free_pages");
  kvc_status st = check_cache(cache, kNeedBT | kNeedNB);
  if (st != KVC_OK) return st;
  if (m == nullptr) return fail(KVC_ERR_INVALID_ARG, "m is NULL");
  if (alloc == nullptr || alloc->free_ids == nullptr || alloc->free_top == nullptr || alloc->capacity < 0)
    return fail(KVC_ERR_INVALID_ARG, "allocator is NULL or incomplete");
  Plan p;
  if ((st = build_plan(cache, segs, m, &p)) != KVC_OK) return st;
  if ((st = check_plan(cache, p, plan)) != KVC_OK) return st;
  if (p.seqs.empty()) return ok();
  DeviceInfo di;
  if ((st = device_info(&di)) != KVC_OK) return st;
  std::vector<LaunchMeta> pm, rm, cm, fm;
  compact_metas(cache, p, di.num_sms, &pm, &rm, &cm, &fm);
  CompactLaunch cl;
  cl.num_sms = di.num_sms;
  cl.chunks = fm.size();
  cl.free_meta = fm.data();
  cl.block_table_mut = cache->block_table;
  cl.nblocks = cache->nblocks;
  cl.new_rows = plan->new_rows;
  cl.freed = plan->freed;
  cl.free_ids = alloc->free_ids;
  cl.free_top = alloc->free_top;
  cl.capacity = alloc->capacity;
  cl.status = di.status;
  const cudaError_t e = launch_free(cl, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvc_free_pages launch");
  return launched(stream, "kvc_free_pages");
}

// ------------------------------------------------------------- layout variants

namespace {

constexpr int kSentinelChunkHost = 4096;   // positions per sentinel block (layout.cu)

bool fresh_active(const Seq& q) { return q.m < q.n; }

int64_t fresh_returned(const Plan& p) {
  int64_t f = 0;
  for (const Seq& q : p.seqs)
    if (fresh_active(q)) f += q.nb;
  return f;
}

kvc_status check_fresh_plan(const kvc_cache* cache, const Plan& p, const kvc_plan* plan) {
  if (plan == nullptr) return fail(KVC_ERR_INVALID_ARG, "plan is NULL");
  const int64_t LH = (int64_t)cache->num_layers * cache->num_kv_heads;
  struct { const int32_t* ptr; int64_t have, need; const char* name; } bufs[] = {
      {plan->moves, plan->moves_len, 2 * LH * p.Mtot, "moves"},
      {plan->move_count, plan->units_len, LH * cache->batch, "move_count"},
      {plan->dead, plan->dead_len, LH * cache->batch * cache->page_size, "dead"},
      {plan->dead_count, plan->units_len, LH * cache->batch, "dead_count"},
      {plan->freed, plan->freed_len, fresh_returned(p), "freed"},
      {plan->new_rows, plan->new_rows_len, (int64_t)cache->batch * cache->max_blocks, "new_rows"},
  };
  for (const auto& b : bufs) {
    if (b.need > 0 && (b.ptr == nullptr || b.have < b.need))
      return fail(KVC_ERR_WORKSPACE, "fresh plan buffer %s needs %lld elements (have %lld)", b.name,
                  (long long)b.need, (long long)b.have);
  }
  return KVC_OK;
}

// Metas of the fresh-page plan/commit: per-unit blocks (moves) and per-sequence
// blocks (rows); the pop offsets (xoff) and return offsets (foff) run over
// the whole call.
void fresh_metas(const kvc_cache* cache, const Plan& p, std::vector<LaunchMeta>* mv,
                 std::vector<LaunchMeta>* rows) {
  const int64_t LH = (int64_t)cache->num_layers * cache->num_kv_heads;
  int64_t Xtot = 0;
  for (const Seq& q : p.seqs)
    if (fresh_active(q)) Xtot += q.X;
  int64_t xoff = 0, foff = 0;
  for (auto [lo, hi] : chunks_of(p)) {
    LaunchMeta a = base_meta(cache, p), r = base_meta(cache, p);
    a.nseq = r.nseq = (int)(hi - lo);
    a.Xtot = r.Xtot = Xtot;
    int64_t it = 0;
    for (size_t i = lo; i < hi; ++i) {
      const size_t j = i - lo;
      fill_seq(&a.seq[j], p, i);
      fill_seq(&r.seq[j], p, i);
      const Seq& q = p.seqs[i];
      a.seq[j].xoff = r.seq[j].xoff = (int32_t)xoff;
      a.seq[j].foff = r.seq[j].foff = foff;
      if (fresh_active(q)) {
        xoff += q.X;
        foff += q.nb;
      }
      a.seq[j].item0 = it;
      it += LH * std::max<int64_t>(1, ceil_div(q.m, kFreshMovesPerBlock));
    }
    a.items = it;
    mv->push_back(a);
    rows->push_back(r);
  }
}

kvc_status check_allocator(const kvc_allocator* alloc) {
  if (alloc == nullptr || alloc->free_ids == nullptr || alloc->free_top == nullptr || alloc->capacity < 0)
    return fail(KVC_ERR_INVALID_ARG, "allocator is NULL or incomplete");
  return KVC_OK;
}

}  // namespace

kvc_status kvc_evict_sentinel(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m,
                              const int32_t* keep, kvc_stream_t stream) {
  const NvtxRange nvtx_range("kvc_evict_sentinel");
  kvc_status st = check_cache(cache, kNeedK | kNeedV | kNeedTags | kNeedBT);
  if (st != KVC_OK) return st;
  if (m == nullptr) return fail(KVC_ERR_INVALID_ARG, "m is NULL");
  Plan p;
  if ((st = build_plan(cache, segs, m, &p)) != KVC_OK) return st;
  if (p.seqs.empty()) return ok();
  if (p.Mtot > 0 && keep == nullptr) return fail(KVC_ERR_INVALID_ARG, "keep is NULL");
  DeviceInfo di;
  if ((st = device_info(&di)) != KVC_OK) return st;
  const int64_t LH = (int64_t)cache->num_layers * cache->num_kv_heads;
  std::vector<LaunchMeta> metas;
  for (auto [lo, hi] : chunks_of(p)) {
    LaunchMeta a = base_meta(cache, p);
    a.nseq = (int)(hi - lo);
    int64_t it = 0;
    for (size_t i = lo; i < hi; ++i) {
      fill_seq(&a.seq[i - lo], p, i);
      a.seq[i - lo].item0 = it;
      it += LH * std::max<int64_t>(1, ceil_div(p.seqs[i].n, kSentinelChunkHost));
    }
    a.items = it;
    metas.push_back(a);
  }
  LayoutLaunch ll;
  ll.chunks = metas.size();
  ll.meta = metas.data();
  ll.block_table = cache->block_table;
  ll.keep = keep;
  ll.k_pool = cache->k_pool;
  ll.v_pool = cache->v_pool;
  ll.tags = cache->tags;
  ll.status = di.status;
  const cudaError_t e = launch_sentinel(ll, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvc_evict_sentinel launch");
  return launched(stream, "kvc_evict_sentinel");
}

kvc_status kvc_plan_fresh_buffer_sizes(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m,
                                       kvc_plan_sizes* out) {
  kvc_status st = kvc_plan_buffer_sizes(cache, segs, m, out);
  if (st != KVC_OK) return st;
  Plan p;
  if ((st = build_plan(cache, segs, m, &p)) != KVC_OK) return st;
  out->freed_len = fresh_returned(p);
  return ok();
}

kvc_status kvc_plan_fresh(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m,
                          const int32_t* keep, const kvc_allocator* alloc, const kvc_plan* plan,
                          kvc_stream_t stream) {
  const NvtxRange nvtx_range("kvc_plan_fresh");
  kvc_status st = check_cache(cache, kNeedBT | kNeedNB);
  if (st != KVC_OK) return st;
  if (m == nullptr) return fail(KVC_ERR_INVALID_ARG, "m is NULL");
  if ((st = check_allocator(alloc)) != KVC_OK) return st;
  Plan p;
  if ((st = build_plan(cache, segs, m, &p)) != KVC_OK) return st;
  if ((st = check_fresh_plan(cache, p, plan)) != KVC_OK) return st;
  if (p.seqs.empty()) return ok();
  if (p.Mtot > 0 && keep == nullptr) return fail(KVC_ERR_INVALID_ARG, "keep is NULL");
  DeviceInfo di;
  if ((st = device_info(&di)) != KVC_OK) return st;
  std::vector<LaunchMeta> mv, rows;
  fresh_metas(cache, p, &mv, &rows);
  LayoutLaunch ll;
  ll.chunks = mv.size();
  ll.meta = mv.data();
  ll.rows = rows.data();
  ll.block_table = cache->block_table;
  ll.nblocks = cache->nblocks;
  ll.keep = keep;
  ll.moves = plan->moves;
  ll.move_count = plan->move_count;
  ll.dead = plan->dead;
  ll.dead_count = plan->dead_count;
  ll.freed = plan->freed;
  ll.new_rows = plan->new_rows;
  ll.free_ids = alloc->free_ids;
  ll.free_top = alloc->free_top;
  ll.status = di.status;
  const cudaError_t e = launch_fresh_plan(ll, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvc_plan_fresh launch");
  return launched(stream, "kvc_plan_fresh");
}

kvc_status kvc_commit_fresh(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m,
                            const kvc_allocator* alloc, const kvc_plan* plan, kvc_stream_t stream) {
  const NvtxRange nvtx_range("kvc_commit_fresh");
  kvc_status st = check_cache(cache, kNeedBT | kNeedNB);
  if (st != KVC_OK) return st;
  if (m == nullptr) return fail(KVC_ERR_INVALID_ARG, "m is NULL");
  if ((st = check_allocator(alloc)) != KVC_OK) return st;
  Plan p;
  if ((st = build_plan(cache, segs, m, &p)) != KVC_OK) return st;
  if ((st = check_fresh_plan(cache, p, plan)) != KVC_OK) return st;
  if (p.seqs.empty()) return ok();
  DeviceInfo di;
  if ((st = device_info(&di)) != KVC_OK) return st;
  std::vector<LaunchMeta> mv, rows;
  fresh_metas(cache, p, &mv, &rows);
  LayoutLaunch ll;
  ll.chunks = rows.size();
  ll.rows = rows.data();
  ll.block_table_mut = cache->block_table;
  ll.nblocks = cache->nblocks;
  ll.freed = plan->freed;
  ll.new_rows = plan->new_rows;
  ll.free_ids = alloc->free_ids;
  ll.free_top = alloc->free_top;
  ll.capacity = alloc->capacity;
  ll.Ftot_all = fresh_returned(p);
  ll.status = di.status;
  const cudaError_t e = launch_fresh_commit(ll, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvc_commit_fresh launch");
  return launched(stream, "kvc_commit_fresh");
}

// ------------------------------------------------------------- ActKV LRFU

kvc_status kvc_lrfu_update(const kvc_cache* cache, const kvc_segments* segs, const float* attn, float frac,
                           float lambda, float* crf_out, uint8_t* hits, kvc_stream_t stream) {
  const NvtxRange nvtx_range("kvc_lrfu_update");
  kvc_status st = check_cache(cache, kNeedBT);
  if (st != KVC_OK) return st;
  if (cache->aux == nullptr) return fail(KVC_ERR_INVALID_ARG, "cache->aux (the per-slot LRFU values) is NULL");
  if (attn == nullptr || crf_out == nullptr) return fail(KVC_ERR_INVALID_ARG, "attn or crf_out is NULL");
  if (!(frac >= 0.0f && frac <= 1.0f)) return fail(KVC_ERR_INVALID_ARG, "frac must lie in [0, 1]");
  if (!std::isfinite(lambda) || lambda < 0.0f) return fail(KVC_ERR_INVALID_ARG, "lambda must be finite and >= 0");
  Plan p;
  if ((st = build_plan(cache, segs, nullptr, &p)) != KVC_OK) return st;
  if (p.seqs.empty()) return ok();
  for (const Seq& q : p.seqs)
    if (q.n > kLrfuMaxSegment)
      return fail(KVC_ERR_UNSUPPORTED, "segment of %d positions exceeds %d (LRFU mass histograms)", q.n,
                  kLrfuMaxSegment);
  DeviceInfo di;
  if ((st = device_info(&di)) != KVC_OK) return st;
  const int64_t LH = (int64_t)cache->num_layers * cache->num_kv_heads;
  std::vector<LaunchMeta> metas;
  for (auto [lo, hi] : chunks_of(p)) {
    LaunchMeta a = base_meta(cache, p);
    a.nseq = (int)(hi - lo);
    int64_t it = 0;
    for (size_t i = lo; i < hi; ++i) {
      fill_seq(&a.seq[i - lo], p, i);
      a.seq[i - lo].item0 = it;
      it += LH;
    }
    a.items = it;
    metas.push_back(a);
  }
  LrfuLaunch ll;
  ll.chunks = metas.size();
  ll.meta = metas.data();
  ll.block_table = cache->block_table;
  ll.attn = attn;
  ll.crf_pool = cache->aux;
  ll.crf_out = crf_out;
  ll.hits = hits;
  ll.frac = frac;
  ll.decay = (float)std::exp2(-(double)lambda);
  ll.status = di.status;
  const cudaError_t e = launch_lrfu(ll, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvc_lrfu_update launch");
  return launched(stream, "kvc_lrfu_update");
}

}  // extern "C"

namespace kvc {
namespace {

// Launch chunks and workspace offsets of Attention Matching: units are the
// (sequence, layer, head) triples of the sequences with m > 0.
struct AmPlan {
  std::vector<AmMeta> metas;
  int64_t floats = 0;
};

void build_am_plan(const kvc_cache* c, const Plan& p, int R, float scale, int sweeps, AmPlan* out) {
  const int64_t LH = (int64_t)c->num_layers * c->num_kv_heads;
  std::vector<size_t> act;
  for (size_t i = 0; i < p.seqs.size(); ++i)
    if (p.seqs[i].m > 0) act.push_back(i);
  int64_t wsf = 0;
  for (size_t a0 = 0; a0 < act.size(); a0 += kMaxSeqPerLaunch) {
    AmMeta am;
    std::memset(&am, 0, sizeof am);
    am.L = c->num_layers;
    am.H = c->num_kv_heads;
    am.P = c->page_size;
    am.d = c->head_dim;
    am.num_pages = c->num_pages;
    am.max_blocks = c->max_blocks;
    am.R = R;
    am.sweeps = sweeps;
    am.scale = scale;
    am.bm_parts = std::min(kAmBmParts, (R + 15) / 16);  // at most one range per 16-row chunk
    am.Mtot = p.Mtot;
    const size_t a1 = std::min(act.size(), a0 + (size_t)kMaxSeqPerLaunch);
    am.nseq = (int)(a1 - a0);
    for (size_t k = a0; k < a1; ++k) am.max_m = std::max(am.max_m, p.seqs[act[k]].m);
    // every unit of the launch is laid out for its largest m (one row stride,
    // one unit stride), so that one tensor map per operand covers the launch
    const int ldE = (am.max_m + 1 + 3) & ~3;
    const int64_t unit_floats = am_unit_floats(R, am.max_m, ldE, c->head_dim);
    int64_t units = 0;
    for (size_t k = a0; k < a1; ++k) {
      const size_t i = act[k];
      const Seq& q = p.seqs[i];
      AmSeq& s = am.seq[k - a0];
      s.b = q.b;
      s.s0 = q.s0;
      s.n = q.n;
      s.m = q.m;
      s.ldE = ldE;
      s.moff = p.moff[i];
      s.unit0 = units;
      s.ws = wsf;
      s.unit_floats = unit_floats;
      units += LH;
      wsf += LH * s.unit_floats;
    }
    am.units = units;
    out->metas.push_back(am);
  }
  out->floats = wsf;
}

// Attention Matching workspace: the units' fits, then the scoring LSE pass's
// workspace, then the LSE of every proxy row ([B][L][H][R] floats).
size_t am_lse_rows_bytes(const kvc_cache* c, int R) {
  return (size_t)c->batch * c->num_layers * c->num_kv_heads * R * sizeof(float);
}
size_t am_workspace_bytes(const kvc_cache* c, const AmPlan& ap, size_t score_bytes, int R) {
  return align256((size_t)ap.floats * sizeof(float)) + align256(score_bytes) + align256(am_lse_rows_bytes(c, R));
}

kvc_status check_am_args(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m, int32_t R, Plan* p) {
  kvc_status st = check_cache(cache, kNeedK | kNeedV | kNeedBT);
  if (st != KVC_OK) return st;
  if (m == nullptr) return fail(KVC_ERR_INVALID_ARG, "m is NULL");
  if (R < 1 || R > kAmMaxR) return fail(KVC_ERR_UNSUPPORTED, "R = %d (supported: 1..%d)", R, kAmMaxR);
  if ((st = build_plan(cache, segs, m, p)) != KVC_OK) return st;
  for (const Seq& q : p->seqs)
    if (q.m > kAmMaxM)
      return fail(KVC_ERR_UNSUPPORTED, "budget m = %d exceeds %d (Attention Matching's m x m Gram matrices)", q.m,
                  kAmMaxM);
  return KVC_OK;
}

}  // namespace
}  // namespace kvc

extern "C" {

kvc_status kvc_am_workspace_size(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m, int32_t R,
                                 size_t* bytes) {
  if (bytes == nullptr) return fail(KVC_ERR_INVALID_ARG, "bytes is NULL");
  Plan p;
  kvc_status st = check_am_args(cache, segs, m, R, &p);
  if (st != KVC_OK) return st;
  AmPlan ap;
  build_am_plan(cache, p, R, 1.0f, 0, &ap);
  if (p.Mtot == 0) {  // nothing to fit
    *bytes = 0;
    return ok();
  }
  size_t score_bytes = 0;
  if ((st = kvc_score_workspace_size(cache, segs, R, &score_bytes)) != KVC_OK) return st;
  *bytes = am_workspace_bytes(cache, ap, score_bytes, R);
  return ok();
}

kvc_status kvc_am_fit(const kvc_cache* cache, const kvc_segments* segs, const int32_t* m, const uint16_t* q,
                      int32_t R, float scale, const float* lse, const int32_t* keep, int32_t sweeps, float* beta,
                      float* vc, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  const NvtxRange nvtx_range("kvc_am_fit");
  Plan p;
  kvc_status st = check_am_args(cache, segs, m, R, &p);
  if (st != KVC_OK) return st;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return fail(KVC_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (sweeps < 0 || sweeps > 1000) return fail(KVC_ERR_INVALID_ARG, "sweeps = %d (allowed: 0..1000)", sweeps);
  if (p.Mtot == 0) return ok();
  if (q == nullptr || !aligned16(q)) return fail(KVC_ERR_INVALID_ARG, "q is NULL or not 16-byte aligned");
  if (keep == nullptr) return fail(KVC_ERR_INVALID_ARG, "keep is NULL");
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(KVC_ERR_INVALID_ARG, "lse is not 4-byte aligned");
  const int64_t qrows = (int64_t)cache->batch * cache->num_layers * cache->num_kv_heads * R;
  if (qrows >= (int64_t(1) << 31)) return fail(KVC_ERR_UNSUPPORTED, "B*L*H*R >= 2^31");
  AmPlan ap;
  build_am_plan(cache, p, R, scale, sweeps, &ap);
  size_t score_bytes = 0;
  if ((st = kvc_score_workspace_size(cache, segs, R, &score_bytes)) != KVC_OK) return st;
  const size_t need = am_workspace_bytes(cache, ap, score_bytes, R);
  if (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(KVC_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", need, ws_bytes);
  DeviceInfo di;
  if ((st = device_info(&di)) != KVC_OK) return st;
  // the LSE of every proxy row over its segment's keys: the caller's (the scoring
  // LSE pass's own output for the same rows), else the scoring LSE pass here
  uint8_t* score_ws = static_cast<uint8_t*>(ws) + align256((size_t)ap.floats * sizeof(float));
  const float* lse_rows = lse;
  if (lse_rows == nullptr) {
    float* own = reinterpret_cast<float*>(score_ws + align256(score_bytes));
    if ((st = score_common("kvc_am_fit", kPhaseLse, 2.0f, cache, segs, q, R, scale, nullptr, own, nullptr,
                           score_ws, align256(score_bytes), stream)) != KVC_OK)
      return st;
    lse_rows = own;
  }
  const int64_t krows = (int64_t)cache->num_layers * cache->num_pages * cache->num_kv_heads * cache->page_size;
  CUtensorMap tmK, tmV, tmQ;
  if ((st = make_kmap(&tmK, cache->k_pool, krows, cache->head_dim, cache->page_size)) != KVC_OK) return st;
  if ((st = make_kmap(&tmV, cache->v_pool, krows, cache->head_dim, cache->page_size)) != KVC_OK) return st;
  if ((st = make_tmap(&tmQ, q, qrows, cache->head_dim, kScoreTile)) != KVC_OK) return st;
  // per launch chunk: the units' E / Ph and Y for the Gram products
  const size_t nc = ap.metas.size();
  std::vector<CUtensorMap> tmX(nc), tmY(nc), tmH(nc), tmX0(nc);
  for (size_t ci = 0; ci < nc; ++ci) {
    const AmMeta& am = ap.metas[ci];
    const float* base = static_cast<const float*>(ws) + am.seq[0].ws;
    const int ldE = am.seq[0].ldE, d = cache->head_dim;
    const int64_t uf = am.seq[0].unit_floats;
    if ((st = make_amap(&tmX[ci], base, ldE, R, am.units, ldE, uf)) != KVC_OK ||
        (st = make_amap(&tmY[ci], base + am_off_Y(R, am.max_m, ldE), d, R, am.units, d, uf)) != KVC_OK ||
        (st = make_amap(&tmH[ci], base + am_off_G(R, ldE), ldE, am.max_m, am.units, ldE, uf)) != KVC_OK ||
        (st = make_amap(&tmX0[ci], base + am_off_X(R, am.max_m, ldE, d), d, am.max_m, am.units, d, uf)) != KVC_OK)
      return st;
  }
  AmLaunch al;
  al.chunks = ap.metas.size();
  al.meta = ap.metas.data();
  al.tmK = &tmK;
  al.tmVpool = &tmV;
  al.tmQ = &tmQ;
  al.tmX = tmX.data();
  al.tmY = tmY.data();
  al.tmH = tmH.data();
  al.tmX0 = tmX0.data();
  al.lse_rows = lse_rows;
  al.block_table = cache->block_table;
  al.k_pool = cache->k_pool;
  al.v_pool = cache->v_pool;
  al.q = q;
  al.keep = keep;
  al.ws = static_cast<float*>(ws);
  al.aux = cache->aux;
  al.beta = beta;
  al.vc = vc;
  al.status = di.status;
  const cudaError_t e = launch_am(al, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvc_am_fit launch");
  return launched(stream, "kvc_am_fit");
}

kvc_status kvc_read_device_status(uint32_t* out, int32_t clear, kvc_stream_t stream) {
  if (out == nullptr) return fail(KVC_ERR_INVALID_ARG, "out is NULL");
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol(status)");
  if (clear) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol(status)");
  }
  *out = v;
  return ok();
}

kvc_status kvc_validate_cache_host(const int32_t* block_table, const int32_t* nblocks, const int32_t* seq_len,
                                   int32_t batch, int32_t max_blocks, int32_t num_pages, int32_t page_size,
                                   const int32_t* free_ids, int32_t free_top) {
  if (block_table == nullptr || nblocks == nullptr || batch <= 0 || max_blocks <= 0 || num_pages <= 0 ||
      page_size <= 0)
    return fail(KVC_ERR_INVALID_ARG, "bad arguments");
  std::vector<int32_t> owner(num_pages, -1);  // -1 free/unknown, b = mapped by b, -2 on the free stack
  for (int b = 0; b < batch; ++b) {
    const int nb = nblocks[b];
    if (nb < 0 || nb > max_blocks) return fail(KVC_ERR_INVALID_ARG, "nblocks[%d] = %d out of range", b, nb);
    if (seq_len != nullptr && (seq_len[b] < 0 || ceil_div(seq_len[b], page_size) > nb))
      return fail(KVC_ERR_INVALID_ARG, "seq_len[%d] = %d needs more than %d blocks", b, seq_len[b], nb);
    for (int j = 0; j < max_blocks; ++j) {
      const int32_t pg = block_table[(int64_t)b * max_blocks + j];
      if (j >= nb) {
        if (pg != -1) return fail(KVC_ERR_INVALID_ARG, "block_table[%d][%d] = %d past nblocks is not -1", b, j, pg);
        continue;
      }
      if (pg < 0 || pg >= num_pages)
        return fail(KVC_ERR_INVALID_ARG, "block_table[%d][%d] = %d outside the pool", b, j, pg);
      if (owner[pg] != -1)
        return fail(KVC_ERR_INVALID_ARG, "page %d mapped twice (sequence %d block %d)", pg, b, j);
      owner[pg] = b;
    }
  }
  if (free_ids != nullptr) {
    if (free_top < 0 || free_top > num_pages) return fail(KVC_ERR_INVALID_ARG, "free_top = %d out of range", free_top);
    for (int i = 0; i < free_top; ++i) {
      const int32_t pg = free_ids[i];
      if (pg < 0 || pg >= num_pages) return fail(KVC_ERR_INVALID_ARG, "free_ids[%d] = %d outside the pool", i, pg);
      if (owner[pg] >= 0) return fail(KVC_ERR_INVALID_ARG, "page %d is both mapped and free", pg);
      if (owner[pg] == -2) return fail(KVC_ERR_INVALID_ARG, "page %d is free twice", pg);
      owner[pg] = -2;
    }
  }
  return ok();
}

}  // extern "C"
