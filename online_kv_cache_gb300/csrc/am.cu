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
// Work is fp32 on the CUDA cores: the fits are ill-conditioned (exp of
// logits), so their Gram matrices cannot take the 8-bit-mantissa rounding of a
// bf16 or tf32 tensor-core contraction.  Per unit the kernels run
//   am_targets_kernel  Y = softmax(L) V and LSE over all n keys (online softmax)
//   am_exp_kernel      E = exp(L_C - c) over the kept keys, s = exp(LSE - c)
//   am_atb_kernel      G = E^T [E | s]              (mode 0)
//   am_mass_kernel     w by projected coordinate descent; beta = ln w
//   am_probs_kernel    Ph = rows of E diag(w), normalised (in place)
//   am_atb_kernel      H = Ph^T Ph, Bm = Ph^T Y     (modes 1, 2)
//   am_value_kernel    V_C by coordinate descent; written to the pool (bf16)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int kAmThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
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

__device__ __forceinline__ void unpack8(const uint4 v, float* out) {
  out[0] = bf16_bits_to_float(v.x & 0xffffu);
  out[1] = bf16_bits_to_float(v.x >> 16);
  out[2] = bf16_bits_to_float(v.y & 0xffffu);
  out[3] = bf16_bits_to_float(v.y >> 16);
  out[4] = bf16_bits_to_float(v.z & 0xffffu);
  out[5] = bf16_bits_to_float(v.z >> 16);
  out[6] = bf16_bits_to_float(v.w & 0xffffu);
  out[7] = bf16_bits_to_float(v.w >> 16);
}

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
  u.base = ws + q.ws + (int64_t)r * q.unit_floats;
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

// 64 rows x D of a bf16 matrix into shared memory (fp32, row stride D + 1),
// zero rows where row_of(i) < 0.  16-byte loads, consecutive threads along a row.
template <int D, typename RowOf>
__device__ __forceinline__ void load_rows64(float* dst, const uint16_t* src, RowOf row_of) {
  constexpr int kChunks = D / 8;
  for (int ci = threadIdx.x; ci < 64 * kChunks; ci += kAmThreads) {
    const int i = ci / kChunks, dc = ci % kChunks;
    const int64_t row = row_of(i);
    float v[8];
    if (row >= 0) {
      unpack8(*reinterpret_cast<const uint4*>(src + row * D + dc * 8), v);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) dst[i * (D + 1) + dc * 8 + e] = v[e];
  }
}

// acc[a][b] = sum_k A[ty + 16a][k] * B[tx + 16b][k] over 64 x 64 tiles (stride D + 1).
template <int D>
__device__ __forceinline__ void dot64(const float* As, const float* Bs, int ty, int tx, float acc[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;
#pragma unroll 4
  for (int k = 0; k < D; ++k) {
    float qa[4], kb[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) qa[a] = As[(ty + 16 * a) * (D + 1) + k];
#pragma unroll
    for (int b = 0; b < 4; ++b) kb[b] = Bs[(tx + 16 * b) * (D + 1) + k];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(qa[a], kb[b], acc[a][b]);
  }
}

__device__ __forceinline__ float max16(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float sum16(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Targets tiling: 128 proxy rows per block, keys in tiles of 64.
constexpr int kTgRows = 128;
constexpr int kTgKeys = 64;
constexpr int kTgPs = kTgRows + 1;  // row stride of the probability tile (fewer bank conflicts)

template <int D>
constexpr int targets_kp_floats() {  // Kt [D][64], later Pt [64][129] in the same place
  return D * kTgKeys > kTgKeys * kTgPs ? D * kTgKeys : kTgKeys * kTgPs;
}

template <int D>
constexpr int targets_smem_bytes() {  // Qt [D][128], Kt / Pt, Vs [64][D]
  return (D * kTgRows + targets_kp_floats<D>() + kTgKeys * D) * 4;
}

// ------------------------------------------------------------------ targets
// Block = (unit, 128 proxy rows), 16 x 16 threads.  Online softmax over all n
// keys of the segment in tiles of 64.  Thread (ty, tx) forms the logits of rows
// 8 ty .. 8 ty + 7 against keys 4 tx .. 4 tx + 3 of the tile from Q and K held
// dimension-major in shared memory (three 128-bit loads per 32 multiply-adds),
// keeps the rows' running max (common to the 16 threads of a row, through
// shuffles) and its own share of their running sums, and accumulates Y rows
// 8 ty .. 8 ty + 7, columns tx D/16 .. tx D/16 + D/16 - 1 from the tile's
// probabilities (key-major, over the key tile once the logits are formed) and
// values.  Writes LSE (natural log) and Y = softmax(L) V to the unit's workspace.
template <int D>
__global__ void __launch_bounds__(kAmThreads) am_targets_kernel(const AmMeta meta, const int32_t* __restrict__ bt,
                                                                const uint16_t* __restrict__ kp,
                                                                const uint16_t* __restrict__ vp,
                                                                const uint16_t* __restrict__ q, float* ws,
                                                                unsigned* status) {
  extern __shared__ __align__(16) float am_smem[];
  constexpr int kCpt = D / 16;  // Y columns per thread
  constexpr int kChunks = D / 8;
  float* Qt = am_smem;                            // [D][128]
  float* Kt = Qt + D * kTgRows;                   // [D][64]
  float* Pt = Kt;                                 // [64][129]
  float* Vs = Kt + targets_kp_floats<D>();        // [64][D]
  const int rb = (meta.R + kTgRows - 1) / kTgRows;
  const int64_t unit = blockIdx.x / rb;
  const int r0 = (int)(blockIdx.x % rb) * kTgRows;
  const AmUnit u = am_unit(meta, unit, ws);
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int64_t qrow0 = (((int64_t)u.b * meta.L + u.l) * meta.H + u.h) * meta.R;
  for (int ci = threadIdx.x; ci < kTgRows * kChunks; ci += kAmThreads) {  // Q (zero past R)
    const int i = ci % kTgRows, dc = ci / kTgRows;
    float v[8];
    if (r0 + i < meta.R) {
      unpack8(*reinterpret_cast<const uint4*>(q + (qrow0 + r0 + i) * D + dc * 8), v);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) Qt[(dc * 8 + e) * kTgRows + i] = v[e];
  }
  const float c2 = meta.scale * kLog2e;
  float mx[8], sm[8], y[8][kCpt];
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    mx[a] = -INFINITY;
    sm[a] = 0.0f;
#pragma unroll
    for (int e = 0; e < kCpt; ++e) y[a][e] = 0.0f;
  }
  // The next tile's keys and values are loaded into registers while this
  // tile's products run (kLd 16-byte chunks of each per thread).
  constexpr int kLd = kTgKeys * kChunks / kAmThreads;
  static_assert(kLd * kAmThreads == kTgKeys * kChunks, "tile chunks split evenly over the threads");
  uint4 kr[kLd], vr[kLd];
  auto fetch = [&](int t0) {
#pragma unroll
    for (int c = 0; c < kLd; ++c) {
      const int ci = threadIdx.x + c * kAmThreads;
      const int ik = ci % kTgKeys, dk = ci / kTgKeys;  // keys: consecutive threads on consecutive keys
      const int iv = ci / kChunks, dv = ci % kChunks;  // values: consecutive threads along a row
      const int64_t rk = t0 + ik < u.n ? am_row(meta, u, bt, t0 + ik, status) : -1;
      const int64_t rv = t0 + iv < u.n ? am_row(meta, u, bt, t0 + iv, status) : -1;
      kr[c] = rk >= 0 ? *reinterpret_cast<const uint4*>(kp + rk * D + dk * 8) : make_uint4(0u, 0u, 0u, 0u);
      vr[c] = rv >= 0 ? *reinterpret_cast<const uint4*>(vp + rv * D + dv * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  fetch(0);
  for (int j0 = 0; j0 < u.n; j0 += kTgKeys) {
    __syncthreads();  // the previous tile's Pt and Vs are fully read
#pragma unroll
    for (int c = 0; c < kLd; ++c) {  // keys dimension-major, values key-major; bf16 bits -> fp32 (zero rows stay zero)
      const int ci = threadIdx.x + c * kAmThreads;
      const int ik = ci % kTgKeys, dk = ci / kTgKeys;
      const int iv = ci / kChunks, dv = ci % kChunks;
      float v[8];
      unpack8(kr[c], v);
#pragma unroll
      for (int e = 0; e < 8; ++e) Kt[(dk * 8 + e) * kTgKeys + ik] = v[e];
      unpack8(vr[c], v);
      float4* dst = reinterpret_cast<float4*>(Vs + iv * D + dv * 8);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    __syncthreads();
    if (j0 + kTgKeys < u.n) fetch(j0 + kTgKeys);
    float acc[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;
#pragma unroll 2
    for (int k = 0; k < D; ++k) {
      const float4 q0 = *reinterpret_cast<const float4*>(Qt + k * kTgRows + ty * 8);
      const float4 q1 = *reinterpret_cast<const float4*>(Qt + k * kTgRows + ty * 8 + 4);
      const float4 k0 = *reinterpret_cast<const float4*>(Kt + k * kTgKeys + tx * 4);
      const float qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      const float kv[4] = {k0.x, k0.y, k0.z, k0.w};
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(qv[a], kv[b], acc[a][b]);
    }
    __syncthreads();  // every thread's logits are formed: Kt is free for Pt
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      float t[4], tmax = -INFINITY;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        t[b] = (j0 + tx * 4 + b < u.n) ? acc[a][b] * c2 : -INFINITY;
        tmax = fmaxf(tmax, t[b]);
      }
      const float mnew = fmaxf(mx[a], max16(tmax));  // finite: key j0 is in the segment
      const float alpha = exp2f(mx[a] - mnew);        // 0 on the first tile (mx = -inf)
      float ps = 0.0f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float p = exp2f(t[b] - mnew);
        Pt[(tx * 4 + b) * kTgPs + ty * 8 + a] = p;
        ps += p;
      }
      sm[a] = sm[a] * alpha + ps;
      mx[a] = mnew;
#pragma unroll
      for (int e = 0; e < kCpt; ++e) y[a][e] *= alpha;
    }
    __syncthreads();
#pragma unroll 2
    for (int j = 0; j < kTgKeys; ++j) {
      float pv[8], vv[kCpt];
#pragma unroll
      for (int a = 0; a < 8; ++a) pv[a] = Pt[j * kTgPs + ty * 8 + a];
#pragma unroll
      for (int e = 0; e < kCpt; e += 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(Vs + j * D + tx * kCpt + e);
        vv[e] = v4.x;
        vv[e + 1] = v4.y;
        vv[e + 2] = v4.z;
        vv[e + 3] = v4.w;
      }
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int e = 0; e < kCpt; ++e) y[a][e] = fmaf(pv[a], vv[e], y[a][e]);
    }
  }
  float* Y = u.base + am_off_Y(meta.R, u.m, u.ldE);
  float* lse = u.base + am_off_lse(meta.R, u.m, u.ldE, D);
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const float s = sum16(sm[a]);  // every lane takes part in the shuffles
    const int i = r0 + ty * 8 + a;
    if (i >= meta.R) continue;
    const float inv = 1.0f / s;
#pragma unroll
    for (int e = 0; e < kCpt; e += 4)
      *reinterpret_cast<float4*>(Y + (int64_t)i * D + tx * kCpt + e) =
          make_float4(y[a][e] * inv, y[a][e + 1] * inv, y[a][e + 2] * inv, y[a][e + 3] * inv);
    if (tx == 0) lse[i] = (mx[a] + log2f(s)) * kLn2;
  }
}

template <int D>
constexpr int exp_smem_bytes() {
  return (2 * 64 * (D + 1) + 8) * 4;
}

// ------------------------------------------------------------------ exp
// Block = (unit, 64 proxy rows, 64 kept keys): E[i][j] = exp(L_ij - c) with
// c = max_i LSE_i, and (key block 0) column m = s_i = exp(LSE_i - c).
template <int D>
__global__ void __launch_bounds__(kAmThreads) am_exp_kernel(const AmMeta meta, const int32_t* __restrict__ bt,
                                                            const uint16_t* __restrict__ kp,
                                                            const uint16_t* __restrict__ q,
                                                            const int32_t* __restrict__ keep, float* ws,
                                                            unsigned* status) {
  extern __shared__ __align__(16) float am_smem[];
  float* Qs = am_smem;            // [64][D + 1]
  float* Ks = Qs + 64 * (D + 1);  // [64][D + 1]
  float* red = Ks + 64 * (D + 1); // [8]
  const int rb = (meta.R + 63) / 64;
  const int cb = (meta.max_m + 63) / 64;
  const int cblk = (int)(blockIdx.x % cb);
  const int64_t rest = blockIdx.x / cb;
  const int r0 = (int)(rest % rb) * 64;
  const AmUnit u = am_unit(meta, rest / rb, ws);
  if (cblk * 64 >= u.m) return;
  const float* lse = u.base + am_off_lse(meta.R, u.m, u.ldE, D);
  // c = max_i LSE_i of the unit
  float c = -INFINITY;
  for (int i = threadIdx.x; i < meta.R; i += kAmThreads) c = fmaxf(c, lse[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int64_t qrow0 = (((int64_t)u.b * meta.L + u.l) * meta.H + u.h) * meta.R;
  load_rows64<D>(Qs, q, [&](int i) -> int64_t { return r0 + i < meta.R ? qrow0 + r0 + i : -1; });
  const int j0 = cblk * 64;
  load_rows64<D>(Ks, kp, [&](int i) -> int64_t {
    if (j0 + i >= u.m) return -1;
    const int pos = am_kept(meta, u, keep, j0 + i, status);
    return pos < 0 ? -1 : am_row(meta, u, bt, pos, status);
  });
  __syncthreads();
  c = red[0];
#pragma unroll
  for (int w = 1; w < kAmThreads / 32; ++w) c = fmaxf(c, red[w]);
  float acc[4][4];
  dot64<D>(Qs, Ks, ty, tx, acc);
  const float c2 = meta.scale * kLog2e, cc = c * kLog2e;
  float* E = u.base;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = r0 + ty + 16 * a;
    if (i >= meta.R) continue;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int j = j0 + tx + 16 * b;
      if (j < u.m) E[(int64_t)i * u.ldE + j] = exp2f(fmaf(acc[a][b], c2, -cc));
    }
    if (cblk == 0 && tx == 0) E[(int64_t)i * u.ldE + u.m] = exp2f((lse[i] - c) * kLog2e);
  }
}

// ------------------------------------------------------------------ A^T B
// Block = (unit, 128 x 128 tile of C): C[p][q] = sum_i A[i][p] B[i][q] over the
// R proxy rows, 16 rows per step through shared memory; each thread holds an
// 8 x 8 sub-tile (rows ty*4 + {0..3, 64..67}, columns tx*4 + {0..3, 64..67}) and
// reads its operands with 128-bit shared loads (4 loads per 64 multiply-adds).
//   mode 0: A = E (m columns), B = [E | s] (m + 1), C = G        (stride ldE)
//   mode 1: A = B = Ph (m columns),                 C = H in G's place
//   mode 2: A = Ph, B = Y (d columns, stride d),    C = Bm       (stride d)
constexpr int kAtbTile = 128;

__global__ void __launch_bounds__(kAmThreads) am_atb_kernel(const AmMeta meta, float* ws, int mode) {
  __shared__ __align__(16) float As[16][kAtbTile];
  __shared__ __align__(16) float Bs[16][kAtbTile];
  const int mt = (meta.max_m + kAtbTile - 1) / kAtbTile;
  const int nt = mode == 2 ? (meta.d + kAtbTile - 1) / kAtbTile : (meta.max_m + 1 + kAtbTile - 1) / kAtbTile;
  const int ni = (int)(blockIdx.x % nt);
  const int mi = (int)((blockIdx.x / nt) % mt);
  const AmUnit u = am_unit(meta, blockIdx.x / ((int64_t)nt * mt), ws);
  const int M = u.m;
  const int N = mode == 0 ? u.m + 1 : (mode == 1 ? u.m : meta.d);
  const int p0 = mi * kAtbTile, q0 = ni * kAtbTile;
  if (p0 >= M || q0 >= N) return;
  const float* A = u.base;
  const int lda = u.ldE;
  const float* B = mode == 2 ? u.base + am_off_Y(meta.R, u.m, u.ldE) : u.base;
  const int ldb = mode == 2 ? meta.d : u.ldE;
  float* C = mode == 2 ? u.base + am_off_Bm(meta.R, u.m, u.ldE, meta.d) : u.base + am_off_G(meta.R, u.ldE);
  const int ldc = mode == 2 ? meta.d : u.ldE;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  float acc[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.0f;
  for (int i0 = 0; i0 < meta.R; i0 += 16) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {  // 16 x 128 of A and of B, consecutive threads along a row
      const int e = threadIdx.x + r * kAmThreads;
      const int ii = e >> 7, pp = e & 127;
      const bool in = i0 + ii < meta.R;
      As[ii][pp] = (in && p0 + pp < M) ? A[(int64_t)(i0 + ii) * lda + p0 + pp] : 0.0f;
      Bs[ii][pp] = (in && q0 + pp < N) ? B[(int64_t)(i0 + ii) * ldb + q0 + pp] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[i][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[i][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[i][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[i][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(av[a], bv[b], acc[a][b]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const int p = p0 + (a < 4 ? ty * 4 + a : 64 + ty * 4 + a - 4);
    if (p >= M) continue;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int qq = q0 + (b < 4 ? tx * 4 + b : 64 + tx * 4 + b - 4);
      if (qq < N) C[(int64_t)p * ldc + qq] = acc[a][b];
    }
  }
}

// ------------------------------------------------------------------ row ring
// The descents read one row of a Gram matrix per step.  Rows stream from L2
// into a ring of kRing shared-memory buffers, kAhead = kRing - 2 steps ahead
// of use.  The buffer refilled at step st was last read at step st - 2, and
// every thread has passed step st - 1's barriers before it issues the copy,
// so no copy lands in a buffer that is still being read.  (Two buffers with
// the copy one step ahead would refill the buffer of step st - 1 while slower
// threads may still be reading it.)  Deeper rings (4, 6 buffers) measured no
// faster.
constexpr int kRing = 3;
constexpr int kAhead = kRing - 2;

struct RowRing {
  float* rows;      // [kRing][m] shared
  const float* Mx;  // the Gram matrix, leading dimension ld
  int64_t ld;
  int m;
  int row = 0, buf = 0;  // row and buffer of the next copy
  // Issue the next row's copy when `live`; commit a group either way, so that
  // group k always belongs to step k.
  __device__ __forceinline__ void issue(bool live) {
    if (live) {
      const float* src = Mx + (int64_t)row * ld;
      float* dst = rows + buf * m;
      for (int i = threadIdx.x; i < m; i += kAmThreads) cp_async_4(dst + i, src + i);
    }
    cp_async_commit();
    row = (row + 1 == m) ? 0 : row + 1;
    buf = (buf + 1 == kRing) ? 0 : buf + 1;
  }
};

// ------------------------------------------------------------------ mass fit
// Block = unit.  Projected cyclic coordinate descent on min_{w >= 0} ||E w - s||^2
// from w = 1: with g = G w - b, coordinate j moves to max(0, w_j - g_j / G_jj)
// and g follows by the change times column j of G (= row j, G symmetric).
// Coordinate j moves only when |g_j| > 2^-17 b_j (every term of G w and of
// b = E^T s is >= 0, so b_j is their scale).  Rows of G stream through the
// row ring.  Two barriers per step: every thread reads g_j and w_j before any
// of them is updated.
// Writes w (workspace), beta = ln w (-inf at 0) to `beta` and to the per-slot
// state of each kept entry.
__global__ void __launch_bounds__(kAmThreads) am_mass_kernel(const AmMeta meta, const int32_t* __restrict__ bt,
                                                             const int32_t* __restrict__ keep, float* ws,
                                                             float* aux, float* beta, unsigned* status) {
  extern __shared__ __align__(16) float am_smem[];
  const AmUnit u = am_unit(meta, blockIdx.x, ws);
  const int m = u.m;
  float* g = am_smem;         // [m]
  float* w = g + m;           // [m]
  float* diag = w + m;        // [m]
  float* bvec = diag + m;     // [m] b = E^T s
  float* rows = bvec + m;     // [kRing][m]
  const float* G = u.base + am_off_G(meta.R, u.ldE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < m; i += kAmThreads / 32) {  // g = G 1 - b, one warp per row
    const float* gr = G + (int64_t)i * u.ldE;
    float acc = 0.0f;
    for (int k = lane; k < m; k += 32) acc += gr[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      g[i] = acc - gr[m];
      bvec[i] = gr[m];
      diag[i] = gr[i];
      w[i] = 1.0f;
    }
  }
  const int64_t steps = (int64_t)meta.sweeps * m;
  RowRing ring{rows, G, u.ldE, m};
  for (int p = 0; p < kAhead; ++p) ring.issue(p < steps);
  int j = 0, cb = 0;  // step st's row and ring buffer
  for (int64_t st = 0; st < steps; ++st) {
    ring.issue(st + kAhead < steps);
    cp_async_wait_group<kAhead>();  // this thread's copies of step st's row are in
    __syncthreads();
    const float gj = g[j], wj = w[j], Gjj = diag[j];
    const float nw = (Gjj > 0.0f && fabsf(gj) > kAmGuard * bvec[j]) ? fmaxf(0.0f, wj - gj / Gjj) : wj;
    const float dl = nw - wj;
    __syncthreads();
    if (dl != 0.0f) {
      const float* rj = rows + cb * m;
      for (int i = threadIdx.x; i < m; i += kAmThreads) g[i] = fmaf(dl, rj[i], g[i]);
      if (threadIdx.x == 0) w[j] = nw;
    }
    j = (j + 1 == m) ? 0 : j + 1;
    cb = (cb + 1 == kRing) ? 0 : cb + 1;
  }
  cp_async_wait_all();
  __syncthreads();
  float* wout = u.base + am_off_w(meta.R, m, u.ldE, meta.d);
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
// Ph_ij = E_ij w_j / z_i in place (a row without mass stays zero).
__global__ void __launch_bounds__(kAmThreads) am_probs_kernel(const AmMeta meta, float* ws) {
  const int rb = (meta.R + 7) / 8;
  const AmUnit u = am_unit(meta, blockIdx.x / rb, ws);
  const int i = (int)(blockIdx.x % rb) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= meta.R) return;
  float* E = u.base + (int64_t)i * u.ldE;
  const float* w = u.base + am_off_w(meta.R, u.m, u.ldE, meta.d);
  float z = 0.0f;
  for (int j = lane; j < u.m; j += 32) z = fmaf(E[j], w[j], z);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  const float inv = z > 0.0f ? 1.0f / z : 0.0f;
  for (int j = lane; j < u.m; j += 32) E[j] = E[j] * w[j] * inv;
}

constexpr int kValueCols = 8;  // value-fit columns per block (32 row slices x 8 columns)

__host__ __device__ constexpr int value_smem_bytes(int m) {
  return (2 * m * kValueCols + (2 + kRing) * m + (kAmThreads / kValueCols + 1) * kValueCols) * 4;
}
__host__ __device__ constexpr int mass_smem_bytes(int m) { return (4 + kRing) * m * 4; }
static_assert(value_smem_bytes(kAmMaxM) <= 227 * 1024 && mass_smem_bytes(kAmMaxM) <= 227 * 1024,
              "descent working sets fit one CTA's shared memory at the largest m");

// ------------------------------------------------------------------ value fit
// Block = (unit, 8 of the d value columns).  The columns are independent
// least-squares problems sharing H = Ph^T Ph: cyclic coordinate descent from
// X = the kept values, gradient Gv = H X - Bm kept in shared memory; row j of
// X moves by -Gv_j / H_jj and Gv follows by column j of H (= row j) times the
// change, when |Gv_jc| > 2^-17 pi_j S_c (pi_j = sum_k H_jk, S_c = max_i |Y_ic|
// + max_k |X0_kc|: the scale of the gradient's terms in column c).  Rows of H
// stream through the row ring.  At the end V_C is
// written to `vc` (fp32) and over the kept entries' V rows (bf16, round to
// nearest even).
template <int D>
__global__ void __launch_bounds__(kAmThreads) am_value_kernel(const AmMeta meta, const int32_t* __restrict__ bt,
                                                              const int32_t* __restrict__ keep, uint16_t* vp,
                                                              float* ws, float* vc, unsigned* status) {
  extern __shared__ __align__(16) float am_smem[];
  constexpr int kCb = D / kValueCols;
  const AmUnit u = am_unit(meta, blockIdx.x / kCb, ws);
  const int col0 = (int)(blockIdx.x % kCb) * kValueCols;
  const int m = u.m;
  float* Gv = am_smem;                 // [m][8]
  float* X = Gv + m * kValueCols;      // [m][8]
  float* hdiag = X + m * kValueCols;   // [m]
  float* pi = hdiag + m;               // [m]
  float* rows = pi + m;                // [kRing][m]
  float* red = rows + kRing * m;       // [32][8] partial column scales, then S[8]
  const float* Hm = u.base + am_off_G(meta.R, u.ldE);
  const float* Bm = u.base + am_off_Bm(meta.R, m, u.ldE, D);
  const int c = threadIdx.x & (kValueCols - 1), r = threadIdx.x / kValueCols;
  constexpr int kSlices = kAmThreads / kValueCols;
  for (int j = threadIdx.x; j < m; j += kAmThreads) {  // start: the kept entries' values
    const int pos = am_kept(meta, u, keep, j, status);
    const int64_t row = pos < 0 ? -1 : am_row(meta, u, bt, pos, status);
    float v[8];
    if (row >= 0) {
      unpack8(*reinterpret_cast<const uint4*>(vp + row * D + col0), v);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) X[j * kValueCols + e] = v[e];
    hdiag[j] = Hm[(int64_t)j * u.ldE + j];
  }
  __syncthreads();
  {  // S_c = max_i |Y_ic| + max_k |X0_kc|
    const float* Y = u.base + am_off_Y(meta.R, m, u.ldE);
    float ym = 0.0f, xm = 0.0f;
    for (int i = r; i < meta.R; i += kSlices) ym = fmaxf(ym, fabsf(Y[(int64_t)i * D + col0 + c]));
    for (int k = r; k < m; k += kSlices) xm = fmaxf(xm, fabsf(X[k * kValueCols + c]));
    red[r * kValueCols + c] = ym;
    __syncthreads();
    if (r == 0) {
      for (int t = 1; t < kSlices; ++t) ym = fmaxf(ym, red[t * kValueCols + c]);
    }
    __syncthreads();
    red[r * kValueCols + c] = xm;
    __syncthreads();
    if (r == 0) {
      for (int t = 1; t < kSlices; ++t) xm = fmaxf(xm, red[t * kValueCols + c]);
      red[kSlices * kValueCols + c] = ym + xm;
    }
  }
  for (int i = r; i < m; i += kSlices) {  // Gv = H X - Bm and pi = H 1
    const float* hr = Hm + (int64_t)i * u.ldE;
    float acc = 0.0f, ps = 0.0f;
    for (int k = 0; k < m; ++k) {
      acc = fmaf(hr[k], X[k * kValueCols + c], acc);
      ps += hr[k];
    }
    Gv[i * kValueCols + c] = acc - Bm[(int64_t)i * D + col0 + c];
    if (c == 0) pi[i] = ps;
  }
  __syncthreads();
  const float Sc = red[kSlices * kValueCols + c];
  const int64_t steps = (int64_t)meta.sweeps * m;
  RowRing ring{rows, Hm, u.ldE, m};
  for (int p = 0; p < kAhead; ++p) ring.issue(p < steps);
  int j = 0, cb = 0;  // step st's row and ring buffer
  for (int64_t st = 0; st < steps; ++st) {
    ring.issue(st + kAhead < steps);
    cp_async_wait_group<kAhead>();  // this thread's copies of step st's row are in
    __syncthreads();
    const float Hjj = hdiag[j];
    const float gv = Gv[j * kValueCols + c];
    const float dl = (Hjj > 0.0f && fabsf(gv) > kAmGuard * pi[j] * Sc) ? -gv / Hjj : 0.0f;
    __syncthreads();
    if (dl != 0.0f) {
      const float* rj = rows + cb * m;
      for (int i = r; i < m; i += kSlices) Gv[i * kValueCols + c] = fmaf(rj[i], dl, Gv[i * kValueCols + c]);
      if (r == 0) X[j * kValueCols + c] += dl;
    }
    j = (j + 1 == m) ? 0 : j + 1;
    cb = (cb + 1 == kRing) ? 0 : cb + 1;
  }
  cp_async_wait_all();
  __syncthreads();
  const int64_t orow = ((int64_t)u.l * meta.H + u.h) * meta.Mtot + u.moff;
  for (int j = r; j < m; j += kSlices) {
    const float x = X[j * kValueCols + c];
    if (vc != nullptr) vc[(orow + j) * D + col0 + c] = x;
    const int pos = am_kept(meta, u, keep, j, status);
    const int64_t row = pos < 0 ? -1 : am_row(meta, u, bt, pos, status);
    if (row >= 0) {
      const __nv_bfloat16 hb = __float2bfloat16_rn(x);
      vp[row * D + col0 + c] = *reinterpret_cast<const uint16_t*>(&hb);
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
    if ((e = set_smem(am_targets_kernel<D>, targets_smem_bytes<D>())) != cudaSuccess) return e;
    if ((e = set_smem(am_exp_kernel<D>, exp_smem_bytes<D>())) != cudaSuccess) return e;
    if ((e = set_smem(am_mass_kernel, mass_smem_bytes(kAmMaxM))) != cudaSuccess) return e;
    if ((e = set_smem(am_value_kernel<D>, value_smem_bytes(kAmMaxM))) != cudaSuccess) return e;
    if (dev < 64) attr_set[dev] = true;
  }
  const uint16_t* kp = static_cast<const uint16_t*>(al.k_pool);
  uint16_t* vp = static_cast<uint16_t*>(al.v_pool);
  auto check = [&]() {
    count_launch();
    return cudaGetLastError();
  };
  for (size_t ci = 0; ci < al.chunks; ++ci) {
    const AmMeta& m = al.meta[ci];
    if (m.units <= 0) continue;
    const int rb64 = (m.R + 63) / 64;
    const int mt = (m.max_m + 63) / 64;
    const int rbt = (m.R + kTgRows - 1) / kTgRows;
    am_targets_kernel<D><<<(unsigned)(m.units * rbt), kAmThreads, targets_smem_bytes<D>(), stream>>>(
        m, al.block_table, kp, vp, al.q, al.ws, al.status);
    if ((e = check()) != cudaSuccess) return e;
    am_exp_kernel<D><<<(unsigned)(m.units * rb64 * mt), kAmThreads, exp_smem_bytes<D>(), stream>>>(
        m, al.block_table, kp, al.q, al.keep, al.ws, al.status);
    if ((e = check()) != cudaSuccess) return e;
    const int mt128 = (m.max_m + kAtbTile - 1) / kAtbTile;
    const int nt0 = (m.max_m + 1 + kAtbTile - 1) / kAtbTile;
    am_atb_kernel<<<(unsigned)(m.units * mt128 * nt0), kAmThreads, 0, stream>>>(m, al.ws, 0);
    if ((e = check()) != cudaSuccess) return e;
    am_mass_kernel<<<(unsigned)m.units, kAmThreads, mass_smem_bytes(m.max_m), stream>>>(
        m, al.block_table, al.keep, al.ws, al.aux, al.beta, al.status);
    if ((e = check()) != cudaSuccess) return e;
    am_probs_kernel<<<(unsigned)(m.units * ((m.R + 7) / 8)), kAmThreads, 0, stream>>>(m, al.ws);
    if ((e = check()) != cudaSuccess) return e;
    am_atb_kernel<<<(unsigned)(m.units * mt128 * nt0), kAmThreads, 0, stream>>>(m, al.ws, 1);
    if ((e = check()) != cudaSuccess) return e;
    am_atb_kernel<<<(unsigned)(m.units * mt128 * ((D + kAtbTile - 1) / kAtbTile)), kAmThreads, 0, stream>>>(m, al.ws, 2);
    if ((e = check()) != cudaSuccess) return e;
    am_value_kernel<D><<<(unsigned)(m.units * (D / kValueCols)), kAmThreads, value_smem_bytes(m.max_m), stream>>>(
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
