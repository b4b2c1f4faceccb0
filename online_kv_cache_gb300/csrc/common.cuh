// common.cuh -- launch metadata shared by the kernels and the host front end.
//
// The host knows every segment length and budget, so it sizes all grids and
// offsets itself and passes them by value in the kernel parameter block (no
// host->device copy, no device->host read on the hot path).  Sequences are
// processed in chunks of at most kMaxSeqPerLaunch per launch.
#pragma once

#include <cstdint>

#include "kvc.h"

namespace kvc {

constexpr int kMaxSeqPerLaunch = 128;

// Keys per K tile and rows per Q row tile of the scoring passes, as the host
// sizes their work split, workspaces and tensor-map boxes (score.cu's kTile).
constexpr int kScoreTile = 128;

struct SeqMeta {
  int32_t b;      // sequence index (block-table row)
  int32_t s0;     // first slot of the segment
  int32_t n;      // segment length (slots)
  int32_t m;      // budget, clamped to n
  int32_t nb;     // ceil(n / P): blocks of the segment
  int32_t X;      // ceil(m / P): blocks of the target region
  int32_t split;  // score pass 1: key splits per unit
  int32_t xoff;   // fresh-page compaction: first of the sequence's popped pages
  int64_t off;    // offset of the sequence in the [L][H][Ntot] score rows
  int64_t moff;   // offset in the [L][H][Mtot] keep / move rows
  int64_t foff;   // offset in the freed-page list
  int64_t item0;  // first work item of the sequence in this launch
  int64_t item1;  // first work item of the sequence in a companion launch
};

struct LaunchMeta {
  int32_t nseq;  // sequences in this launch
  int32_t L, H, P, d;
  int32_t num_pages, max_blocks, B;
  int32_t R;        // proxy rows per unit
  int32_t R_pad;    // R rounded up to nchunks * W
  int32_t rowtiles; // ceil(R / 128) (score pass 1)
  int32_t W;        // Q rows per pass-2 chunk (multiple of 32, <= 256)
  int32_t nchunks;  // R_pad / W
  int32_t ngroups;  // row groups of a scoring pass (each resident in shared memory)
  int32_t gsub;     // jobs per K tile of a full group (row tiles or chunks)
  int32_t kst;      // K-tile ring stages of a scoring pass
  int32_t qbytes;   // shared-memory bytes of one resident row group
  int32_t log2P;    // log2(P)
  int32_t words;    // plan: 32-bit bitmap words covering the largest target region
  int32_t mpb;      // copy: moves per block
  float scale;      // logit scale
  float pw;         // score pass 2: power of alpha summed per key (2: eviction score, 1: action attention)
  int64_t Ntot, Mtot, Ftot;
  int64_t Xtot;     // fresh-page compaction: pages popped by the whole call
  int64_t items;    // work items of this launch
  int64_t stall_ns; // scoring passes, failure-path test only: > 0 withholds the proxy-row loads
                    // and limits every wait between the kernel's roles to stall_ns (0: normal)
  SeqMeta seq[kMaxSeqPerLaunch];
};

// Index of the sequence owning work item `item` (seq[i].item0 ascending).
__device__ __forceinline__ int find_seq(const LaunchMeta& meta, int64_t item) {
  int lo = 0, hi = meta.nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (meta.seq[mid].item0 <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace kvc
