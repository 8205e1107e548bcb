// Split-KV plan of the sparse decode attention, shared by the kernels and the host.
#pragma once

#include "bs_internal.cuh"

namespace bsi {

constexpr int kStagePages = 4;                     // pages staged per pipeline step
constexpr int kStageTokens = kStagePages * kPage;  // 64 tokens
constexpr int kClusterSplits = 16;                 // most splits of a unit in one thread-block cluster
constexpr int kClusterMaxPages = 1024;             // largest selection (pages) the cluster mode takes
constexpr int kAttnMaxSplits = 32;                 // splits of a unit in the workspace mode

// One partial record per (unit, split, head) in the workspace mode: o[D]
// (unnormalised), m (log2 units), l, 2 pad.
__host__ __device__ constexpr int attn_record_floats(int D) { return D + 4; }

// The workspace starts with four int32 words per unit, padded to 16 bytes:
//   [0, U)    selection tickets of the fused step's front kernel;
//   [U, 2U)   arrival tickets of the attention's splits;
//   [2U, 3U)  the fused step's published selections: (epoch << 16) | count;
//   [3U, 4U)  the epoch the next published selection carries, minus one (kept by the
//             attention of the fused step).
// After them: in cluster mode the fused step's page lists (int32 [units][max gather
// pages]: the physical pages of each unit's selected blocks in attention order); in
// workspace mode the split records.
__host__ __device__ constexpr size_t attn_counter_floats(size_t units) { return (4 * units + 3) / 4 * 4; }
__host__ __device__ constexpr size_t attn_plist_ints(size_t units, int max_gather) {
  return (units * static_cast<size_t>(max_gather) + 3) / 4 * 4;
}
constexpr int kEpochMask = 0x7fff;  // epochs of published selections wrap at 2^15

// Counter words of unit u inside the workspace's first block.
struct StepWords {
  int32_t *tickets, *arrivals, *pub, *expect;
};
__host__ __device__ inline StepWords step_words(void *workspace, size_t units) {
  int32_t *w = static_cast<int32_t *>(workspace);
  return StepWords{w, w + units, w + 2 * units, w + 3 * units};
}

constexpr int kMidSplitPages = 24;     // workspace mode up to 1024 pages: pages per split, at least
constexpr int kClusterSmallPages = 256; // cluster mode for any unit count up to this selection
constexpr int kClusterUnitsMax = 19; // cluster mode while units x 16 splits fit one wave of ~304 CTAs ...
constexpr int kManyUnits = 304;      // ... or once the units alone fill it (then one split each)

// Attention modes, chosen from the dims only.
//   cluster:   selections up to 1024 pages with few units (<= 19), many units (>= 304)
//              or selections up to 256 pages; a unit's S splits are one thread-block
//              cluster and merge through distributed shared memory; every unit has the
//              same number of splits;
//   workspace: the rest (selections above 1024 pages, or 20..303 units with selections
//              that may exceed 256 pages, whose page counts can then differ a lot
//              between units): each unit's splits are sized by its own pages (at least
//              24 per split up to 1024 pages, 4 beyond, so a long unit gets more
//              splits), up to 32, and merge
//              through records in the workspace.
enum AttnMode { kModeCluster = 0, kModeWorkspace = 1 };

__host__ __device__ inline bool attn_cluster_mode(int units, int max_gather_pages) {
  if (max_gather_pages > kClusterMaxPages) return false;
  return units <= kClusterUnitsMax || units >= kManyUnits || max_gather_pages <= kClusterSmallPages;
}

__host__ __device__ inline int attn_mode(int units, int max_gather_pages) {
  return attn_cluster_mode(units, max_gather_pages) ? kModeCluster : kModeWorkspace;
}

// The fused decode step selects in a kernel of its own (three launches: scores,
// selection, attention) in workspace mode when a unit can have more candidates than
// kFrontSelectMaxCandidates (eight per thread of a front CTA); otherwise the front
// kernel's CTA that finishes a unit's last score tile selects it (two launches).
constexpr int kFrontSelectMaxCandidates = 2048;
__host__ __device__ inline bool step_selects_apart(int units, int max_gather_pages, int max_blocks) {
  // (the tail block is always forced: at most max_blocks - 1 candidates)
  return attn_mode(units, max_gather_pages) == kModeWorkspace && max_blocks - 1 > kFrontSelectMaxCandidates;
}

// Floats of the workspace before the split records (the counters), and the floats of
// the records themselves (workspace mode: 32 per unit, index unit, split).
__host__ __device__ inline size_t attn_records_offset(size_t units) { return attn_counter_floats(units); }
__host__ __device__ inline size_t attn_record_area_floats(size_t units, int G, int D, int mode) {
  return mode == kModeWorkspace ? units * 32 * static_cast<size_t>(G) * (D + 4) : 0;
}

// Smallest split (pages) in workspace mode.
__host__ __device__ inline int attn_min_split_pages(int max_gather_pages) {
  return max_gather_pages > kClusterMaxPages ? kStagePages : kMidSplitPages;
}

// Splits of a unit in cluster mode: the largest power of two (at most 16) that keeps
// the launch within one wave of `slots` CTAs (about two per SM), at least 1. Few units:
// 16 short splits each; many units: one wave of long splits, so the fixed latency of
// a CTA's start (count, row, page table, first copy) is paid once per many pages.
__host__ __device__ inline int attn_cluster_splits(int units, int max_gather_pages, int slots) {
  (void)max_gather_pages;
  int s = kClusterSplits;
  while (s > 1 && static_cast<long long>(units) * s > slots) s >>= 1;
  return s;
}

// Splits launched per unit.
__host__ __device__ inline int attn_grid_splits(int units, int max_gather_pages, int slots) {
  if (attn_cluster_mode(units, max_gather_pages)) return attn_cluster_splits(units, max_gather_pages, slots);
  const int mn = attn_min_split_pages(max_gather_pages);
  int splits = (max_gather_pages + mn - 1) / mn;
  if (splits > kAttnMaxSplits) splits = kAttnMaxSplits;
  return splits < 1 ? 1 : splits;
}

// Pages covered by a unit's selection: every selected block but the last is complete
// (only the tail block can be partial and it has the largest index).
struct UnitPages {
  int n_pages;   // gathered pages (0 when the unit has nothing to attend or is invalid)
  int ppb;       // pages per block
  int pps;       // pages per split
  int n_split;
};

// The split plan depends only on the unit's own page count and the launch's splits per
// unit in cluster mode (cluster_splits; 0 in workspace mode, where splits hold at least
// min_pps pages).
__device__ __forceinline__ UnitPages unit_pages(int T, int g, int cnt, int last_blk, int cluster_splits,
                                                int min_pps) {
  UnitPages p;
  p.ppb = g / kPage;
  p.n_pages = 0;
  p.pps = kStagePages;
  p.n_split = 0;
  if (cnt <= 0 || T < 1 || last_blk < 0 || last_blk * g >= T) return p;
  const int rem_pages = (T - last_blk * g + kPage - 1) / kPage;
  const int last_pages = rem_pages < p.ppb ? rem_pages : p.ppb;
  p.n_pages = (cnt - 1) * p.ppb + last_pages;
  if (cluster_splits > 0) {
    p.pps = (p.n_pages + cluster_splits - 1) / cluster_splits;
  } else {
    int per = (p.n_pages + kStagePages * kAttnMaxSplits - 1) / (kStagePages * kAttnMaxSplits);
    if (per < 1) per = 1;
    p.pps = kStagePages * per;
    if (p.pps < min_pps) p.pps = min_pps;
  }
  p.n_split = (p.n_pages + p.pps - 1) / p.pps;
  return p;
}

}  // namespace bsi
