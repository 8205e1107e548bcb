// Device code of the block scores (a2), shared by the stand-alone kernel and the fused
// decode step: the second stage of NOSA's two-stage pooling ("Technisches Resümee:
// NOSA", Methodik / 1. Algorithmus: NOSA, "Blockweise Implementierung": max pooling
// at block level), shared by the query heads of a GQA group ("Technische Samenvatting:
// Fluxion", Systeemcomponenten, "Granularity-Budget Selector").
//
// A CTA of 256 threads scores tiles of 64 consecutive summary rows (64/r whole
// blocks, r = g/s), each arriving in shared memory with one bulk copy (two buffers
// when a CTA takes several tiles: the next tile's copy flies during this one). Each warp
// takes 8 rows; each lane keeps its slice of the G query vectors (pre-scaled by
// 1/sqrt(d)) in registers and reads its slice of every row once, and a butterfly
// reduce-scatter across the lanes completes the dot products: shared memory is read
// once per summary byte.
#pragma once

#include <math.h>

#include "bs_internal.cuh"

namespace bsi {

constexpr int kScoreThreads = 256;
constexpr int kTileRows = 64;

template <int D, int G>
struct ScoreLayout {
  static constexpr int kTileBytes = kTileRows * D * 4;
  // nb tile buffers, then the G query vectors [G][D] and the dot products [64][G].
  __host__ __device__ static constexpr int off_q(int nb) { return nb * kTileBytes; }
  __host__ __device__ static constexpr int off_dots(int nb) { return off_q(nb) + G * D * 4; }
  __host__ __device__ static constexpr int bytes(int nb) { return off_dots(nb) + kTileRows * G * 4; }
  static constexpr int kBytes = kTileRows * D * 4 + G * D * 4 + kTileRows * G * 4;  // one buffer
};

// Blocks of a unit's candidate range covered by one tile, and the tile count.
__host__ __device__ __forceinline__ int score_blocks_per_tile(int g, int s) { return kTileRows / (g / s); }
__host__ __device__ __forceinline__ int score_tiles(const Geom &ge) {
  const int bpt = score_blocks_per_tile(ge.g, ge.s);
  return (ge.c_hi - ge.c_lo + bpt - 1) / bpt;
}

// Thread 0 initialises nb copy barriers; the caller synchronises before their use.
__device__ __forceinline__ void score_bars_init(uint64_t *bars, int nb) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < nb; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
}

// Starts (thread 0) the bulk copy of summary rows [row0, min(row0 + 64, row_end)) of a
// unit (summ_unit: its first row, 16-byte aligned) into `buf` on barrier `bar` and
// returns the row count to every thread (0: nothing in flight).
template <int D>
__device__ __forceinline__ int score_copy(const float *summ_unit, int64_t row0, int64_t row_end, void *buf,
                                          uint64_t *bar) {
  const int64_t left = row_end - row0;
  const int n = row0 < 0 ? 0 : static_cast<int>(left < kTileRows ? (left > 0 ? left : 0) : kTileRows);
  if (threadIdx.x == 0 && n > 0) {
    const uint32_t bytes = static_cast<uint32_t>(n) * D * sizeof(float);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(buf, summ_unit + row0 * D, bytes, bar);
  }
  return n;
}

// The G query vectors of the unit, pre-scaled by 1/sqrt(d), into shared memory.
template <int D, int G>
__device__ __forceinline__ void score_load_q(float *qs, const void *qrow, int q_dtype) {
  const float scale = rsqrtf(static_cast<float>(D));
  for (int i = threadIdx.x; i < G * D; i += kScoreThreads) qs[i] = load_scalar(qrow, i, q_dtype) * scale;
}

// Waits for a copy of n_loaded rows on `bar` (phase `parity`); false (for every
// thread) when it timed out. All threads call it.
__device__ __forceinline__ bool score_wait(uint64_t *bar, uint32_t parity, int n_loaded, int32_t *st) {
  const bool ok = n_loaded == 0 || mbar_wait_bounded(bar, parity, st);
  return !__syncthreads_or(!ok);
}

// Scores tile `tile` of the unit's candidates from `tile_sm` (rows from c_lo * r + 64 *
// tile, n_loaded of them, covering the tile) into row_out[c] (c = block index). qs holds
// the scaled queries (visible to all threads). All 256 threads call it; the tile buffer
// is no longer read when it returns.
//
// Dot products: warp w takes rows 8w .. 8w+7 of the tile; lane l owns dimensions
// [l*DPL, (l+1)*DPL) and keeps the G query slices of them in registers, so shared
// memory is read once per row (a contiguous row per warp). Each lane forms the 8 x G
// partial sums of its dimensions; a butterfly reduce-scatter over the 32 lanes (values
// halved at each of 5 stages) leaves lane l with the full sums of entries
// [l*NF, (l+1)*NF) of the row-major (row, head) list.
template <int D, int G>
__device__ void score_compute(const float *tile_sm, const float *qs, float *dots, const Geom &ge, int tile,
                              int reduce, int n_loaded, float *row_out) {
  const int tid = threadIdx.x;
  const int r = ge.g / ge.s;
  const int bpt = kTileRows / r;
  const int c_first = ge.c_lo + tile * bpt;
  const int nb = min(bpt, ge.c_hi - c_first);
  const int nrows = min(nb * r, n_loaded);
  static_assert(D % 32 == 0 && D / 32 <= 4, "head_dim 32..128");
  constexpr int DPL = D / 32;
  constexpr int GP = G <= 4 ? 4 : 8;  // heads padded to a power of two
  constexpr int PV = 8 * GP;          // partials per lane: 32 or 64
  constexpr int NF = PV / 32;         // full sums per lane after the reduction
  const int lane = tid & 31, warp = tid >> 5;
  float qv[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < DPL; ++j) qv[h][j] = qs[h * D + lane * DPL + j];
  float part[PV];
#pragma unroll
  for (int i = 0; i < PV; ++i) part[i] = 0.0f;
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int row = warp * 8 + rr;
    if (row < nrows) {
      float kv[DPL];
      const float *rp = tile_sm + row * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 k4 = *reinterpret_cast<const float4 *>(rp);
        kv[0] = k4.x;
        kv[1] = k4.y;
        kv[2] = k4.z;
        kv[3] = k4.w;
      } else if constexpr (DPL == 2) {
        const float2 k2 = *reinterpret_cast<const float2 *>(rp);
        kv[0] = k2.x;
        kv[1] = k2.y;
      } else {
#pragma unroll
        for (int j = 0; j < DPL; ++j) kv[j] = rp[j];
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc = fmaf(qv[h][j], kv[j], acc);
        part[rr * GP + h] = acc;
      }
    }
  }
  // Reduce-scatter: at offset o the lane keeps the half of its values selected by
  // (lane & o) and adds the partner's copy of that half.
#pragma unroll
  for (int o = 16, n = PV; o >= 1; o >>= 1, n >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < PV / 2; ++i) {
      if (i < n / 2) {
        const float send = upper ? part[i] : part[i + n / 2];
        const float keep = upper ? part[i + n / 2] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NF; ++j) {
    const int idx = lane * NF + j;
    const int rr = idx / GP, h = idx % GP;
    const int row = warp * 8 + rr;
    if (h < G && row < nrows) dots[row * G + h] = part[j];
  }
  __syncthreads();
  // Max over the r sub-blocks of a block per head, then over (or mean across) heads.
  if (tid < nb) {
    float red = reduce == BS_GROUP_MAX ? -INFINITY : 0.0f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float m = -INFINITY;
      for (int j = 0; j < r; ++j) m = fmaxf(m, dots[(tid * r + j) * G + h]);
      red = reduce == BS_GROUP_MAX ? fmaxf(red, m) : red + m;
    }
    if (reduce != BS_GROUP_MAX) red = red / static_cast<float>(G);
    row_out[c_first + tid] = red;
  }
  __syncthreads();  // dots are free again
}

}  // namespace bsi
