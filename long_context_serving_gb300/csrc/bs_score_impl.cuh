// Device code of the block scores (a2), shared by the stand-alone kernel and the fused
// decode step: the second stage of NOSA's two-stage pooling ("Technisches Resümee:
// NOSA", Methodik / 1. Algorithmus: NOSA, "Blockweise Implementierung": max pooling
// at block level), shared by the query heads of a GQA group ("Technische Samenvatting:
// Fluxion", Systeemcomponenten, "Granularity-Budget Selector").
//
// One CTA of 256 threads scores a tile of 64 consecutive summary rows (64/r whole
// blocks, r = g/s). The tile arrives in shared memory with one bulk copy. Each warp
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
  static constexpr int kOffQ = kTileRows * D * 4;
  static constexpr int kOffDots = kOffQ + G * D * 4;
  static constexpr int kBytes = kOffDots + kTileRows * G * 4;
};

// Blocks of a unit's candidate range covered by one tile, and the tile count.
__host__ __device__ __forceinline__ int score_blocks_per_tile(int g, int s) { return kTileRows / (g / s); }
__host__ __device__ __forceinline__ int score_tiles(const Geom &ge) {
  const int bpt = score_blocks_per_tile(ge.g, ge.s);
  return (ge.c_hi - ge.c_lo + bpt - 1) / bpt;
}

// Starts the bulk copy of summary rows [row0, min(row0 + 64, row_end)) of a unit
// (summ_unit: its first row, 16-byte aligned) into the tile buffer and returns the row
// count (0: nothing in flight). The barrier is initialised either way; every thread
// calls it, and every thread must call score_tile_finish afterwards, which waits for
// the copy, before the shared memory is reused or the CTA exits.
template <int D, int G>
__device__ __forceinline__ int score_tile_issue(const float *summ_unit, int64_t row0, int64_t row_end,
                                                unsigned char *smem, uint64_t *bar) {
  const int64_t left = row_end - row0;
  const int n = row0 < 0 ? 0 : static_cast<int>(left < kTileRows ? (left > 0 ? left : 0) : kTileRows);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    if (n > 0) {
      const uint32_t bytes = static_cast<uint32_t>(n) * D * sizeof(float);
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(smem, summ_unit + row0 * D, bytes, bar);
    }
  }
  __syncthreads();
  return n;
}

// Waits for the copy started by score_tile_issue (n_loaded rows) and, if `score`,
// scores tile `tile` of the unit's candidates into row_out[c] (c = block index): the
// copied rows must start at row c_lo * r + 64 * tile and cover the tile. qrow points at
// the unit's G query vectors. Returns false when the copy timed out. All 256 threads
// call it with the same arguments.
template <int D, int G>
__device__ bool score_tile_finish(int n_loaded, bool score, const void *qrow, int q_dtype, const Geom &ge, int tile,
                                  int reduce, float *row_out, unsigned char *smem, uint64_t *bar, int32_t *st) {
  using L = ScoreLayout<D, G>;
  float *tile_sm = reinterpret_cast<float *>(smem);          // [64][D]
  float *qs = reinterpret_cast<float *>(smem + L::kOffQ);     // [G][D]
  float *dots = reinterpret_cast<float *>(smem + L::kOffDots);  // [64][G]
  const int tid = threadIdx.x;
  const float scale = rsqrtf(static_cast<float>(D));
  if (score)
    for (int i = tid; i < G * D; i += kScoreThreads) qs[i] = load_scalar(qrow, i, q_dtype) * scale;
  const bool ok = n_loaded == 0 || mbar_wait_bounded(bar, 0, st);
  if (__syncthreads_or(!ok)) return false;
  if (!score) return true;
  const int r = ge.g / ge.s;
  const int bpt = kTileRows / r;
  const int c_first = ge.c_lo + tile * bpt;
  const int nb = min(bpt, ge.c_hi - c_first);
  const int nrows = min(nb * r, n_loaded);

  // Dot products. Warp w takes rows 8w .. 8w+7 of the tile; lane l owns dimensions
  // [l*DPL, (l+1)*DPL) and keeps the G query slices of them in registers, so shared
  // memory is read once per row (a contiguous row per warp). Each lane forms the
  // 8 x G partial sums of its dimensions; a butterfly reduce-scatter over the 32
  // lanes (values halved at each of 5 stages) leaves lane l with the full sums of
  // entries [l*NF, (l+1)*NF) of the row-major (row, head) list.
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
  return true;
}

// Scores tile `tile` of a unit's candidates into row_out[c] (c = block index).
// summ_unit points at the unit's first summary row (16-byte aligned); qrow at its G
// query vectors. Returns false when the bulk copy timed out. All 256 threads call it
// with the same arguments; the tile must exist.
template <int D, int G>
__device__ bool score_tile(const float *summ_unit, const void *qrow, int q_dtype, const Geom &ge, int tile,
                           int reduce, float *row_out, unsigned char *smem, uint64_t *bar, int32_t *st) {
  const int r = ge.g / ge.s;
  const int bpt = kTileRows / r;
  const int c_first = ge.c_lo + tile * bpt;
  const int nb = min(bpt, ge.c_hi - c_first);
  const int64_t row0 = static_cast<int64_t>(c_first) * r;
  const int n = score_tile_issue<D, G>(summ_unit, row0, row0 + nb * r, smem, bar);
  return score_tile_finish<D, G>(n, true, qrow, q_dtype, ge, tile, reduce, row_out, smem, bar, st);
}

}  // namespace bsi
