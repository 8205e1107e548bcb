// Device code of the block scores (a2), shared by the stand-alone kernel and the fused
// decode step: the second stage of NOSA's two-stage pooling ("Technisches Resümee:
// NOSA", Methodik / 1. Algorithmus: NOSA, "Blockweise Implementierung": max pooling
// at block level), shared by the query heads of a GQA group ("Technische Samenvatting:
// Fluxion", Systeemcomponenten, "Granularity-Budget Selector").
//
// One CTA of 256 threads scores a tile of 64 consecutive summary rows (64/r whole
// blocks, r = g/s). The tile arrives in shared memory with one bulk copy; four threads
// share a row, each taking every fourth 16-byte chunk in a row-rotated order so that
// the 8 lanes of a shared-memory phase hit 8 different bank groups. The G query vectors
// (pre-scaled by 1/sqrt(d)) sit in shared memory and are read as broadcasts.
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

// Scores tile `tile` of a unit's candidates into row_out[c] (c = block index).
// summ_unit points at the unit's first summary row (16-byte aligned); qrow at its G
// query vectors. Returns false when the bulk copy timed out. All 256 threads call it
// with the same arguments; the tile must exist.
template <int D, int G>
__device__ bool score_tile(const float *summ_unit, const void *qrow, int q_dtype, const Geom &ge, int tile,
                           int reduce, float *row_out, unsigned char *smem, uint64_t *bar, int32_t *st) {
  using L = ScoreLayout<D, G>;
  float *tile_sm = reinterpret_cast<float *>(smem);          // [64][D]
  float *qs = reinterpret_cast<float *>(smem + L::kOffQ);     // [G][D]
  float *dots = reinterpret_cast<float *>(smem + L::kOffDots);  // [64][G]
  const int tid = threadIdx.x;
  const int r = ge.g / ge.s;
  const int bpt = kTileRows / r;
  const int c_first = ge.c_lo + tile * bpt;
  const int nb = min(bpt, ge.c_hi - c_first);
  const int nrows = nb * r;
  const int64_t row0 = static_cast<int64_t>(c_first) * r;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = static_cast<uint32_t>(nrows) * D * sizeof(float);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(tile_sm, summ_unit + row0 * D, bytes, bar);
  }
  const float scale = rsqrtf(static_cast<float>(D));
  for (int i = tid; i < G * D; i += kScoreThreads) qs[i] = load_scalar(qrow, i, q_dtype) * scale;
  const bool ok = mbar_wait_bounded(bar, 0, st);
  if (__syncthreads_or(!ok)) return false;

  // Dot products: thread (row, quarter).
  constexpr int kChunks = D / 4;     // float4 chunks per row
  constexpr int kPer = kChunks / 4;  // chunks per quarter (power of two)
  const int row = tid >> 2, qq = tid & 3;
  float acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = 0.0f;
  if (row < nrows) {
    const float4 *rp = reinterpret_cast<const float4 *>(tile_sm + row * D);
#pragma unroll
    for (int c = 0; c < kPer; ++c) {
      const int ch = qq + 4 * ((c + row) & (kPer - 1));
      const float4 k4 = rp[ch];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float4 q4 = reinterpret_cast<const float4 *>(qs + h * D)[ch];
        acc[h] = fmaf(q4.x, k4.x, acc[h]);
        acc[h] = fmaf(q4.y, k4.y, acc[h]);
        acc[h] = fmaf(q4.z, k4.z, acc[h]);
        acc[h] = fmaf(q4.w, k4.w, acc[h]);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
    acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 2);
  }
  if (row < nrows && qq == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) dots[row * G + h] = acc[h];
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

}  // namespace bsi
