// Device code of the block scores (a2), shared by the stand-alone kernel and the fused
// decode step: the second stage of NOSA's two-stage pooling ("Technisches Resümee:
// NOSA", Methodik / 1. Algorithmus: NOSA, "Blockweise Implementierung": max pooling
// at block level), shared by the query heads of a GQA group ("Technische Samenvatting:
// Fluxion", Systeemcomponenten, "Granularity-Budget Selector").
//
// A CTA of 256 threads scores tiles of 64 consecutive summary rows (64/r whole
// blocks, r = g/s), each arriving in shared memory with one bulk copy (two or three
// buffers when a CTA takes several tiles: the next tiles' copies fly during this one).
// The dot products of a tile are a (64 rows x d) by (d x G heads) product: they run on
// the tensor cores (mma.sync m16n8k8, tf32) with each fp32 operand split into a tf32
// high part and a tf32 remainder and three products summed (hi*hi + hi*lo + lo*hi), which
// keeps the dot products at about fp32 accuracy; each warp takes 16 rows and half of
// the dimensions.
#pragma once

#include <math.h>

#include "bs_internal.cuh"

namespace bsi {

constexpr int kScoreThreads = 256;
constexpr int kTileRows = 64;

template <int D, int G>
struct ScoreLayout {
  static constexpr int kTileBytes = kTileRows * D * 4;
  // nb tile buffers, then the G query vectors as tf32 high parts [G][D] and remainders
  // [G][D], then the partial dot products of the two halves of the dimensions [2][64][8].
  __host__ __device__ static constexpr int off_q(int nb) { return nb * kTileBytes; }
  __host__ __device__ static constexpr int off_dots(int nb) { return off_q(nb) + 2 * G * D * 4; }
  __host__ __device__ static constexpr int bytes(int nb) { return off_dots(nb) + 2 * kTileRows * 8 * 4; }
  static constexpr int kBytes = bytes(1);  // one buffer
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

// fp32 to tf32, rounded to nearest (ties away from zero); the result is exact in fp32.
__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// The G query vectors of the unit, pre-scaled by 1/sqrt(d), into shared memory as tf32
// high parts qs[0, G*D) and remainders qs[G*D, 2*G*D) (x - hi is exact in fp32).
template <int D, int G>
__device__ __forceinline__ void score_load_q(float *qs, const void *qrow, int q_dtype) {
  const float scale = rsqrtf(static_cast<float>(D));
  for (int i = threadIdx.x; i < G * D; i += kScoreThreads) {
    const float x = load_scalar(qrow, i, q_dtype) * scale;
    const float hi = tf32_rna(x);
    qs[i] = hi;
    qs[G * D + i] = tf32_rna(x - hi);
  }
}

// d += a * b on one m16n8k8 tf32 tile (fp32 accumulators).
__device__ __forceinline__ void mma_tf32(float (&d)[4], float a0, float a1, float a2, float a3, float b0, float b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(__float_as_uint(a0)), "r"(__float_as_uint(a1)), "r"(__float_as_uint(a2)), "r"(__float_as_uint(a3)),
        "r"(__float_as_uint(b0)), "r"(__float_as_uint(b1)));
}

// The query fragments of a warp (tf32 high parts and remainders) for score_compute,
// kept in registers across tiles: lane (g, t) holds query head g's dimensions [c, c+4),
// c = 16p + 4t within the warp's half of the dimensions (zero for heads g >= G).
template <int D, int G>
struct ScoreQ {
  float4 hi[D / 32], lo[D / 32];
};

// Loads the warp's query fragments from qs (written by score_load_q and made visible by a
// CTA barrier since).
template <int D, int G>
__device__ __forceinline__ ScoreQ<D, G> score_qfrag(const float *qs) {
  ScoreQ<D, G> f;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, tq = lane & 3, kh = warp >> 2;
  const bool head = gq < G;
  const float *qh = qs + (head ? gq : 0) * D + kh * (D / 2) + 4 * tq;
#pragma unroll
  for (int p = 0; p < D / 32; ++p) {
    f.hi[p] = head ? *reinterpret_cast<const float4 *>(qh + 16 * p) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    f.lo[p] = head ? *reinterpret_cast<const float4 *>(qh + G * D + 16 * p) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  return f;
}

// Waits for a copy of n_loaded rows on `bar` (phase `parity`); false (for every
// thread) when it timed out. All threads call it.
__device__ __forceinline__ bool score_wait(uint64_t *bar, uint32_t parity, int n_loaded, int32_t *st) {
  const bool ok = n_loaded == 0 || mbar_wait_bounded(bar, parity, st);
  return !__syncthreads_or(!ok);
}

// Scores tile `tile` of the unit's candidates from `tile_sm` (rows from c_lo * r + 64 *
// tile, n_loaded of them, covering the tile) into row_out[c] (c = block index). qf holds
// the warp's query fragments (score_qfrag). All 256 threads call it. Once every warp has
// read the tile (a CTA barrier), it calls refill() in every thread, so that the caller can
// start the next copy into the tile's buffer while the block scores are reduced. The
// caller passes a CTA barrier (score_wait is one) before the next call or any other use of
// `dots`.
//
// Dot products: warp w takes rows 16*(w%4) .. +15 (the MMA's M) and dimensions
// [(w/4)*d/2, (w/4+1)*d/2) (its K), with the heads as N (padded to 8 by zero columns).
// The order in which dimensions fill the k-slots is free as long as A and B agree: lane
// (g, t) loads one float4 of dimensions [c, c+4), c = 16p + 4t within the warp's half,
// of rows g and g+8 and of query g; its elements fill slots t and t+4 of k-steps 2p
// (.x, .y) and 2p+1 (.z, .w), which is where the m16n8k8 fragments want lane (g, t).
// A summary value x splits into hi = x with its 13 low mantissa bits cleared (a tf32
// value) and lo = x - hi (exact in fp32); the tensor core reads lo's top tf32 bits, so
// what is dropped is below 2^-20 |x|. The two halves' partial sums meet in shared memory.
template <int D, int G, class Refill>
__device__ void score_compute(const float *tile_sm, const ScoreQ<D, G> &qf, float *dots, const Geom &ge, int tile,
                              int reduce, int n_loaded, float *row_out, Refill refill) {
  (void)n_loaded;  // rows past the copied ones feed only their own (unread) dot products
  const int tid = threadIdx.x;
  const int r = ge.g / ge.s;
  const int bpt = kTileRows / r;
  const int c_first = ge.c_lo + tile * bpt;
  const int nb = min(bpt, ge.c_hi - c_first);
  static_assert(D % 32 == 0 && D / 32 <= 4, "head_dim 32..128");
  static_assert(G >= 1 && G <= 8, "1..8 query heads per KV head");
  static_assert(kScoreThreads == 256 && kTileRows == 64, "8 warps: 4 row tiles x 2 halves of the dimensions");
  constexpr int KH = D / 2;   // dimensions per warp
  constexpr int NP = D / 32;  // float4 loads (two k-steps each) per row per warp
  const int lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  const int mt = warp & 3, kh = warp >> 2;
  const float *ra = tile_sm + (mt * 16 + gq) * D + kh * KH + 4 * tq;
  const float *rb = ra + 8 * D;
  // Four independent accumulator chains: (hi*hi, the two cross terms) x (even, odd k-step).
  float big0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, big1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float sm0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sm1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const float4 x0 = *reinterpret_cast<const float4 *>(ra + 16 * p);
    const float4 x1 = *reinterpret_cast<const float4 *>(rb + 16 * p);
    const float4 bh = qf.hi[p], bl = qf.lo[p];
    const float a0[4] = {x0.x, x0.y, x0.z, x0.w}, a1[4] = {x1.x, x1.y, x1.z, x1.w};
    float h0[4], l0[4], h1[4], l1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h0[e] = __uint_as_float(__float_as_uint(a0[e]) & 0xffffe000u);
      l0[e] = a0[e] - h0[e];
      h1[e] = __uint_as_float(__float_as_uint(a1[e]) & 0xffffe000u);
      l1[e] = a1[e] - h1[e];
    }
    // k-step 2p: (.x, .y); k-step 2p+1: (.z, .w). A = {row g slot t, row g+8 slot t,
    // row g slot t+4, row g+8 slot t+4}; B = {slot t, slot t+4} of head g.
    mma_tf32(sm0, l0[0], l1[0], l0[1], l1[1], bh.x, bh.y);
    mma_tf32(sm1, l0[2], l1[2], l0[3], l1[3], bh.z, bh.w);
    mma_tf32(big0, h0[0], h1[0], h0[1], h1[1], bh.x, bh.y);
    mma_tf32(big1, h0[2], h1[2], h0[3], h1[3], bh.z, bh.w);
    mma_tf32(sm0, h0[0], h1[0], h0[1], h1[1], bl.x, bl.y);
    mma_tf32(sm1, h0[2], h1[2], h0[3], h1[3], bl.z, bl.w);
  }
  // Accumulators: (row g, heads 2t, 2t+1) and (row g+8, heads 2t, 2t+1).
  float acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = (big0[i] + big1[i]) + (sm0[i] + sm1[i]);
  float *dw = dots + kh * (kTileRows * 8) + (mt * 16 + gq) * 8 + 2 * tq;
  *reinterpret_cast<float2 *>(dw) = make_float2(acc[0], acc[1]);
  *reinterpret_cast<float2 *>(dw + 64) = make_float2(acc[2], acc[3]);
  __syncthreads();  // every warp has read the tile and written its partial sums
  refill();
  // Max over the r sub-blocks of a block per head, then over (or mean across) heads:
  // 8 lanes per block (one per head), 4 blocks per warp, 32 per pass of the CTA.
  const float *d0 = dots, *d1 = dots + kTileRows * 8;
  const int h = lane & 7;
  for (int c0 = warp * 4; c0 < nb; c0 += 32) {
    const int c = c0 + (lane >> 3);
    float m = -INFINITY;
    if (c < nb && h < G) {
      for (int j = 0; j < r; ++j) {
        const int i = (c * r + j) * 8 + h;
        m = fmaxf(m, d0[i] + d1[i]);
      }
    }
    float red = reduce == BS_GROUP_MAX ? m : (h < G ? m : 0.0f);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const float other = __shfl_xor_sync(0xffffffffu, red, o);
      red = reduce == BS_GROUP_MAX ? fmaxf(red, other) : red + other;
    }
    if (reduce != BS_GROUP_MAX) red = red / static_cast<float>(G);
    if (h == 0 && c < nb) row_out[c_first + c] = red;
  }
}

}  // namespace bsi
